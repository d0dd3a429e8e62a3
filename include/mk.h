/*
 * mk.h — C ABI of the GB300 persistent megakernel library (libmk.so).
 *
 * A caller builds a static op graph over its own device buffers, compiles it once into a
 * plan (a flat list of fixed-size tile instructions, per-tile dependency counters and a node
 * table), and runs the plan as ONE persistent kernel launch per call on its own stream.
 *
 * Where the operations come from (page title, section):
 *  - graph of ops with fused epilogue flags, lowered to tile tasks:
 *      "Implementing a Mega Kernel for B300", §1 "Build the graph", §2 "Lower each op into tasks"
 *  - flat instruction list, per-tile integer counters, round-robin placement, counter zeroing
 *    per call: "MegaKittens Internals", §04 "Scheduler", §05 "The real schedule", §07
 *    "Dispatcher, JIT and launch", §11 "The TMEM token and global barriers"
 *  - the GEMM tile (TMA, mbarriers, TMEM, tcgen05): "Hand-writing a Blackwell GEMM", steps 1-8
 *  - split-KV attention partial + combine: "Implementing a Mega Kernel for B300", §2 and §8
 *  - buffer pool with reuse counters for plan-owned intermediates: "MegaKittens Internals", §04
 *    phase 2 and phase 3 (reuse barriers)
 *
 * Conventions
 *  - Every function returns an mk_status; MK_OK is 0. On failure mk_last_error() returns a
 *    message (thread-local, valid until the next call on the same thread). No function aborts.
 *  - Tensors registered with mk_add_tensor are caller-owned device memory, registered by
 *    pointer; the library never frees or allocates them, and a plan is bound to the pointers
 *    given at compile time. Transients (mk_add_transient) are plan-owned: they live in the
 *    plan's buffer pool.
 *  - Tensor ids and node ids are small non-negative integers local to one graph.
 *  - Element types: MK_F16 (IEEE half), MK_BF16 (bfloat16), MK_F32; MK_I32 for the indices an
 *    ARGMAX node writes.
 *  - Row-major 2-D view of every tensor: the innermost dimension is the column dimension and
 *    must have stride 1; all outer dimensions fold into rows and must be contiguous with each
 *    other. Row stride (elements) = strides[rank-2].
 *  - Threading: a graph or plan must not be used from two threads at once. Different plans
 *    may run concurrently on different streams.
 */
#ifndef MK_H_
#define MK_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MK_ABI_VERSION 2

typedef struct mk_graph* mk_graph_t;
typedef struct mk_plan* mk_plan_t;
typedef int32_t mk_status;

enum {
  MK_OK = 0,
  MK_ERR_INVALID_ARG = 1,   /* bad id, shape mismatch, null pointer */
  MK_ERR_UNSUPPORTED = 2,   /* valid graph the kernel cannot run: dtype, alignment, sizes */
  MK_ERR_HAZARD = 3,        /* a node writes a region an earlier node reads or writes */
  MK_ERR_OOM = 4,           /* device or host allocation failed */
  MK_ERR_CUDA = 5,          /* a CUDA runtime/driver call failed (message has the name) */
  MK_ERR_TIMEOUT = 6,       /* a device-side wait exceeded its limit; see mk_device_status */
  MK_ERR_DEVICE_CHECK = 7,  /* a device-side consistency check failed; see mk_device_status */
};

enum { MK_F16 = 0, MK_BF16 = 1, MK_F32 = 2, MK_I32 = 3 };

/* ---------------------------------------------------------------- graph construction */

/* Create an empty graph. *out receives the handle (owned by the caller; free with
 * mk_graph_destroy). */
mk_status mk_graph_create(mk_graph_t* out);
mk_status mk_graph_destroy(mk_graph_t g);

/* Register a caller-owned device tensor.
 *   dev_ptr  device address (16-byte aligned for any tensor read or written by TMA: GEMM and
 *            GEMV operands). May be NULL only for plans compiled with dry_run.
 *   dtype    MK_F16 / MK_BF16 / MK_F32 / MK_I32 (int32: ARGMAX outputs only)
 *   rank     1..4; shape[rank], strides[rank] in elements (strides may be NULL: contiguous)
 * The tensor is seen as rows x cols with cols = shape[rank-1]. */
mk_status mk_add_tensor(mk_graph_t g, void* dev_ptr, int32_t dtype, int32_t rank,
                        const int64_t* shape, const int64_t* strides, int32_t* tensor_id);

/* A plan-owned intermediate of rows x cols elements (no caller memory; rows start 16-byte
 * aligned). mk_compile places transients in the plan's buffer pool, where one whose accesses are
 * all finished a wave of instructions earlier (every node touching it ends at least n_sm
 * instructions before the next writer starts) hands its memory to a later transient of the same
 * shape and dtype; a reuse counter orders the new writes after the old accesses. Exactly one
 * node may write a transient (through any of its views), and every node reading it comes later.
 * mk_plan_tensor_ptr gives its device address once the plan exists; its contents are defined
 * until its buffer is reused by a later node of the same run. */
mk_status mk_add_transient(mk_graph_t g, int32_t dtype, int64_t rows, int64_t cols,
                           int32_t* tensor_id);

/* A rows x cols window of a registered tensor starting at (r0, c0) of its 2-D view; used to
 * name a layer of stacked weights, a slice of columns (q | k | v), a cache row, ... */
mk_status mk_add_view(mk_graph_t g, int32_t base, int64_t r0, int64_t c0, int64_t rows,
                      int64_t cols, int32_t* view_id);

/* Epilogue flags of a matmul ("Implementing a Mega Kernel for B300", §2: SILU_MUL,
 * ADD_RESIDUAL, RMS_NORM_INPUT; bias + ReLU: "MegaKittens Internals", §02). */
enum {
  MK_EPI_BIAS = 1u << 0,           /* + bias[m, n]; bias is a full M x N tensor */
  MK_EPI_RELU = 1u << 1,           /* max(., 0) after the bias */
  MK_EPI_RESIDUAL = 1u << 2,       /* + residual[m, n] after ReLU */
  MK_EPI_RMSNORM_INPUT = 1u << 3,  /* A := A / sqrt(mean(A^2) + eps) * gamma, row-wise (GEMV only) */
  MK_EPI_SILU_MUL = 1u << 4,       /* out = silu(A B) * (A b_up) */
};

typedef struct {
  uint32_t flags;     /* MK_EPI_* */
  int32_t bias;       /* tensor id or -1 */
  int32_t residual;   /* tensor id or -1 */
  int32_t gamma;      /* tensor id (1 x K) or -1 */
  int32_t b_up;       /* tensor id (K x N) or -1: second weight of SILU_MUL */
  float eps;          /* RMS_NORM_INPUT epsilon */
} mk_epilogue;

/* out[M x N] = epilogue(a[M x K] @ b[K x N]). a, b, out (and bias, residual, b_up) share one
 * dtype, MK_F16 or MK_BF16; accumulation is fp32. epi may be NULL (plain product). */
mk_status mk_add_matmul(mk_graph_t g, int32_t a, int32_t b, int32_t out, const mk_epilogue* epi,
                        int32_t* node_id);

/* Elementwise and row operations ("MegaKittens Internals", §12; "Implementing a Mega Kernel
 * for B300", §8 RMSNORM and ATTENTION_APPEND). Inputs and outputs of ADD/RELU/COPY/SILU_MUL
 * have the same shape (no broadcasting). */
enum {
  MK_EW_ADD = 0,        /* out = in0 + in1 */
  MK_EW_RELU = 1,       /* out = max(in0, 0) */
  MK_EW_COPY = 2,       /* out = in0 */
  MK_EW_SILU_MUL = 3,   /* out = silu(in0) * in1 */
  MK_EW_RMSNORM = 16,   /* out = in0 / sqrt(mean(in0^2) + eps) * gamma (row-wise) */
  MK_EW_ROPE = 17,      /* rotary embedding of q and k heads (+ copy of v), see mk_ew_params */
  MK_EW_ARGMAX = 18,    /* out[r] (MK_I32, R x 1) = the first column of in0's row r (f16 / bf16,
                           R x C) holding its largest value; NaN entries are ignored, a row
                           without a number gives -1 (greedy sampling of logits) */
};

typedef struct {
  float eps;            /* RMSNORM */
  int32_t gamma;        /* RMSNORM: tensor id (1 x cols) */
  /* ROPE: in0 = x [R x (Hq + Hkv) * d (+ Hkv * d)], columns [q | k (| v)]; row r is position
   * pos0 + r. out = rotated q [R x Hq*d]; out_k = rotated k [R x Hkv*d]; out_v (or -1) =
   * copy of v [R x Hkv*d]. Pairs (i, i + d/2) of each head rotate by pos * theta^(-2i/d). */
  int32_t n_q_heads, n_kv_heads, head_dim;
  int32_t pos0;
  float theta;
  int32_t out_k, out_v;
} mk_ew_params;

mk_status mk_add_elementwise(mk_graph_t g, int32_t op, const int32_t* ins, int32_t n_in,
                             int32_t out, const mk_ew_params* p, int32_t* node_id);

/* Attention out = softmax(q k^T * scale [+ causal mask]) v with grouped kv heads.
 *   q [Tq x Hq*d], k and v [Tk x Hkv*d], out [Tq x Hq*d], all MK_BF16.
 *   Query row i is at position q_pos0 + i, key row j at position j; causal: j <= q_pos0 + i.
 *   Tq == 1 lowers to split-KV partial + reduce tiles ("Implementing a Mega Kernel for B300",
 *   §2); Tq > 1 to causal prefill tiles. scale 0 means 1/sqrt(d). */
typedef struct {
  int32_t n_q_heads, n_kv_heads, head_dim;
  int32_t causal;
  int32_t q_pos0;
  float scale;
} mk_attn_params;

mk_status mk_add_attention(mk_graph_t g, int32_t q, int32_t k, int32_t v, int32_t out,
                           const mk_attn_params* p, int32_t* node_id);

/* ---------------------------------------------------------------- compile and run */

typedef struct {
  int32_t n_sm;          /* placement stride = persistent grid size; 0 = the device's SM count */
  int32_t gemm_tile_m;   /* GEMM output tile rows: 128 (one CTA), or 256 with cluster 2 */
  int32_t gemm_tile_n;   /* GEMM output tile columns: 64, 128 or 256 (halved for SILU_MUL) */
  int32_t cluster;       /* instructions per GEMM tile: 1 (default), or 2 for CTA pairs (the
                            256-row tile runs on both CTAs of a 2-CTA cluster, tcgen05
                            cta_group::2; needs gemm_tile_m 256 and no prefill attention) */
  int32_t ew_rows, ew_cols, ew_tiles;   /* elementwise instruction = ew_rows x ew_cols*ew_tiles */
  int32_t norm_rows;     /* rows per RMSNORM / ROPE instruction */
  int32_t gemv_max_m;    /* matmuls with M <= this lower to GEMV tiles */
  int32_t gemv_tile_n;   /* GEMV output columns per tile: 256 (halved for SILU_MUL) */
  int32_t gemv_splits;   /* K splits per GEMV tile; 0 = max(1, n_sm / column tiles) */
  int32_t gemv_kstep;    /* GEMV K chunks are multiples of this */
  int32_t attn_chunk;    /* keys per split-KV partial */
  int32_t attn_tile_q;   /* query rows per prefill attention tile */
  int32_t dry_run;       /* 1: lower only (no device, no kernel-support checks) */
  int32_t timeout_ms;    /* limit of every device-side wait; 0 = 2000 */
  int32_t device;        /* CUDA device ordinal; -1 = current */
  int32_t debug_counter; /* test hook: counter whose target is raised by debug_extra (-1: none) */
  int32_t debug_extra;
  int32_t snapshot_counters; /* 1: keep each run's final counter values for mk_get_counters */
  int32_t trace;         /* 1: record per-instruction timestamps for mk_get_trace */
  int32_t gemm_split_tail; /* 1: the GEMM tiles of a matmul's last, partly filled wave are
                            split along K. With two splits and no SILU_MUL each split stores
                            the half of its fp32 partial the other finishes and both finish
                            their half (the later one releases the counters); otherwise the
                            last split to finish sums the partials and runs the epilogue.
                            0 (default): never split */
  int32_t fuse_rope;     /* 1 (default): a ROPE node right after a matmul that lowers to GEMV
                            tiles, reading exactly its output (head_dim 64, output width a
                            multiple of gemv_tile_n), runs inside those tiles; 0: never */
  int32_t fuse_attn_reduce; /* 1 (default): the last split-KV partial of each key/value head
                            to finish combines the head's partials (no reduce phase); 0: a
                            separate reduce instruction per key/value head */
  int32_t kernel_set;    /* 0 (default): launch the smallest specialisation of the kernel whose
                            instruction kinds cover the plan (GEMM tiles only; decode: GEMV,
                            split-KV attention and row instructions; prefill: GEMM, prefill
                            attention and row instructions); 1: the general kernel. Both give
                            bit-identical results; a specialisation compiles without the code
                            of the kinds it never runs */
  int32_t gemv_pack;     /* 1 (default): the weights of GEMV tiles that no node of the graph
                            writes are copied at mk_compile into a plan-owned packed layout
                            (each 64-row stage of a tile contiguous, in its shared-memory
                            layout) and streamed from there with one bulk copy per stage; the
                            copy follows mk_run_host copies into the weight, and mk_plan_repack
                            refreshes it after any other change to such a weight. 0: stream
                            them from the tensors through tensor maps */
  int32_t argmax_chunk;  /* columns per ARGMAX partial instruction (multiple of 8); a reduce
                            instruction per row block picks the winner of the partials */
  int32_t gemm_group_m;  /* GEMM tile order: groups of this many row tiles, column by column
                            inside a group (L2 reuse of the B and A panels of a wave);
                            1: row-major. Default 8 */
  int32_t wave_pack;     /* 1 (default): consecutive independent GEMM nodes are placed as one
                            run, tiles longest K first on the least loaded SM (or CTA pair),
                            padded with Noops; 0: each node's tiles in order */
  int32_t row_stage;     /* 1 (default): RMSNorm and RoPE row instructions of single-CTA plans
                            get their input rows copied into the operand ring by the loader warp
                            (bulk copies), when a row fits one ring stage; 0: the compute
                            warpgroup loads them itself */
  int32_t pool_waves;    /* buffer pool reuse distance: a transient takes an earlier buffer only
                            when its writer starts at least pool_waves * n_sm instructions past
                            the end of every node that touched the old occupant. Default 1 (one
                            wave); larger values keep more buffers and wait less */
} mk_compile_opts;

/* Fill *o with the defaults (the values listed above for each field). */
mk_status mk_default_opts(mk_compile_opts* o);

/* Lower the graph and, unless dry_run, upload the plan to the device: instruction list, node
 * table, dependency lists, tensor maps, counters, scratch, status word, packed GEMV weight copies
 * (gemv_pack) and the transients' buffer pool, all in one plan-owned allocation. The graph may
 * be destroyed afterwards. */
mk_status mk_compile(mk_graph_t g, const mk_compile_opts* opts, mk_plan_t* out);

/* Enqueue one run on `stream` (a cudaStream_t; NULL = legacy default stream): ONE persistent
 * kernel launch. The CTA that finishes last resets the counters for the next run (also after a
 * device-side failure) and moves the run's status to where mk_sync_status reads it (keeping an
 * earlier failure that has not been read).
 * Asynchronous; errors of the launch itself are returned, device-side failures are reported by
 * mk_sync_status. Runs of one plan must not overlap (use one stream, or order the streams). */
mk_status mk_run(mk_plan_t p, void* stream);

/* One copy between a registered tensor (or view) and host memory. */
typedef struct {
  int32_t tensor;      /* tensor or view id of the compiled graph */
  void* host;          /* rows x cols elements, densely packed (pinned memory for overlap) */
  int32_t to_device;   /* 1: host -> tensor before the launch; 0: tensor -> host after it */
} mk_host_copy;

/* End-to-end call with host buffers: the host->device copies (in order), mk_run, then the
 * device->host copies, all enqueued on `stream`. */
mk_status mk_run_host(mk_plan_t p, const mk_host_copy* copies, int32_t n_copies, void* stream);

typedef struct {
  int32_t code;       /* MK_OK, MK_ERR_TIMEOUT or MK_ERR_DEVICE_CHECK */
  int32_t instr;      /* instruction index being processed */
  int32_t counter;    /* counter waited on (-1: an on-chip barrier) */
  int32_t observed;   /* its value when the wait gave up */
  int32_t expected;   /* the value waited for */
  int32_t sm;         /* CTA index */
  int32_t role;       /* 0 scheduler, 1 loader, 2 MMA, 3 compute */
  int32_t where;      /* wait site id (kernel-internal) */
} mk_device_status;

/* Device address of a registered tensor (a transient's place in the buffer pool included) in
 * plan p; *ptr = NULL for a dry-run plan's transients. */
mk_status mk_plan_tensor_ptr(mk_plan_t p, int32_t tensor, void** ptr);

/* Re-read every weight the plan holds a packed copy of (gemv_pack = 1) into that copy, on
 * `stream` (ordered before later work on it). Needed after a change to such a weight made
 * outside mk_run_host; without it mk_run keeps using the weight as it was when packed. */
mk_status mk_plan_repack(mk_plan_t p, void* stream);

/* Synchronise the device and read the plan's status: the first device-side failure of any run
 * since the previous mk_sync_status (its record is then cleared), or MK_OK with the last run's
 * record. Returns st->code as the status. */
mk_status mk_sync_status(mk_plan_t p, mk_device_status* st);

mk_status mk_plan_destroy(mk_plan_t p);

/* Allocation-free matrix product for a few rows: out[m x n] = x[m x k] @ w[k x n], run by the
 * same persistent kernel as split-K GEMV tiles. The pages have no counterpart of this entry
 * point; it exists for callers that cannot allocate device memory when they need the product
 * (a serving loop whose device memory an up-front pool owns, code inside that pool's callbacks,
 * paths where cudaMalloc / cudaFree would synchronise the device). It calls no cudaMalloc,
 * cudaFree or allocating library routine: all run state (instruction records, node entry,
 * tensor map, split semaphores, status, fp32 split partials) lives in one file-scope device
 * array of 4 MiB that every GPU using the library holds until the process exits.
 *   x, w, out  caller-owned device memory, row-major and contiguous, 16-byte aligned.
 *   m 1..8; n >= 1 and k >= 0 multiples of 8; n <= 262144 (the array holds 1024 column tiles of
 *              256); larger sizes return MK_ERR_UNSUPPORTED with a message.
 *   dtype      MK_F16 or MK_BF16 (fp32 accumulation, one rounding at the end).
 *   stream     cudaStream_t (NULL = legacy default stream). Asynchronous unless `status` is
 *              non-NULL: then the call synchronises the stream and fills *status.
 * The first call on each device, with that device current, looks up the array's device address
 * (cudaGetSymbolAddress) and sets the kernel's shared-memory limit; make that first call before
 * any stream capture. A call on a capturing stream must pass status == NULL and come after that
 * first call; otherwise it returns MK_ERR_UNSUPPORTED with a message and records nothing. A
 * captured call replays with the arguments it was captured with. Every call shares the array and clears the parts that must start at zero;
 * the rest keeps the previous call's contents. A call writes its records into the array with a
 * small set-up kernel that receives them by value, so it reads no host buffer after it returns
 * and calls from different host threads share no host state. Calls on one stream run one after
 * the other; calls that can overlap on the same device (different streams, or host threads
 * calling at once for that device) race on that device's array and must not be issued. */
mk_status mk_gemv_noalloc(const void* x, const void* w, void* out, int32_t m, int32_t n,
                          int32_t k, int32_t dtype, void* stream, mk_device_status* status);

/* ---------------------------------------------------------------- introspection */

typedef struct {
  int64_t n_instr;       /* instructions in the list, Noop padding included */
  int64_t n_counters;    /* dependency counters */
  int64_t n_sems;        /* split-K semaphores (after the counters in the counter array) */
  int64_t n_sm;          /* placement stride */
  int64_t n_iter;        /* ceil(n_instr / n_sm): iterations of the longest SM queue */
  double waves;          /* n_instr / n_sm */
  int64_t n_src;         /* entries of the source list (pairs) */
  int64_t n_dst;         /* entries of the arrival list */
  int64_t per_op[16];    /* instructions per op code */
  int64_t smem_bytes;    /* dynamic shared memory of the launch (0 when dry_run) */
  int64_t scratch_bytes; /* plan-owned device scratch */
  int64_t kernel_set;    /* specialisation mk_run launches: 0 general, 1 GEMM tiles only,
                            2 decode, 3 prefill */
  int64_t packed_bytes;  /* device bytes of packed GEMV weight copies (gemv_pack) */
  int64_t pool_bytes;    /* device bytes of the transient buffer pool */
  int64_t n_reuse;       /* transients placed in a buffer an earlier transient used */
} mk_stats;

mk_status mk_plan_stats(mk_plan_t p, mk_stats* s);

/* Instruction records, 64 bytes each, little-endian:
 *   u16 op, u16 flags, i32 node, i32 m0, n0, k0, klen, aux0, aux1, sem,
 *   i32 n_src, src_off, n_dst, dst_off, i32 pad[3].
 * bytes must be >= n_instr * 64. */
mk_status mk_get_instructions(mk_plan_t p, void* host_buf, size_t bytes);
/* Source list: n_src pairs (counter, target) as int32; n = number of int32 slots. */
mk_status mk_get_src_list(mk_plan_t p, int32_t* host_buf, size_t n);
/* Arrival list: n_dst counter ids. */
mk_status mk_get_dst_list(mk_plan_t p, int32_t* host_buf, size_t n);
/* Target of every dependency counter (n_counters values). */
mk_status mk_get_counter_targets(mk_plan_t p, int32_t* host_buf, size_t n);
/* Counter array at the end of the last run (n_counters + n_sems values): each dependency
 * counter equals its target and each split semaphore its number of K splits. Needs a plan
 * compiled with snapshot_counters = 1; synchronises. */
mk_status mk_get_counters(mk_plan_t p, int32_t* host_buf, size_t n);

/* Per-instruction timestamps of the last run (plans compiled with trace = 1), %globaltimer ns:
 * for instruction i, buf[8i..8i+7] = {the compute warpgroup took the descriptor, the scheduler
 * saw every source counter complete, the compute warpgroup saw that, the instruction's body
 * ended, the instruction was published, the SM index, the accumulation ended (GEMM: the
 * accumulator is complete in tensor memory; GEMV: the last weight stage is consumed; split-KV
 * partial: its partial is stored), and for a split-KV partial whose combine is fused the time
 * its semaphore decided which partial combines (0 otherwise)}.
 * A slot an op does not reach stays 0. n >= 8 * n_instr; synchronises. */
mk_status mk_get_trace(mk_plan_t p, uint64_t* host_buf, size_t n);

const char* mk_last_error(void);
int32_t mk_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MK_H_ */
