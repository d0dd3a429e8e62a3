// Host/device layouts of a compiled plan: instruction records, node table, kernel parameters.
//
// The instruction record is a fixed-size POD written by the host compiler and read by the
// persistent kernel, in the manner of the 64-byte TaskDescriptor of "Implementing a Mega Kernel
// for B300" (§2: op id, flags, indices instead of pointers, static_asserts on the layout) and the
// fixed-size instruction of "MegaKittens Internals" §06. Source and arrival counter lists live
// out of line (offsets into two int32 arrays) so no instruction has a fan-in or fan-out limit.
#pragma once
#include <stddef.h>
#include <stdint.h>

#ifdef __CUDACC__
#define MK_HD __host__ __device__
#else
#define MK_HD
#endif

namespace mk {

enum Op : uint16_t {
  OP_NOOP = 0,
  OP_GEMM = 1,          // tcgen05 output tile of a matmul
  OP_GEMV = 2,          // split-K column tile of a small-M matmul (CUDA cores)
  OP_EW = 3,            // elementwise tile
  OP_RMSNORM = 4,       // block of rows
  OP_ROPE = 5,          // block of rows: rotary q/k (+ v copy)
  OP_ATTN_PARTIAL = 6,  // split-KV partial (m, l, o) for one kv group and key chunk
  OP_ATTN_REDUCE = 7,   // LSE merge of one kv group's partials
  OP_ATTN_PREFILL = 8,  // causal attention for one (q tile, head)
  OP_ARGMAX = 9,        // block of rows x column chunk: (max, first index) partials
  OP_ARGMAX_REDUCE = 10,  // block of rows: the winner of the row's partials
  OP_END = 0xFFFF,      // past the end of an SM's queue (never stored in the list)
};

enum : uint16_t { IFLAG_B_DEP = 1 };  // the B operand is produced inside the graph

struct Instr {
  uint16_t op;
  uint16_t flags;
  int32_t node;
  int32_t m0, n0, k0, klen;
  int32_t aux0, aux1;
  int32_t sem;
  int32_t n_src, src_off;
  int32_t n_dst, dst_off;
  int32_t slot;   // GEMM split tail: scratch slot of split 0 (this rank); slot of split s = slot + s * cluster
  int32_t split;  // GEMM split tail: this instruction's split index
  int32_t pad;
};
static_assert(sizeof(Instr) == 64, "instruction record is 64 bytes");
static_assert(offsetof(Instr, node) == 4 && offsetof(Instr, sem) == 32 &&
                  offsetof(Instr, dst_off) == 48,
              "instruction field offsets are part of the ABI");

enum DType : int32_t { DT_F16 = 0, DT_BF16 = 1, DT_F32 = 2, DT_I32 = 3 };

enum : uint32_t {
  EPI_BIAS = 1u << 0,
  EPI_RELU = 1u << 1,
  EPI_RESIDUAL = 1u << 2,
  EPI_RMSNORM_INPUT = 1u << 3,
  EPI_SILU_MUL = 1u << 4,
  NF_B_PANELS = 1u << 16,  // B (and b2) maps are 3D panel maps: one box per stage, all panels
  NF_ROPE = 1u << 17,      // GEMV tiles also write RoPE's outputs (out_q, out_k, out_v)
  NF_ATTN_FUSED = 1u << 18, // split-KV partials: the last one of a key/value head combines
  NF_B_PACKED = 1u << 19,   // GEMV: b / b2 point at the plan's packed copies (ld = 64-row blocks
                            // per column tile), one contiguous unit per weight stage
};

enum : int32_t { EWOP_ADD = 0, EWOP_RELU = 1, EWOP_COPY = 2, EWOP_SILU_MUL = 3 };

// One operand: pointer to the first element of the window and its row stride (elements).
struct Operand {
  uint64_t ptr;
  int32_t ld;
  int32_t tmap;  // index into the plan's tensor-map array, -1 when not read through TMA
};
static_assert(sizeof(Operand) == 16, "operand is 16 bytes");

// Node table entry: everything an instruction body needs about its graph node. 256 bytes; the
// scheduler warp copies it into the instruction slot next to the instruction record.
struct Node {
  int32_t kind;     // Op of the node's (first) phase family
  int32_t dtype;    // DType of A/B/out
  uint32_t flags;   // EPI_* for matmuls
  int32_t M, N, K;  // matmul: out M x N, reduction K; rows/cols for row ops
  int32_t tile_n;   // output columns per GEMM/GEMV tile
  int32_t ewop;     // EWOP_* for elementwise nodes
  Operand a, b, b2, out;        // 64 B
  Operand bias, res, gamma;     // 48 B (gamma also RMSNORM's weight)
  Operand out_k, out_v;         // 32 B: ROPE k / v outputs
  Operand scratch;              // 16 B: fp32 partials (GEMV split-K, attention)
  float eps, scale, theta;
  int32_t hq, hkv, hd;          // heads and head dim
  int32_t pos0;                 // ROPE first position / attention q_pos0
  int32_t causal;
  int32_t n_chunks;             // attention decode: chunks per kv group
  int32_t n_splits;             // GEMV: K splits per tile
  int32_t ldp;                  // GEMV partial stride (elements per split: M * N * (1 or 2))
  int32_t tile_m;               // rows per instruction of row/elementwise ops
  Operand out_q;                // 16 B: RoPE fused into a GEMV: rotated q output
};
static_assert(sizeof(Node) == 256, "node entry is 256 bytes");

constexpr int kMaxTmaps = 1024;
constexpr int kXrFloats = 5120;  // shared-memory staging of GEMV activations / RoPE angle tables

// Kernel parameters (plain pointers into plan-owned device memory).
struct Params {
  const Instr* instrs;
  const Node* nodes;
  const int32_t* src_list;  // pairs (counter, target)
  const int32_t* dst_list;
  int32_t* counters;        // dependency counters, then split semaphores
  int32_t* status;          // 8 int32: mk_device_status
  const void* tmaps;        // CUtensorMap array (64-byte aligned), global memory
  int32_t* done;            // CTAs finished in this run (the last one resets the run state)
  int32_t* last_status;     // status of the last completed run (read by the host)
  int32_t* snapshot;        // copy of the counters at the end of a run, or null
  uint64_t* trace;          // per instruction kTraceWords timestamps (see mk_get_trace), or null
  int32_t n_instr;
  int32_t n_sm;             // placement stride
  int32_t n_tmaps;
  int32_t n_counters;       // dependency counters + split semaphores
  int32_t stages;           // operand ring depth: 4 stages of 48 KB, or 6 of 32 KB (CTA pairs)
  uint64_t timeout_ns;
};

// Device status record (mirrors mk_device_status).
enum : int32_t { ST_CODE = 0, ST_INSTR, ST_COUNTER, ST_OBSERVED, ST_EXPECTED, ST_SM, ST_ROLE, ST_WHERE };
constexpr int kStatusWords = 8;
constexpr int kTraceWords = 8;

// Kernel geometry shared with the host (launch configuration and shared-memory budget).
constexpr int kThreads = 256;          // 8 warps: scheduler, loader, MMA, spare, 4 compute
constexpr int kRingBytes = 192 * 1024; // operand ring, split into equal 1024-byte-aligned stages
constexpr int kStages = 4;              // single-CTA GEMM tiles: A 128x64 (16 KB) + B 64x256 (32 KB)
constexpr int kPairStages = 6;          // CTA pairs: A 128x64 + half of B (16 KB) per CTA, 32 KB
constexpr int kMaxStages = kPairStages;
constexpr int kSlots = 8;              // instruction slots (scheduler lookahead)
constexpr int kSlotBytes = 64 + 256;   // Instr + Node
constexpr int kGemmTileM = 128;
constexpr int kGemmBK = 64;            // K per stage for GEMM (128-byte rows of 16-bit elements)
constexpr int kGemvRows = 64;          // K rows per stage for GEMV (x 256 columns = 32 KB)
constexpr int kAttnChunkMax = 128;     // keys per split-KV partial handled by one instruction
constexpr int kAttnTileQ = 128;        // query rows of one prefill attention instruction
constexpr int kAttnKeyBlock = 64;      // keys per ring stage of prefill attention (Q + K + V = 32 KB)
constexpr int kAttnPCol = 192;         // single CTA: P tiles in TMEM, two of 32 columns

// Specialisations of the kernel by the instruction kinds they run. The host launches the
// smallest one that covers every instruction of a plan: a specialisation leaves out the code,
// and with it the register pressure, of every role path it never meets.
enum KernelSet : int32_t {
  KS_ALL = 0,      // every instruction kind
  KS_GEMM = 1,     // tcgen05 GEMM tiles only
  KS_DECODE = 2,   // GEMV tiles, split-KV attention partials and combines, row instructions
  KS_PREFILL = 3,  // GEMM tiles, causal prefill attention, row instructions
};
MK_HD constexpr bool ks_has_gemm(int ks) { return ks != KS_DECODE; }
MK_HD constexpr bool ks_has_gemv(int ks) { return ks == KS_ALL || ks == KS_DECODE; }
MK_HD constexpr bool ks_has_attn_prefill(int ks) { return ks == KS_ALL || ks == KS_PREFILL; }
MK_HD constexpr bool ks_has_rows(int ks) { return ks != KS_GEMM; }
// RMSNorm and RoPE rows staged through the operand ring by the loader (Instr.pad = stages)
MK_HD constexpr bool ks_stages_rows(int ks) { return ks == KS_ALL || ks == KS_PREFILL; }
MK_HD constexpr bool ks_has_tmem(int ks) {
  return ks_has_gemm(ks) || ks_has_attn_prefill(ks) || ks_has_gemv(ks);  // GEMV: tensor cores
}
MK_HD constexpr bool ks_covers(int ks, int op) {
  return op == OP_NOOP || op == OP_END                ? true
         : op == OP_GEMM                              ? ks_has_gemm(ks)
         : op == OP_GEMV || op == OP_ATTN_PARTIAL ||
                   op == OP_ATTN_REDUCE               ? ks_has_gemv(ks)
         : op == OP_ATTN_PREFILL                      ? ks_has_attn_prefill(ks)
                                                      : ks_has_rows(ks);
}

}  // namespace mk
