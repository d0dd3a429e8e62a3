// Plan compilation (device half), launch, status and introspection of the C ABI.
//
// mk_compile uploads once: instruction list, node table, dependency lists, tensor maps and a
// zero-initialised counter array ("Implementing a Mega Kernel for B300" §6 uploads descriptors
// and a pointer table once; "MegaKittens Internals" §07 builds tensor maps on the host with
// cuTensorMapEncodeTiled). Every mk_run launches the persistent kernel once on the caller's
// stream (§07 "Every call: launch"); the counters need no reset per call, because the last CTA
// of each run to finish zeroes them (and the run's other state) for the next run.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <string.h>

#include <algorithm>
#include <new>

#include "mk_internal.h"
#include "mk_launch.h"

using namespace mk;

struct mk_plan {
  HostPlan hp;
  mk_compile_opts opts{};
  std::vector<Node> nodes;
  bool on_device = false;
  int device = 0;
  char* d_mem = nullptr;
  size_t scratch_bytes = 0;
  size_t smem = 0;
  int grid = 0;
  int kernel_set = KS_ALL;  // specialisation launched by mk_run
  // Packed copies of GEMV weights (see mk_pack.cu): one job per (node, weight), refreshed by
  // mk_plan_repack and by mk_run_host copies into the weight's tensor.
  struct PackJob {
    int node = -1, tensor = -1;  // graph node; weight tensor id (a base tensor or a view)
    const void* src = nullptr;
    long long ld = 0;
    int K = 0, N = 0, tw = 0;
    size_t off = 0;  // offset of the packed copy in d_mem
  };
  std::vector<PackJob> packs;
  size_t packed_bytes = 0;
  Params params{};
};

namespace mk {
size_t packed_gemv_bytes(int K, int N, int tw);
cudaError_t pack_gemv_weight(const void* w, long long ld, int K, int N, int tw, void* dst,
                             cudaStream_t stream);
}  // namespace mk

static cudaError_t run_packs(mk_plan* p, cudaStream_t s, int base_tensor = -1) {
  for (const auto& j : p->packs) {
    if (base_tensor >= 0 && p->hp.tensors[j.tensor].base != base_tensor) continue;
    const cudaError_t e = pack_gemv_weight(j.src, j.ld, j.K, j.N, j.tw, p->d_mem + j.off, s);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// The smallest kernel specialisation that runs every instruction of the list (KS_ALL when
// kernel_set = 1 asks for the general kernel); CTA-pair decode plans run KS_ALL.
static int pick_kernel_set(const std::vector<Instr>& instrs, const mk_compile_opts& o) {
  if (o.kernel_set == 1) return KS_ALL;
  int ks = KS_ALL;
  for (int cand : {KS_GEMM, KS_DECODE, KS_PREFILL}) {
    bool ok = true;
    for (const Instr& in : instrs) ok = ok && ks_covers(cand, in.op);
    if (ok) {
      ks = cand;
      break;
    }
  }
  return launched_kernel_set(ks, o.cluster == 2);
}

#define CUDA_TRY(call)                                                                    \
  do {                                                                                    \
    cudaError_t e_ = (call);                                                              \
    if (e_ != cudaSuccess) {                                                              \
      set_error("%s failed: %s (%s:%d)", #call, cudaGetErrorString(e_), __FILE__, __LINE__); \
      return MK_ERR_CUDA;                                                                 \
    }                                                                                     \
  } while (0)

// ------------------------------------------------------------------ validation

static void node_regions(const mk_graph* g, const NodeRec& nd, std::vector<int>& reads,
                         std::vector<int>& writes) {
  reads.clear();
  writes.clear();
  for (int id : {nd.a, nd.b, nd.b2, nd.bias, nd.res, nd.gamma, nd.ins[0], nd.ins[1]})
    if (id >= 0) reads.push_back(id);
  for (int id : {nd.out, nd.out_k, nd.out_v})
    if (id >= 0) writes.push_back(id);
  (void)g;
}

static Box full_box(const std::vector<TensorRec>& ts, int id) {
  const TensorRec& v = ts[id];
  Box b;
  b.t = v.base;
  b.r0 = v.r0;
  b.r1 = v.r0 + v.rows;
  b.c0 = v.c0;
  b.c1 = v.c0 + v.cols;
  return b;
}

// No node may write a region that it or an earlier node reads or writes: every dependency is
// then read-after-write and carried by a counter, and a run never races with itself.
static mk_status check_hazards(const mk_graph* g) {
  std::vector<int> r_i, w_i, r_j, w_j;
  for (size_t i = 0; i < g->nodes.size(); ++i) {
    node_regions(g, g->nodes[i], r_i, w_i);
    for (size_t j = 0; j <= i; ++j) {
      node_regions(g, g->nodes[j], r_j, w_j);
      for (int w : w_i) {
        const Box bw = full_box(g->tensors, w);
        for (int other : r_j)
          if (meets(bw, full_box(g->tensors, other))) {
            set_error("mk_compile: node %zu writes tensor %d over a region node %zu reads", i, w, j);
            return MK_ERR_HAZARD;
          }
        if (j == i) continue;
        for (int other : w_j)
          if (meets(bw, full_box(g->tensors, other))) {
            set_error("mk_compile: nodes %zu and %zu write overlapping regions", j, i);
            return MK_ERR_HAZARD;
          }
      }
    }
  }
  return MK_OK;
}

// A transient (plan-owned) tensor is defined by exactly one node, and every node reading it
// (through any view) comes after that node: its buffer may hold an earlier transient's data
// until the writer runs.
static mk_status check_transients(const mk_graph* g) {
  std::vector<int> writer(g->tensors.size(), -1), r, w;
  for (size_t i = 0; i < g->nodes.size(); ++i) {
    node_regions(g, g->nodes[i], r, w);
    for (int id : r) {
      const int b = g->tensors[id].base;
      if (g->tensors[b].transient && writer[b] < 0) {
        set_error("mk_compile: node %zu reads transient tensor %d before a node writes it", i, b);
        return MK_ERR_INVALID_ARG;
      }
    }
    for (int id : w) {
      const int b = g->tensors[id].base;
      if (!g->tensors[b].transient) continue;
      if (writer[b] >= 0 && writer[b] != (int)i) {
        set_error("mk_compile: transient tensor %d is written by nodes %d and %zu (one writer)", b,
                  writer[b], i);
        return MK_ERR_INVALID_ARG;
      }
      writer[b] = (int)i;
    }
  }
  return MK_OK;
}

static bool aligned16(const TensorRec& t) {
  return ((uintptr_t)t.ptr % 16) == 0 && (t.ld * dtype_size(t.dtype)) % 16 == 0;
}

// Transients have no address before mk_compile places them: their alignment is that of the
// element offset within the pool buffer (which starts 1 KB aligned).
static bool aligned16_transient(const TensorRec& t) {
  const size_t es = dtype_size(t.dtype);
  return ((t.r0 * t.ld + t.c0) * es) % 16 == 0 && (t.ld * es) % 16 == 0;
}

namespace mk {
mk_status check_kernel_support(const std::vector<TensorRec>& ts, const std::vector<NodeRec>& nodes,
                               const mk_compile_opts& o) {
  const bool pair = o.cluster == 2;
  if (!((o.gemm_tile_m == kGemmTileM && o.cluster == 1) ||
        (o.gemm_tile_m == 2 * kGemmTileM && pair))) {
    set_error("mk_compile: GEMM tiles are 128 rows on one CTA (cluster 1) or 256 rows on a CTA "
              "pair (cluster 2)");
    return MK_ERR_UNSUPPORTED;
  }
  if (o.gemm_tile_n != (pair ? 128 : 64) && o.gemm_tile_n != 128 && o.gemm_tile_n != 256) {
    set_error("mk_compile: gemm_tile_n must be 64, 128 or 256 (128 or 256 on CTA pairs)");
    return MK_ERR_UNSUPPORTED;
  }
  if (pair && o.n_sm % 2) {
    set_error("mk_compile: CTA pairs need an even n_sm");
    return MK_ERR_UNSUPPORTED;
  }
  if (o.gemv_pack != 0 && o.gemv_pack != 1) {
    set_error("mk_compile: gemv_pack is 0 or 1");
    return MK_ERR_UNSUPPORTED;
  }
  if (o.row_stage != 0 && o.row_stage != 1) {
    set_error("mk_compile: row_stage is 0 or 1");
    return MK_ERR_UNSUPPORTED;
  }
  if (o.kernel_set != 0 && o.kernel_set != 1) {
    set_error("mk_compile: kernel_set is 0 (smallest specialisation) or 1 (general kernel)");
    return MK_ERR_UNSUPPORTED;
  }
  if (o.gemv_tile_n != 256 || o.gemv_kstep % kGemvRows || o.gemv_max_m > 8 || o.gemv_max_m < 0) {
    set_error("mk_compile: the kernel runs 256-column GEMV tiles (128 with SILU_MUL), K chunks a "
              "multiple of %d, M <= 8", kGemvRows);
    return MK_ERR_UNSUPPORTED;
  }
  if (o.attn_chunk > kAttnChunkMax || o.attn_chunk % 8) {
    set_error("mk_compile: attn_chunk must be a multiple of 8, at most %d", kAttnChunkMax);
    return MK_ERR_UNSUPPORTED;
  }
  for (size_t i = 0; i < nodes.size(); ++i) {
    const NodeRec& nd = nodes[i];
    std::vector<int> all;
    for (int id : {nd.a, nd.b, nd.b2, nd.bias, nd.res, nd.gamma, nd.ins[0], nd.ins[1], nd.out,
                   nd.out_k, nd.out_v})
      if (id >= 0) all.push_back(id);
    for (int id : all) {
      if (ts[id].rows * ts[id].cols == 0) continue;  // never accessed
      const bool transient = ts[ts[id].base].transient;
      if (!transient && !ts[id].ptr) {
        set_error("mk_compile: node %zu uses tensor %d with a NULL device pointer", i, id);
        return MK_ERR_INVALID_ARG;
      }
      const bool al = transient ? aligned16_transient(ts[id]) : aligned16(ts[id]);
      // ARGMAX reads rows that are not 16-byte aligned element by element and stores one int32
      if (nd.kind != NK_ARGMAX && (!al || ts[id].cols % 8)) {
        set_error("mk_compile: node %zu tensor %d: start address and row stride must be 16-byte "
                  "aligned and cols a multiple of 8", i, id);
        return MK_ERR_UNSUPPORTED;
      }
    }
    if (nd.kind == NK_MATMUL) {
      if ((nd.flags & MK_EPI_SILU_MUL) && ts[nd.a].rows > o.gemv_max_m &&
          o.gemm_tile_n < (o.cluster == 2 ? 256 : 128)) {
        set_error("mk_compile: SILU_MUL GEMM tiles need gemm_tile_n >= 128 (256 on CTA pairs)");
        return MK_ERR_UNSUPPORTED;
      }
      if ((nd.flags & MK_EPI_RMSNORM_INPUT) && ts[nd.a].rows > o.gemv_max_m) {
        set_error("mk_compile: RMS_NORM_INPUT is fused into GEMV tiles only (M <= gemv_max_m); "
                  "use an RMSNORM node before a GEMM");
        return MK_ERR_UNSUPPORTED;
      }
    }
    if (nd.kind == NK_ROPE && nd.hd % 16) {
      set_error("mk_compile: ROPE runs head_dim a multiple of 16");
      return MK_ERR_UNSUPPORTED;
    }
    if (nd.kind == NK_ATTN) {
      if (nd.hd != 64) {
        set_error("mk_compile: attention runs head_dim 64");
        return MK_ERR_UNSUPPORTED;
      }
      for (int id : {nd.a, nd.b, nd.b2, nd.out})
        if (ts[id].dtype != DT_BF16) {
          set_error("mk_compile: attention tensors are bf16");
          return MK_ERR_UNSUPPORTED;
        }
      if (ts[nd.a].rows > 1 && o.attn_tile_q != kAttnTileQ) {
        // prefill tiles: 128 query rows per CTA (256 on a CTA pair), 64-key blocks
        set_error("mk_compile: prefill attention runs attn_tile_q %d", kAttnTileQ);
        return MK_ERR_UNSUPPORTED;
      }
    }
  }
  return MK_OK;
}
}  // namespace mk

// ------------------------------------------------------------------ tensor maps

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
  }
  return fn;
}

struct MapKey {
  uintptr_t ptr;
  int64_t rows, cols, ld;
  int dtype, box_c, box_r, swz, panels;
  bool operator==(const MapKey& o) const {
    return ptr == o.ptr && rows == o.rows && cols == o.cols && ld == o.ld && dtype == o.dtype &&
           box_c == o.box_c && box_r == o.box_r && swz == o.swz && panels == o.panels;
  }
};

// A 2D tiled map (box_c columns x box_r rows), or with panels > 0 a 3D "panel" map of a matrix
// whose column count is a multiple of 64: dimensions (column within a 64-column panel, row,
// panel), strides (row pitch, 128 bytes), box (64, box_r, panels). One copy through it writes
// `panels` consecutive 64-column atoms, each box_r rows of 128 bytes, the same bytes and layout
// as `panels` 2D copies of 64 x box_r boxes.
// swz: shared-memory swizzle span in bytes (0, 64 or 128; true = 128).
static mk_status add_map(std::vector<MapKey>& keys, std::vector<CUtensorMap>& maps,
                         const TensorRec& t, int box_c, int box_r, int swz, int* idx,
                         int panels = 0) {
  if (swz == 1) swz = 128;
  MapKey k{(uintptr_t)t.ptr, t.rows, t.cols, t.ld, t.dtype, box_c, box_r, swz, panels};
  for (size_t i = 0; i < keys.size(); ++i)
    if (keys[i] == k) {
      *idx = (int)i;
      return MK_OK;
    }
  if ((int)maps.size() >= kMaxTmaps) {
    set_error("mk_compile: more than %d distinct TMA operands", kMaxTmaps);
    return MK_ERR_UNSUPPORTED;
  }
  auto fn = encode_fn();
  if (!fn) {
    set_error("mk_compile: cuTensorMapEncodeTiled is unavailable (no CUDA driver?)");
    return MK_ERR_CUDA;
  }
  CUtensorMap m;
  memset(&m, 0, sizeof m);
  const cuuint64_t pitch = (cuuint64_t)(t.ld * dtype_size(t.dtype));
  cuuint64_t dims[3] = {(cuuint64_t)t.cols, (cuuint64_t)t.rows, 1};
  cuuint64_t strides[2] = {pitch, 0};
  cuuint32_t box[3] = {(cuuint32_t)box_c, (cuuint32_t)box_r, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  cuuint32_t rank = 2;
  if (panels > 0) {
    dims[0] = 64;
    dims[2] = (cuuint64_t)(t.cols / 64);
    strides[1] = 128;
    box[0] = 64;
    box[2] = (cuuint32_t)panels;
    rank = 3;
  }
  CUresult r = fn(&m, t.dtype == DT_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                         : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                  rank, t.ptr, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swz == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                  : swz == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                              : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("mk_compile: cuTensorMapEncodeTiled failed (%d) for a %lldx%lld tensor, box %dx%d, "
              "%d panels", (int)r, (long long)t.rows, (long long)t.cols, box_r, box_c, panels);
    return MK_ERR_CUDA;
  }
  keys.push_back(k);
  maps.push_back(m);
  *idx = (int)maps.size() - 1;
  return MK_OK;
}

static Operand operand(const std::vector<TensorRec>& ts, int id) {
  Operand o;
  o.ptr = id >= 0 ? (uint64_t)(uintptr_t)ts[id].ptr : 0;
  o.ld = id >= 0 ? (int32_t)ts[id].ld : 0;
  o.tmap = -1;
  return o;
}

// Node table and tensor maps for a device plan.
static mk_status build_nodes(const mk_graph* g, mk_plan* p, std::vector<CUtensorMap>& maps,
                             const std::vector<uint64_t>& scratch_ptr) {
  std::vector<MapKey> keys;
  const auto& ts = p->hp.tensors;
  p->nodes.assign(g->nodes.size(), Node{});
  for (size_t i = 0; i < g->nodes.size(); ++i) {
    const NodeRec& nd = g->nodes[i];
    Node& n = p->nodes[i];
    memset(&n, 0, sizeof n);
    n.flags = nd.flags;
    n.eps = nd.eps;
    n.theta = nd.theta;
    n.hq = nd.hq;
    n.hkv = nd.hkv;
    n.hd = nd.hd;
    n.pos0 = nd.pos0;
    n.causal = nd.causal;
    n.ewop = nd.ewop;
    n.tile_n = p->hp.node_tile_n[i];
    n.n_splits = p->hp.node_splits[i];
    n.n_chunks = p->hp.node_chunks[i];
    n.out = operand(ts, nd.out);
    n.out_k = operand(ts, nd.out_k);
    n.out_v = operand(ts, nd.out_v);
    n.bias = operand(ts, nd.bias);
    n.res = operand(ts, nd.res);
    n.gamma = operand(ts, nd.gamma);
    n.scratch.ptr = scratch_ptr[i];
    n.scratch.tmap = -1;
    switch (nd.kind) {
      case NK_MATMUL: {
        const TensorRec &A = ts[nd.a], &B = ts[nd.b];
        n.dtype = A.dtype;
        n.M = (int)A.rows;
        n.K = (int)A.cols;
        n.N = (int)B.cols;
        n.a = operand(ts, nd.a);
        n.b = operand(ts, nd.b);
        n.b2 = operand(ts, nd.b2);
        const bool gemv = A.rows <= p->opts.gemv_max_m;
        n.kind = gemv ? OP_GEMV : OP_GEMM;
        if (gemv) n.ldp = n.M * n.N * ((nd.flags & MK_EPI_SILU_MUL) ? 2 : 1);
        if (p->hp.node_rope[i] >= 0) {
          // the next node's RoPE runs in this matmul's GEMV or GEMM tiles (the lowering's rule)
          const NodeRec& r = g->nodes[p->hp.node_rope[i]];
          n.flags |= NF_ROPE;
          n.hq = r.hq;
          n.hkv = r.hkv;
          n.hd = r.hd;
          n.pos0 = r.pos0;
          n.theta = r.theta;
          n.out_q = operand(ts, r.out);
          n.out_k = operand(ts, r.out_k);
          n.out_v = operand(ts, r.out_v);
        }
        if (!gemv && n.M > 0 && n.N > 0) {
          // GEMM tiles store through TMA in 32 x 32 blocks (one per compute warp), 64-byte
          // swizzled; K = 0 tiles too (they store the epilogue of zero)
          mk_status st;
          if ((st = add_map(keys, maps, ts[nd.out], 32, 32, 64, &n.out.tmap))) return st;
          if (n.flags & NF_ROPE) {  // the fused rope's outputs leave the epilogue the same way
            const NodeRec& r = g->nodes[p->hp.node_rope[i]];
            if ((st = add_map(keys, maps, ts[r.out], 32, 32, 64, &n.out_q.tmap))) return st;
            if ((st = add_map(keys, maps, ts[r.out_k], 32, 32, 64, &n.out_k.tmap))) return st;
            if (r.out_v >= 0 &&
                (st = add_map(keys, maps, ts[r.out_v], 32, 32, 64, &n.out_v.tmap)))
              return st;
          }
        }
        if (n.M > 0 && n.N > 0 && n.K > 0) {
          mk_status st;
          // B (and b2) move as 64-column panels of 64 rows, 128-byte swizzled: one 3D copy
          // for all of a stage's panels when every weight has a multiple of 64 columns, else
          // one 2D copy per panel.
          const bool dual = nd.b2 >= 0;
          const bool panel = B.cols % 64 == 0 && (!dual || ts[nd.b2].cols % 64 == 0);
          int np;
          if (!gemv) {
            const int tnw = n.tile_n;  // columns per weight of one tile
            np = (p->opts.cluster == 2 ? tnw / 2 : tnw) / 64;
            if ((st = add_map(keys, maps, A, kGemmBK, kGemmTileM, true, &n.a.tmap))) return st;
          } else {
            np = dual ? 2 : 4;  // a 32 KB stage: 256 columns, or 128 gate + 128 up
          }
          const int rows = gemv ? kGemvRows : kGemmBK;
          if ((st = add_map(keys, maps, B, 64, rows, true, &n.b.tmap, panel ? np : 0))) return st;
          if (dual &&
              (st = add_map(keys, maps, ts[nd.b2], 64, rows, true, &n.b2.tmap, panel ? np : 0)))
            return st;
          if (panel) n.flags |= NF_B_PANELS;
          int w = 0;  // the node's packed weights, b then b2
          for (const auto& j : p->packs) {
            if (j.node != (int)i) continue;
            Operand& op = w++ == 0 ? n.b : n.b2;
            op.ptr = (uint64_t)(uintptr_t)(p->d_mem + j.off);
            op.ld = (j.K + 63) / 64;  // 64-row blocks per column tile
            n.flags |= NF_B_PACKED;
          }
        }
        break;
      }
      case NK_EW:
        n.kind = OP_EW;
        n.tile_m = p->opts.ew_rows;
        n.tile_n = p->opts.ew_cols * p->opts.ew_tiles;
        n.dtype = ts[nd.out].dtype;
        n.M = (int)ts[nd.out].rows;
        n.N = (int)ts[nd.out].cols;
        n.a = operand(ts, nd.ins[0]);
        n.b = operand(ts, nd.ins[1]);
        break;
      case NK_RMSNORM:
        n.kind = OP_RMSNORM;
        n.tile_m = p->opts.norm_rows;
        n.dtype = ts[nd.out].dtype;
        n.M = (int)ts[nd.out].rows;
        n.N = (int)ts[nd.out].cols;
        n.a = operand(ts, nd.ins[0]);
        break;
      case NK_ROPE:
        n.kind = OP_ROPE;
        n.tile_m = p->opts.norm_rows;
        n.dtype = ts[nd.out].dtype;
        n.M = (int)ts[nd.ins[0]].rows;
        n.N = (int)ts[nd.ins[0]].cols;
        n.a = operand(ts, nd.ins[0]);
        break;
      case NK_ARGMAX:
        n.kind = OP_ARGMAX;
        n.tile_m = p->opts.norm_rows;
        n.dtype = ts[nd.ins[0]].dtype;
        n.M = (int)ts[nd.ins[0]].rows;
        n.N = (int)ts[nd.ins[0]].cols;
        n.a = operand(ts, nd.ins[0]);
        n.n_chunks = p->hp.node_chunks[i];
        if (p->hp.node_scratch[i] >= 0) n.scratch.ld = (int)ts[p->hp.node_scratch[i]].ld;
        break;
      case NK_ATTN:
        n.kind = ts[nd.a].rows == 1 ? OP_ATTN_PARTIAL : OP_ATTN_PREFILL;
        n.dtype = DT_BF16;
        n.M = (int)ts[nd.a].rows;   // Tq
        n.K = (int)ts[nd.b].rows;   // Tk
        n.N = (int)ts[nd.a].cols;
        n.a = operand(ts, nd.a);
        n.b = operand(ts, nd.b);
        n.b2 = operand(ts, nd.b2);
        n.scale = nd.scale != 0.f ? nd.scale : 1.0f / sqrtf((float)nd.hd);
        if (p->hp.node_scratch[i] >= 0) n.scratch.ld = (int)ts[p->hp.node_scratch[i]].ld;
        if (n.M == 1) {
          if (p->opts.fuse_attn_reduce) n.flags |= NF_ATTN_FUSED;
          // key / value chunks stream by TMA: one head (64 columns) x attn_chunk rows
          n.tile_m = p->opts.attn_chunk;
          mk_status st;
          if ((st = add_map(keys, maps, ts[nd.b], 64, n.tile_m, true, &n.b.tmap))) return st;
          if ((st = add_map(keys, maps, ts[nd.b2], 64, n.tile_m, true, &n.b2.tmap))) return st;
        } else if (n.M > 0 && n.K > 0) {
          // prefill: the query tile (64 columns of one head x 128 rows) and 64-key blocks of
          // keys and values, all 128-byte swizzled
          // CTA pairs: each CTA loads half the keys of a block (32 x 64 columns) and half the
          // value columns (64 keys x 32 columns, 64-byte rows, 64-byte swizzled)
          const bool pr = p->opts.cluster == 2;
          n.tile_m = kAttnKeyBlock;
          mk_status st;
          if ((st = add_map(keys, maps, ts[nd.a], 64, kAttnTileQ, true, &n.a.tmap))) return st;
          if ((st = add_map(keys, maps, ts[nd.b], 64, pr ? kAttnKeyBlock / 2 : kAttnKeyBlock, true,
                            &n.b.tmap)))
            return st;
          if ((st = pr ? add_map(keys, maps, ts[nd.b2], 32, kAttnKeyBlock, 64, &n.b2.tmap)
                       : add_map(keys, maps, ts[nd.b2], 64, kAttnKeyBlock, true, &n.b2.tmap)))
            return st;
        }
        break;
    }
  }
  return MK_OK;
}

// ------------------------------------------------------------------ C ABI: compile/run

extern "C" mk_status mk_compile(mk_graph_t g, const mk_compile_opts* opts_in, mk_plan_t* out) {
  if (!g || !out) {
    set_error("mk_compile: NULL graph or output");
    return MK_ERR_INVALID_ARG;
  }
  *out = nullptr;
  mk_compile_opts o;
  if (opts_in) {
    o = *opts_in;
  } else {
    mk_default_opts(&o);
  }
  mk_status st = check_hazards(g);
  if (st == MK_OK) st = check_transients(g);
  if (st) return st;
  mk_plan* p = new (std::nothrow) mk_plan();
  if (!p) {
    set_error("mk_compile: out of host memory");
    return MK_ERR_OOM;
  }
  int sm_count = 0;
  if (!o.dry_run) {
    int dev = o.device;
    if (dev < 0 && cudaGetDevice(&dev) != cudaSuccess) dev = 0;
    cudaError_t e = cudaSetDevice(dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sm_count, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) {
      set_error("mk_compile: no usable CUDA device (%s)", cudaGetErrorString(e));
      delete p;
      return MK_ERR_CUDA;
    }
    p->device = dev;
    if (o.n_sm <= 0) o.n_sm = sm_count;
    if (o.n_sm > sm_count) {
      set_error("mk_compile: n_sm %d exceeds the device's %d SMs (CTAs must be co-resident)",
                o.n_sm, sm_count);
      delete p;
      return MK_ERR_UNSUPPORTED;
    }
    if ((st = check_kernel_support(g->tensors, g->nodes, o))) {
      delete p;
      return st;
    }
  } else if (o.n_sm <= 0) {
    set_error("mk_compile: dry_run needs an explicit n_sm");
    delete p;
    return MK_ERR_INVALID_ARG;
  }
  if (o.pool_waves < 1) {
    set_error("mk_compile: pool_waves must be at least 1");
    delete p;
    return MK_ERR_INVALID_ARG;
  }
  p->opts = o;
  if ((st = lower_graph(g->tensors, g->nodes, o, &p->hp))) {
    delete p;
    return st;
  }
  if (o.debug_counter >= 0) {
    if (o.debug_counter >= p->hp.n_dep) {
      set_error("mk_compile: debug_counter %d out of range", o.debug_counter);
      delete p;
      return MK_ERR_INVALID_ARG;
    }
    // Test hook: raise one counter's target so that its consumers wait on a count nothing
    // will reach (the device wait limit then ends the run with MK_ERR_TIMEOUT).
    p->hp.targets[o.debug_counter] += o.debug_extra;
    for (auto& in : p->hp.instrs)
      for (int s = 0; s < in.n_src; ++s)
        if (p->hp.src_list[2 * (in.src_off + s)] == o.debug_counter)
          p->hp.src_list[2 * (in.src_off + s) + 1] += o.debug_extra;
  }
  p->kernel_set = pick_kernel_set(p->hp.instrs, o);
  if (o.gemv_pack) {
    // GEMV weights that no instruction of the plan writes get a packed copy
    std::vector<char> bdep(g->nodes.size(), 0);
    for (const Instr& in : p->hp.instrs)
      if (in.op == OP_GEMV && (in.flags & IFLAG_B_DEP)) bdep[in.node] = 1;
    size_t off = 0;
    for (size_t i = 0; i < g->nodes.size(); ++i) {
      const NodeRec& nd = g->nodes[i];
      if (nd.kind != NK_MATMUL || bdep[i]) continue;
      const TensorRec &A = p->hp.tensors[nd.a], &B = p->hp.tensors[nd.b];
      if (A.rows > o.gemv_max_m || A.rows == 0 || A.cols == 0 || B.cols == 0) continue;
      const int tw = nd.b2 >= 0 ? 128 : 256;  // columns per weight of one GEMV tile
      for (int w : {nd.b, nd.b2}) {
        if (w < 0) continue;
        const TensorRec& W = p->hp.tensors[w];
        mk_plan::PackJob j;
        j.node = (int)i;
        j.tensor = w;
        j.src = W.ptr;
        j.ld = W.ld;
        j.K = (int)A.cols;
        j.N = (int)W.cols;
        j.tw = tw;
        j.off = off;
        off = (off + packed_gemv_bytes(j.K, j.N, tw) + 1023) & ~(size_t)1023;
        p->packs.push_back(j);
      }
    }
    p->packed_bytes = off;
  }
  if (o.dry_run) {
    *out = p;
    return MK_OK;
  }

  // Scratch per node: GEMV split partials (fp32) and attention partials (fp32).
  const auto& ts = p->hp.tensors;
  std::vector<size_t> scratch_off(g->nodes.size(), 0), scratch_len(g->nodes.size(), 0);
  size_t scratch = 0;
  auto align = [](size_t x) { return (x + 255) & ~(size_t)255; };
  for (size_t i = 0; i < g->nodes.size(); ++i) {
    const NodeRec& nd = g->nodes[i];
    size_t bytes = 0;
    if (nd.kind == NK_MATMUL && p->hp.node_splits[i] > 0) {
      bytes = (size_t)p->hp.node_splits[i] * ts[nd.a].rows * ts[nd.out].cols * 4 *
              ((nd.flags & MK_EPI_SILU_MUL) ? 2 : 1);
    } else if (nd.kind == NK_MATMUL && p->hp.node_gsplit_slots[i] > 0) {
      // GEMM split tails: one fp32 partial of a CTA's 128 rows x tile columns per slot
      bytes = (size_t)p->hp.node_gsplit_slots[i] * kGemmTileM * p->hp.node_tile_n[i] * 4 *
              ((nd.flags & MK_EPI_SILU_MUL) ? 2 : 1);
    } else if (p->hp.node_scratch[i] >= 0) {
      const TensorRec& s = ts[p->hp.node_scratch[i]];
      bytes = (size_t)s.rows * s.ld * 4;
    }
    scratch_off[i] = scratch;
    scratch_len[i] = bytes;
    scratch = align(scratch + bytes);
  }
  p->scratch_bytes = scratch;

  std::vector<CUtensorMap> maps;
  std::vector<uint64_t> scratch_ptr(g->nodes.size(), 0);  // patched after allocation
  const size_t n_ctr = (size_t)p->hp.n_dep + p->hp.n_sem;
  const size_t off_instr = 0;
  const size_t off_nodes = align(off_instr + p->hp.instrs.size() * sizeof(Instr));
  const size_t off_src = align(off_nodes + g->nodes.size() * sizeof(Node));
  const size_t off_dst = align(off_src + p->hp.src_list.size() * 4);
  const size_t off_ctr = align(off_dst + p->hp.dst_list.size() * 4);
  const size_t off_status = align(off_ctr + n_ctr * 4);
  const size_t off_last = off_status + kStatusWords * 4;  // last_status, then `done`
  const size_t off_snap = align(off_last + (kStatusWords + 1) * 4);
  const size_t off_trace = align(off_snap + (o.snapshot_counters ? n_ctr * 4 : 0));
  const size_t trace_bytes = o.trace ? p->hp.instrs.size() * kTraceWords * sizeof(uint64_t) : 0;
  const size_t off_maps = align(off_trace + trace_bytes);
  const size_t off_scratch = align(off_maps + kMaxTmaps * sizeof(CUtensorMap));
  const size_t off_pack = (off_scratch + scratch + 1023) & ~(size_t)1023;
  const size_t off_pool = off_pack + p->packed_bytes;  // packed copies end 1 KB aligned
  const size_t total = off_pool + (size_t)p->hp.pool_bytes;
  for (auto& j : p->packs) j.off += off_pack;
  if (cudaMalloc((void**)&p->d_mem, total) != cudaSuccess) {
    cudaGetLastError();
    set_error("mk_compile: cudaMalloc of %zu plan bytes failed", total);
    delete p;
    return MK_ERR_OOM;
  }
  for (size_t i = 0; i < g->nodes.size(); ++i)
    scratch_ptr[i] = scratch_len[i] ? (uint64_t)(uintptr_t)(p->d_mem + off_scratch + scratch_off[i]) : 0;
  for (size_t t = 0; t < p->hp.pool_off.size(); ++t)  // transients (and their views) get addresses
    if (p->hp.pool_off[t] >= 0) p->hp.tensors[t].ptr = p->d_mem + off_pool + p->hp.pool_off[t];
  if ((st = build_nodes(g, p, maps, scratch_ptr))) {
    cudaFree(p->d_mem);
    delete p;
    return st;
  }
  // 48 KB stages only where a single-CTA GEMM tile needs them; every other ring user (a GEMV
  // weight tile, an attention key/value chunk or prefill block, staged rows) fits 32 KB, so such
  // plans prefetch 192 KB of operands per SM instead of 128 KB.
  bool single_gemm = false;
  for (const Instr& in : p->hp.instrs) single_gemm |= in.op == OP_GEMM;
  single_gemm &= o.cluster != 2;
  const int stages = single_gemm ? kStages : kPairStages;
  const int64_t stage_bytes = kRingBytes / stages;
  if (o.row_stage && o.cluster == 1 && ks_stages_rows(p->kernel_set)) {
    // staged rows: the ring stages each RMSNorm / RoPE instruction fills (Instr.pad)
    for (Instr& in : p->hp.instrs) {
      if (in.op != OP_RMSNORM && in.op != OP_ROPE) continue;
      const Node& n = p->nodes[in.node];
      if (n.dtype != DT_F16 && n.dtype != DT_BF16) continue;
      const int64_t w = n.N;  // the whole row of x (RoPE: q, k and v heads)
      // RoPE: the angle table fits, and whole heads of 16-byte chunks fall in one warp
      if (in.op == OP_ROPE && (2 * (int64_t)n.tile_m * (n.hd / 2) > kXrFloats || n.hd % 16 ||
                               32 % (n.hd / 8)))
        continue;
      const int64_t rows = std::min<int64_t>(n.tile_m, n.M - in.m0);
      const int64_t rps = w > 0 ? stage_bytes / (w * 2) : 0;
      if (rps == 0 || rows <= 0) continue;
      in.pad = (int32_t)((rows + rps - 1) / rps);
    }
  }
  auto up = [&](size_t off, const void* src, size_t bytes) -> cudaError_t {
    return bytes ? cudaMemcpy(p->d_mem + off, src, bytes, cudaMemcpyHostToDevice) : cudaSuccess;
  };
  cudaError_t e = up(off_instr, p->hp.instrs.data(), p->hp.instrs.size() * sizeof(Instr));
  if (e == cudaSuccess) e = up(off_nodes, p->nodes.data(), p->nodes.size() * sizeof(Node));
  if (e == cudaSuccess) e = up(off_src, p->hp.src_list.data(), p->hp.src_list.size() * 4);
  if (e == cudaSuccess) e = up(off_dst, p->hp.dst_list.data(), p->hp.dst_list.size() * 4);
  if (e == cudaSuccess) e = up(off_maps, maps.data(), maps.size() * sizeof(CUtensorMap));
  if (e == cudaSuccess) e = cudaMemset(p->d_mem + off_ctr, 0, off_maps - off_ctr);
  if (e == cudaSuccess && !p->packs.empty()) {
    e = run_packs(p, 0);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
  }
  if (e == cudaSuccess) {
    p->smem = megakernel_smem_bytes();
    e = configure_megakernel(p->smem);
  }
  if (e == cudaSuccess && o.cluster == 2) {
    int clusters = 0;
    e = pair_clusters_resident(p->smem, p->kernel_set, &clusters);
    if (e == cudaSuccess && clusters < o.n_sm / 2) {
      set_error("mk_compile: only %d CTA pairs can be resident, %d needed", clusters, o.n_sm / 2);
      cudaFree(p->d_mem);
      delete p;
      return MK_ERR_UNSUPPORTED;
    }
  }
  if (e != cudaSuccess) {
    set_error("mk_compile: device upload failed: %s", cudaGetErrorString(e));
    cudaFree(p->d_mem);
    delete p;
    return MK_ERR_CUDA;
  }
  Params& pr = p->params;
  pr.instrs = (const Instr*)(p->d_mem + off_instr);
  pr.nodes = (const Node*)(p->d_mem + off_nodes);
  pr.src_list = (const int32_t*)(p->d_mem + off_src);
  pr.dst_list = (const int32_t*)(p->d_mem + off_dst);
  pr.counters = (int32_t*)(p->d_mem + off_ctr);
  pr.status = (int32_t*)(p->d_mem + off_status);
  pr.last_status = (int32_t*)(p->d_mem + off_last);
  pr.done = pr.last_status + kStatusWords;
  pr.snapshot = o.snapshot_counters ? (int32_t*)(p->d_mem + off_snap) : nullptr;
  pr.trace = o.trace ? (uint64_t*)(p->d_mem + off_trace) : nullptr;
  pr.tmaps = (const void*)(p->d_mem + off_maps);
  pr.n_instr = (int32_t)p->hp.instrs.size();
  pr.n_sm = o.n_sm;
  pr.n_tmaps = (int32_t)maps.size();
  pr.n_counters = (int32_t)n_ctr;
  pr.stages = stages;
  pr.timeout_ns = (uint64_t)(o.timeout_ms > 0 ? o.timeout_ms : 2000) * 1000000ull;
  p->grid = o.n_sm;
  p->on_device = true;
  *out = p;
  return MK_OK;
}

extern "C" mk_status mk_run(mk_plan_t p, void* stream) {
  if (!p || !p->on_device) {
    set_error("mk_run: plan is NULL or was compiled with dry_run");
    return MK_ERR_INVALID_ARG;
  }
  cudaStream_t s = (cudaStream_t)stream;
  if (p->params.n_instr == 0) return MK_OK;
  CUDA_TRY(launch_megakernel(p->params, p->grid, p->smem, s, p->opts.cluster == 2,
                             p->kernel_set));
  return MK_OK;
}

static mk_status host_copy(mk_plan_t p, const mk_host_copy& c, cudaStream_t s) {
  const auto& ts = p->hp.tensors;
  if (c.tensor < 0 || c.tensor >= (int)ts.size() || ts[c.tensor].internal || !c.host) {
    set_error("mk_run_host: bad tensor id %d or NULL host pointer", c.tensor);
    return MK_ERR_INVALID_ARG;
  }
  if (c.to_device && ts[ts[c.tensor].base].transient) {
    set_error("mk_run_host: tensor %d is a transient, which its writer node defines", c.tensor);
    return MK_ERR_INVALID_ARG;
  }
  const TensorRec& t = ts[c.tensor];
  const size_t es = dtype_size(t.dtype);
  if (t.rows == 0 || t.cols == 0) return MK_OK;
  if (c.to_device)
    CUDA_TRY(cudaMemcpy2DAsync(t.ptr, t.ld * es, c.host, t.cols * es, t.cols * es, t.rows,
                               cudaMemcpyHostToDevice, s));
  else
    CUDA_TRY(cudaMemcpy2DAsync(c.host, t.cols * es, t.ptr, t.ld * es, t.cols * es, t.rows,
                               cudaMemcpyDeviceToHost, s));
  return MK_OK;
}

extern "C" mk_status mk_run_host(mk_plan_t p, const mk_host_copy* copies, int32_t n,
                                 void* stream) {
  if (!p || (n > 0 && !copies) || n < 0 || !p->on_device) {
    set_error("mk_run_host: NULL plan or copies, or a dry-run plan");
    return MK_ERR_INVALID_ARG;
  }
  cudaStream_t s = (cudaStream_t)stream;
  mk_status st;
  for (int i = 0; i < n; ++i) {
    if (!copies[i].to_device) continue;
    if ((st = host_copy(p, copies[i], s))) return st;
    if (p->on_device && !p->packs.empty())  // a packed GEMV weight follows its tensor
      CUDA_TRY(run_packs(p, s, p->hp.tensors[copies[i].tensor].base));
  }
  if ((st = mk_run(p, stream))) return st;
  for (int i = 0; i < n; ++i)
    if (!copies[i].to_device && (st = host_copy(p, copies[i], s))) return st;
  return MK_OK;
}

extern "C" mk_status mk_plan_repack(mk_plan_t p, void* stream) {
  if (!p || !p->on_device) {
    set_error("mk_plan_repack: NULL plan or dry-run plan");
    return MK_ERR_INVALID_ARG;
  }
  CUDA_TRY(run_packs(p, (cudaStream_t)stream));
  return MK_OK;
}

extern "C" mk_status mk_sync_status(mk_plan_t p, mk_device_status* st) {
  if (!p || !st || !p->on_device) {
    set_error("mk_sync_status: NULL plan/status or dry-run plan");
    return MK_ERR_INVALID_ARG;
  }
  CUDA_TRY(cudaDeviceSynchronize());
  int32_t w[kStatusWords];
  CUDA_TRY(cudaMemcpy(w, p->params.last_status, sizeof w, cudaMemcpyDeviceToHost));
  st->code = w[ST_CODE];
  st->instr = w[ST_INSTR];
  st->counter = w[ST_COUNTER];
  st->observed = w[ST_OBSERVED];
  st->expected = w[ST_EXPECTED];
  st->sm = w[ST_SM];
  st->role = w[ST_ROLE];
  st->where = w[ST_WHERE];
  if (st->code) {
    // read: the next runs report afresh
    CUDA_TRY(cudaMemset(p->params.last_status, 0, sizeof w));
    set_error("device reported %s at instruction %d (SM %d, role %d, site %d): counter %d "
              "observed %d, expected %d",
              st->code == MK_ERR_TIMEOUT ? "a wait timeout" : "a failed check", st->instr, st->sm,
              st->role, st->where, st->counter, st->observed, st->expected);
  }
  return st->code;
}

extern "C" mk_status mk_plan_destroy(mk_plan_t p) {
  if (p && p->d_mem) cudaFree(p->d_mem);
  delete p;
  return MK_OK;
}

extern "C" mk_status mk_plan_stats(mk_plan_t p, mk_stats* s) {
  if (!p || !s) {
    set_error("mk_plan_stats: NULL");
    return MK_ERR_INVALID_ARG;
  }
  memset(s, 0, sizeof *s);
  s->n_instr = (int64_t)p->hp.instrs.size();
  s->n_counters = p->hp.n_dep;
  s->n_sems = p->hp.n_sem;
  s->n_sm = p->hp.n_sm;
  s->n_iter = p->hp.n_sm ? (s->n_instr + p->hp.n_sm - 1) / p->hp.n_sm : 0;
  s->waves = p->hp.n_sm ? (double)s->n_instr / p->hp.n_sm : 0.0;
  s->n_src = (int64_t)p->hp.src_list.size() / 2;
  s->n_dst = (int64_t)p->hp.dst_list.size();
  for (const auto& in : p->hp.instrs)
    if (in.op < 16) s->per_op[in.op]++;
  s->smem_bytes = (int64_t)p->smem;
  s->scratch_bytes = (int64_t)p->scratch_bytes;
  s->kernel_set = p->kernel_set;
  s->packed_bytes = (int64_t)p->packed_bytes;
  s->pool_bytes = p->hp.pool_bytes;
  s->n_reuse = p->hp.n_reuse;
  return MK_OK;
}

extern "C" mk_status mk_plan_tensor_ptr(mk_plan_t p, int32_t tensor, void** ptr) {
  if (!p || !ptr || tensor < 0 || tensor >= (int)p->hp.tensors.size() ||
      p->hp.tensors[tensor].internal) {
    set_error("mk_plan_tensor_ptr: NULL plan/pointer or bad tensor id %d", tensor);
    return MK_ERR_INVALID_ARG;
  }
  *ptr = p->hp.tensors[tensor].ptr;
  return MK_OK;
}

extern "C" mk_status mk_get_instructions(mk_plan_t p, void* buf, size_t bytes) {
  if (!p || !buf || bytes < p->hp.instrs.size() * sizeof(Instr)) {
    set_error("mk_get_instructions: NULL or buffer smaller than n_instr * 64");
    return MK_ERR_INVALID_ARG;
  }
  memcpy(buf, p->hp.instrs.data(), p->hp.instrs.size() * sizeof(Instr));
  return MK_OK;
}

extern "C" mk_status mk_get_src_list(mk_plan_t p, int32_t* buf, size_t n) {
  if (!p || (!buf && !p->hp.src_list.empty()) || n < p->hp.src_list.size()) {
    set_error("mk_get_src_list: NULL or buffer too small");
    return MK_ERR_INVALID_ARG;
  }
  if (!p->hp.src_list.empty()) memcpy(buf, p->hp.src_list.data(), p->hp.src_list.size() * 4);
  return MK_OK;
}

extern "C" mk_status mk_get_dst_list(mk_plan_t p, int32_t* buf, size_t n) {
  if (!p || (!buf && !p->hp.dst_list.empty()) || n < p->hp.dst_list.size()) {
    set_error("mk_get_dst_list: NULL or buffer too small");
    return MK_ERR_INVALID_ARG;
  }
  if (!p->hp.dst_list.empty()) memcpy(buf, p->hp.dst_list.data(), p->hp.dst_list.size() * 4);
  return MK_OK;
}

extern "C" mk_status mk_get_counter_targets(mk_plan_t p, int32_t* buf, size_t n) {
  if (!p || (!buf && p->hp.n_dep) || n < (size_t)p->hp.n_dep) {
    set_error("mk_get_counter_targets: NULL or buffer too small");
    return MK_ERR_INVALID_ARG;
  }
  if (p->hp.n_dep) memcpy(buf, p->hp.targets.data(), (size_t)p->hp.n_dep * 4);
  return MK_OK;
}

extern "C" mk_status mk_get_trace(mk_plan_t p, uint64_t* buf, size_t n) {
  if (!p || !p->on_device || !p->params.trace) {
    set_error("mk_get_trace: NULL plan, dry-run plan, or compiled without trace");
    return MK_ERR_INVALID_ARG;
  }
  const size_t need = p->hp.instrs.size() * kTraceWords;
  if ((!buf && need) || n < need) {
    set_error("mk_get_trace: buffer smaller than 8 * n_instr");
    return MK_ERR_INVALID_ARG;
  }
  CUDA_TRY(cudaDeviceSynchronize());
  if (need) CUDA_TRY(cudaMemcpy(buf, p->params.trace, need * 8, cudaMemcpyDeviceToHost));
  return MK_OK;
}

extern "C" mk_status mk_get_counters(mk_plan_t p, int32_t* buf, size_t n) {
  if (!p || !p->on_device) {
    set_error("mk_get_counters: NULL or dry-run plan");
    return MK_ERR_INVALID_ARG;
  }
  const size_t need = (size_t)p->hp.n_dep + p->hp.n_sem;
  if ((!buf && need) || n < need || !p->params.snapshot) {
    set_error("mk_get_counters: buffer too small, or the plan was compiled without "
              "snapshot_counters");
    return MK_ERR_INVALID_ARG;
  }
  CUDA_TRY(cudaDeviceSynchronize());
  if (need) CUDA_TRY(cudaMemcpy(buf, p->params.snapshot, need * 4, cudaMemcpyDeviceToHost));
  return MK_OK;
}
