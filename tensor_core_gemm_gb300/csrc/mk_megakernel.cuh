// The persistent megakernel: one CTA per SM walks its share of the instruction list.
//
// This header holds the kernel template, megakernel<PAIR, KS>: PAIR selects CTA-pair GEMM tiles,
// KS the instruction kinds compiled in (KernelSet). Each specialisation is instantiated by one
// small translation unit, so they compile in parallel.
//
// Roles inside a CTA (256 threads):
//   warp 0      scheduler: publishes instruction descriptors into an 8-slot ring ahead of the
//               roles and polls the global dependency counters of the oldest published one
//               ("MegaKittens Internals" §09 controller; §11 barrier wait with acquire).
//   warp 1      TMA loader: streams operand tiles into a shared-memory ring (4 stages of 48 KB,
//               or 6 of 32 KB); weight (B) tiles of an instruction are issued before its
//               activations are ready ("Beating torch.compile with Megakernels", "TMA Compute
//               Overlap"; MegaKittens §00); packed GEMV weights move as one bulk copy per stage.
//   warp 2      MMA issuer: tcgen05.mma into TMEM: GEMM tiles into a double-buffered accumulator
//               ("Hand-writing a Blackwell GEMM", steps 3 and 8: warp specialisation, persistent
//               kernel with two accumulator slots), GEMV tiles with swapped operands, and the
//               S = QK^T and O += PV products of prefill attention.
//   warp 3      spare.
//   warps 4-7   compute warpgroup: GEMM epilogue (TMEM -> registers -> fused epilogue -> TMA
//               store), GEMV activation staging and split-K epilogue, elementwise / RMSNorm /
//               RoPE / ARGMAX rows, split-KV attention partial and combine, prefill attention
//               softmax; publishes finished tiles on the global counters (release).
// Every wait is bounded: past `timeout_ns` the waiter records MK_ERR_TIMEOUT in the status word,
// every role drains what it has in flight and the CTA exits normally.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "mk.h"
#include "mk_ptx.cuh"
#include "mk_types.h"

namespace mk {
using namespace ptx;

// Device code has internal linkage: every specialisation's translation unit holds its own copy.
namespace {

enum RoleId { R_SCHED = 0, R_LOAD = 1, R_MMA = 2, R_COMPUTE = 3 };
constexpr unsigned FULL = 0xffffffffu;
constexpr int kCompute = 128;   // threads of the compute warpgroup
constexpr int kBarCompute = 1;  // named barrier of the compute warpgroup

struct __align__(1024) Smem {
  uint8_t ring[kRingBytes];             // operand ring (stages 1024-byte aligned: 128-byte swizzle)
  float xr[kXrFloats];                  // GEMV activations, then its output exchange
  float red_small[8][4];                // per-row, per-warp partial sums
  uint8_t slot[kSlots][kSlotBytes];     // instruction record + node entry per slot
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t go;                          // pair mode, odd CTA: released by the even CTA once per GEMM
  uint64_t gx_full;                     // tensor-core GEMV: the activation operand is staged
  // prefill attention: scores S and P double-buffered in TMEM (P in a stage on pairs), O in TMEM
  uint64_t att_s_full[2], att_s_free[2], att_p_full[2], att_o_full[2];
  uint64_t att_q_full;                  // CTA pairs: both CTAs' query tiles are in xr
  uint64_t att_done;                    // CTA pairs: both CTAs have read O (once per tile)
  uint64_t instr_ready[kSlots];
  uint64_t deps_ready[kSlots];
  uint64_t slot_free[kSlots];
  uint64_t drain;
  float rstd[8];
  uint32_t tmem_base;
  int32_t flag;
};
static_assert(sizeof(Smem) + 1024 <= 232448, "shared memory budget of one CTA");

constexpr size_t kMegakernelSmem = sizeof(Smem) + 1024;  // dynamic smem of a launch

// ------------------------------------------------------------------ small helpers

__device__ __forceinline__ const Instr& slot_instr(const Smem& s, int slot) {
  return *reinterpret_cast<const Instr*>(s.slot[slot]);
}
__device__ __forceinline__ const Node& slot_node(const Smem& s, int slot) {
  return *reinterpret_cast<const Node*>(s.slot[slot] + sizeof(Instr));
}
__device__ __forceinline__ const void* tmap_at(const Params& p, int i) {
  return static_cast<const char*>(p.tmaps) + (size_t)i * 128;
}
// Ring geometry of this launch: 4 stages of 48 KB, or 6 of 32 KB when GEMM tiles run on CTA pairs
// (every other ring user, a GEMV weight tile or an attention key/value chunk, fits in 32 KB).
__device__ __forceinline__ uint32_t ring_n(const Params& p) { return (uint32_t)p.stages; }
__device__ __forceinline__ uint32_t stage_bytes(const Params& p) {
  return p.stages == kPairStages ? 32768u : 49152u;
}
__device__ __forceinline__ uint8_t* stage_ptr(Smem& s, const Params& p, int st) {
  return s.ring + (size_t)st * stage_bytes(p);
}
// Position in the operand ring: stage index and the parity of the current pass over the ring
// (use count / depth, mod 2), advanced incrementally so hot loops do no division.
struct RingPos {
  uint32_t st = 0, ph = 0;
  __device__ __forceinline__ void next(uint32_t ns) {
    if (++st == ns) {
      st = 0;
      ph ^= 1u;
    }
  }
  __device__ __forceinline__ void advance(uint32_t n, uint32_t ns) {
    const uint32_t t = st + n;
    st = t % ns;
    ph ^= (t / ns) & 1u;
  }
  __device__ __forceinline__ void align() {  // to the start of the next pass
    if (st) {
      st = 0;
      ph ^= 1u;
    }
  }
};
// A plain use count rounded up to the start of the next pass (the compute warpgroup's count).
__device__ __forceinline__ uint32_t ring_align(uint32_t v, uint32_t ns) {
  return (v + ns - 1) / ns * ns;
}
__device__ __forceinline__ int ring_stages(const Instr& in) {
  if (in.op == OP_GEMM) return (in.klen + kGemmBK - 1) / kGemmBK;
  if (in.op == OP_GEMV) return (in.klen + kGemvRows - 1) / kGemvRows;
  if (in.op == OP_ATTN_PARTIAL) return 1;  // the key/value chunk
  if (in.op == OP_ATTN_PREFILL) return (in.klen + kAttnKeyBlock - 1) / kAttnKeyBlock;
  if (in.op == OP_RMSNORM || in.op == OP_ROPE) return in.pad;  // staged rows (0: direct)
  return 0;
}
// Columns of each input row a staged row instruction copies: the whole row of x (RMSNorm: the
// normalised columns; RoPE: the q and k heads, then the v heads when it copies v).
__device__ __forceinline__ int row_stage_cols(const Node& nd) { return nd.N; }
__device__ __forceinline__ int instr_index(const Params& p, int it) {
  return it * p.n_sm + (int)blockIdx.x;
}

__device__ void report(const Params& p, int code, int instr, int counter, int observed,
                       int expected, int role, int where) {
  if (atomicCAS(p.status + ST_CODE, 0, code) == 0) {
    p.status[ST_INSTR] = instr;
    p.status[ST_COUNTER] = counter;
    p.status[ST_OBSERVED] = observed;
    p.status[ST_EXPECTED] = expected;
    p.status[ST_SM] = (int)blockIdx.x;
    p.status[ST_ROLE] = role;
    p.status[ST_WHERE] = where;
    __threadfence();
  }
}

// Bounded mbarrier wait; false when the limit passed (reported) or another waiter aborted.
// On-chip waits get four times the counter-wait limit: when a dependency never completes, the
// scheduler's counter wait runs out first and the report names the counter.
__device__ bool wait_mbar(const Params& p, uint32_t bar, uint32_t parity, int role, int where,
                          int instr, bool cluster_scope = false) {
  auto probe = [&]() { return cluster_scope ? mbar_try_cluster(bar, parity) : mbar_try(bar, parity); };
  if (probe()) return true;
  const uint64_t t0 = globaltimer();
  const uint64_t limit = 4 * p.timeout_ns;
  for (uint32_t n = 1;; ++n) {
    if (probe()) return true;
    if ((n & 15u) == 0) {
      if (ld_volatile(p.status + ST_CODE) != 0) return false;
      if (globaltimer() - t0 > limit) {
        report(p, MK_ERR_TIMEOUT, instr, -1, 0, (int)parity, role, where);
        return false;
      }
    }
  }
}
// Warp-converged variant for roles run by a whole warp: every lane polls the same barrier and
// all lanes leave together (lane 0's view of the limit decides), so the code after it stays
// converged and its values warp-uniform.
__device__ __noinline__ bool wait_warp_slow(const Params& p, uint32_t bar, uint32_t parity,
                                            int role, int where, int instr, bool cluster_scope) {
  const uint64_t t0 = globaltimer();
  const uint64_t limit = 4 * p.timeout_ns;
  for (uint32_t n = 1;; ++n) {
    const bool done = cluster_scope ? mbar_try_cluster(bar, parity) : mbar_try(bar, parity);
    if (__all_sync(FULL, done)) return true;
    if ((n & 15u) == 0) {
      int stop = 0;
      if ((threadIdx.x & 31) == 0) {
        if (ld_volatile(p.status + ST_CODE) != 0) stop = 1;
        else if (globaltimer() - t0 > limit) stop = 2;
      }
      stop = __shfl_sync(FULL, stop, 0);
      if (stop) {
        if (stop == 2 && (threadIdx.x & 31) == 0)
          report(p, MK_ERR_TIMEOUT, instr, -1, 0, (int)parity, role, where);
        return false;
      }
    }
  }
}
__device__ __forceinline__ bool wait_warp(const Params& p, uint32_t bar, uint32_t parity, int role,
                                          int where, int instr, bool cluster_scope = false) {
  const bool done = cluster_scope ? mbar_try_cluster(bar, parity) : mbar_try(bar, parity);
  if (__all_sync(FULL, done)) return true;
  return wait_warp_slow(p, bar, parity, role, where, instr, cluster_scope);
}
// Wait used while draining after an abort: ignores the status word, short fixed limit.
__device__ void wait_mbar_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try(bar, parity))
    if (globaltimer() - t0 > 200000000ull) return;
}
// Compute warpgroup: its first thread polls a global counter until it reaches `target`
// (acquire, bounded like every wait), then all threads agree on the outcome.
__device__ bool cw_wait_counter(const Params& p, const int32_t* ctr, int target, int where,
                                int instr) {
  bool ok = true;
  if (threadIdx.x == kThreads - kCompute && ld_acquire(ctr) < target) {
    const uint64_t t0 = globaltimer();
    for (uint32_t n = 1;; ++n) {
      if (ld_acquire(ctr) >= target) break;
      if ((n & 15u) == 0) {
        if (ld_volatile(p.status + ST_CODE) != 0) {
          ok = false;
          break;
        }
        if (globaltimer() - t0 > p.timeout_ns) {
          report(p, MK_ERR_TIMEOUT, instr, (int)(ctr - p.counters), ld_volatile(ctr), target,
                 R_COMPUTE, where);
          ok = false;
          break;
        }
      }
    }
  }
  return bar_and(kBarCompute, kCompute, ok);
}

// Compute-warpgroup wait: every thread waits (bounded), then all agree on the outcome so no
// thread is left alone at a later named barrier.
__device__ __forceinline__ bool cw_wait(const Params& p, uint32_t bar, uint32_t parity, int where,
                                        int instr) {
  const bool ok = wait_mbar(p, bar, parity, R_COMPUTE, where, instr);
  return bar_and(kBarCompute, kCompute, ok);
}
__device__ __forceinline__ void cw_sync() { bar_sync(kBarCompute, kCompute); }
// Trace point `k` of instruction `idx` (compute warpgroup, thread 0), when tracing is on.
__device__ __forceinline__ void trace_mark(const Params& p, int idx, int k) {
  if (p.trace && threadIdx.x == kThreads - kCompute) p.trace[(size_t)idx * kTraceWords + k] = globaltimer();
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(FULL, v, o));
  return v;
}
// silu(z) = z * sigmoid(z), with the fast exponential and division intrinsics: for z below
// about -87 the denominator passes 2^126 and the quotient is 0 (true value below 1e-36).
__device__ __forceinline__ float silu(float z) { return __fdividef(z, 1.0f + __expf(-z)); }
// sin and cos of a RoPE angle (|a| up to ~1e5 rad): Cody and Waite's additive reduction to
// [-pi, pi], 2*pi split into its fp32 rounding and the remainder of that rounding (two fused
// multiply-adds, the remainder's term below 1e-7 rad for these angles), then the hardware sine
// and cosine approximations, which hold 2^-21 absolute accuracy on that interval. Every RoPE
// path (rows, fused into GEMV and GEMM tiles) takes the same steps, so they agree bit for bit.
__device__ __forceinline__ void rope_sincos(float a, float* sn, float* cs) {
  const float k = rintf(a * 0.15915493667125702f);  // a / (2 pi), nearest integer
  float r = fmaf(-k, 6.2831854820251465f, a);
  r = fmaf(-k, -1.7484555314695172e-07f, r);
  __sincosf(r, sn, cs);
}
// One rotate_half pair (x1 in the first half of the head, x2 its partner in the second):
// z1 = x1 cos - x2 sin and z2 = x2 cos + x1 sin, each as one rounded product and one fused
// multiply-add, so that every RoPE path rounds the same way.
__device__ __forceinline__ float rope_z1(float x1, float x2, float c, float s) {
  return fmaf(x1, c, -__fmul_rn(x2, s));
}
__device__ __forceinline__ float rope_z2(float x1, float x2, float c, float s) {
  return fmaf(x2, c, __fmul_rn(x1, s));
}

// 16-bit element conversions (dt: DT_F16 or DT_BF16).
__device__ __forceinline__ float h2f(uint16_t v, int dt) {
  return dt == DT_BF16 ? __uint_as_float((uint32_t)v << 16)
                       : __half2float(__ushort_as_half(v));
}
// 8 packed elements <-> 8 floats. The element type is uniform, so one branch picks the path;
// conversions go two elements at a time (one paired instruction each way), the same rounding
// as element by element.
__device__ __forceinline__ void unpack8(const uint4 raw, int dt, float* x) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
  if (dt == DT_BF16) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = __uint_as_float(w[i] << 16);
      x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
      x[2 * i] = f.x;
      x[2 * i + 1] = f.y;
    }
  }
}
__device__ __forceinline__ uint4 pack8(const float* x, int dt) {
  uint32_t w[4];
  if (dt == DT_BF16) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat162 t = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
      w[i] = *reinterpret_cast<const uint32_t*>(&t);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __half2 t = __floats2half2_rn(x[2 * i], x[2 * i + 1]);
      w[i] = *reinterpret_cast<const uint32_t*>(&t);
    }
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}
// 8 consecutive elements of an operand at (row, col); data produced inside the kernel is read
// at L2 (ld.global.cg) so no SM can see a stale L1 line.
__device__ __forceinline__ void load8(const Operand& o, int row, int col, int dt, float* x) {
  const uint16_t* ptr = reinterpret_cast<const uint16_t*>(o.ptr) + (size_t)row * o.ld + col;
  unpack8(__ldcg(reinterpret_cast<const uint4*>(ptr)), dt, x);
}
__device__ __forceinline__ void store8(const Operand& o, int row, int col, int dt, const float* x) {
  uint16_t* ptr = reinterpret_cast<uint16_t*>(o.ptr) + (size_t)row * o.ld + col;
  *reinterpret_cast<uint4*>(ptr) = pack8(x, dt);
}
__device__ __forceinline__ float load1(const Operand& o, int row, int col, int dt) {
  const uint16_t* ptr = reinterpret_cast<const uint16_t*>(o.ptr) + (size_t)row * o.ld + col;
  return h2f(__ldcg(reinterpret_cast<const unsigned short*>(ptr)), dt);
}
__device__ __forceinline__ uint32_t pack2(float v0, float v1, int dt) {
  if (dt == DT_BF16) {
    const __nv_bfloat162 t = __floats2bfloat162_rn(v0, v1);
    return *reinterpret_cast<const uint32_t*>(&t);
  }
  const __half2 t = __floats2half2_rn(v0, v1);
  return *reinterpret_cast<const uint32_t*>(&t);
}
// a and b rounded to the element type and back: the values a later reader of the stored pair
// sees
__device__ __forceinline__ void round2(float& a, float& b, int dt) {
  float2 f;
  if (dt == DT_BF16)
    f = __bfloat1622float2(__floats2bfloat162_rn(a, b));
  else
    f = __half22float2(__floats2half2_rn(a, b));
  a = f.x;
  b = f.y;
}
__device__ __forceinline__ void store2(const Operand& o, int row, int col, int dt, float v0,
                                       float v1) {
  uint16_t* ptr = reinterpret_cast<uint16_t*>(o.ptr) + (size_t)row * o.ld + col;
  *reinterpret_cast<uint32_t*>(ptr) = pack2(v0, v1, dt);
}

// ------------------------------------------------------------------ scheduler warp

template <int KS>
__device__ void run_scheduler(const Params& p, Smem& s) {
  const int lane = threadIdx.x & 31;
  int fetched = 0, ready = 0;
  bool end_published = false;
  uint32_t idle = 0;
  uint64_t idle_since = 0;
  int pend_ctr = -1, pend_obs = 0, pend_tgt = 0;
  while (true) {
    bool progress = false;
    // Publish the next descriptor as soon as its slot is free: roles may run ahead of the
    // dependency resolution by up to kSlots instructions (the loader prefetches weights).
    if (!end_published && fetched < ready + kSlots) {
      const int slot = fetched % kSlots;
      const uint32_t use = (uint32_t)(fetched / kSlots);
      if (mbar_try(smem_u32(&s.slot_free[slot]), (use & 1u) ^ 1u)) {
        uint32_t* dst = reinterpret_cast<uint32_t*>(s.slot[slot]);
        const int idx = instr_index(p, fetched);
        if (idx < p.n_instr) {
          const uint32_t* si = reinterpret_cast<const uint32_t*>(p.instrs + idx);
          const uint32_t w = lane < 16 ? __ldg(si + lane) : 0u;
          const int node = __shfl_sync(FULL, (int)w, 1);
          const int op = (int)(__shfl_sync(FULL, w, 0) & 0xffffu);
          if (!ks_covers(KS, op)) {  // the host launches a specialisation that covers the plan
            if (lane == 0) report(p, MK_ERR_DEVICE_CHECK, idx, -1, op, KS, R_SCHED, 2);
            break;
          }
          if (lane < 16) dst[lane] = w;
          const uint32_t* sn = reinterpret_cast<const uint32_t*>(p.nodes + node);
          dst[16 + lane] = __ldg(sn + lane);
          dst[48 + lane] = __ldg(sn + 32 + lane);
          ++fetched;
        } else {
          if (lane == 0) dst[0] = (uint32_t)OP_END;
          end_published = true;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&s.instr_ready[slot]));
        progress = true;
      }
    }
    // Resolve the oldest published instruction's sources (one pass, lanes in parallel).
    if (ready < fetched) {
      const int slot = ready % kSlots;
      const Instr& in = slot_instr(s, slot);
      bool ok = true;
      pend_ctr = -1;
      for (int j = lane; j < in.n_src; j += 32) {
        const int ctr = __ldg(p.src_list + 2 * (in.src_off + j));
        const int tgt = __ldg(p.src_list + 2 * (in.src_off + j) + 1);
        const int v = ld_acquire(p.counters + ctr);
        if (v < tgt) {
          ok = false;
          pend_ctr = ctr;
          pend_obs = v;
          pend_tgt = tgt;
        }
      }
      if (__all_sync(FULL, ok)) {
        if (lane == 0) {
          // later TMA (async-proxy) reads of the producers' data are ordered after the acquire
          fence_proxy_async_global();
          mbar_arrive(smem_u32(&s.deps_ready[slot]));
          if (p.trace) p.trace[(size_t)instr_index(p, ready) * kTraceWords + 1] = globaltimer();
        }
        ++ready;
        progress = true;
      }
    }
    if (end_published && ready == fetched) break;
    if (progress) {
      idle = 0;
      continue;
    }
    if (idle++ == 0) {
      idle_since = globaltimer();
    } else if ((idle & 15u) == 0) {
      if (ld_volatile(p.status + ST_CODE) != 0) break;
      if (globaltimer() - idle_since > p.timeout_ns) {
        const unsigned who = __ballot_sync(FULL, pend_ctr >= 0);
        const int src = who ? __ffs(who) - 1 : 0;
        const int c = __shfl_sync(FULL, pend_ctr, src), o = __shfl_sync(FULL, pend_obs, src),
                  t = __shfl_sync(FULL, pend_tgt, src);
        if (lane == 0) report(p, MK_ERR_TIMEOUT, instr_index(p, ready), c, o, t, R_SCHED, 1);
        break;
      }
    }
  }
}

// ------------------------------------------------------------------ TMA loader (one warp)

// The loader runs on a whole warp, converged: every lane polls the barriers, ring positions and
// coordinates are warp-uniform, and one elected lane issues each barrier operation and copy.
// The issuing thread's own latency bounds how fast stages are refilled, so the per-stage work is
// one or two copies and a few uniform integer operations.

// `panels` 64-column panels of B (64 rows each, 8 KB atoms in the 128-byte swizzled layout) from
// column `col`, row `k`, into consecutive atoms at `dst`. A panel map (3D: column within the
// panel, row, panel) moves them in one copy; a plain 2D map takes one copy per panel. PC: the
// copy counts on the even CTA's barrier of a CTA pair.
template <bool PC>
__device__ __forceinline__ void load_panels(uint32_t dst, const void* map, bool panel_map,
                                            uint32_t bar, int col, int k, int panels) {
  if (panel_map) {
    if (PC)
      tma_load_3d_pair(dst, map, bar, 0, k, col >> 6);
    else
      tma_load_3d(dst, map, bar, 0, k, col >> 6);
  } else {
    for (int j = 0; j < panels; ++j) {
      if (PC)
        tma_load_2d_pair(dst + j * 8192, map, bar, col + 64 * j, k);
      else
        tma_load_2d(dst + j * 8192, map, bar, col + 64 * j, k);
    }
  }
}

// Everything the k-loop of one GEMM tile's loads needs, as plain values.
struct LoadTile {
  uint32_t full0, tx0, empty0, deps, deps_par, ring0, sb, ns, own;
  int nk, npre, arow, bcol, k0, nbox;
  const void *ta, *tb, *tb2;
  bool leader, panel;
};

// The loads of one GEMM tile, from ring position (st, ph). Out of line so the hot loop compiles
// on its own. Weights first: the first npre stages get their B operand before the activations
// are known to be ready (they depend on nothing inside the graph), then A follows for those and
// both for the rest. Each stage is armed by the CTA whose barrier counts the bytes: the even CTA
// of a pair expects both CTAs' bytes; the odd CTA arrives on its own barrier only to keep its
// phase count in step.
template <bool PAIR, bool DUAL>
__device__ __noinline__ bool load_tile(const Params& p, const LoadTile& tp, uint32_t st,
                                       uint32_t ph, int idx) {
  const LoadTile t = tp;  // a private copy: its fields stay in registers
  auto arm = [&](uint32_t s_) {
    if (t.leader)
      mbar_expect_tx(t.full0 + s_ * 8u, PAIR ? 2 * t.own : t.own);
    else
      mbar_arrive(t.full0 + s_ * 8u);
  };
  auto issue_b = [&](uint32_t s_, int kb) {
    const uint32_t dst = t.ring0 + s_ * t.sb + kGemmTileM * kGemmBK * 2;
    const int k = t.k0 + kb * kGemmBK;
    load_panels<PAIR>(dst, t.tb, t.panel, t.tx0 + s_ * 8u, t.bcol, k, t.nbox);
    if (DUAL) load_panels<PAIR>(dst + t.nbox * 8192, t.tb2, t.panel, t.tx0 + s_ * 8u, t.bcol, k, t.nbox);
  };
  auto issue_a = [&](uint32_t s_, int kb) {
    if (PAIR)
      tma_load_2d_pair(t.ring0 + s_ * t.sb, t.ta, t.tx0 + s_ * 8u, t.k0 + kb * kGemmBK, t.arow);
    else
      tma_load_2d(t.ring0 + s_ * t.sb, t.ta, t.tx0 + s_ * 8u, t.k0 + kb * kGemmBK, t.arow);
  };
  const uint32_t st0 = st;
  for (int kb = 0; kb < t.npre; ++kb) {
    if (!wait_warp(p, t.empty0 + st * 8u, ph ^ 1u, R_LOAD, 11, idx)) return false;
    if (elect_one()) {
      arm(st);
      issue_b(st, kb);
    }
    __syncwarp();
    if (++st == t.ns) {
      st = 0;
      ph ^= 1u;
    }
  }
  if (!wait_warp(p, t.deps, t.deps_par, R_LOAD, 12, idx)) return false;
  if (elect_one()) {
    fence_proxy_async_global();
    uint32_t q = st0;
    for (int kb = 0; kb < t.npre; ++kb) {
      issue_a(q, kb);
      if (++q == t.ns) q = 0;
    }
  }
  __syncwarp();
  for (int kb = t.npre; kb < t.nk; ++kb) {
    if (!wait_warp(p, t.empty0 + st * 8u, ph ^ 1u, R_LOAD, 13, idx)) return false;
    if (elect_one()) {
      arm(st);
      issue_b(st, kb);
      issue_a(st, kb);
    }
    __syncwarp();
    if (++st == t.ns) {
      st = 0;
      ph ^= 1u;
    }
  }
  return true;
}

// Pair-mode ring sync before a pair instruction (a GEMM or attention tile both CTAs of a pair
// run together) that fills nst stages. `synced` holds while every instruction since the last
// resync was such a pair instruction (all roles of both CTAs see the same instruction kinds per
// iteration, so they agree); then both CTAs consumed the same stages from the same position and
// every stage's last use was a pair MMA that released it in both CTAs: the instruction streams
// straight on. Otherwise both CTAs move to the start of the next pass over the ring (each
// skipped stage waited free, both its barriers arrived on so their phase counts stay equal to
// the use count every role tracks), and, when the instruction fills stages, the handshake below.
template <bool PAIR>
__device__ bool pair_ring_sync(const Params& p, Smem& s, RingPos& rp, uint32_t& nfill,
                               uint32_t& go_par, bool& synced, int nst, int idx) {
  if (!PAIR || synced) return true;
  const uint32_t NS = ring_n(p);
  while (rp.st != 0) {
    if (!wait_warp(p, smem_u32(&s.empty[rp.st]), rp.ph ^ 1u, R_LOAD, 18, idx)) return false;
    if (elect_one()) {
      mbar_arrive(smem_u32(&s.full[rp.st]));
      mbar_arrive(smem_u32(&s.empty[rp.st]));
    }
    __syncwarp();
    rp.next(NS);
    ++nfill;
  }
  if (nst == 0) return true;
  // After other instructions the two CTAs' rings differ, so the odd CTA's bytes must not reach
  // the even CTA's full barriers while one of them still carries an earlier load. The even CTA
  // waits until every stage of the pass is free (every earlier use consumed), then releases the
  // odd CTA once. Later stages need no handshake: the odd CTA reuses a stage only after the
  // pair MMA that read it committed, which is after the even CTA's barrier for it completed.
  // Bytes that land before the even CTA's expect_tx leave the transaction count negative
  // until it arrives.
  if (cluster_ctarank() == 0) {
    for (int j = 0; j < (int)NS; ++j)
      if (!wait_warp(p, smem_u32(&s.empty[j]), rp.ph ^ 1u, R_LOAD, 17, idx)) return false;
    if (elect_one()) mbar_arrive_cluster(mapa_shared(smem_u32(&s.go), 1));
    __syncwarp();
  } else {
    if (!wait_warp(p, smem_u32(&s.go), go_par & 1u, R_LOAD, 19, idx, true)) return false;
    go_par ^= 1u;
  }
  synced = true;
  return true;
}

template <bool PAIR>
__device__ bool load_gemm(const Params& p, Smem& s, const Instr& in, const Node& nd, int slot,
                          uint32_t use, RingPos& rp, uint32_t& nfill, uint32_t& go_par,
                          bool& synced, int idx) {
  const uint32_t NS = ring_n(p);
  const int nk = ring_stages(in);
  if (!pair_ring_sync<PAIR>(p, s, rp, nfill, go_par, synced, nk, idx)) return false;
  if (nk == 0) return true;
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const bool dual = (nd.flags & EPI_SILU_MUL) != 0;
  const bool panel = (nd.flags & NF_B_PANELS) != 0;
  const int tn = nd.tile_n;
  const int ncol = PAIR ? tn / 2 : tn;  // B columns this CTA loads per weight
  LoadTile t;
  t.full0 = smem_u32(&s.full[0]);
  // bytes of both CTAs of a pair complete on the even CTA's full barrier
  t.tx0 = PAIR ? mapa_shared(t.full0, 0) : t.full0;
  t.empty0 = smem_u32(&s.empty[0]);
  t.deps = smem_u32(&s.deps_ready[slot]);
  t.deps_par = use & 1u;
  t.ring0 = smem_u32(s.ring);
  t.sb = stage_bytes(p);
  t.ns = NS;
  t.nk = nk;
  t.npre = (in.flags & IFLAG_B_DEP) ? 0 : (nk < (int)NS ? nk : (int)NS);
  t.ta = tmap_at(p, nd.a.tmap);
  t.tb = tmap_at(p, nd.b.tmap);
  t.tb2 = dual ? tmap_at(p, nd.b2.tmap) : nullptr;
  t.arow = in.m0 + (int)rank * kGemmTileM;
  t.bcol = in.n0 + (int)rank * ncol;
  t.k0 = in.k0;
  t.nbox = ncol / 64;
  t.own = (uint32_t)(kGemmTileM * kGemmBK * 2 + (dual ? 2 : 1) * ncol * kGemmBK * 2);
  t.leader = !PAIR || rank == 0;
  t.panel = panel;
  const bool ok = dual ? load_tile<PAIR, true>(p, t, rp.st, rp.ph, idx)
                       : load_tile<PAIR, false>(p, t, rp.st, rp.ph, idx);
  rp.advance((uint32_t)nk, NS);
  nfill += (uint32_t)nk;
  return ok;
}

// Staged row instruction (RMSNorm, RoPE): once the sources are complete, the instruction's input
// rows are copied into consecutive ring stages, as many whole rows per stage as fit, by bulk
// copies (one per row, one lane each; one per stage when the rows are contiguous). Deep queues
// of bytes in flight without holding registers: the compute warpgroup reads the rows from
// shared memory.
__device__ bool load_rows(const Params& p, Smem& s, const Instr& in, const Node& nd, int slot,
                          uint32_t use, RingPos& rp, uint32_t& nfill, int idx) {
  const uint32_t NS = ring_n(p);
  const int nst = ring_stages(in);
  if (nst == 0) return true;
  if (!wait_warp(p, smem_u32(&s.deps_ready[slot]), use & 1u, R_LOAD, 36, idx)) return false;
  if (elect_one()) fence_proxy_async_global();
  __syncwarp();
  const int lane = (int)(threadIdx.x & 31u);
  const int rows = min(nd.tile_m, nd.M - in.m0);
  const uint32_t rb = (uint32_t)row_stage_cols(nd) * 2u, sb = stage_bytes(p);
  const int rps = (int)(sb / rb);
  const size_t lda = (size_t)nd.a.ld * 2u;
  const uint8_t* a = reinterpret_cast<const uint8_t*>(nd.a.ptr) + (size_t)in.m0 * lda;
  const uint32_t ring0 = smem_u32(s.ring);
  for (int j = 0; j < nst; ++j) {
    if (!wait_warp(p, smem_u32(&s.empty[rp.st]), rp.ph ^ 1u, R_LOAD, 37, idx)) return false;
    const int r0 = j * rps, nr = min(rps, rows - r0);
    const uint32_t bar = smem_u32(&s.full[rp.st]), dst = ring0 + rp.st * sb;
    if (elect_one()) mbar_expect_tx(bar, (uint32_t)nr * rb);
    __syncwarp();
    if (lda == rb) {
      if (lane == 0) bulk_load(dst, a + (size_t)r0 * lda, (uint32_t)nr * rb, bar);
    } else {
      for (int r = lane; r < nr; r += 32) bulk_load(dst + r * rb, a + (size_t)(r0 + r) * lda, rb, bar);
    }
    __syncwarp();
    rp.next(NS);
    ++nfill;
  }
  return true;
}

__device__ bool load_gemv(const Params& p, Smem& s, const Instr& in, const Node& nd, int slot,
                          uint32_t use, RingPos& rp, uint32_t& nfill, int idx) {
  const uint32_t NS = ring_n(p);
  const int nk = ring_stages(in);
  if (nk == 0) return true;
  const bool dual = (nd.flags & EPI_SILU_MUL) != 0;
  const bool panel = (nd.flags & NF_B_PANELS) != 0;
  // a stage is four 64-row x 64-column panels, 128-byte swizzled (8 KB each): the tile's 256
  // columns, or 128 gate columns then 128 up columns
  const uint32_t bytes = 4u * 64u * kGemvRows * 2u;
  const void* tb = tmap_at(p, nd.b.tmap);
  const void* tb2 = dual ? tmap_at(p, nd.b2.tmap) : nullptr;
  const uint32_t ring0 = smem_u32(s.ring), sb = stage_bytes(p);
  // packed weights: each stage is one contiguous unit per weight, already in the swizzled layout
  const bool packed = (nd.flags & NF_B_PACKED) != 0;
  const uint32_t unit = dual ? 16384u : 32768u;
  const uint8_t* pb = nullptr;
  const uint8_t* pb2 = nullptr;
  if (packed) {
    const size_t first = (size_t)(in.n0 / (dual ? 128 : 256)) * (size_t)nd.b.ld + in.k0 / 64;
    pb = reinterpret_cast<const uint8_t*>(nd.b.ptr) + first * unit;
    if (dual) pb2 = reinterpret_cast<const uint8_t*>(nd.b2.ptr) + first * unit;
  }
  if (in.flags & IFLAG_B_DEP) {
    if (!wait_warp(p, smem_u32(&s.deps_ready[slot]), use & 1u, R_LOAD, 14, idx)) return false;
    if (elect_one()) fence_proxy_async_global();
    __syncwarp();
  }
  for (int kb = 0; kb < nk; ++kb) {
    if (!wait_warp(p, smem_u32(&s.empty[rp.st]), rp.ph ^ 1u, R_LOAD, 15, idx)) return false;
    if (elect_one()) {
      const uint32_t bar = smem_u32(&s.full[rp.st]);
      const uint32_t dst = ring0 + rp.st * sb;
      const int k = in.k0 + kb * kGemvRows;
      mbar_expect_tx(bar, bytes);
      if (packed) {
        bulk_load(dst, pb + (size_t)kb * unit, unit, bar);
        if (dual) bulk_load(dst + unit, pb2 + (size_t)kb * unit, unit, bar);
      } else if (dual) {
        load_panels<false>(dst, tb, panel, bar, in.n0, k, 2);
        load_panels<false>(dst + 2 * 8192, tb2, panel, bar, in.n0, k, 2);
      } else {
        load_panels<false>(dst, tb, panel, bar, in.n0, k, 4);
      }
    }
    __syncwarp();
    rp.next(NS);
    ++nfill;
  }
  return true;
}

// Split-KV partial: the chunk's keys and values (head g = n0, 64 columns each) land in one
// stage, 128-byte swizzled: keys at offset 0, values at 16 KB. A chunk that does not contain a
// row appended inside the graph streams before the query is ready.
__device__ bool load_attn(const Params& p, Smem& s, const Instr& in, const Node& nd, int slot,
                          uint32_t use, RingPos& rp, uint32_t& nfill, int idx) {
  const uint32_t NS = ring_n(p);
  if (in.flags & IFLAG_B_DEP) {
    if (!wait_warp(p, smem_u32(&s.deps_ready[slot]), use & 1u, R_LOAD, 16, idx)) return false;
    if (elect_one()) fence_proxy_async_global();
    __syncwarp();
  }
  if (!wait_warp(p, smem_u32(&s.empty[rp.st]), rp.ph ^ 1u, R_LOAD, 17, idx)) return false;
  if (elect_one()) {
    const uint32_t bar = smem_u32(&s.full[rp.st]);
    const uint32_t dst = smem_u32(s.ring) + rp.st * stage_bytes(p);
    mbar_expect_tx(bar, (uint32_t)(2 * nd.tile_m * 128));
    tma_load_2d(dst, tmap_at(p, nd.b.tmap), bar, in.n0 * 64, in.k0);
    tma_load_2d(dst + 16384, tmap_at(p, nd.b2.tmap), bar, in.n0 * 64, in.k0);
  }
  __syncwarp();
  rp.next(NS);
  ++nfill;
  return true;
}

// Causal prefill attention, one (128-row query tile, query head) instruction: per 64-key block a
// stage holds the query tile (16 KB), the block's keys (8 KB) and values (8 KB) of the head's
// key/value head, all 128-byte swizzled; the block's P tile goes to TMEM. The query tile is
// fetched again with every block (from L2) so each stage is self-contained. All three operands
// are produced inside the graph, so the loads start once the sources are ready. On a CTA pair (a
// 256-row query tile, rank r holding rows 128r..) the query rows stay in the staging buffer for
// the whole instruction (loaded by the compute warpgroup) and a stage holds keys 32r..32r+31 of
// the block (the N half of S = Q K^T this CTA holds) and value columns 32r..32r+31 (the N half
// of O = P V, 64-byte rows, 64-byte swizzled): 8 KB per CTA, counted on the even CTA's barrier;
// the block's P tile follows at offset 8 KB.
template <bool PAIR>
__device__ bool load_attn_prefill(const Params& p, Smem& s, const Instr& in, const Node& nd,
                                  int slot, uint32_t use, RingPos& rp, uint32_t& nfill,
                                  uint32_t& go_par, bool& synced, int idx) {
  const uint32_t NS = ring_n(p);
  const int nb = ring_stages(in);
  if (!pair_ring_sync<PAIR>(p, s, rp, nfill, go_par, synced, nb, idx)) return false;
  if (nb == 0) return true;
  if (!wait_warp(p, smem_u32(&s.deps_ready[slot]), use & 1u, R_LOAD, 28, idx)) return false;
  if (elect_one()) fence_proxy_async_global();
  __syncwarp();
  const int h = in.n0, g = in.n0 / (nd.hq / nd.hkv);
  const void* tq = PAIR ? nullptr : tmap_at(p, nd.a.tmap);
  const void* tk = tmap_at(p, nd.b.tmap);
  const void* tv = tmap_at(p, nd.b2.tmap);
  const uint32_t ring0 = smem_u32(s.ring), sb = stage_bytes(p);
  const int rank = PAIR ? (int)cluster_ctarank() : 0;
  for (int j = 0; j < nb; ++j) {
    if (!wait_warp(p, smem_u32(&s.empty[rp.st]), rp.ph ^ 1u, R_LOAD, 29, idx)) return false;
    if (elect_one()) {
      const uint32_t bar = smem_u32(&s.full[rp.st]);
      const uint32_t dst = ring0 + rp.st * sb;
      if (PAIR) {
        const uint32_t tx = mapa_shared(bar, 0);  // both CTAs' bytes on the even CTA's barrier
        if (rank == 0)
          mbar_expect_tx(bar, 2u * 8192u);
        else
          mbar_arrive(bar);
        tma_load_2d_pair(dst, tk, tx, g * 64, j * kAttnKeyBlock + rank * 32);
        tma_load_2d_pair(dst + 4096, tv, tx, g * 64 + rank * 32, j * kAttnKeyBlock);
      } else {
        mbar_expect_tx(bar, 32768u);
        tma_load_2d(dst, tq, bar, h * 64, in.m0);
        tma_load_2d(dst + 16384, tk, bar, g * 64, j * kAttnKeyBlock);
        tma_load_2d(dst + 24576, tv, bar, g * 64, j * kAttnKeyBlock);
      }
    }
    __syncwarp();
    rp.next(NS);
    ++nfill;
  }
  return true;
}

template <bool PAIR, int KS>
__device__ void run_loader(const Params& p, Smem& s) {
  const uint32_t NS = ring_n(p);
  for (int i = 0; i < p.n_tmaps; ++i) tensormap_acquire(tmap_at(p, i));
  RingPos rp;
  uint32_t nfill = 0, go_par = 0;
  bool synced = true;  // pair-mode ring sync (see load_gemm)
  for (int it = 0;; ++it) {
    const int slot = it % kSlots;
    const uint32_t use = (uint32_t)(it / kSlots);
    const int idx = instr_index(p, it);
    if (!wait_warp(p, smem_u32(&s.instr_ready[slot]), use & 1u, R_LOAD, 10, idx)) break;
    const Instr& in = slot_instr(s, slot);
    if (in.op == OP_END) break;
    const Node& nd = slot_node(s, slot);
    bool ok = true;
    if (in.op != OP_GEMM && in.op != OP_ATTN_PREFILL) synced = false;
    if (ks_has_gemm(KS) && in.op == OP_GEMM)
      ok = load_gemm<PAIR>(p, s, in, nd, slot, use, rp, nfill, go_par, synced, idx);
    else if (ks_has_gemv(KS) && in.op == OP_GEMV)
      ok = load_gemv(p, s, in, nd, slot, use, rp, nfill, idx);
    else if (ks_has_gemv(KS) && in.op == OP_ATTN_PARTIAL)
      ok = load_attn(p, s, in, nd, slot, use, rp, nfill, idx);
    else if (ks_has_attn_prefill(KS) && in.op == OP_ATTN_PREFILL)
      ok = load_attn_prefill<PAIR>(p, s, in, nd, slot, use, rp, nfill, go_par, synced, idx);
    else if (ks_stages_rows(KS) && (in.op == OP_RMSNORM || in.op == OP_ROPE))
      ok = load_rows(p, s, in, nd, slot, use, rp, nfill, idx);
    if (!ok) break;
    if (elect_one()) mbar_arrive(smem_u32(&s.slot_free[slot]));
    __syncwarp();
  }
  // Every load issued has landed before the CTA may exit (normally already true): the last fill
  // of stage st was in the current pass when st < rp.st, else in the previous one.
  for (uint32_t st = 0; st < NS; ++st) {
    if (nfill <= st) continue;
    wait_mbar_drain(smem_u32(&s.full[st]), st < rp.st ? rp.ph : rp.ph ^ 1u);
  }
  __syncwarp();
}

// ------------------------------------------------------------------ MMA issuer (one warp)

// The MMAs of one GEMM tile: nk k-steps from ring position (st, ph), accumulating into TMEM
// column d. Out of line and with scalar arguments so the hot loop compiles on its own: few live
// values, operands that stay warp-uniform. Software-pipelined: an MMA issue waits while the
// tensor pipe is busy and the pipe queues little ahead, so the next stage's barrier is polled
// after all but the last K slice of the current stage is issued; the pipe keeps executing
// meanwhile. Returns the number of k-steps whose MMAs were issued (nk unless a wait gave up).
template <bool PAIR, bool DUAL>
__device__ __noinline__ int mma_tile(const Params& p, uint32_t full0, uint32_t empty0,
                                     uint32_t st, uint32_t ph, uint32_t ns, int nk,
                                     uint64_t adesc0, uint64_t bdesc0, uint32_t units, uint32_t d,
                                     uint32_t idesc, int tn, uint64_t up, int idx) {
  auto slice = [&](uint64_t so, int j, uint32_t acc) {
    const uint64_t ad = adesc0 + so + (uint64_t)(j * 2);
    const uint64_t bd = bdesc0 + so + (uint64_t)(j * 128);
    if (PAIR)
      tc_mma_f16_pair(d, ad, bd, idesc, acc);
    else
      tc_mma_f16(d, ad, bd, idesc, acc);
    if (DUAL) {
      if (PAIR)
        tc_mma_f16_pair(d + (uint32_t)tn, ad, bd + up, idesc, acc);
      else
        tc_mma_f16(d + (uint32_t)tn, ad, bd + up, idesc, acc);
    }
  };
  if (!wait_warp(p, full0 + st * 8u, ph, R_MMA, 22, idx)) return 0;
  tc_fence_after();
  for (int kb = 0; kb < nk; ++kb) {
    const uint64_t so = (uint64_t)(st * units);
    uint32_t nst = st + 1, nph = ph;
    if (nst == ns) {
      nst = 0;
      nph ^= 1u;
    }
    if (elect_one()) {
#pragma unroll
      for (int j = 0; j < kGemmBK / 16 - 1; ++j) slice(so, j, (kb | j) != 0);
    }
    __syncwarp();
    if (kb + 1 < nk) {
      if (!wait_warp(p, full0 + nst * 8u, nph, R_MMA, 22, idx)) return kb + 1;
      tc_fence_after();
    }
    if (elect_one()) {
      slice(so, kGemmBK / 16 - 1, 1u);
      // the stage is free (in both CTAs of a pair) once these MMAs complete
      if (PAIR)
        tc_commit_pair(empty0 + st * 8u, 3);
      else
        tc_commit(empty0 + st * 8u);
    }
    __syncwarp();
    st = nst;
    ph = nph;
  }
  return nk;
}

// GEMV tiles run on the tensor cores with the operands swapped: D [256 weight columns x 16] =
// W^T x^T as two M = 128 halves, N = 16 >= M activation rows, K = 16 per MMA. The weight stage
// is the A operand exactly as TMA wrote it (MN-major); the compute warpgroup stages the K chunk's
// activations as the K-major B operand in the staging buffer, one 1 KB block (8 rows x 64 K) per
// weight stage. The chunk must fit that buffer with one spare block (rows 8-15 of the last block's
// MMAs read past it), and CTA-pair kernels keep the CUDA-core path (a kernel uses one cta_group).
constexpr int kGemvTensorBlocks = kXrFloats * 4 / 1024 - 1;
template <bool PAIR>
__device__ __forceinline__ bool gemv_on_tensor(const Instr& in, const Node& nd) {
  const int nk = ring_stages(in);
  return !PAIR && nk > 0 && nk <= kGemvTensorBlocks && nd.M <= 8;
}

// The MMAs of one tensor-core GEMV tile: per weight stage, 4 K slices x 2 column halves. A: the
// stage (64-column atoms 8 KB apart, 8-row K groups 1 KB apart; a 16-row K slice is 128 units,
// the second half of the columns 1024 units on). B: block kb of the staged activations (2 units
// per K slice). Rows 8-15 of B are the next block's rows 0-7: they only fill accumulator columns
// 8-15, which nobody reads (M <= 8). A stage is released when its MMAs complete. Returns the
// number of stages whose MMAs were issued (nk unless a wait gave up).
__device__ __noinline__ int mma_gemv(const Params& p, uint32_t full0, uint32_t empty0,
                                     uint32_t st, uint32_t ph, uint32_t ns, int nk,
                                     uint64_t adesc0, uint64_t bdesc0, uint32_t units, uint32_t d,
                                     uint32_t idesc, int idx) {
  for (int kb = 0; kb < nk; ++kb) {
    if (!wait_warp(p, full0 + st * 8u, ph, R_MMA, 23, idx)) return kb;
    tc_fence_after();
    if (elect_one()) {
      const uint64_t so = (uint64_t)(st * units);
#pragma unroll
      for (int j = 0; j < kGemvRows / 16; ++j) {
        const uint64_t ad = adesc0 + so + (uint64_t)(j * 128);
        const uint64_t bd = bdesc0 + (uint64_t)(kb * 64 + j * 2);
        const uint32_t acc = (kb | j) != 0;
        tc_mma_f16(d, ad, bd, idesc, acc);
        tc_mma_f16(d + 16u, ad + 1024u, bd, idesc, acc);
      }
      tc_commit(empty0 + st * 8u);
    }
    __syncwarp();
    if (++st == ns) {
      st = 0;
      ph ^= 1u;
    }
  }
  return nk;
}

// Prefill attention MMAs of one instruction: nb key blocks from ring position (st, ph). Block j:
// S_j = Q K_j^T into TMEM S[n&1] (M = 128 query rows, N = 64 keys, K = 64 dims; the keys are a
// K-major B operand), then, once the compute warps have written P_j (bf16: into TMEM on a single
// CTA, 128-byte swizzled K-major in the stage on a pair), O += P_j V_j into the one TMEM output
// (N = 64 dims, K = 64 keys; the values are an N-major B operand; block 0 overwrites it).
// S_{j+1} is issued before P_j is awaited, so the tensor pipe computes the next scores while the
// softmax of the current block runs. A stage is released when the block's P V completes. `n`
// counts attention blocks on this SM: it gives every barrier's phase. TMEM columns: S at 0 and
// 64, O at 128, P at 192 and 224 (single CTA).
template <bool PAIR>
__device__ __noinline__ bool mma_attn(const Params& p, Smem& s, uint32_t st, uint32_t ph,
                                      uint32_t ns, int nb, uint32_t tmem, uint32_t& n,
                                      uint32_t q_par, int idx) {
  const uint32_t ring0 = smem_u32(s.ring), units = stage_bytes(p) >> 4;
  const uint32_t xr = smem_u32(s.xr);
  // Single CTA: a stage holds Q (128 rows of 128 B), K (64 rows of 128 B) and V (N-major, 64
  // rows of 128 B); P_j is the A operand of P V straight from TMEM (two buffers of 32 columns,
  // a row per lane, two keys per column). Pair: Q in xr; a stage holds this CTA's 32 keys
  // (rows of 128 B), its 32 value columns (N-major, 64 rows of 64 B) and the block's P (128
  // rows of 128 B).
  const uint64_t qd = sdesc_sw128(PAIR ? xr : ring0, 16, 1024);
  const uint64_t kd = sdesc_sw128(ring0 + (PAIR ? 0 : 16384), 16, 1024);
  const uint64_t vd = PAIR ? sdesc_sw64(ring0 + 4096, 4096, 512)
                           : sdesc_sw128(ring0 + 24576, 8192, 1024);
  const uint64_t vk = PAIR ? 64 : 128;  // a 16-key slice of V, 16-byte units
  const uint64_t pd = sdesc_sw128(ring0 + 8192, 16, 1024);  // pair: P in the stage
  const uint64_t qs = PAIR ? 0 : 1;     // Q moves with the stage (single CTA) or stays in xr
  const int mrows = PAIR ? 2 * kAttnTileQ : kAttnTileQ;
  const uint32_t is = idesc_f16_bk(1, kAttnKeyBlock, mrows), io = idesc_f16(1, 64, mrows);
  const uint32_t n0 = n;
  RingPos rs, ro;
  rs.st = ro.st = st;
  rs.ph = ro.ph = ph;
  // pair: both CTAs' query tiles are loaded (the compute warpgroups load them)
  if (PAIR && !wait_warp(p, smem_u32(&s.att_q_full), q_par, R_MMA, 26, idx, true)) return false;
  auto issue_s = [&](int j) -> bool {
    const uint32_t nn = n0 + (uint32_t)j, b = nn & 1u;
    if (!wait_warp(p, smem_u32(&s.full[rs.st]), rs.ph, R_MMA, 23, idx)) return false;
    // S_j reuses the buffer of S_{j-2}. Single CTA: its reads are signalled on their own. Pair:
    // every arrival on the even CTA is a cluster-scope release that holds the arriving warp, so
    // a block arrives once (P_j); S_j is issued after P V_{j-2}, which waited for P_{j-2}, which
    // the warps wrote after reading S_{j-2}.
    if (!PAIR &&
        !wait_warp(p, smem_u32(&s.att_s_free[b]), ((nn >> 1) & 1u) ^ 1u, R_MMA, 24, idx))
      return false;
    tc_fence_after();
    const uint64_t so = (uint64_t)(rs.st * units);
    if (elect_one()) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        if (PAIR)
          tc_mma_f16_pair(tmem + b * 64u, qd + so * qs + (uint64_t)(kk * 2),
                          kd + so + (uint64_t)(kk * 2), is, kk != 0);
        else
          tc_mma_f16(tmem + b * 64u, qd + so * qs + (uint64_t)(kk * 2),
                     kd + so + (uint64_t)(kk * 2), is, kk != 0);
      }
      if (PAIR)
        tc_commit_pair(smem_u32(&s.att_s_full[b]), 3);
      else
        tc_commit(smem_u32(&s.att_s_full[b]));
    }
    __syncwarp();
    rs.next(ns);
    return true;
  };
  if (!issue_s(0)) return false;
  for (int j = 0; j < nb; ++j) {
    if (j + 1 < nb && !issue_s(j + 1)) return false;
    const uint32_t nn = n0 + (uint32_t)j, b = nn & 1u;
    // P_j is written (and any rescale of O by the compute warps is stored) before p_full. Two
    // barriers by block parity: the compute warps can arrive for block j + 1 before this warp
    // has seen block j's arrival (S_{j+1} is issued first), which would move one barrier two
    // phases past the one awaited.
    if (!wait_warp(p, smem_u32(&s.att_p_full[b]), (nn >> 1) & 1u, R_MMA, 25, idx, PAIR))
      return false;
    tc_fence_after();
    const uint64_t so = (uint64_t)(ro.st * units);
    if (elect_one()) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        if (PAIR)
          tc_mma_f16_pair(tmem + 128u, pd + so + (uint64_t)(kk * 2),
                          vd + so + (uint64_t)kk * vk, io, (j | kk) != 0);
        else  // P_j from TMEM: 16 keys are 8 columns
          tc_mma_f16_ts(tmem + 128u, tmem + kAttnPCol + b * 32u + (uint32_t)(kk * 8),
                        vd + so + (uint64_t)kk * vk, io, (j | kk) != 0);
      }
      if (PAIR) {
        tc_commit_pair(smem_u32(&s.att_o_full[b]), 3);
        tc_commit_pair(smem_u32(&s.empty[ro.st]), 3);
      } else {
        tc_commit(smem_u32(&s.att_o_full[b]));
        tc_commit(smem_u32(&s.empty[ro.st]));
      }
    }
    __syncwarp();
    ro.next(ns);
  }
  // The compute warps have read every S and O block of this instruction before TMEM is reused.
  if (!wait_warp(p, smem_u32(&s.att_done), q_par, R_MMA, 27, idx, PAIR)) return false;
  n = n0 + (uint32_t)nb;
  return true;
}

template <bool PAIR, int KS>
__device__ void run_mma(const Params& p, Smem& s, uint32_t tmem) {
  // The whole warp runs this loop, converged: ring position, descriptors and flags are
  // warp-uniform and one elected lane issues each tcgen05 operation. Per k-step the issuer does
  // a barrier poll, a fence and the MMAs of the stage; descriptors are the stage-0 descriptors
  // plus the stage's offset in 16-byte units.
  const uint32_t NS = ring_n(p);
  const uint32_t units = stage_bytes(p) >> 4;
  const uint32_t ring0 = smem_u32(s.ring);
  // A: K-major, 128-byte rows, 8-row groups 1024 B apart; a 16-wide K slice is 32 B (2 units).
  const uint64_t adesc0 = sdesc_sw128(ring0, 16, 1024);
  // B: N-major, 64-column atoms 8 KB apart (LBO), 8-row K groups 1024 B apart (SBO); a 16-deep
  // K slice is 16 rows of 128 B (128 units).
  const uint64_t bdesc0 = sdesc_sw128(ring0 + kGemmTileM * kGemmBK * 2, 8192, 1024);
  RingPos rp;
  uint32_t acc_n = 0, att_n = 0, att_i = 0, gx_n = 0;  // att_i: pair attention instructions
  bool issued = false, synced = true;
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  for (int it = 0;; ++it) {
    const int slot = it % kSlots;
    const uint32_t u = (uint32_t)(it / kSlots);
    const int idx = instr_index(p, it);
    if (!wait_warp(p, smem_u32(&s.instr_ready[slot]), u & 1u, R_MMA, 20, idx)) break;
    const Instr& in = slot_instr(s, slot);
    if (in.op == OP_END) break;
    const Node& nd = slot_node(s, slot);
    bool ok = true;
    if (ks_has_gemm(KS) && in.op == OP_GEMM) {
      const int nk = ring_stages(in);
      if (PAIR && !synced) rp.align();  // mirrors the loader's ring sync
      if (nk > 0) synced = true;
      if (nk > 0 && PAIR && rank != 0) {
        rp.advance((uint32_t)nk, NS);  // the even CTA issues the pair's MMAs
        ++acc_n;
      } else if (nk > 0) {
        const uint32_t as = acc_n & 1u;
        // the slot is free once every epilogue that read it (both CTAs' in pair mode) is done
        if (!wait_warp(p, smem_u32(&s.acc_empty[as]), ((acc_n >> 1) & 1u) ^ 1u, R_MMA, 21, idx,
                       PAIR))
          break;
        tc_fence_after();
        const bool dual = (nd.flags & EPI_SILU_MUL) != 0;
        const int tn = nd.tile_n;
        const int ncol = PAIR ? tn / 2 : tn;  // B columns held by each CTA per weight
        const uint32_t idesc = idesc_f16(nd.dtype == DT_BF16, tn, PAIR ? 256 : 128);
        const uint32_t d = tmem + as * 256u;
        const uint64_t up = (uint64_t)((ncol / 64) * (8192 >> 4));  // up-weight atoms
        const uint32_t full0 = smem_u32(&s.full[0]), empty0 = smem_u32(&s.empty[0]);
        const int done = dual ? mma_tile<PAIR, true>(p, full0, empty0, rp.st, rp.ph, NS, nk,
                                                     adesc0, bdesc0, units, d, idesc, tn, up, idx)
                              : mma_tile<PAIR, false>(p, full0, empty0, rp.st, rp.ph, NS, nk,
                                                      adesc0, bdesc0, units, d, idesc, tn, up, idx);
        if (done > 0) issued = true;
        ok = done == nk;
        rp.advance((uint32_t)nk, NS);
        if (!ok) break;  // MMAs in flight are drained below
        if (elect_one()) {
          if (PAIR)
            tc_commit_pair(smem_u32(&s.acc_full[as]), 3);
          else
            tc_commit(smem_u32(&s.acc_full[as]));
        }
        __syncwarp();
        ++acc_n;
      }
    } else if (ks_has_attn_prefill(KS) && in.op == OP_ATTN_PREFILL) {
      const int nb = ring_stages(in);
      if (PAIR && !synced) rp.align();  // mirrors the loader's ring sync
      if (nb > 0) synced = true;
      if (nb > 0 && PAIR && rank != 0) {
        rp.advance((uint32_t)nb, NS);  // the even CTA issues the pair's MMAs
      } else if (nb > 0) {
        // TMEM columns 0..255 are reused: every GEMM epilogue still reading them is done first
        bool w = true;
        for (uint32_t k = 0; k < 2 && w; ++k)
          w = wait_warp(p, smem_u32(&s.acc_empty[(acc_n + k) & 1u]),
                        (((acc_n + k) >> 1) & 1u) ^ 1u, R_MMA, 21, idx, PAIR);
        if (!w) break;
        tc_fence_after();
        if (!mma_attn<PAIR>(p, s, rp.st, rp.ph, NS, nb, tmem, att_n, att_i & 1u, idx)) {
          issued = true;
          break;
        }
        issued = true;
        ++att_i;
        rp.advance((uint32_t)nb, NS);
      }
    } else if (ks_has_gemv(KS) && in.op == OP_GEMV && gemv_on_tensor<PAIR>(in, nd)) {
      synced = false;
      const int nk = ring_stages(in);
      const uint32_t as = acc_n & 1u;
      // the accumulator slot is free, and the activations are staged
      if (!wait_warp(p, smem_u32(&s.acc_empty[as]), ((acc_n >> 1) & 1u) ^ 1u, R_MMA, 21, idx))
        break;
      if (!wait_warp(p, smem_u32(&s.gx_full), gx_n & 1u, R_MMA, 24, idx)) break;
      ++gx_n;
      tc_fence_after();
      const uint32_t ring0 = smem_u32(s.ring);
      const int done = mma_gemv(p, smem_u32(&s.full[0]), smem_u32(&s.empty[0]), rp.st, rp.ph, NS,
                                nk, sdesc_sw128(ring0, 8192, 1024),
                                sdesc_sw128(smem_u32(s.xr), 16, 1024), units, tmem + as * 256u,
                                idesc_f16_amn(nd.dtype == DT_BF16, 16, 128), idx);
      if (done > 0) issued = true;
      rp.advance((uint32_t)nk, NS);
      if (done != nk) break;
      if (elect_one()) tc_commit(smem_u32(&s.acc_full[as]));
      __syncwarp();
      ++acc_n;
    } else {
      synced = false;
      rp.advance((uint32_t)ring_stages(in), NS);  // stages consumed by the compute warpgroup
    }
    if (elect_one()) mbar_arrive(smem_u32(&s.slot_free[slot]));
    __syncwarp();
  }
  if (ks_has_tmem(KS) && issued) {
    if (elect_one()) {
      if (PAIR)
        tc_commit_pair(smem_u32(&s.drain), 1);
      else
        tc_commit(smem_u32(&s.drain));
    }
    __syncwarp();
    wait_mbar_drain(smem_u32(&s.drain), 0);
  }
  __syncwarp();
}

// ------------------------------------------------------------------ compute warpgroup bodies

// The column chunks of one warp's 32 rows of a GEMM tile, after the accumulator is complete:
// per 32-column chunk, TMEM -> registers (lane = row) -> bias, ReLU, residual or SiLU·mul ->
// 16-bit values in a 32 x 32 block of shared memory (64-byte rows, 64-byte swizzle: 16-byte
// chunk j of row r at j ^ ((r >> 1) & 3), conflict-free) -> one TMA store by lane 0. Two 2 KB
// buffers at xr alternate; a buffer is rewritten once the store issued from it has read it.
// The next chunk's bias / residual loads are in flight while the current chunk is processed.
// Out of line with scalar arguments, like the mainloops: compiled inside the kernel function
// the same loop took about a microsecond per chunk. nk == 0 (K = 0) stores the epilogue of 0.
template <bool DUAL, bool SIDE, bool AHEAD = true>
__device__ __noinline__ void epi_chunks(uint32_t tb, int tn, int nk, uint32_t flags, int dt,
                                        const uint16_t* bias, int ldb, const uint16_t* res,
                                        int ldr, const void* omap, uint32_t xr, int row0, int n0,
                                        int M, int N) {
  const int lane = threadIdx.x & 31;
  const int row = row0 + lane;
  const bool has_bias = SIDE && (flags & EPI_BIAS) != 0, relu = (flags & EPI_RELU) != 0,
             has_res = SIDE && (flags & EPI_RESIDUAL) != 0;
  // bias / residual vectors of a chunk (4 groups of 8 columns), loaded one chunk ahead (AHEAD)
  // or at the start of the chunk, before its TMEM loads
  uint4 sb[SIDE ? 4 : 1], sr[SIDE ? 4 : 1], nb[SIDE && AHEAD ? 4 : 1], nr[SIDE && AHEAD ? 4 : 1];
  auto load_side = [&](int c, uint4* b, uint4* rr) {
#pragma unroll
    for (int g = 0; g < (SIDE ? 4 : 0); ++g) {
      const int col = n0 + c + g * 8;
      const bool inside = row < M && col < N;
      b[g] = rr[g] = make_uint4(0u, 0u, 0u, 0u);
      if (has_bias && inside)
        b[g] = __ldcg(reinterpret_cast<const uint4*>(bias + (size_t)row * ldb + col));
      if (has_res && inside)
        rr[g] = __ldcg(reinterpret_cast<const uint4*>(res + (size_t)row * ldr + col));
    }
  };
  if (SIDE && AHEAD) load_side(0, sb, sr);
  // without the register copies of the next chunk, this row's side vectors of the chunk after
  // next are fetched into L1 (a hint: no registers held)
  auto prefetch_side = [&](int c) {
    if (!SIDE || AHEAD || c >= tn || row >= M || n0 + c >= N) return;
    if (has_bias) asm volatile("prefetch.global.L1 [%0];" ::"l"(bias + (size_t)row * ldb + n0 + c));
    if (has_res) asm volatile("prefetch.global.L1 [%0];" ::"l"(res + (size_t)row * ldr + n0 + c));
  };
  prefetch_side(0);
  prefetch_side(32);
  for (int c = 0; c < tn; c += 32) {
    if (SIDE && AHEAD && c + 32 < tn) load_side(c + 32, nb, nr);
    prefetch_side(c + 64);
    if (SIDE && !AHEAD) load_side(c, sb, sr);
    uint32_t r[32], r2[DUAL ? 32 : 1];
    if (nk > 0) {
      tmem_ld32(tb + (uint32_t)c, r);
      if (DUAL) tmem_ld32(tb + (uint32_t)(tn + c), r2);
      tmem_ld_wait();
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) r[i] = 0u;
#pragma unroll
      for (int i = 0; i < (DUAL ? 32 : 1); ++i) r2[i] = 0u;
    }
    if (DUAL) {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        r[i] = __float_as_uint(silu(__uint_as_float(r[i])) * __uint_as_float(r2[i]));
    }
    const uint32_t buf = xr + (uint32_t)((c >> 5) & 1) * 2048u;
    if (c >= 64) {
      if (lane == 0) bulk_wait_read_1();
      __syncwarp();
    }
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const bool inside = row < M && n0 + c + g * 8 < N;
      float w[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) w[e] = __uint_as_float(r[g * 8 + e]);
      if (has_bias && inside) {
        float b[8];
        unpack8(sb[g], dt, b);
#pragma unroll
        for (int e = 0; e < 8; ++e) w[e] += b[e];
      }
      if (relu) {
#pragma unroll
        for (int e = 0; e < 8; ++e) w[e] = fmaxf(w[e], 0.0f);
      }
      if (has_res && inside) {
        float b[8];
        unpack8(sr[g], dt, b);
#pragma unroll
        for (int e = 0; e < 8; ++e) w[e] += b[e];
      }
      const uint4 pk = pack8(w, dt);
      const uint32_t dst = buf + (uint32_t)lane * 64u + (uint32_t)((g ^ ((lane >> 1) & 3)) << 4);
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(pk.x), "r"(pk.y),
                   "r"(pk.z), "r"(pk.w)
                   : "memory");
    }
    fence_proxy_async_shared();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(omap, buf, n0 + c, row0);
      bulk_commit();
    }
    if (SIDE && AHEAD) {
#pragma unroll
      for (int g = 0; g < (SIDE && AHEAD ? 4 : 0); ++g) {
        sb[g] = nb[g];
        sr[g] = nr[g];
      }
    }
  }
}

// One call site for the four epilogue loops (SiLU·mul or not, bias / residual or not); the
// node's fields are read here, so few values are live across the call.
__device__ __noinline__ void epi_tile(const Node& nd, int n0, int tn, uint32_t tb, int nk,
                                      const void* omap, uint32_t xr, int row0) {
  const uint32_t flags = nd.flags;
  const int dt = nd.dtype, M = nd.M, N = nd.N;
  const uint16_t* bias = reinterpret_cast<const uint16_t*>(nd.bias.ptr);
  const uint16_t* res = reinterpret_cast<const uint16_t*>(nd.res.ptr);
  const int ldb = nd.bias.ld, ldr = nd.res.ld;
  const bool dual = (flags & EPI_SILU_MUL) != 0;
  const bool side = (flags & (EPI_BIAS | EPI_RESIDUAL)) != 0;
  if (dual && side)
    epi_chunks<true, true>(tb, tn, nk, flags, dt, bias, ldb, res, ldr, omap, xr, row0, n0, M, N);
  else if (dual)
    epi_chunks<true, false>(tb, tn, nk, flags, dt, bias, ldb, res, ldr, omap, xr, row0, n0, M, N);
  else if (side)
    epi_chunks<false, true>(tb, tn, nk, flags, dt, bias, ldb, res, ldr, omap, xr, row0, n0, M, N);
  else
    epi_chunks<false, false>(tb, tn, nk, flags, dt, bias, ldb, res, ldr, omap, xr, row0, n0, M,
                             N);
}

// Split-tail partials. A (split, rank) slot holds a CTA's 128 rows x W fp32 columns warp by
// warp and, inside a warp's 32 rows, column group by column group: the float4 of columns
// 4j..4j+3 of lane l (row 32q + l) is element (q * W / 4 + j) * 32 + l, so every warp-wide load
// or store is 512 contiguous bytes. `dst` points at this warp's block and lane; columns
// [c0, c1) are stored.
__device__ __noinline__ void split_store(uint32_t tb, int c0, int c1, int nk, float4* dst) {
  for (int c = c0; c < c1; c += 32) {
    uint32_t r[32];
    if (nk > 0) {
      tmem_ld32(tb + (uint32_t)c, r);
      tmem_ld_wait();
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) r[i] = 0u;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i)
      __stcg(dst + (size_t)(c / 4 + i) * 32,
             make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                         __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3])));
  }
}

// The epilogue of a split-tail tile's last split. Each 32-column chunk is the sum of the splits'
// partials in split order, starting from zero (this split's own from TMEM, so neither the order
// nor the result depends on which split finishes last), followed by the fused epilogue and the
// TMA store of epi_chunks. With two splits (no SiLU·mul) the partner's partial of the next chunk
// is in flight while a chunk is finished; otherwise each chunk's loads of one partial go out
// together.
// `parts` is this warp's block and lane in split 0's slot; pstride the float4 between splits.
// Columns [c0, c1) of the tile are finished (of each weight's tn with SiLU·mul).
template <bool DUAL, bool SIDE>
__device__ __noinline__ void epi_split(uint32_t tb, int tn, int c0, int c1, int nk,
                                       uint32_t flags, int dt,
                                       const uint16_t* bias, int ldb, const uint16_t* res,
                                       int ldr, const void* omap, uint32_t xr, int row0, int n0,
                                       int M, int N, const float4* parts, int S, int mine,
                                       size_t pstride) {
  constexpr int V = DUAL ? 16 : 8;  // float4 of one chunk of one partial
  const int lane = threadIdx.x & 31;
  const int row = row0 + lane;
  const bool has_bias = SIDE && (flags & EPI_BIAS) != 0, relu = (flags & EPI_RELU) != 0,
             has_res = SIDE && (flags & EPI_RESIDUAL) != 0;
  auto issue = [&](int c, const float4* src, float4* v) {
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __ldcg(src + (size_t)(c / 4 + i) * 32);
    if (DUAL) {
#pragma unroll
      for (int i = 0; i < 8; ++i) v[8 + i] = __ldcg(src + (size_t)((tn + c) / 4 + i) * 32);
    }
  };
  auto add_part = [&](float* w, float* u, const float4* v) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      w[4 * i] += v[i].x;
      w[4 * i + 1] += v[i].y;
      w[4 * i + 2] += v[i].z;
      w[4 * i + 3] += v[i].w;
      if (DUAL) {
        u[4 * i] += v[8 + i].x;
        u[4 * i + 1] += v[8 + i].y;
        u[4 * i + 2] += v[8 + i].z;
        u[4 * i + 3] += v[8 + i].w;
      }
    }
  };
  auto add_own = [&](int c, float* w, float* u) {
    uint32_t r[32], r2[DUAL ? 32 : 1];
    if (nk > 0) {
      tmem_ld32(tb + (uint32_t)c, r);
      if (DUAL) tmem_ld32(tb + (uint32_t)(tn + c), r2);
      tmem_ld_wait();
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) r[i] = 0u;
#pragma unroll
      for (int i = 0; i < (DUAL ? 32 : 1); ++i) r2[i] = 0u;
    }
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      w[i] += __uint_as_float(r[i]);
      if (DUAL) u[i] += __uint_as_float(r2[i]);
    }
  };
  auto finish = [&](int c, float* w, const float* u) {
    if (DUAL) {
#pragma unroll
      for (int i = 0; i < 32; ++i) w[i] = silu(w[i]) * u[i];
    }
    uint4 sb[SIDE ? 4 : 1], sr[SIDE ? 4 : 1];
#pragma unroll
    for (int g = 0; g < (SIDE ? 4 : 0); ++g) {
      const int col = n0 + c + g * 8;
      const bool inside = row < M && col < N;
      sb[g] = sr[g] = make_uint4(0u, 0u, 0u, 0u);
      if (has_bias && inside)
        sb[g] = __ldcg(reinterpret_cast<const uint4*>(bias + (size_t)row * ldb + col));
      if (has_res && inside)
        sr[g] = __ldcg(reinterpret_cast<const uint4*>(res + (size_t)row * ldr + col));
    }
    const uint32_t buf = xr + (uint32_t)((c >> 5) & 1) * 2048u;
    if (c - c0 >= 64) {
      if (lane == 0) bulk_wait_read_1();
      __syncwarp();
    }
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const bool inside = row < M && n0 + c + g * 8 < N;
      float* x = w + g * 8;
      if (has_bias && inside) {
        float b[8];
        unpack8(sb[g], dt, b);
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] += b[e];
      }
      if (relu) {
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = fmaxf(x[e], 0.0f);
      }
      if (has_res && inside) {
        float b[8];
        unpack8(sr[g], dt, b);
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] += b[e];
      }
      const uint4 pk = pack8(x, dt);
      const uint32_t dst = buf + (uint32_t)lane * 64u + (uint32_t)((g ^ ((lane >> 1) & 3)) << 4);
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(pk.x), "r"(pk.y),
                   "r"(pk.z), "r"(pk.w)
                   : "memory");
    }
    fence_proxy_async_shared();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(omap, buf, n0 + c, row0);
      bulk_commit();
    }
  };
  if (!DUAL && S == 2) {
    // the partner's partial of the next chunk is in flight while a chunk is finished (a deeper
    // prefetch raises this callee's registers enough to make the kernel function spill)
    const float4* other = parts + (size_t)(1 - mine) * pstride;
    float4 a[V];
    issue(c0, other, a);
    for (int c = c0; c < c1; c += 32) {
      float w[32], u[1];
#pragma unroll
      for (int i = 0; i < 32; ++i) w[i] = 0.f;
      if (mine == 0) {
        add_own(c, w, u);
        add_part(w, u, a);
      } else {
        add_part(w, u, a);
        add_own(c, w, u);
      }
      if (c + 32 < c1) issue(c + 32, other, a);
      finish(c, w, u);
    }
  } else {
    for (int c = c0; c < c1; c += 32) {
      float w[32], u[DUAL ? 32 : 1];
#pragma unroll
      for (int i = 0; i < 32; ++i) w[i] = 0.f;
#pragma unroll
      for (int i = 0; i < (DUAL ? 32 : 1); ++i) u[i] = 0.f;
      for (int sp = 0; sp < S; ++sp) {
        if (sp == mine) {
          add_own(c, w, u);
        } else {
          float4 v[V];
          issue(c, parts + (size_t)sp * pstride, v);
          add_part(w, u, v);
        }
      }
      finish(c, w, u);
    }
  }
}

// The epilogue of a GEMM tile whose output feeds a fused RoPE (plain matmul, head_dim 64): per
// 64-column head, TMEM -> registers, the output rounded and stored as usual, then the following
// rope node's rotation of those rounded values (rotate_half pairing (j, j + 32), position =
// pos0 + output row, theta^(-2i/64) frequencies, the angle formula of the row path) stored to
// out_q / out_k, or the value copied to out_v for v heads when the node has one. Each 32 x 32
// block goes through one of the warp's two staging buffers to a TMA store; a buffer is rewritten
// once the store issued from it two blocks earlier has read it.
__device__ __noinline__ void epi_rope(const Params& p, const Node& nd, int n0, uint32_t tb,
                                      int nk, uint32_t xr, int row0) {
  const int tn = nd.tile_n, dt = nd.dtype, hq = nd.hq, hkv = nd.hkv, pos0 = nd.pos0;
  const float l2t = log2f(nd.theta);
  const void* omap = tmap_at(p, nd.out.tmap);
  const void* qmap = tmap_at(p, nd.out_q.tmap);
  const void* kmap = tmap_at(p, nd.out_k.tmap);
  const void* vmap = nd.out_v.tmap >= 0 ? tmap_at(p, nd.out_v.tmap) : nullptr;
  const int lane = threadIdx.x & 31;
  const float pos = (float)(pos0 + row0 + lane);
  // the row's 32 angles are the same for every head of the tile: their sines and cosines once
  const float my_inv = exp2f(-(2.0f * (float)lane / 64.0f) * l2t);  // lane i: frequency i
  float cs[32], sn[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) rope_sincos(pos * __shfl_sync(FULL, my_inv, i), &sn[i], &cs[i]);
  int nb = 0;  // blocks stored so far by this warp
  auto store_block = [&](const void* map, int col, const float* v) {
    const uint32_t buf = xr + (uint32_t)(nb & 1) * 2048u;
    if (nb >= 2) {
      if (lane == 0) bulk_wait_read_1();
      __syncwarp();
    }
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const uint4 pk = pack8(v + g * 8, dt);
      const uint32_t dst = buf + (uint32_t)lane * 64u + (uint32_t)((g ^ ((lane >> 1) & 3)) << 4);
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(pk.x), "r"(pk.y),
                   "r"(pk.z), "r"(pk.w)
                   : "memory");
    }
    fence_proxy_async_shared();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(map, buf, col, row0);
      bulk_commit();
    }
    ++nb;
  };
  for (int c = 0; c < tn; c += 64) {
    float lo[32], hi[32];
    if (nk > 0) {
      uint32_t r[32], r2[32];
      tmem_ld32(tb + (uint32_t)c, r);
      tmem_ld32(tb + (uint32_t)(c + 32), r2);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        lo[i] = __uint_as_float(r[i]);
        hi[i] = __uint_as_float(r2[i]);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) lo[i] = hi[i] = 0.f;
    }
    const int col = n0 + c, h = col >> 6;
    store_block(omap, col, lo);
    store_block(omap, col + 32, hi);
#pragma unroll
    for (int i = 0; i < 32; i += 2) {  // the values the rope node reads: the stored outputs
      round2(lo[i], lo[i + 1], dt);
      round2(hi[i], hi[i + 1], dt);
    }
    if (h < hq + hkv) {
#pragma unroll
      for (int i = 0; i < 32; ++i) {  // fully unrolled: the arrays stay in registers
        const float a = lo[i], b = hi[i];
        lo[i] = rope_z1(a, b, cs[i], sn[i]);  // first half: x cos - x' sin
        hi[i] = rope_z2(a, b, cs[i], sn[i]);  // second half: x cos + x' sin
      }
      const bool q = h < hq;
      const void* map = q ? qmap : kmap;
      const int oc = q ? col : col - hq * 64;
      store_block(map, oc, lo);
      store_block(map, oc + 32, hi);
    } else if (vmap && h < hq + 2 * hkv) {
      const int oc = col - (hq + hkv) * 64;
      store_block(vmap, oc, lo);
      store_block(vmap, oc + 32, hi);
    }
  }
}

// One call site for the four split epilogues, like epi_tile.
__device__ __noinline__ void epi_split_tile(const Node& nd, int n0, int c0, int c1, uint32_t tb,
                                            int nk, const void* omap, uint32_t xr, int row0,
                                            const float4* parts, int S, int mine,
                                            size_t pstride) {
  const uint32_t flags = nd.flags;
  const int tn = nd.tile_n, dt = nd.dtype, M = nd.M, N = nd.N;
  const uint16_t* bias = reinterpret_cast<const uint16_t*>(nd.bias.ptr);
  const uint16_t* res = reinterpret_cast<const uint16_t*>(nd.res.ptr);
  const int ldb = nd.bias.ld, ldr = nd.res.ld;
  const bool dual = (flags & EPI_SILU_MUL) != 0;
  const bool side = (flags & (EPI_BIAS | EPI_RESIDUAL)) != 0;
  if (dual && side)
    epi_split<true, true>(tb, tn, c0, c1, nk, flags, dt, bias, ldb, res, ldr, omap, xr, row0, n0,
                          M, N, parts, S, mine, pstride);
  else if (dual)
    epi_split<true, false>(tb, tn, c0, c1, nk, flags, dt, bias, ldb, res, ldr, omap, xr, row0,
                           n0, M, N, parts, S, mine, pstride);
  else if (side)
    epi_split<false, true>(tb, tn, c0, c1, nk, flags, dt, bias, ldb, res, ldr, omap, xr, row0,
                           n0, M, N, parts, S, mine, pstride);
  else
    epi_split<false, false>(tb, tn, c0, c1, nk, flags, dt, bias, ldb, res, ldr, omap, xr, row0,
                            n0, M, N, parts, S, mine, pstride);
}

// GEMM epilogue: TMEM -> registers (one row per thread), fused epilogue, then per 32-column chunk
// a 32 x 32 block per warp staged in shared memory and stored with TMA. In pair mode each CTA
// drains its own 128 rows of the 256-row tile. A split-tail tile (aux1 = number of K splits)
// first writes its fp32 partial to scratch and releases TMEM; the last split to finish (tile
// semaphore) sums the partials in split order and runs the epilogue; the others do not publish.
template <bool PAIR, int KS>
__device__ bool gemm_epilogue(const Params& p, Smem& s, const Instr& in, const Node& nd, int slot,
                              uint32_t use, uint32_t tmem, uint32_t& acc_n, bool* publish,
                              int idx) {
  const int ct = (int)threadIdx.x - (kThreads - kCompute);
  const int q = ct >> 5, lane = ct & 31;
  if (!cw_wait(p, smem_u32(&s.deps_ready[slot]), use & 1u, 30, idx)) return false;
  trace_mark(p, idx, 2);
  const int nk = ring_stages(in);
  const uint32_t as = acc_n & 1u;
  if (nk > 0) {
    if (!cw_wait(p, smem_u32(&s.acc_full[as]), (acc_n >> 1) & 1u, 31, idx)) return false;
    tc_fence_after();
  }
  trace_mark(p, idx, 6);
  const int dt = nd.dtype;
  const bool dual = (nd.flags & EPI_SILU_MUL) != 0;
  const int tn = nd.tile_n;
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const int row0 = in.m0 + (int)rank * kGemmTileM + q * 32;  // this warp's 32 rows
  const uint32_t tb = tmem + as * 256u + ((uint32_t)(q * 32) << 16);
  auto release_tmem = [&]() {
    if (nk > 0) {
      tc_fence_before();
      cw_sync();
      if (ct == 0) {
        if (PAIR && rank != 0)
          mbar_arrive_cluster(mapa_shared(smem_u32(&s.acc_empty[as]), 0));
        else
          mbar_arrive(smem_u32(&s.acc_empty[as]));
      }
      ++acc_n;
    }
  };
  if (nd.out.tmap < 0) {  // the host builds the output map of every GEMM node
    if (ct == 0) report(p, MK_ERR_DEVICE_CHECK, idx, -1, nd.out.tmap, 0, R_COMPUTE, 36);
    return false;
  }
  // Each warp stages its 32 x 32 block of a chunk in one of two 2 KB buffers (64-byte rows,
  // 64-byte swizzle: 16-byte chunk j of row r at j ^ ((r >> 1) & 3), conflict-free) and one lane
  // stores it with TMA; a buffer is rewritten once the store issued from it has read it.
  const uint32_t xr0 = smem_u32(s.xr) + (uint32_t)q * 4096u;
  const void* omap = tmap_at(p, nd.out.tmap);
  if (in.aux1 == 2 && !dual) {
    // Two-split tail, both splits finishing: split s owns columns [s h, s h + h) of the tile
    // (h = tn / 2). Each stores the half of its fp32 partial the other owns, meets the other at
    // the tile's semaphore (count 2: the two splits are consecutive instructions, so neither
    // waits on work queued behind the other), sums its half in split order and runs that half's
    // epilogue. A second round on the semaphore (count 4) lets the split that finishes last
    // publish, once both halves' stores are in global memory.
    const int h = tn / 2, own0 = in.split * h, cl = PAIR ? 2 : 1;
    const size_t slot_f4 = (size_t)kGemmTileM * tn / 4;  // float4 per (split, rank) slot
    const size_t pstride = (size_t)cl * slot_f4;          // next split, same rank
    float4* part0 = reinterpret_cast<float4*>(nd.scratch.ptr) + (size_t)in.slot * slot_f4 +
                    (size_t)q * 8 * tn + lane;  // this warp's block of split 0, this lane
    split_store(tb, h - own0, tn - own0, nk, part0 + (size_t)in.split * pstride);
    cw_sync();
    if (ct == 0) {
      fence_acq_rel_gpu();
      red_relaxed_add(p.counters + in.sem, 1);
    }
    if (!cw_wait_counter(p, p.counters + in.sem, 2, 47, idx)) return false;
    trace_mark(p, idx, 7);
    epi_split_tile(nd, in.n0, own0, own0 + h, tb, nk, omap, xr0, row0, part0, 2, in.split,
                   pstride);
    release_tmem();
    if (in.n_dst == 0) {  // nothing to publish: the second round only counts
      if (ct == 0) red_relaxed_add(p.counters + in.sem, 1);
      if (lane == 0) bulk_wait_read_all();
      *publish = false;
      return true;
    }
    if (lane == 0) {
      bulk_wait_all();
      fence_proxy_async_global();
    }
    cw_sync();
    if (ct == 0) {
      fence_acq_rel_gpu();
      s.flag = atomicAdd(p.counters + in.sem, 1) == 3;
      fence_acq_rel_gpu();
    }
    cw_sync();
    if (!s.flag) {
      *publish = false;
      return true;
    }
  } else if (in.aux1 > 0) {
    // Split tail: every split stores its fp32 partial (gate columns, then up columns with
    // SiLU·mul); the last split to reach the tile's semaphore sums them and runs the epilogue.
    const int W = dual ? 2 * tn : tn, S = in.aux1, cl = PAIR ? 2 : 1;
    const size_t slot_f4 = (size_t)kGemmTileM * W / 4;  // float4 per (split, rank) slot
    const size_t pstride = (size_t)cl * slot_f4;          // next split, same rank
    float4* part0 = reinterpret_cast<float4*>(nd.scratch.ptr) + (size_t)in.slot * slot_f4 +
                    (size_t)q * 8 * W + lane;  // this warp's block of split 0, this lane
    split_store(tb, 0, W, nk, part0 + (size_t)in.split * pstride);
    cw_sync();
    if (ct == 0) {
      fence_acq_rel_gpu();
      s.flag = atomicAdd(p.counters + in.sem, 1) == S - 1;
      fence_acq_rel_gpu();
    }
    cw_sync();
    if (!s.flag) {
      release_tmem();
      *publish = false;
      return true;
    }
    epi_split_tile(nd, in.n0, 0, tn, tb, nk, omap, xr0, row0, part0, S, in.split, pstride);
    release_tmem();
  } else if (nd.flags & NF_ROPE) {
    epi_rope(p, nd, in.n0, tb, nk, xr0, row0);
    release_tmem();
  } else {
    if constexpr (KS == KS_GEMM) {
      epi_tile(nd, in.n0, tn, tb, nk, omap, xr0, row0);
    } else {
      const uint16_t* bp = reinterpret_cast<const uint16_t*>(nd.bias.ptr);
      const uint16_t* rp = reinterpret_cast<const uint16_t*>(nd.res.ptr);
      // fewer registers in the callee: fewer values saved around the call in these kernels
      if (dual)
        epi_chunks<true, true, false>(tb, tn, nk, nd.flags, dt, bp, nd.bias.ld, rp, nd.res.ld,
                                      omap, xr0, row0, in.n0, nd.M, nd.N);
      else
        epi_chunks<false, true, false>(tb, tn, nk, nd.flags, dt, bp, nd.bias.ld, rp, nd.res.ld,
                                       omap, xr0, row0, in.n0, nd.M, nd.N);
    }
    release_tmem();
  }
  // the tile's stores are in global memory before its counters are released; with no counter
  // to release, the staging buffers need only have been read
  if (lane == 0) {
    if (in.n_dst > 0) {
      bulk_wait_all();
      fence_proxy_async_global();
    } else {
      bulk_wait_read_all();
    }
  }
  return true;
}

// One 64-row weight stage of a GEMV for MT activation rows (compile-time), element type BF
// (compile-time): acc[m][0..1] += sum_kk x[m][kk] * W[kk][col..col+1], W read from a 64-column
// box in the 128-byte swizzled layout TMA writes. Four activations per shared-memory read; the
// weight pair of each row is one 4-byte read (a warp covers one 128-byte row: no conflicts).
template <int MT, bool BF, int UNROLL = 2>
__device__ __forceinline__ void gemv_stage(const uint8_t* B, int ch, const float* xs,
                                           int xstride, float (&acc)[8][2]) {
#pragma unroll UNROLL
  for (int kk = 0; kk < kGemvRows; kk += 4) {
    float xv[MT][4];
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      const float4 x4 = *reinterpret_cast<const float4*>(xs + m * xstride + kk);
      xv[m][0] = x4.x;
      xv[m][1] = x4.y;
      xv[m][2] = x4.z;
      xv[m][3] = x4.w;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int r = kk + u;  // 128-byte row r of the box; 16-byte chunk ch sits at ch ^ (r & 7)
      const uint32_t raw = *reinterpret_cast<const uint32_t*>(B + r * 128 + ((ch ^ (r & 7)) << 4));
      float f0, f1;
      if (BF) {
        f0 = __uint_as_float(raw << 16);
        f1 = __uint_as_float(raw & 0xffff0000u);
      } else {
        f0 = __half2float(__ushort_as_half((uint16_t)(raw & 0xffffu)));
        f1 = __half2float(__ushort_as_half((uint16_t)(raw >> 16)));
      }
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        acc[m][0] = fmaf(xv[m][u], f0, acc[m][0]);
        acc[m][1] = fmaf(xv[m][u], f1, acc[m][1]);
      }
    }
  }
}

template <bool BF>
__device__ __forceinline__ void gemv_stage_rows(int M, const uint8_t* B, int ch, const float* xs,
                                                int xstride, float (&acc)[8][2]) {
  switch (M) {
    case 1: gemv_stage<1, BF>(B, ch, xs, xstride, acc); break;
    case 2: gemv_stage<2, BF>(B, ch, xs, xstride, acc); break;
    case 3: gemv_stage<3, BF>(B, ch, xs, xstride, acc); break;
    case 4: gemv_stage<4, BF>(B, ch, xs, xstride, acc); break;
    case 5: gemv_stage<5, BF>(B, ch, xs, xstride, acc); break;
    case 6: gemv_stage<6, BF>(B, ch, xs, xstride, acc); break;
    case 7: gemv_stage<7, BF>(B, ch, xs, xstride, acc); break;
    default: gemv_stage<8, BF>(B, ch, xs, xstride, acc); break;
  }
}

// The weight stages of a GEMV tile whose activations are all staged in shared memory: nk stages
// from ring position (st, ph), each consumed and released in turn. Out of line with scalar
// arguments, so the stage loop compiles on its own (inside the single large kernel function it ran
// several times slower); the 2·MT sums leave through `out` once.
template <int MT, bool BF>
__device__ __noinline__ bool gemv_staged(const Params& p, uint32_t full0, uint32_t empty0,
                                         const uint8_t* b0, uint32_t sb, uint32_t ns, uint32_t st,
                                         uint32_t ph, int nk, int ch, const float* xs0, int kpad,
                                         float* out, int idx) {
  const int ct = (int)threadIdx.x - (kThreads - kCompute);
  float acc[8][2];
#pragma unroll
  for (int m = 0; m < 8; ++m) acc[m][0] = acc[m][1] = 0.f;
  for (int kb = 0; kb < nk; ++kb) {
    if (!cw_wait(p, full0 + st * 8u, ph, 41, idx)) return false;
    // all 64 rows unrolled: the stage's shared-memory reads issue ahead of their FMAs
    gemv_stage<MT, BF, 16>(b0 + (size_t)st * sb, ch, xs0 + kb * kGemvRows, kpad, acc);
    cw_sync();
    if (ct == 0) mbar_arrive(empty0 + st * 8u);
    if (++st == ns) {
      st = 0;
      ph ^= 1u;
    }
  }
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    out[2 * m] = acc[m][0];
    out[2 * m + 1] = acc[m][1];
  }
  return true;
}

template <bool BF>
__device__ bool gemv_staged_rows(int M, const Params& p, uint32_t full0, uint32_t empty0,
                                 const uint8_t* b0, uint32_t sb, uint32_t ns, uint32_t st,
                                 uint32_t ph, int nk, int ch, const float* xs0, int kpad,
                                 float* out, int idx) {
  switch (M) {
    case 1: return gemv_staged<1, BF>(p, full0, empty0, b0, sb, ns, st, ph, nk, ch, xs0, kpad, out, idx);
    case 2: return gemv_staged<2, BF>(p, full0, empty0, b0, sb, ns, st, ph, nk, ch, xs0, kpad, out, idx);
    case 3: return gemv_staged<3, BF>(p, full0, empty0, b0, sb, ns, st, ph, nk, ch, xs0, kpad, out, idx);
    case 4: return gemv_staged<4, BF>(p, full0, empty0, b0, sb, ns, st, ph, nk, ch, xs0, kpad, out, idx);
    case 5: return gemv_staged<5, BF>(p, full0, empty0, b0, sb, ns, st, ph, nk, ch, xs0, kpad, out, idx);
    case 6: return gemv_staged<6, BF>(p, full0, empty0, b0, sb, ns, st, ph, nk, ch, xs0, kpad, out, idx);
    case 7: return gemv_staged<7, BF>(p, full0, empty0, b0, sb, ns, st, ph, nk, ch, xs0, kpad, out, idx);
    default: return gemv_staged<8, BF>(p, full0, empty0, b0, sb, ns, st, ph, nk, ch, xs0, kpad, out, idx);
  }
}

// GEMV tile: out[0..M) x [n0, n0 + w) for one K chunk; split partials reduced by the last
// split to finish. The chunk's activations (normalised when the norm is fused) are staged once
// in shared memory with batched loads. Each thread owns two adjacent output columns of the tile
// (with SILU_MUL: threads 0-63 the gate columns, 64-127 the up columns) over every K row, so a
// stage needs no cross-thread reduction. Weight stages arrive as 128-byte swizzled boxes:
// unswizzled TMA writes of rows 128 bytes apart land on the same shared-memory banks ("Hand-
// writing a Blackwell GEMM", step 4).
// Sum of a column pair over the S split partials of a GEMV tile, in split order (the result
// does not depend on which split finished last). Up to 24 partials are loaded at once, so the
// usual split counts (at most 19 on 152 SMs) cost one round trip to L2 instead of one per few
// partials.
__device__ __noinline__ float2 sum_splits(const float* c0, int S, size_t ld) {
  constexpr int B = 24;
  float2 t = make_float2(0.f, 0.f);
  for (int q0 = 0; q0 < S; q0 += B) {
    float2 v[B];
#pragma unroll
    for (int u = 0; u < B; ++u)
      v[u] = q0 + u < S ? __ldcg(reinterpret_cast<const float2*>(c0 + (size_t)(q0 + u) * ld))
                        : make_float2(0.f, 0.f);
#pragma unroll
    for (int u = 0; u < B; ++u) {
      if (q0 + u < S) {
        t.x += v[u].x;
        t.y += v[u].y;
      }
    }
  }
  return t;
}

template <bool PAIR>
__device__ bool gemv(const Params& p, Smem& s, const Instr& in, const Node& nd, int slot,
                     uint32_t use, uint32_t& ring, bool* publish, int idx, uint32_t tmem,
                     uint32_t& acc_n) {
  const uint32_t NS = ring_n(p);
  const int ct = (int)threadIdx.x - (kThreads - kCompute);
  const int wp = ct >> 5, lane = ct & 31;
  if (!cw_wait(p, smem_u32(&s.deps_ready[slot]), use & 1u, 40, idx)) return false;
  trace_mark(p, idx, 2);
  const int M = nd.M, dt = nd.dtype;
  const bool dual = (nd.flags & EPI_SILU_MUL) != 0;
  const bool norm = (nd.flags & EPI_RMSNORM_INPUT) != 0;
  const int nk = ring_stages(in);
  const int kpad = nk * kGemvRows;
  const int kend = in.k0 + in.klen;
  const bool staged = M * kpad <= kXrFloats;
  const bool tensor = gemv_on_tensor<PAIR>(in, nd);
  // One row whose K range is at most one 16-byte item per thread (every decode GEMV): the loads
  // for the RMS statistic, the K range and gamma are all issued before any is used, so staging
  // waits on one round trip to L2 instead of two.
  const bool onepass = tensor && M == 1 && kpad / 8 <= kCompute;
  if (norm && !onepass) {
    // RMS statistic of each whole input row (the norm is a flag of this GEMV)
    for (int m = 0; m < M; ++m) {
      float ss = 0.f;
      for (int k = ct * 8; k < nd.K; k += kCompute * 8) {
        float x[8];
        load8(nd.a, m, k, dt, x);
#pragma unroll
        for (int e = 0; e < 8; ++e) ss = fmaf(x[e], x[e], ss);
      }
      ss = warp_sum(ss);
      if (lane == 0) s.red_small[m][wp] = ss;
    }
    cw_sync();
    if (ct < M)
      s.rstd[ct] = rsqrtf((s.red_small[ct][0] + s.red_small[ct][1] + s.red_small[ct][2] +
                           s.red_small[ct][3]) / (float)nd.K + nd.eps);
    cw_sync();
  }
  auto stage_x = [&](int k_first, int rows, int stride) {
    const int nv = rows / 8;
    for (int v = ct; v < M * nv; v += kCompute) {
      const int m = v / nv, kk = (v % nv) * 8, k = k_first + kk;
      float x[8];
      if (k < kend) {
        load8(nd.a, m, k, dt, x);
        if (norm) {
          float g[8];
          load8(nd.gamma, 0, k, dt, g);
          const float r = s.rstd[m];
#pragma unroll
          for (int e = 0; e < 8; ++e) x[e] = x[e] * r * g[e];
        }
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = 0.f;
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) s.xr[m * stride + kk + e] = x[e];
    }
    cw_sync();
  };
  const int which = dual ? (ct >> 6) : 0;
  const int col = dual ? 2 * (ct & 63) : 2 * ct;  // column pair inside this thread's weight
  // the residual pair of a one-row tile is read now, off the critical path of the last split
  float res0 = 0.f, res1 = 0.f;
  if (M == 1 && (nd.flags & EPI_RESIDUAL) && which == 0 && in.n0 + col < nd.N) {
    res0 = load1(nd.res, 0, in.n0 + col, dt);
    res1 = load1(nd.res, 0, in.n0 + col + 1, dt);
  }
  if (onepass) {
    // the B operand as below (one 1 KB atom per 64-K block, chunk c of row 0 at c), one item
    // per thread; the statistic's loads of the whole row go out together with it
    uint8_t* xb = reinterpret_cast<uint8_t*>(s.xr);
    const int kk = ct * 8, k = in.k0 + kk;
    const bool item = kk < kpad, have = item && k < kend;
    const uint16_t* xrow = reinterpret_cast<const uint16_t*>(nd.a.ptr);
    uint4 xv = make_uint4(0u, 0u, 0u, 0u), gv = xv;
    if (have) {
      xv = __ldcg(reinterpret_cast<const uint4*>(xrow + k));
      if (norm) gv = __ldcg(reinterpret_cast<const uint4*>(
                    reinterpret_cast<const uint16_t*>(nd.gamma.ptr) + k));
    }
    float r = 1.f;
    if (norm) {
      constexpr int kRowItems = 4;  // rows up to 4 * 128 * 8 = 4096 elements in one round
      uint4 rv[kRowItems];
#pragma unroll
      for (int u = 0; u < kRowItems; ++u) {
        const int kr = (ct + u * kCompute) * 8;
        rv[u] = kr < nd.K ? __ldcg(reinterpret_cast<const uint4*>(xrow + kr))
                          : make_uint4(0u, 0u, 0u, 0u);
      }
      float ss = 0.f;
#pragma unroll
      for (int u = 0; u < kRowItems; ++u) {
        float x[8];
        unpack8(rv[u], dt, x);
#pragma unroll
        for (int e = 0; e < 8; ++e) ss = fmaf(x[e], x[e], ss);
      }
      for (int kr = (ct + kRowItems * kCompute) * 8; kr < nd.K; kr += kCompute * 8) {
        float x[8];
        load8(nd.a, 0, kr, dt, x);
#pragma unroll
        for (int e = 0; e < 8; ++e) ss = fmaf(x[e], x[e], ss);
      }
      ss = warp_sum(ss);
      if (lane == 0) s.red_small[0][wp] = ss;
      cw_sync();
      r = rsqrtf((s.red_small[0][0] + s.red_small[0][1] + s.red_small[0][2] +
                  s.red_small[0][3]) / (float)nd.K + nd.eps);
    }
    if (item) {
      float x[8];
      unpack8(xv, dt, x);
      if (norm) {
        float g[8];
        unpack8(gv, dt, g);
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = x[e] * r * g[e];
      }
      *reinterpret_cast<uint4*>(xb + (kk >> 6) * 1024 + (((kk & 63) >> 3) << 4)) = pack8(x, dt);
    }
    fence_proxy_async_shared();
    cw_sync();
    if (ct == 0) mbar_arrive(smem_u32(&s.gx_full));
  } else if (tensor) {
    // the K-major B operand of the tensor-core tile: per 64-K block a 1 KB atom of 8 rows x 128
    // bytes, 16-byte chunk c of row m at c ^ m; the activations rounded to the weight type
    uint8_t* xb = reinterpret_cast<uint8_t*>(s.xr);
    const int nv = kpad / 8;
    for (int v = ct; v < M * nv; v += kCompute) {
      const int m = v / nv, kk = (v % nv) * 8, k = in.k0 + kk;
      float x[8];
      if (k < kend) {
        load8(nd.a, m, k, dt, x);
        if (norm) {
          float g[8];
          load8(nd.gamma, 0, k, dt, g);
          const float r = s.rstd[m];
#pragma unroll
          for (int e = 0; e < 8; ++e) x[e] = x[e] * r * g[e];
        }
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = 0.f;
      }
      *reinterpret_cast<uint4*>(xb + (kk >> 6) * 1024 + m * 128 + ((((kk & 63) >> 3) ^ m) << 4)) =
          pack8(x, dt);
    }
    fence_proxy_async_shared();
    cw_sync();
    if (ct == 0) mbar_arrive(smem_u32(&s.gx_full));
  } else if (staged && nk > 0) {
    stage_x(in.k0, kpad, kpad);
  }
  float acc[8][2];
#pragma unroll
  for (int m = 0; m < 8; ++m) acc[m][0] = acc[m][1] = 0.f;
  if (tensor) {
    const uint32_t as = acc_n & 1u;
    if (!cw_wait(p, smem_u32(&s.acc_full[as]), (acc_n >> 1) & 1u, 42, idx)) return false;
    tc_fence_after();
    trace_mark(p, idx, 6);
    // accumulator lanes are the tile's weight columns (this warp: 32 of each half), its columns
    // the activation rows; through the staging buffer into the column-pair layout below
    uint32_t r[32];
    tmem_ld32(tmem + as * 256u + ((uint32_t)(wp * 32) << 16), r);
    tmem_ld_wait();
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int m = 0; m < 8; ++m)
        if (m < M) s.xr[m * 256 + h * 128 + wp * 32 + lane] = __uint_as_float(r[h * 16 + m]);
    tc_fence_before();
    cw_sync();
    if (ct == 0) mbar_arrive(smem_u32(&s.acc_empty[as]));
    ++acc_n;
#pragma unroll
    for (int m = 0; m < 8; ++m)
      if (m < M) {
        acc[m][0] = s.xr[m * 256 + which * 128 + col];
        acc[m][1] = s.xr[m * 256 + which * 128 + col + 1];
      }
    ring += (uint32_t)nk;  // the MMA issuer consumed and released the stages
  } else if (staged && nk > 0) {
    // this thread's column pair: box (which * 2 + col / 64), column col % 64 inside it
    const int box = (dual ? which * 2 : 0) + (col >> 6), lc = col & 63;
    float sums[16];
    const bool ok =
        dt == DT_BF16
            ? gemv_staged_rows<true>(M, p, smem_u32(&s.full[0]), smem_u32(&s.empty[0]),
                                     s.ring + box * 8192 + (lc & 7) * 2, stage_bytes(p), NS,
                                     ring % NS, (ring / NS) & 1u, nk, lc >> 3, s.xr, kpad, sums,
                                     idx)
            : gemv_staged_rows<false>(M, p, smem_u32(&s.full[0]), smem_u32(&s.empty[0]),
                                      s.ring + box * 8192 + (lc & 7) * 2, stage_bytes(p), NS,
                                      ring % NS, (ring / NS) & 1u, nk, lc >> 3, s.xr, kpad, sums,
                                      idx);
    if (!ok) return false;
    trace_mark(p, idx, 6);
#pragma unroll
    for (int m = 0; m < 8; ++m)
      if (m < M) {
        acc[m][0] = sums[2 * m];
        acc[m][1] = sums[2 * m + 1];
      }
    ring += (uint32_t)nk;
  }
  for (int kb = 0; kb < nk && !staged && !tensor; ++kb) {
    const float* xs;
    int xstride;
    if (staged) {
      xs = s.xr + kb * kGemvRows;
      xstride = kpad;
    } else {
      stage_x(in.k0 + kb * kGemvRows, kGemvRows, kGemvRows);
      xs = s.xr;
      xstride = kGemvRows;
    }
    const int st = (int)(ring % NS);
    if (!cw_wait(p, smem_u32(&s.full[st]), (ring / NS) & 1u, 41, idx)) return false;
    // this thread's column pair: box (which * 2 + col / 64), column col % 64 inside it
    const int box = (dual ? which * 2 : 0) + (col >> 6), lc = col & 63;
    const uint8_t* B = stage_ptr(s, p, st) + box * 8192 + (lc & 7) * 2;
    if (dt == DT_BF16)
      gemv_stage_rows<true>(M, B, lc >> 3, xs, xstride, acc);
    else
      gemv_stage_rows<false>(M, B, lc >> 3, xs, xstride, acc);
    cw_sync();
    if (ct == 0) mbar_arrive(smem_u32(&s.empty[st]));
    ++ring;
  }
  const int S = in.aux1;
  const int n = in.n0 + col;
  const bool colok = n < nd.N;  // N is a multiple of 8: both columns are in or both out
  if (S == 1) {
    if (ct == 0) atomicAdd(p.counters + in.sem, 1);  // the semaphore counts every split
  } else {
    float* part = reinterpret_cast<float*>(nd.scratch.ptr);
    if (colok) {
#pragma unroll
      for (int m = 0; m < 8; ++m)
        if (m < M)
          __stcg(reinterpret_cast<float2*>(part + (size_t)in.aux0 * nd.ldp +
                                           ((size_t)which * M + m) * nd.N + n),
                 make_float2(acc[m][0], acc[m][1]));
    }
    // one thread releases the warpgroup's partials (ordered before it by the barrier) and, as
    // the last split, acquires the others'
    cw_sync();
    if (ct == 0) {
      fence_acq_rel_gpu();
      s.flag = (atomicAdd(p.counters + in.sem, 1) == S - 1);
      fence_acq_rel_gpu();
    }
    cw_sync();
    if (!s.flag) {
      *publish = false;
      return true;
    }
    if (colok) {
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        if (m >= M) continue;
        const float2 t = sum_splits(part + ((size_t)which * M + m) * nd.N + n, S, nd.ldp);
        acc[m][0] = t.x;
        acc[m][1] = t.y;
      }
    }
  }
  if (dual) {
    // gate and up halves of a column pair live in threads t and t + 64: exchange via smem
    cw_sync();
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      if (m < M) {
        s.xr[m * 256 + which * 128 + col] = acc[m][0];
        s.xr[m * 256 + which * 128 + col + 1] = acc[m][1];
      }
    }
    cw_sync();
    if (which == 0) {
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        if (m < M) {
          acc[m][0] = silu(s.xr[m * 256 + col]) * s.xr[m * 256 + 128 + col];
          acc[m][1] = silu(s.xr[m * 256 + col + 1]) * s.xr[m * 256 + 128 + col + 1];
        }
      }
    }
  }
  if (which == 0 && colok) {
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      if (m >= M) continue;
      float y0 = acc[m][0], y1 = acc[m][1];
      if (nd.flags & EPI_BIAS) {
        y0 += load1(nd.bias, m, n, dt);
        y1 += load1(nd.bias, m, n + 1, dt);
      }
      if (nd.flags & EPI_RELU) {
        y0 = fmaxf(y0, 0.f);
        y1 = fmaxf(y1, 0.f);
      }
      if (nd.flags & EPI_RESIDUAL) {
        y0 += M == 1 ? res0 : load1(nd.res, m, n, dt);
        y1 += M == 1 ? res1 : load1(nd.res, m, n + 1, dt);
      }
      store2(nd.out, m, n, dt, y0, y1);
      if (nd.flags & NF_ROPE) {
        // RoPE of the following node, on the rounded outputs it would read: the pair partner of
        // column j of a 64-column head is j ^ 32, held by lane ^ 16 (whole heads per tile, every
        // lane active: the host fuses only full-width tiles without a second weight)
        float r0 = y0, r1 = y1;
        round2(r0, r1, dt);
        const float p0 = __shfl_xor_sync(FULL, r0, 16), p1 = __shfl_xor_sync(FULL, r1, 16);
        const int qend = nd.hq * 64, kend = (nd.hq + nd.hkv) * 64;
        if (n < kend) {
          const int j = n & 63, i = j & 31;
          const float pos = (float)(nd.pos0 + m), l2t = log2f(nd.theta);
          float sn0, cs0, sn1, cs1;
          rope_sincos(pos * exp2f(-(2.0f * (float)i / 64.0f) * l2t), &sn0, &cs0);
          rope_sincos(pos * exp2f(-(2.0f * (float)(i + 1) / 64.0f) * l2t), &sn1, &cs1);
          const float z0 = j < 32 ? rope_z1(r0, p0, cs0, sn0) : rope_z2(p0, r0, cs0, sn0);
          const float z1 = j < 32 ? rope_z1(r1, p1, cs1, sn1) : rope_z2(p1, r1, cs1, sn1);
          if (n < qend)
            store2(nd.out_q, m, n, dt, z0, z1);
          else
            store2(nd.out_k, m, n - qend, dt, z0, z1);
        } else if (nd.out_v.ptr) {
          store2(nd.out_v, m, n - kend, dt, r0, r1);
        }
      }
    }
  }
  *publish = true;
  return true;
}

__device__ void ew_body(const Instr& in, const Node& nd) {
  const int ct = (int)threadIdx.x - (kThreads - kCompute);
  const int rows = min(nd.tile_m, nd.M - in.m0), cols = min(nd.tile_n, nd.N - in.n0);
  const int nv = cols / 8, dt = nd.dtype;
  for (int v = ct; v < rows * nv; v += kCompute) {
    const int m = in.m0 + v / nv, n = in.n0 + (v % nv) * 8;
    float a[8], b[8], y[8];
    load8(nd.a, m, n, dt, a);
    if (nd.ewop == EWOP_ADD || nd.ewop == EWOP_SILU_MUL) load8(nd.b, m, n, dt, b);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      switch (nd.ewop) {
        case EWOP_ADD: y[e] = a[e] + b[e]; break;
        case EWOP_RELU: y[e] = fmaxf(a[e], 0.f); break;
        case EWOP_SILU_MUL: y[e] = silu(a[e]) * b[e]; break;
        default: y[e] = a[e]; break;
      }
    }
    store8(nd.out, m, n, dt, y);
  }
}

// RMSNorm rows of one instruction (tile_m rows from m0), one warp per row, read directly from
// global memory: a pass for the statistic, then a pass that scales by rstd and gamma. Lane l
// takes the 16-byte vectors l, l + 32, ... of the row (the summation order the staged form
// keeps too).
__device__ __forceinline__ void rmsnorm_body(const Instr& in, const Node& nd) {
  const int ct = (int)threadIdx.x - (kThreads - kCompute);
  const int wp = ct >> 5, lane = ct & 31;
  const int rows = min(nd.tile_m, nd.M - in.m0), dt = nd.dtype, N = nd.N;
  const float eps = nd.eps;
  for (int r = wp; r < rows; r += 4) {
    const int m = in.m0 + r;
    float s0 = 0.f, s1 = 0.f;  // two chains, as the staged path sums them
    for (int k = lane * 8; k < N; k += 256) {
      float x[8];
      load8(nd.a, m, k, dt, x);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        s0 += x[e] * x[e];
        s1 += x[e + 4] * x[e + 4];
      }
    }
    const float rstd = rsqrtf(warp_sum(s0 + s1) / (float)N + eps);
    for (int k = lane * 8; k < N; k += 256) {
      float x[8], g[8];
      load8(nd.a, m, k, dt, x);
      load8(nd.gamma, 0, k, dt, g);
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] = x[e] * rstd * g[e];
      store8(nd.out, m, k, dt, x);
    }
  }
}

// RoPE rows read directly from global memory: thread work item = (row, head, 8 consecutive
// pair indices); both halves of the pairs arrive as 16-byte vectors and leave the same way, the
// angles computed inline. The v heads, when the node copies them, follow as 16-byte copies.
__device__ __forceinline__ void rope_body(const Instr& in, const Node& nd) {
  const int ct = (int)threadIdx.x - (kThreads - kCompute);
  const int rows = min(nd.tile_m, nd.M - in.m0), dt = nd.dtype;
  const int hd = nd.hd, half = hd / 2, nh = nd.hq + nd.hkv;
  const int groups = half / 8;                 // 8-pair groups per head
  const int items = nh * groups;
  const float l2t = log2f(nd.theta);
  const uint16_t* a = reinterpret_cast<const uint16_t*>(nd.a.ptr);
  const size_t lda = (size_t)nd.a.ld;
  const int total = rows * items;
  for (int v = ct; v < total; v += kCompute) {
    const int m = in.m0 + v / items, it = v % items;
    const int h = it / groups, i0 = (it % groups) * 8;
    const uint16_t* src = a + m * lda + h * hd + i0;
    float x1[8], x2[8], y1[8], y2[8];
    unpack8(__ldcg(reinterpret_cast<const uint4*>(src)), dt, x1);
    unpack8(__ldcg(reinterpret_cast<const uint4*>(src + half)), dt, x2);
    const float pos = (float)(nd.pos0 + m);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      float sn, cs;
      const float inv = exp2f(-(2.0f * (float)(i0 + e) / (float)hd) * l2t);
      rope_sincos(pos * inv, &sn, &cs);
      y1[e] = rope_z1(x1[e], x2[e], cs, sn);
      y2[e] = rope_z2(x1[e], x2[e], cs, sn);
    }
    const Operand& o = h < nd.hq ? nd.out : nd.out_k;
    const int hh = h < nd.hq ? h : h - nd.hq;
    store8(o, m, hh * hd + i0, dt, y1);
    store8(o, m, hh * hd + i0 + half, dt, y2);
  }
  if (nd.out_v.ptr) {
    const int nvv = nd.hkv * hd / 8, tv = rows * nvv;
    for (int v = ct; v < tv; v += kCompute)
      *reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(nd.out_v.ptr) +
                                (size_t)(in.m0 + v / nvv) * nd.out_v.ld + (v % nvv) * 8) =
          __ldcg(reinterpret_cast<const uint4*>(a + (in.m0 + v / nvv) * lda + nh * hd +
                                                (v % nvv) * 8));
  }
}

// Staged row instruction (see load_rows): stage j holds rows [j * rps, j * rps + nr) of the
// instruction, W elements each. RMSNorm: a warp per row, two rows per warp at a time; the
// statistic and the scaling both read the row from shared memory (lane l takes 16-byte vectors
// l, l + 32, ...: the summation order of the direct path), gamma is copied to shared memory
// once, while the rows are in flight. RoPE: a thread per 16-byte chunk (8 elements) of a head;
// the pair partners sit in the chunk of the other half of the head, held by lane ^ (head_dim /
// 16) (the host stages RoPE only when head_dim / 8 divides 32, so heads never straddle warps);
// angles from a table of the instruction's rows computed while the first stage is in flight; v
// is copied through.
template <bool ROPE>
__device__ bool rows_staged(const Params& p, Smem& s, const Instr& in, const Node& nd,
                            uint32_t& ring, int idx) {
  const uint32_t NS = ring_n(p);
  const int ct = (int)threadIdx.x - (kThreads - kCompute);
  const int wp = ct >> 5, lane = ct & 31;
  const int rows = min(nd.tile_m, nd.M - in.m0), dt = nd.dtype;
  const int W = row_stage_cols(nd), nst = ring_stages(in);
  const int rps = (int)(stage_bytes(p) / (uint32_t)(W * 2));
  const int hd = nd.hd, half = hd / 2, nh = nd.hq + nd.hkv;
  float* tcos = s.xr;
  float* tsin = s.xr + rows * half;
  const uint4* gm = reinterpret_cast<const uint4*>(nd.gamma.ptr);
  uint4* gs = reinterpret_cast<uint4*>(s.xr);
  const bool gshared = !ROPE && W * 2 <= kXrFloats * 4;
  if (ROPE) {
    const float l2t = log2f(nd.theta);
    for (int v = ct; v < rows * half; v += kCompute) {
      const int r = v / half, i = v % half;
      const float inv = exp2f(-(2.0f * (float)i / (float)hd) * l2t);
      rope_sincos((float)(nd.pos0 + in.m0 + r) * inv, &tsin[v], &tcos[v]);
    }
    cw_sync();
  } else if (gshared) {
    for (int v = ct; v < W / 8; v += kCompute) gs[v] = __ldg(gm + v);
    cw_sync();
  }
  for (int j = 0; j < nst; ++j) {
    const int st = (int)(ring % NS);
    if (!cw_wait(p, smem_u32(&s.full[st]), (ring / NS) & 1u, 46, idx)) return false;
    if (j == 0) trace_mark(p, idx, 6);
    const uint8_t* base = stage_ptr(s, p, st);
    const int r0 = j * rps, nr = min(rps, rows - r0);
    if (!ROPE) {
      // Rows r, r + 4 and r + 8 of the stage together (three independent rows per warp, each
      // row's squares summed in two chains, the same order as the unstaged path).
      uint16_t* out = reinterpret_cast<uint16_t*>(nd.out.ptr);
      const int nv = W / 8;
      for (int r = wp; r < nr; r += 12) {
        const uint4* xq[3];
        bool live[3];
#pragma unroll
        for (int k = 0; k < 3; ++k) {
          live[k] = r + 4 * k < nr;
          xq[k] = reinterpret_cast<const uint4*>(base + (size_t)(live[k] ? r + 4 * k : r) * W * 2);
        }
        float s0[3] = {0.f, 0.f, 0.f}, s1[3] = {0.f, 0.f, 0.f};
        for (int v = lane; v < nv; v += 32) {
#pragma unroll
          for (int k = 0; k < 3; ++k) {
            float f[8];
            unpack8(xq[k][v], dt, f);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              s0[k] += f[e] * f[e];
              s1[k] += f[e + 4] * f[e + 4];
            }
          }
        }
        float rs[3];
#pragma unroll
        for (int k = 0; k < 3; ++k) rs[k] = rsqrtf(warp_sum(s0[k] + s1[k]) / (float)W + nd.eps);
#pragma unroll 2
        for (int v = lane; v < nv; v += 32) {
          float gf[8];
          unpack8(gshared ? gs[v] : __ldg(gm + v), dt, gf);
#pragma unroll
          for (int k = 0; k < 3; ++k) {
            if (!live[k]) continue;
            float f[8];
            unpack8(xq[k][v], dt, f);
#pragma unroll
            for (int e = 0; e < 8; ++e) f[e] = f[e] * rs[k] * gf[e];
            *reinterpret_cast<uint4*>(out + (size_t)(in.m0 + r0 + r + 4 * k) * nd.out.ld + v * 8) =
                pack8(f, dt);
          }
        }
      }
    } else {
      // cpr = head_dim / 8 chunks per head, a power of two dividing 32 (host-checked): whole
      // heads fall in one warp, and the partner chunk is held by lane ^ cph
      const int cpr = hd / 8, cph = cpr / 2, lc = 31 - __clz(cpr);
      const int per_row = nh * cpr;
      for (int r = 0; r < nr; ++r) {
        const uint8_t* rowp = base + (size_t)r * W * 2;
        const float* tc = tcos + (r0 + r) * half;
        const float* ts = tsin + (r0 + r) * half;
        const int m = in.m0 + r0 + r;
        for (int c0 = 0; c0 < per_row; c0 += kCompute) {  // warp-uniform (shuffles)
          const int cix = c0 + ct;
          const bool live = cix < per_row;
          uint4 x = make_uint4(0u, 0u, 0u, 0u);
          if (live) x = *reinterpret_cast<const uint4*>(rowp + (size_t)cix * 16);
          uint4 q;
          q.x = __shfl_xor_sync(FULL, x.x, cph);
          q.y = __shfl_xor_sync(FULL, x.y, cph);
          q.z = __shfl_xor_sync(FULL, x.z, cph);
          q.w = __shfl_xor_sync(FULL, x.w, cph);
          if (!live) continue;
          const int h = cix >> lc, c = cix & (cpr - 1);
          const bool first = c < cph;
          const int i0 = (first ? c : c - cph) * 8;
          const float4 c_lo = *reinterpret_cast<const float4*>(tc + i0);
          const float4 c_hi = *reinterpret_cast<const float4*>(tc + i0 + 4);
          const float4 s_lo = *reinterpret_cast<const float4*>(ts + i0);
          const float4 s_hi = *reinterpret_cast<const float4*>(ts + i0 + 4);
          const float cs[8] = {c_lo.x, c_lo.y, c_lo.z, c_lo.w, c_hi.x, c_hi.y, c_hi.z, c_hi.w};
          const float sn[8] = {s_lo.x, s_lo.y, s_lo.z, s_lo.w, s_hi.x, s_hi.y, s_hi.z, s_hi.w};
          float xf[8], pf[8], y[8];
          unpack8(x, dt, xf);
          unpack8(q, dt, pf);
          // first half: x cos - x' sin; second half: x cos + x' sin (x' the partner element)
#pragma unroll
          for (int e = 0; e < 8; ++e) y[e] = first ? rope_z1(xf[e], pf[e], cs[e], sn[e])
                                                   : rope_z2(pf[e], xf[e], cs[e], sn[e]);
          const Operand& o = h < nd.hq ? nd.out : nd.out_k;
          const int hh = h < nd.hq ? h : h - nd.hq;
          store8(o, m, hh * hd + c * 8, dt, y);
        }
        if (nd.out_v.ptr) {
          const int nvv = nd.hkv * hd / 8;
          uint16_t* ov = reinterpret_cast<uint16_t*>(nd.out_v.ptr) + (size_t)m * nd.out_v.ld;
          for (int c = ct; c < nvv; c += kCompute)
            *reinterpret_cast<uint4*>(ov + c * 8) =
                *reinterpret_cast<const uint4*>(rowp + (size_t)(nh * hd + c * 8) * 2);
        }
      }
    }
    cw_sync();
    if (ct == 0) mbar_arrive(smem_u32(&s.empty[st]));
    ++ring;
  }
  return true;
}

// ARGMAX: (value, column) pairs where a larger value wins and equal values go to the lower
// column; a column < 0 marks "no number yet" and loses to any number (NaN entries are skipped).
__device__ __forceinline__ void argmax_take(float& bv, int& bi, float v, int i) {
  if (i >= 0 && (bi < 0 || v > bv || (v == bv && i < bi))) {
    bv = v;
    bi = i;
  }
}
__device__ __forceinline__ void argmax_warp(float& bv, int& bi) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const float v = __shfl_xor_sync(FULL, bv, o);
    const int i = __shfl_xor_sync(FULL, bi, o);
    argmax_take(bv, bi, v, i);
  }
}

// ARGMAX partial: rows [m0, m0 + tile_m) x columns [n0, n0 + klen) of x. Per row the largest
// value and the first column holding it go to the node's fp32 scratch as two floats at columns
// 2 * aux0 (a column as a float is exact below 2^24). A warp per row; each lane scans its
// 8-column vectors in increasing column order, four vectors in flight.
__device__ __forceinline__ void argmax_partial_body(const Instr& in, const Node& nd) {
  const int ct = (int)threadIdx.x - (kThreads - kCompute);
  const int wp = ct >> 5, lane = ct & 31;
  const int rows = min(nd.tile_m, nd.M - in.m0), dt = nd.dtype;
  const int c1 = in.n0 + in.klen;
  const uint16_t* x = reinterpret_cast<const uint16_t*>(nd.a.ptr);
  float* sc = reinterpret_cast<float*>(nd.scratch.ptr);
  for (int r = wp; r < rows; r += 4) {
    const uint16_t* row = x + (size_t)(in.m0 + r) * nd.a.ld;
    const bool vec = ((uintptr_t)row & 15u) == 0;  // 16-byte loads need an aligned row
    float bv = -INFINITY;
    int bi = -1;
    for (int v0 = in.n0 + lane * 8; v0 < c1; v0 += 4 * 256) {
      uint4 q[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int c = v0 + u * 256;
        if (c < c1 && vec && c + 8 <= c1) q[u] = __ldcg(reinterpret_cast<const uint4*>(row + c));
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int c = v0 + u * 256;
        if (c >= c1) continue;
        float f[8];
        if (vec && c + 8 <= c1) {
          unpack8(q[u], dt, f);
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) f[e] = c + e < c1 ? h2f(__ldcg(row + c + e), dt) : NAN;
        }
#pragma unroll
        for (int e = 0; e < 8; ++e)
          if (f[e] == f[e]) argmax_take(bv, bi, f[e], c + e);
      }
    }
    argmax_warp(bv, bi);
    if (lane == 0) {
      float* o = sc + (size_t)(in.m0 + r) * nd.scratch.ld + 2 * in.aux0;
      o[0] = bv;
      o[1] = (float)bi;
    }
  }
}

// ARGMAX reduce: per row of the block, the winner of the aux1 chunk partials, as int32 (-1 when
// the row holds no number).
__device__ __forceinline__ void argmax_reduce_body(const Instr& in, const Node& nd) {
  const int ct = (int)threadIdx.x - (kThreads - kCompute);
  const int wp = ct >> 5, lane = ct & 31;
  const int rows = min(nd.tile_m, nd.M - in.m0), C = in.aux1;
  const float* sc = reinterpret_cast<const float*>(nd.scratch.ptr);
  int32_t* out = reinterpret_cast<int32_t*>(nd.out.ptr);
  for (int r = wp; r < rows; r += 4) {
    const float* pr = sc + (size_t)(in.m0 + r) * nd.scratch.ld;
    float bv = -INFINITY;
    int bi = -1;
    for (int c = lane; c < C; c += 32) {
      const float2 vi = __ldcg(reinterpret_cast<const float2*>(pr + 2 * c));
      argmax_take(bv, bi, vi.x, (int)vi.y);
    }
    argmax_warp(bv, bi);
    if (lane == 0) out[(size_t)(in.m0 + r) * nd.out.ld] = bi;
  }
}

// Split-KV partial for kv group g = n0 and keys [k0, k0 + klen): per query head of the group
// m = max s, l = sum e^{s - m}, o = sum e^{s - m} v   (head_dim 64, up to 128 keys).
// Keys and values arrive by TMA in one ring stage, 128-byte swizzled (16-byte chunk c of row r
// sits at chunk c ^ (r & 7)).
__device__ __noinline__ bool attn_partial_body(const Params& p, Smem& s, const Instr& in,
                                               const Node& nd, uint32_t& ring, int idx) {
  const uint32_t NS = ring_n(p);
  const int ct = (int)threadIdx.x - (kThreads - kCompute);
  const int wp = ct >> 5, lane = ct & 31;
  const int g = in.n0, G = nd.hq / nd.hkv, C = in.aux1, c = in.aux0;
  const int kl = in.klen;
  const int st = (int)(ring % NS);
  // the query head's 64 values are in flight while the key/value chunk lands (a warp per head;
  // G <= 4 heads per key/value head keeps this one pass)
  uint4 qraw[8];
  if (wp < G) {
    const uint16_t* qp = reinterpret_cast<const uint16_t*>(nd.a.ptr) + (g * G + wp) * 64;
#pragma unroll
    for (int i = 0; i < 8; ++i) qraw[i] = __ldcg(reinterpret_cast<const uint4*>(qp + i * 8));
  }
  if (!cw_wait(p, smem_u32(&s.full[st]), (ring / NS) & 1u, 42, idx)) return false;
  const uint32_t kb = smem_u32(stage_ptr(s, p, st)), vb = kb + 16384;
  for (int hh = wp; hh < G; hh += 4) {
    const int h = g * G + hh;
    float qv[64];
    if (hh == wp) {
#pragma unroll
      for (int i = 0; i < 8; ++i) unpack8(qraw[i], DT_BF16, qv + i * 8);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) load8(nd.a, 0, h * 64 + i * 8, DT_BF16, qv + i * 8);
    }
    // scores: lane holds keys lane + 32t; each key's eight 16-byte chunks are loaded before its
    // dot product, which sums in four interleaved partial sums
    float sc[4], pr[4];
    float mx = -INFINITY;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int j = lane + 32 * t;
      float sv = -INFINITY;
      if (32 * t < kl) {
        uint4 kr[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          kr[i] = j < kl ? lds_u128(kb + j * 128 + ((i ^ (j & 7)) << 4)) : make_uint4(0, 0, 0, 0);
        float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          float kx[8];
          unpack8(kr[i], DT_BF16, kx);
#pragma unroll
          for (int e = 0; e < 8; ++e) d[e & 3] = fmaf(qv[i * 8 + e], kx[e], d[e & 3]);
        }
        if (j < kl) sv = ((d[0] + d[1]) + (d[2] + d[3])) * nd.scale;
      }
      sc[t] = sv;
      mx = fmaxf(mx, sv);
    }
    mx = warp_max(mx);
    float l = 0.f;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      pr[t] = (lane + 32 * t < kl) ? expf(sc[t] - mx) : 0.f;
      l += pr[t];
    }
    l = warp_sum(l);
    // lane owns value columns 2*lane, 2*lane+1: 16-byte chunk lane/4, 4-byte word lane%4; four
    // interleaved partial sums over the keys
    float oa[4][2];
#pragma unroll
    for (int u = 0; u < 4; ++u) oa[u][0] = oa[u][1] = 0.f;
    const int chunk = lane >> 2, word = lane & 3;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      if (32 * t >= kl) continue;
#pragma unroll 8
      for (int jj = 0; jj < 32; ++jj) {
        const int j = t * 32 + jj;
        const float pj = __shfl_sync(FULL, pr[t], jj);
        if (j < kl) {
          const uint32_t vv = lds_u32(vb + j * 128 + ((chunk ^ (j & 7)) << 4) + word * 4);
          oa[jj & 3][0] = fmaf(pj, __uint_as_float(vv << 16), oa[jj & 3][0]);
          oa[jj & 3][1] = fmaf(pj, __uint_as_float(vv & 0xffff0000u), oa[jj & 3][1]);
        }
      }
    }
    const float o0 = (oa[0][0] + oa[1][0]) + (oa[2][0] + oa[3][0]);
    const float o1 = (oa[0][1] + oa[1][1]) + (oa[2][1] + oa[3][1]);
    float* row = reinterpret_cast<float*>(nd.scratch.ptr) +
                 ((size_t)(g * C + c) * G + hh) * nd.scratch.ld;
    __stcg(reinterpret_cast<float2*>(row + lane * 2), make_float2(o0, o1));
    if (lane == 0) {
      __stcg(row + 64, mx);
      __stcg(row + 65, l);
    }
  }
  cw_sync();
  if (ct == 0) mbar_arrive(smem_u32(&s.empty[st]));
  ++ring;
  return true;
}

// LSE merge of one kv group's partials: M = max m_c, L = sum l_c e^{m_c-M},
// O = sum o_c e^{m_c-M} / L, one warp per query head. Up to 32 chunks: chunk c's statistics in
// lane c and every chunk's output pair of the lane's columns are loaded at once (one round trip
// to L2), the weights e^{m_c-M} broadcast by shuffles. More chunks: lanes stride over the
// chunks' statistics and value loads are batched by 8. Both sum in chunk order.
__device__ __noinline__ void attn_reduce_body(const Instr& in, const Node& nd) {
  const int ct = (int)threadIdx.x - (kThreads - kCompute);
  const int wp = ct >> 5, lane = ct & 31;
  const int g = in.n0, G = nd.hq / nd.hkv, C = in.aux1;
  const float* sc = reinterpret_cast<const float*>(nd.scratch.ptr);
  const int ld = nd.scratch.ld;
  for (int hh = wp; hh < G && C <= 32; hh += 4) {
    const int h = g * G + hh;
    auto row = [&](int c) { return sc + ((size_t)(g * C + c) * G + hh) * ld; };
    float mc = -INFINITY, lc = 0.f;
    if (lane < C) {
      mc = __ldcg(row(lane) + 64);
      lc = __ldcg(row(lane) + 65);
    }
    float2 ov[32];
#pragma unroll
    for (int u = 0; u < 32; ++u)
      ov[u] = u < C ? __ldcg(reinterpret_cast<const float2*>(row(u) + lane * 2))
                    : make_float2(0.f, 0.f);
    const float mx = warp_max(mc);
    const float w = lane < C ? expf(mc - mx) : 0.f;
    const float L = warp_sum(lc * w);
    float o0 = 0.f, o1 = 0.f;
#pragma unroll
    for (int u = 0; u < 32; ++u) {
      const float wu = __shfl_sync(FULL, w, u);
      if (u < C) {
        o0 = fmaf(ov[u].x, wu, o0);
        o1 = fmaf(ov[u].y, wu, o1);
      }
    }
    const float inv = 1.0f / L;
    const __nv_bfloat162 y = __floats2bfloat162_rn(o0 * inv, o1 * inv);
    *reinterpret_cast<__nv_bfloat162*>(reinterpret_cast<__nv_bfloat16*>(nd.out.ptr) + h * 64 +
                                       lane * 2) = y;
  }
  for (int hh = wp; hh < G && C > 32; hh += 4) {
    const int h = g * G + hh;
    auto row = [&](int c) { return sc + ((size_t)(g * C + c) * G + hh) * ld; };
    float mx = -INFINITY;
    for (int c = lane; c < C; c += 32) mx = fmaxf(mx, __ldcg(row(c) + 64));
    mx = warp_max(mx);
    float L = 0.f;
    for (int c = lane; c < C; c += 32) L += __ldcg(row(c) + 65) * expf(__ldcg(row(c) + 64) - mx);
    L = warp_sum(L);
    float o0 = 0.f, o1 = 0.f;
    for (int c0 = 0; c0 < C; c0 += 8) {
      float2 ov[8];
      float mv[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (c0 + u < C) {
          ov[u] = __ldcg(reinterpret_cast<const float2*>(row(c0 + u) + lane * 2));
          mv[u] = __ldcg(row(c0 + u) + 64);
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (c0 + u < C) {
          const float w = expf(mv[u] - mx);
          o0 = fmaf(ov[u].x, w, o0);
          o1 = fmaf(ov[u].y, w, o1);
        }
      }
    }
    const float inv = 1.0f / L;
    const __nv_bfloat162 y = __floats2bfloat162_rn(o0 * inv, o1 * inv);
    *reinterpret_cast<__nv_bfloat162*>(reinterpret_cast<__nv_bfloat16*>(nd.out.ptr) + h * 64 +
                                       lane * 2) = y;
  }
}

// Prefill attention, compute side: thread t of the warpgroup owns query row m0 + t (TMEM lane t).
// Per key block j: S_j from TMEM, scaled to the log2 domain and masked (key beyond the causal
// limit of the row or beyond the instruction's key range); P_j = 2^(s - m) as bf16 into shared
// memory for the P V MMA, which accumulates the output in TMEM; l sums the unrounded P. The
// maximum m in use only moves when a block's maximum exceeds it by more than 8 (log2 units):
// then l and the row of O in TMEM are rescaled by 2^(m_old - m_new) (flash attention's rescale,
// taken lazily: P stays <= 2^8, and O / l does not depend on which m was used). A warp rescales
// its rows only when one of its lanes needs it. At the end the row of O is read once, divided by
// l and stored as bf16. `n` counts attention blocks on this SM, as in the MMA warp.
template <bool PAIR>
__device__ __noinline__ bool attn_prefill_body(const Params& p, Smem& s, const Instr& in,
                                               const Node& nd, uint32_t tmem, uint32_t& n,
                                               uint32_t ring, int slot, uint32_t use, int idx) {
  const int ct = (int)threadIdx.x - (kThreads - kCompute);
  const int lane = ct & 31;
  const uint32_t lanes = (uint32_t)((ct >> 5) * 32) << 16;  // this warp's TMEM lane quarter
  const uint32_t otm = tmem + 128u + lanes;                   // this warp's rows of O
  const int nb = ring_stages(in);
  // on a CTA pair rank r runs rows 128r.. of the 256-row tile; the even CTA issues the MMAs and
  // its barriers count both CTAs' warps
  const int row = in.m0 + (PAIR ? (int)cluster_ctarank() * kAttnTileQ : 0) + ct;
  auto arrive_mma = [&](uint64_t& bar) {
    if (PAIR)
      mbar_arrive_cluster(mapa_shared(smem_u32(&bar), 0));
    else
      mbar_arrive(smem_u32(&bar));
  };
  if (PAIR && nb > 0) {
    // this CTA's query rows into xr for the whole instruction, counted on the even CTA's
    // barrier, once the sources are complete (earlier uses of xr by this warpgroup are
    // finished: its generic writes are fenced first)
    if (!cw_wait(p, smem_u32(&s.deps_ready[slot]), use & 1u, 45, idx)) return false;
    fence_proxy_async_shared();
    cw_sync();
    if (ct == 0) {
      fence_proxy_async_global();  // the producers' stores before this copy reads them
      const uint32_t bar = smem_u32(&s.att_q_full);
      if (cluster_ctarank() == 0) mbar_expect_tx(bar, 2u * 16384u);
      tma_load_2d_pair(smem_u32(s.xr), tmap_at(p, nd.a.tmap), mapa_shared(bar, 0), in.n0 * 64,
                       row - ct);
    }
  }
  const uint32_t NS = ring_n(p), sb = stage_bytes(p);
  const int qpos = nd.pos0 + row;
  const int kmax = in.klen;
  const float sl2 = nd.scale * 1.4426950408889634f;  // scores in log2 units
  float m = -INFINITY, l = 0.f;
  const uint32_t n0 = n;
  // Every barrier here takes one arrival per warp and nothing in the body synchronises the
  // warpgroup, so each warp waits on its own (bounded): warps do not run in lockstep, and one
  // whose wait gives up returns while the others' waits end by the same limit.
  // P V of block nn has completed: the P buffer is free and O holds blocks up to nn
  auto o_done = [&](uint32_t nn) -> bool {
    if (!wait_warp(p, smem_u32(&s.att_o_full[nn & 1u]), (nn >> 1) & 1u, R_COMPUTE, 44, idx))
      return false;
    tc_fence_after();
    return true;
  };
  for (int j = 0; j < nb; ++j) {
    const uint32_t nn = n0 + (uint32_t)j, b = nn & 1u;
    if (!wait_warp(p, smem_u32(&s.att_s_full[b]), (nn >> 1) & 1u, R_COMPUTE, 43, idx))
      return false;
    tc_fence_after();
    uint32_t r0[32], r1[32];
    tmem_ld32(tmem + b * 64u + lanes, r0);
    tmem_ld32(tmem + b * 64u + 32u + lanes, r1);
    tmem_ld_wait();
    tc_fence_before();
    __syncwarp();
    // pair: no arrival here (the even CTA's MMA infers it from P_j, below)
    if (!PAIR && lane == 0) arrive_mma(s.att_s_free[b]);
    const int key0 = j * kAttnKeyBlock;
    const int lim = nd.causal ? min(kmax, qpos + 1) : kmax;  // keys [0, lim) are visible
    // raw scores; masked keys only in a block that reaches the row's limit
    float x[64];
#pragma unroll
    for (int c = 0; c < 64; ++c) x[c] = __uint_as_float(c < 32 ? r0[c] : r1[c - 32]);
    if (key0 + 64 > lim) {
#pragma unroll
      for (int c = 0; c < 64; ++c)
        if (key0 + c >= lim) x[c] = -INFINITY;
    }
    float mx4[4] = {x[0], x[1], x[2], x[3]};
#pragma unroll
    for (int c = 4; c < 64; ++c) mx4[c & 3] = fmaxf(mx4[c & 3], x[c]);
    // the scale is positive: the maximum of the scaled scores is the scaled maximum
    const float mj = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])) * sl2;
    const bool need = mj > m + 8.f;          // false while no key is visible (mj = -inf)
    const float mn = need ? mj : m;
    const float alpha = need ? ex2(m - mn) : 1.f;
    const float mo = mn == -INFINITY ? 0.f : mn;  // masked scores give 2^-inf = 0 either way
    float ls4[4] = {0.f, 0.f, 0.f, 0.f};
    uint4 pk[8];
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) {
      float pv[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        pv[e] = ex2(fmaf(x[ch * 8 + e], sl2, -mo));
        ls4[e & 3] += pv[e];
      }
      uint32_t w[4];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const __nv_bfloat162 t = __floats2bfloat162_rn(pv[2 * h], pv[2 * h + 1]);
        w[h] = *reinterpret_cast<const uint32_t*>(&t);
      }
      pk[ch] = make_uint4(w[0], w[1], w[2], w[3]);
    }
    const float ls = (ls4[0] + ls4[1]) + (ls4[2] + ls4[3]);
    l = fmaf(l, alpha, ls);
    m = mn;
    // P_j has a buffer of its own (in the block's stage), so O is waited for only to rescale it
    const bool rescale = __any_sync(FULL, need);
    if (j > 0 && rescale) {
      if (!o_done(nn - 1u)) return false;
      {  // rescale this warp's rows of O (alpha = 1 where not needed)
        uint32_t o0[32], o1[32];
        tmem_ld32(otm, o0);
        tmem_ld32(otm + 32u, o1);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          o0[i] = __float_as_uint(__uint_as_float(o0[i]) * alpha);
          o1[i] = __float_as_uint(__uint_as_float(o1[i]) * alpha);
        }
        tmem_st32(otm, o0);
        tmem_st32(otm + 32u, o1);
        tmem_st_wait();
      }
    }
    if (PAIR) {
      // P_j into the block's stage for the even CTA's pair MMA
      uint8_t* Pj = s.ring + (size_t)((ring + (uint32_t)j) % NS) * sb + 8192;
#pragma unroll
      for (int ch = 0; ch < 8; ++ch)
        *reinterpret_cast<uint4*>(Pj + ct * 128 + ((ch ^ (ct & 7)) << 4)) = pk[ch];
      fence_proxy_async_all();
    } else {
      // P_j into TMEM (this thread's row, two keys per column), in the buffer P V of block
      // nn - 2 read: that MMA is complete first
      if (nn >= 2u && !o_done(nn - 2u)) return false;
      uint32_t pw[32];
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) {
        pw[4 * ch] = pk[ch].x;
        pw[4 * ch + 1] = pk[ch].y;
        pw[4 * ch + 2] = pk[ch].z;
        pw[4 * ch + 3] = pk[ch].w;
      }
      tmem_st32(tmem + kAttnPCol + b * 32u + lanes, pw);
      tmem_st_wait();
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) arrive_mma(s.att_p_full[b]);
  }
  n = n0 + (uint32_t)nb;
  if (nb == 0) return true;
  const uint32_t nl = n0 + (uint32_t)nb - 1u;
  if (!o_done(nl)) return false;
  uint32_t o0[32], o1[32];
  tmem_ld32(otm, o0);
  tmem_ld32(otm + 32u, o1);
  tmem_ld_wait();
  // the tile's TMEM may be reused once the warps (of both CTAs) have read O
  tc_fence_before();
  __syncwarp();
  if (lane == 0) arrive_mma(s.att_done);
  if (row < nd.M) {
    const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) {
      float v[8];
#pragma unroll
      for (int e = 0; e < 8; ++e)
        v[e] = __uint_as_float(ch < 4 ? o0[ch * 8 + e] : o1[ch * 8 - 32 + e]) * inv;
      store8(nd.out, row, in.n0 * 64 + ch * 8, DT_BF16, v);
    }
  }
  return true;
}

template <bool PAIR, int KS>
__device__ void run_compute(const Params& p, Smem& s, uint32_t tmem) {
  const uint32_t NS = ring_n(p);
  const int ct = (int)threadIdx.x - (kThreads - kCompute);
  uint32_t ring = 0, acc_n = 0, att_n = 0;
  bool synced = true;  // pair-mode ring sync (see load_gemm)
  for (int it = 0;; ++it) {
    const int slot = it % kSlots;
    const uint32_t use = (uint32_t)(it / kSlots);
    const int idx = instr_index(p, it);
    if (!cw_wait(p, smem_u32(&s.instr_ready[slot]), use & 1u, 32, idx)) break;
    const Instr& in = slot_instr(s, slot);
    if (in.op == OP_END) break;
    const Node& nd = slot_node(s, slot);
    if (p.trace && ct == 0) p.trace[(size_t)idx * kTraceWords + 0] = globaltimer();
    bool ok = true, publish = true;
    if (in.op != OP_GEMM && in.op != OP_ATTN_PREFILL) synced = false;
    switch (in.op) {
      case OP_GEMM:
        if constexpr (ks_has_gemm(KS)) {
          if (PAIR && !synced) ring = ring_align(ring, NS);  // mirrors the loader's ring sync
          if (ring_stages(in) > 0) synced = true;
          ok = gemm_epilogue<PAIR, KS>(p, s, in, nd, slot, use, tmem, acc_n, &publish, idx);
          ring += (uint32_t)ring_stages(in);
        }
        break;
      case OP_GEMV:
        if constexpr (ks_has_gemv(KS))
          ok = gemv<PAIR>(p, s, in, nd, slot, use, ring, &publish, idx, tmem, acc_n);
        break;
      case OP_NOOP:
        break;
      case OP_ATTN_PARTIAL:
        if constexpr (ks_has_gemv(KS)) {
          ok = cw_wait(p, smem_u32(&s.deps_ready[slot]), use & 1u, 33, idx);
          trace_mark(p, idx, 2);
          ok = ok && attn_partial_body(p, s, in, nd, ring, idx);
          trace_mark(p, idx, 6);
          if (ok && (nd.flags & NF_ATTN_FUSED)) {
            // the last partial of the key/value head to finish combines the head's partials
            cw_sync();
            if (ct == 0) {
              fence_acq_rel_gpu();
              s.flag = atomicAdd(p.counters + in.sem, 1) == in.aux1 - 1;
              fence_acq_rel_gpu();
            }
            cw_sync();
            trace_mark(p, idx, 7);
            if (s.flag) {
              attn_reduce_body(in, nd);
            } else {
              publish = false;
            }
          }
        }
        break;
      case OP_ATTN_PREFILL:
        if constexpr (ks_has_attn_prefill(KS)) {
          if (PAIR && !synced) ring = ring_align(ring, NS);  // mirrors the loader's ring sync
          if (ring_stages(in) > 0) synced = true;
          // inputs reach this warpgroup only through the loader and the MMAs, which wait
          trace_mark(p, idx, 2);
          ok = attn_prefill_body<PAIR>(p, s, in, nd, tmem, att_n, ring, slot, use, idx);
          ok = bar_and(kBarCompute, kCompute, ok);  // its warps waited on their own
          ring += (uint32_t)ring_stages(in);
        }
        break;
      default:
        ok = cw_wait(p, smem_u32(&s.deps_ready[slot]), use & 1u, 33, idx);
        if (!ok) break;
        trace_mark(p, idx, 2);
        if (ks_stages_rows(KS) && in.op == OP_RMSNORM && in.pad > 0)
          ok = rows_staged<false>(p, s, in, nd, ring, idx);
        else if (ks_stages_rows(KS) && in.op == OP_ROPE && in.pad > 0)
          ok = rows_staged<true>(p, s, in, nd, ring, idx);
        else if (ks_has_rows(KS) && in.op == OP_EW) ew_body(in, nd);
        else if (ks_has_rows(KS) && in.op == OP_RMSNORM) rmsnorm_body(in, nd);
        else if (ks_has_rows(KS) && in.op == OP_ROPE) rope_body(in, nd);
        else if (ks_has_gemv(KS) && in.op == OP_ATTN_REDUCE) attn_reduce_body(in, nd);
        else if (ks_has_rows(KS) && in.op == OP_ARGMAX) argmax_partial_body(in, nd);
        else if (ks_has_rows(KS) && in.op == OP_ARGMAX_REDUCE) argmax_reduce_body(in, nd);
        else {
          if (ct == 0) report(p, MK_ERR_DEVICE_CHECK, idx, -1, in.op, 0, R_COMPUTE, 34);
          ok = false;
        }
        break;
    }
    if (!ok) break;
    trace_mark(p, idx, 3);
    // Publish: the barrier orders every thread's stores before the first thread's release
    // (release is cumulative). One counter: a release increment. More: the first warp loads
    // the counter ids together, then one release fence and relaxed increments (a release
    // increment each would wait on the last).
    cw_sync();
    if (ct < 32 && publish && in.n_dst > 1) {
      if (ct == 0) {
        fence_proxy_async_global();
        fence_acq_rel_gpu();
      }
      for (int j0 = 0; j0 < in.n_dst; j0 += 32) {
        const int n = min(32, in.n_dst - j0);
        const int c = ct < n ? __ldg(p.dst_list + in.dst_off + j0 + ct) : 0;
        for (int k = 0; k < n; ++k) {
          const int ck = __shfl_sync(FULL, c, k);
          if (ct == 0) red_relaxed_add(p.counters + ck, 1);
        }
      }
    }
    if (ct == 0) {
      if (publish && in.n_dst == 1) {
        fence_proxy_async_global();
        red_release_add(p.counters + __ldg(p.dst_list + in.dst_off), 1);
      }
      if (p.trace) {
        p.trace[(size_t)idx * kTraceWords + 4] = globaltimer();
        p.trace[(size_t)idx * kTraceWords + 5] = blockIdx.x;
      }
      mbar_arrive(smem_u32(&s.slot_free[slot]));
    }
  }
}

// ------------------------------------------------------------------ the kernel

template <bool PAIR, int KS>
__global__ void __launch_bounds__(kThreads, 1) megakernel(const __grid_constant__ Params p) {
  extern __shared__ uint8_t smem_raw[];
  Smem& s = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                     ~static_cast<uintptr_t>(1023));
  const int warp = (int)threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kMaxStages; ++i) {
      mbar_init(smem_u32(&s.full[i]), 1);
      mbar_init(smem_u32(&s.empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&s.acc_full[i]), 1);
      mbar_init(smem_u32(&s.acc_empty[i]), PAIR ? 2 : 1);  // both epilogues of a pair
    }
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(smem_u32(&s.instr_ready[i]), 1);
      mbar_init(smem_u32(&s.deps_ready[i]), 1);
      mbar_init(smem_u32(&s.slot_free[i]), 3);  // loader, MMA issuer, compute warpgroup
    }
    mbar_init(smem_u32(&s.drain), 1);
    mbar_init(smem_u32(&s.go), 1);
    mbar_init(smem_u32(&s.gx_full), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&s.att_s_full[i]), 1);   // tcgen05.commit
      mbar_init(smem_u32(&s.att_s_free[i]), PAIR ? 8 : 4);  // a lane per compute warp (both CTAs)
      mbar_init(smem_u32(&s.att_o_full[i]), 1);
    }
    for (int i = 0; i < 2; ++i) mbar_init(smem_u32(&s.att_p_full[i]), PAIR ? 8 : 4);
    mbar_init(smem_u32(&s.att_q_full), 1);
    mbar_init(smem_u32(&s.att_done), PAIR ? 8 : 4);  // a lane per compute warp (both CTAs)
    mbar_fence_init();
  }
  if (ks_has_tmem(KS) && warp == 2) {
    if (PAIR) {
      tmem_alloc_pair(smem_u32(&s.tmem_base), 512);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(&s.tmem_base), 512);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync();  // the peer's barriers are initialised before any remote arrive
  tc_fence_after();
  const uint32_t tmem = ks_has_tmem(KS) ? s.tmem_base : 0u;

  if (warp == 0) {
    run_scheduler<KS>(p, s);
  } else if (warp == 1) {
    run_loader<PAIR, KS>(p, s);
  } else if (warp == 2) {
    run_mma<PAIR, KS>(p, s, tmem);
  } else if (warp >= 4) {
    run_compute<PAIR, KS>(p, s, tmem);
  }

  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync();  // neither CTA leaves while its peer may still address it
  if (ks_has_tmem(KS) && warp == 2) {
    tc_fence_after();
    if (PAIR)
      tmem_dealloc_pair(tmem, 512);
    else
      tmem_dealloc(tmem, 512);
  }
  // The CTA that finishes last (after every other CTA's work, including a drained abort)
  // publishes the run's status and zeroes the counters, so the next run needs no host reset.
  if (threadIdx.x == 0) {
    __threadfence();
    s.flag = atomicAdd(p.done, 1) == (int)gridDim.x - 1;
  }
  __syncthreads();
  if (s.flag) {
    __threadfence();
    for (int i = threadIdx.x; i < p.n_counters; i += kThreads) {
      const int v = __ldcg(p.counters + i);
      if (p.snapshot) p.snapshot[i] = v;
      p.counters[i] = 0;
    }
    // the run's status joins the record the host reads unless that already holds an unread
    // failure (the first failure since the last read is kept)
    int prev = 0;
    if (threadIdx.x < kStatusWords) prev = __ldcg(p.last_status + ST_CODE);
    __syncthreads();
    if (threadIdx.x < kStatusWords) {
      if (prev == 0) p.last_status[threadIdx.x] = __ldcg(p.status + threadIdx.x);
      p.status[threadIdx.x] = 0;
    }
    if (threadIdx.x == 0) *p.done = 0;
  }
}

}  // namespace

// ------------------------------------------------------------------ host launch stubs

// The host entry points of one specialisation; each translation unit that instantiates a
// specialisation returns them from a plain function (variant_*), the dispatcher picks one.
struct KernelVariant {
  cudaError_t (*configure)(size_t smem);
  cudaError_t (*launch)(const Params& p, int grid, size_t smem, cudaStream_t stream);
  cudaError_t (*clusters_resident)(size_t smem, int* n);  // 2-CTA clusters resident at once
};

template <bool PAIR, int KS>
cudaError_t configure_variant(size_t smem) {
  return cudaFuncSetAttribute(megakernel<PAIR, KS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)smem);
}

template <bool PAIR, int KS>
cudaError_t clusters_resident_variant(size_t smem, int* n) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(n, megakernel<PAIR, KS>, &cfg);
}

template <bool PAIR, int KS>
cudaError_t launch_variant(const Params& p, int grid, size_t smem, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  if (PAIR) {
    // 2-CTA clusters; co-residency of the whole grid is checked at compile time
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
  } else {
    attr[0].id = cudaLaunchAttributeCooperative;  // all CTAs co-resident (they wait on each other)
    attr[0].val.cooperative = 1;
  }
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, megakernel<PAIR, KS>, p);
}

template <bool PAIR, int KS>
KernelVariant make_variant() {
  return {&configure_variant<PAIR, KS>, &launch_variant<PAIR, KS>,
          &clusters_resident_variant<PAIR, KS>};
}

KernelVariant variant_all(bool pair);
KernelVariant variant_gemm(bool pair);
KernelVariant variant_decode();
KernelVariant variant_prefill(bool pair);
KernelVariant variant_prefill_pair();

}  // namespace mk
