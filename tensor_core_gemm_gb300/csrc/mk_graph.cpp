// Graph construction, validation and the compiler's lowering: ops -> tile instructions ->
// dependency counters -> static per-SM placement. No CUDA here; this file also builds the
// plans that dry-run tests inspect on a machine without a GPU.
//
// Lowering follows "MegaKittens Internals" §04 (phase 1: contiguous per-node ranges rounded to
// the cluster size with Noops; phase 3: a consumer waits on the producer instructions whose
// write boxes meet its read boxes, and each distinct (producer phase, set) is one counter whose
// target is the set size), §05 (instruction i -> SM i mod S, iteration i div S) and the task
// fan-out of "Implementing a Mega Kernel for B300" §2 (one GEMV task per column tile, one
// ATTENTION_PARTIAL per (kv group, chunk) followed by a combine).
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <map>

#include "mk_internal.h"

namespace mk {

static thread_local std::string g_err;

void set_error(const char* fmt, ...) {
  char buf[1024];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
}

int dtype_size(int dt) { return dt == DT_F32 || dt == DT_I32 ? 4 : 2; }
static bool half_type(int dt) { return dt == DT_F16 || dt == DT_BF16; }

static inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Window [r0,r1) x [c0,c1) of tensor/view `id`, clipped to it, in base coordinates.
static Box window(const std::vector<TensorRec>& ts, int id, int64_t r0, int64_t r1, int64_t c0,
                  int64_t c1) {
  const TensorRec& v = ts[id];
  Box b;
  b.t = v.base;
  r1 = std::min(r1, v.rows);
  c1 = std::min(c1, v.cols);
  b.r0 = v.r0 + r0;
  b.r1 = v.r0 + r1;
  b.c0 = v.c0 + c0;
  b.c1 = v.c0 + c1;
  return b;
}
static Box whole(const std::vector<TensorRec>& ts, int id) {
  return window(ts, id, 0, ts[id].rows, 0, ts[id].cols);
}

static HInstr make(uint16_t op, int node, int m0 = 0, int n0 = 0, int k0 = 0, int klen = 0,
                   int aux0 = 0, int aux1 = 0) {
  HInstr h;
  h.rec.op = op;
  h.rec.node = node;
  h.rec.m0 = m0;
  h.rec.n0 = n0;
  h.rec.k0 = k0;
  h.rec.klen = klen;
  h.rec.aux0 = aux0;
  h.rec.aux1 = aux1;
  return h;
}

// RoPE fusion: a ROPE node right after a matmul (no second weight) with head_dim 64 emits no
// instructions when either
//  - the matmul lowers to GEMV tiles, the rope input is exactly its output window and the
//    output width is a multiple of the GEMV tile width: split 0 of every GEMV column tile also
//    writes the rotated q / k (and v) columns it produced; or
//  - the matmul lowers to GEMM tiles without epilogue flags or a split tail, and the rope input
//    is the left part of its output window holding exactly the q, k (and, with out_v, v) heads:
//    every GEMM tile also writes the rotated q / k (and copied v) columns of its rows.
static bool same_window(const std::vector<TensorRec>& ts, int a, int b) {
  const TensorRec &x = ts[a], &y = ts[b];
  return x.base == y.base && x.r0 == y.r0 && x.c0 == y.c0 && x.rows == y.rows &&
         x.cols == y.cols;
}
static bool rope_fusable(const std::vector<TensorRec>& ts, const std::vector<NodeRec>& nodes,
                         int ri, const mk_compile_opts& o) {
  if (!o.fuse_rope || ri == 0 || nodes[ri].kind != NK_ROPE) return false;
  const NodeRec& r = nodes[ri];
  const NodeRec& p = nodes[ri - 1];
  if (p.kind != NK_MATMUL || p.b2 >= 0) return false;
  const int64_t m = ts[p.a].rows;
  if (m <= 0 || r.hd != 64) return false;
  if (m <= o.gemv_max_m)
    return same_window(ts, r.ins[0], p.out) && o.gemv_tile_n % 64 == 0 &&
           ts[p.out].cols % o.gemv_tile_n == 0;
  const TensorRec &x = ts[r.ins[0]], &y = ts[p.out];
  const int64_t w = (int64_t)(r.hq + r.hkv + (r.out_v >= 0 ? r.hkv : 0)) * r.hd;
  return p.flags == 0 && !o.gemm_split_tail && x.base == y.base && x.r0 == y.r0 &&
         x.c0 == y.c0 && x.rows == y.rows && x.cols == w && w <= y.cols;
}

// Boxes of the rope outputs that rows [r0, r1) and columns [c0, c1) of its input produce.
static void rope_writes(const std::vector<TensorRec>& ts, const NodeRec& rope, int64_t r0,
                        int64_t r1, int64_t c0, int64_t c1, std::vector<Box>& out) {
  const int64_t qend = (int64_t)rope.hq * 64, kend = (int64_t)(rope.hq + rope.hkv) * 64;
  if (c0 < qend) out.push_back(window(ts, rope.out, r0, r1, c0, std::min(c1, qend)));
  if (c1 > qend && c0 < kend)
    out.push_back(window(ts, rope.out_k, r0, r1, std::max(c0, qend) - qend,
                         std::min(c1, kend) - qend));
  if (rope.out_v >= 0 && c1 > kend)
    out.push_back(window(ts, rope.out_v, r0, r1, std::max(c0, kend) - kend, c1 - kend));
}

static void lower_matmul(const std::vector<TensorRec>& ts, int ni, const NodeRec& nd,
                         const mk_compile_opts& o, std::vector<std::vector<HInstr>>& phases,
                         int& n_tiles_sem, HostPlan* plan, const NodeRec* rope = nullptr) {
  const int64_t m = ts[nd.a].rows, k = ts[nd.a].cols, n = ts[nd.out].cols;
  const bool dual = nd.b2 >= 0;
  std::vector<HInstr> out;
  if (m == 0 || n == 0) {
    // nothing to compute
  } else if (m <= o.gemv_max_m) {
    const int64_t w = dual ? o.gemv_tile_n / 2 : o.gemv_tile_n;
    const int64_t nct = cdiv(n, w);
    int64_t s0 = o.gemv_splits > 0 ? o.gemv_splits : std::max<int64_t>(1, o.n_sm / nct);
    const int64_t chunk =
        std::max<int64_t>(o.gemv_kstep, cdiv(cdiv(k, s0), o.gemv_kstep) * o.gemv_kstep);
    const int64_t s = std::max<int64_t>(1, cdiv(k, chunk));
    plan->node_splits[ni] = (int)s;
    plan->node_tile_n[ni] = (int)w;
    for (int64_t ct = 0; ct < nct; ++ct) {
      const int64_t n0 = ct * w;
      const int tile = n_tiles_sem++;
      for (int64_t si = 0; si < s; ++si) {
        const int64_t k0 = si * chunk, kl = std::min(chunk, k - k0);
        HInstr h = make(OP_GEMV, ni, 0, (int)n0, (int)k0, (int)kl, (int)si, (int)s);
        h.tile = tile;
        if (nd.gamma >= 0) {
          h.reads.push_back({whole(ts, nd.a), ROLE_A});
          h.reads.push_back({whole(ts, nd.gamma), ROLE_A});
        } else {
          h.reads.push_back({window(ts, nd.a, 0, m, k0, k0 + kl), ROLE_A});
        }
        h.reads.push_back({window(ts, nd.b, k0, k0 + kl, n0, n0 + w), ROLE_B});
        if (dual) h.reads.push_back({window(ts, nd.b2, k0, k0 + kl, n0, n0 + w), ROLE_B});
        if (nd.bias >= 0) h.reads.push_back({window(ts, nd.bias, 0, m, n0, n0 + w), ROLE_E});
        if (nd.res >= 0) h.reads.push_back({window(ts, nd.res, 0, m, n0, n0 + w), ROLE_E});
        if (si == 0) {
          h.writes.push_back(window(ts, nd.out, 0, m, n0, n0 + w));
          if (rope) rope_writes(ts, *rope, 0, m, n0, n0 + w, h.writes);
        }
        out.push_back(std::move(h));
      }
    }
  } else {
    const int64_t tm = o.gemm_tile_m;
    const int64_t tn = dual ? o.gemm_tile_n / 2 : o.gemm_tile_n;
    const int cl = o.cluster;
    const int64_t rope_w =  // columns of the output a fused rope reads
        rope ? (int64_t)(rope->hq + rope->hkv + (rope->out_v >= 0 ? rope->hkv : 0)) * 64 : 0;
    plan->node_tile_n[ni] = (int)tn;
    // Split tail: the tiles of the last, partly filled wave (T mod units) are split along K
    // when at least two splits fit per tile; the last split to finish sums the partials.
    const int64_t nnt = cdiv(n, tn), t_all = cdiv(m, tm) * nnt;
    const int64_t units = o.n_sm / cl, nks = cdiv(k, kGemmBK);
    const int64_t r_tail = units > 0 ? t_all % units : 0;
    const int64_t n_split =
        (o.gemm_split_tail && r_tail) ? std::min<int64_t>(units / r_tail, nks) : 1;
    const int64_t split_from = n_split >= 2 ? t_all - r_tail : t_all;
    const int64_t chunk = n_split >= 2 ? cdiv(nks, n_split) * kGemmBK : k;
    const int64_t n_ranges = n_split >= 2 ? cdiv(k, chunk) : 1;
    int slots = 0;
    // Tile order: groups of gemm_group_m row tiles, column-major inside a group (consecutive
    // tiles share B panels and a group's A panels stay in L2; "Hand-writing a Blackwell GEMM",
    // Experiments, "Threadblock swizzle"); 1 = row-major.
    const int64_t nmt = cdiv(m, tm), gm = std::max(1, o.gemm_group_m);
    for (int64_t t = 0; t < t_all; ++t) {
      const int64_t g = t / (gm * nnt), r = t % (gm * nnt);
      const int64_t rows_g = std::min(gm, nmt - g * gm);
      const int64_t m0 = (g * gm + r % rows_g) * tm, n0 = (r / rows_g) * tn;
      const bool split = t >= split_from;
      const int64_t nr = split ? n_ranges : 1;
      int base = -1, slot0 = 0;
      if (split) {
        base = n_tiles_sem;
        n_tiles_sem += cl;
        slot0 = slots;
        slots += (int)nr * cl;
      }
      for (int64_t si = 0; si < nr; ++si) {
        const int64_t k0 = split ? si * chunk : 0, kl = split ? std::min(chunk, k - k0) : k;
        for (int r = 0; r < cl; ++r) {
          HInstr h = make(OP_GEMM, ni, (int)m0, (int)n0, (int)k0, (int)kl, r,
                          split ? (int)nr : 0);
          if (split) {
            h.tile = base + r;
            h.rec.slot = slot0 + r;
            h.rec.split = (int)si;
          }
          h.reads.push_back({window(ts, nd.a, m0, m0 + tm, k0, k0 + kl), ROLE_A});
          h.reads.push_back({window(ts, nd.b, k0, k0 + kl, n0, n0 + tn), ROLE_B});
          if (dual) h.reads.push_back({window(ts, nd.b2, k0, k0 + kl, n0, n0 + tn), ROLE_B});
          if (nd.bias >= 0)
            h.reads.push_back({window(ts, nd.bias, m0, m0 + tm, n0, n0 + tn), ROLE_E});
          if (nd.res >= 0)
            h.reads.push_back({window(ts, nd.res, m0, m0 + tm, n0, n0 + tn), ROLE_E});
          if (si == 0) {
            h.writes.push_back(window(ts, nd.out, m0, m0 + tm, n0, n0 + tn));
            if (rope) rope_writes(ts, *rope, m0, m0 + tm, n0, std::min<int64_t>(n0 + tn, rope_w),
                                  h.writes);
          }
          out.push_back(std::move(h));
        }
      }
    }
    plan->node_gsplit_slots[ni] = slots;
  }
  phases.push_back(std::move(out));
}

static void lower_ew(const std::vector<TensorRec>& ts, int ni, const NodeRec& nd,
                     const mk_compile_opts& o, std::vector<std::vector<HInstr>>& phases) {
  const int64_t rows = ts[nd.out].rows, cols = ts[nd.out].cols;
  const int64_t er = o.ew_rows, ew = (int64_t)o.ew_cols * o.ew_tiles;
  std::vector<HInstr> out;
  for (int64_t rt = 0; rt < cdiv(rows, er); ++rt) {
    for (int64_t ct = 0; ct < cdiv(cols, ew); ++ct) {
      const int64_t m0 = rt * er, n0 = ct * ew;
      HInstr h = make(OP_EW, ni, (int)m0, (int)n0, 0, 0, nd.ewop, 0);
      for (int i = 0; i < nd.n_in; ++i)
        h.reads.push_back({window(ts, nd.ins[i], m0, m0 + er, n0, n0 + ew), ROLE_E});
      h.writes.push_back(window(ts, nd.out, m0, m0 + er, n0, n0 + ew));
      out.push_back(std::move(h));
    }
  }
  phases.push_back(std::move(out));
}

static void lower_rows(const std::vector<TensorRec>& ts, int ni, const NodeRec& nd,
                       const mk_compile_opts& o, uint16_t op,
                       std::vector<std::vector<HInstr>>& phases) {
  const int x = nd.ins[0];
  const int64_t rows = ts[x].rows, nr = o.norm_rows;
  std::vector<int> outs;
  for (int id : {nd.out, nd.out_k, nd.out_v})
    if (id >= 0) outs.push_back(id);
  std::vector<HInstr> out;
  for (int64_t rt = 0; rt < cdiv(rows, nr); ++rt) {
    const int64_t m0 = rt * nr;
    HInstr h = make(op, ni, (int)m0);
    h.reads.push_back({window(ts, x, m0, m0 + nr, 0, ts[x].cols), ROLE_E});
    if (nd.gamma >= 0) h.reads.push_back({whole(ts, nd.gamma), ROLE_E});
    for (int id : outs) h.writes.push_back(window(ts, id, m0, m0 + nr, 0, ts[id].cols));
    out.push_back(std::move(h));
  }
  phases.push_back(std::move(out));
}

// ARGMAX of every row of x [R x C]: per block of norm_rows rows, one instruction per chunk of
// argmax_chunk columns writes the chunk's (largest value, first column holding it) of each row
// to an internal fp32 tensor [R x 2 * chunks] (the column as a float: exact below 2^24), then
// one instruction per row block picks the winner of the row's partials (ties: the lower
// column) and writes it as int32.
static void lower_argmax(std::vector<TensorRec>& ts, int ni, const NodeRec& nd,
                         const mk_compile_opts& o, std::vector<std::vector<HInstr>>& phases,
                         HostPlan* plan) {
  const int x = nd.ins[0];
  const int64_t rows = ts[x].rows, cols = ts[x].cols, nr = o.norm_rows;
  const int64_t ch = o.argmax_chunk, nc = cdiv(cols, ch);
  TensorRec s;
  s.dtype = DT_F32;
  s.rows = rows;
  s.cols = 2 * nc;
  s.ld = 2 * nc;
  s.base = (int)ts.size();
  s.internal = true;
  const int sid = s.base;
  ts.push_back(s);
  plan->node_scratch[ni] = sid;
  plan->node_chunks[ni] = (int)nc;
  std::vector<HInstr> part, red;
  for (int64_t rt = 0; rt < cdiv(rows, nr); ++rt) {
    const int64_t m0 = rt * nr;
    for (int64_t c = 0; c < nc; ++c) {
      HInstr h = make(OP_ARGMAX, ni, (int)m0, (int)(c * ch), 0, (int)std::min(ch, cols - c * ch));
      h.rec.aux0 = (int)c;
      h.reads.push_back({window(ts, x, m0, m0 + nr, c * ch, c * ch + ch), ROLE_E});
      h.writes.push_back(window(ts, sid, m0, m0 + nr, 2 * c, 2 * c + 2));
      part.push_back(std::move(h));
    }
    HInstr h = make(OP_ARGMAX_REDUCE, ni, (int)m0);
    h.rec.aux1 = (int)nc;
    h.reads.push_back({window(ts, sid, m0, m0 + nr, 0, 2 * nc), ROLE_E});
    h.writes.push_back(window(ts, nd.out, m0, m0 + nr, 0, 1));
    red.push_back(std::move(h));
  }
  phases.push_back(std::move(part));
  phases.push_back(std::move(red));
}

static void lower_attention(std::vector<TensorRec>& ts, int ni, const NodeRec& nd,
                            const mk_compile_opts& o, std::vector<std::vector<HInstr>>& phases,
                            int& n_tiles_sem, HostPlan* plan) {
  const int64_t hq = nd.hq, hkv = nd.hkv, d = nd.hd, g_sz = hq / hkv;
  const int64_t tq = ts[nd.a].rows, tk = ts[nd.b].rows;  // a = q, b = k, b2 = v
  if (tq == 1) {
    const int64_t ch = o.attn_chunk, nc = cdiv(tk, ch);
    TensorRec s;
    s.dtype = DT_F32;
    s.rows = hkv * nc * g_sz;
    s.cols = d + 2;
    s.ld = d + 2;
    s.base = (int)ts.size();
    s.internal = true;
    const int sid = s.base;
    ts.push_back(s);
    plan->node_scratch[ni] = sid;
    plan->node_chunks[ni] = (int)nc;
    std::vector<HInstr> part, red;
    // fused: the last partial of each key/value head combines the head's partials
    const bool fuse = o.fuse_attn_reduce != 0;
    for (int64_t g = 0; g < hkv; ++g) {
      const int tile = fuse ? n_tiles_sem++ : -1;
      for (int64_t c = 0; c < nc; ++c) {
        const int64_t k0 = c * ch, kl = std::min(ch, tk - k0);
        HInstr h = make(OP_ATTN_PARTIAL, ni, 0, (int)g, (int)k0, (int)kl, (int)c, (int)nc);
        h.tile = tile;
        h.reads.push_back({window(ts, nd.a, 0, 1, g * g_sz * d, (g + 1) * g_sz * d), ROLE_A});
        h.reads.push_back({window(ts, nd.b, k0, k0 + kl, g * d, (g + 1) * d), ROLE_B});
        h.reads.push_back({window(ts, nd.b2, k0, k0 + kl, g * d, (g + 1) * d), ROLE_B});
        const int64_t r0 = (g * nc + c) * g_sz;
        h.writes.push_back(window(ts, sid, r0, r0 + g_sz, 0, d + 2));
        if (fuse && c == 0)
          h.writes.push_back(window(ts, nd.out, 0, 1, g * g_sz * d, (g + 1) * g_sz * d));
        part.push_back(std::move(h));
      }
    }
    if (fuse) {
      phases.push_back(std::move(part));
      return;
    }
    for (int64_t g = 0; g < hkv; ++g) {
      HInstr h = make(OP_ATTN_REDUCE, ni, 0, (int)g, 0, 0, 0, (int)nc);
      const int64_t r0 = g * nc * g_sz;
      h.reads.push_back({window(ts, sid, r0, r0 + nc * g_sz, 0, d + 2), ROLE_E});
      h.writes.push_back(window(ts, nd.out, 0, 1, g * g_sz * d, (g + 1) * g_sz * d));
      red.push_back(std::move(h));
    }
    phases.push_back(std::move(part));
    phases.push_back(std::move(red));
  } else {
    // Query tiles of attn_tile_q rows, or on CTA pairs of cluster x attn_tile_q rows with one
    // instruction per rank (aux0), each carrying the whole cluster tile's boxes.
    const int cl = o.cluster;
    const int64_t tt = o.attn_tile_q * cl;
    std::vector<HInstr> out;
    for (int64_t t = cdiv(tq, tt) - 1; t >= 0; --t) {
      const int64_t m0 = t * tt;
      const int64_t kmax = nd.causal ? std::min(tk, (int64_t)nd.pos0 + m0 + tt) : tk;
      for (int64_t h = 0; h < hq; ++h) {
        const int64_t g = h / g_sz;
        for (int r = 0; r < cl; ++r) {
          HInstr hi = make(OP_ATTN_PREFILL, ni, (int)m0, (int)h, 0, (int)kmax, r, 0);
          hi.reads.push_back({window(ts, nd.a, m0, m0 + tt, h * d, (h + 1) * d), ROLE_E});
          hi.reads.push_back({window(ts, nd.b, 0, kmax, g * d, (g + 1) * d), ROLE_E});
          hi.reads.push_back({window(ts, nd.b2, 0, kmax, g * d, (g + 1) * d), ROLE_E});
          hi.writes.push_back(window(ts, nd.out, m0, m0 + tt, h * d, (h + 1) * d));
          out.push_back(std::move(hi));
        }
      }
    }
    phases.push_back(std::move(out));
  }
}

// Wave packing. A run of consecutive phases of one kind, none reading what an earlier phase of
// the run writes, is placed as one phase: GEMM phases without split tails (runs of two or more;
// cost of a tile = K length x B operands) or causal prefill attention phases (runs of one or
// more; cost = keys). Its cluster groups (the `cluster` instructions of a tile), stably sorted by
// cost longest first, each go to the unit (CTA, or CTA pair) with the least cost so far (the
// lowest unit on ties), and the run is laid out row by row, row r holding every unit's r-th group
// in unit order (Noops where a unit has none; trailing Noops dropped), so that with instruction i
// on SM i mod n_sm every group runs on its unit. Equal costs reproduce the tiles' own order.
static void pack_waves(std::vector<std::vector<HInstr>>& phases, const mk_compile_opts& o) {
  const int cl = o.cluster, units = o.n_sm / cl;
  if (units <= 0) return;
  // 1: GEMM phase, 2: prefill attention phase, 0: neither
  auto kind = [&](const std::vector<HInstr>& ph) {
    if (ph.empty() || ph.size() % cl) return 0;
    bool gemm = true, attn = true;
    for (const HInstr& h : ph) {
      gemm = gemm && h.rec.op == OP_GEMM && h.rec.aux1 == 0;
      attn = attn && h.rec.op == OP_ATTN_PREFILL;
    }
    return gemm ? 1 : attn ? 2 : 0;
  };
  // bounding boxes of a phase's reads and writes, per base tensor
  auto bounds = [](const std::vector<HInstr>& ph, bool reads) {
    std::map<int, Box> bb;
    for (const HInstr& h : ph) {
      std::vector<Box> boxes;
      if (reads)
        for (const auto& r : h.reads) boxes.push_back(r.first);
      else
        boxes = h.writes;
      for (const Box& b : boxes) {
        if (b.empty()) continue;
        auto it = bb.find(b.t);
        if (it == bb.end()) {
          bb[b.t] = b;
        } else {
          Box& u = it->second;
          u.r0 = std::min(u.r0, b.r0);
          u.r1 = std::max(u.r1, b.r1);
          u.c0 = std::min(u.c0, b.c0);
          u.c1 = std::max(u.c1, b.c1);
        }
      }
    }
    return bb;
  };
  std::vector<std::vector<HInstr>> out;
  size_t i = 0;
  while (i < phases.size()) {
    const int k0 = kind(phases[i]);
    if (k0 == 0) {
      out.push_back(std::move(phases[i++]));
      continue;
    }
    size_t j = i + 1;
    std::map<int, Box> written = bounds(phases[i], false);
    while (j < phases.size() && kind(phases[j]) == k0) {
      bool dep = false;
      for (const auto& r : bounds(phases[j], true)) {
        auto w = written.find(r.first);
        if (w != written.end() && meets(w->second, r.second)) dep = true;
      }
      if (dep) break;
      for (const auto& w : bounds(phases[j], false)) {
        auto it = written.find(w.first);
        if (it == written.end()) {
          written[w.first] = w.second;
        } else {
          Box& u = it->second;
          u.r0 = std::min(u.r0, w.second.r0);
          u.r1 = std::max(u.r1, w.second.r1);
          u.c0 = std::min(u.c0, w.second.c0);
          u.c1 = std::max(u.c1, w.second.c1);
        }
      }
      ++j;
    }
    if (k0 == 1 && j - i < 2) {
      out.push_back(std::move(phases[i++]));
      continue;
    }
    std::vector<std::vector<HInstr>> groups;
    std::vector<int64_t> cost;
    for (size_t q = i; q < j; ++q)
      for (size_t g = 0; g < phases[q].size(); g += cl) {
        groups.emplace_back();
        for (int r = 0; r < cl; ++r) groups.back().push_back(std::move(phases[q][g + r]));
        int nb = 0;
        for (const auto& rd : groups.back()[0].reads) nb += rd.second == ROLE_B;
        cost.push_back((int64_t)groups.back()[0].rec.klen * (k0 == 1 ? nb : 1));
      }
    std::vector<size_t> order(groups.size());
    for (size_t g = 0; g < order.size(); ++g) order[g] = g;
    std::stable_sort(order.begin(), order.end(),
                     [&](size_t a, size_t b) { return cost[a] > cost[b]; });
    std::vector<int64_t> load(units, 0);
    std::vector<std::vector<size_t>> queue(units);
    for (size_t g : order) {
      int u = 0;
      for (int v = 1; v < units; ++v)
        if (load[v] < load[u]) u = v;
      load[u] += cost[g];
      queue[u].push_back(g);
    }
    size_t rows = 0;
    for (const auto& q : queue) rows = std::max(rows, q.size());
    std::vector<HInstr> run;
    for (size_t r = 0; r < rows; ++r)
      for (int u = 0; u < units; ++u) {
        if (r < queue[u].size()) {
          for (auto& h : groups[queue[u][r]]) run.push_back(std::move(h));
        } else {
          for (int k = 0; k < cl; ++k) run.push_back(make(OP_NOOP, 0));
        }
      }
    while (!run.empty() && run.back().rec.op == OP_NOOP) run.pop_back();
    out.push_back(std::move(run));
    i = j;
  }
  phases = std::move(out);
}

mk_status lower_graph(const std::vector<TensorRec>& tensors_in, const std::vector<NodeRec>& nodes,
                      const mk_compile_opts& o, HostPlan* plan) {
  if (o.n_sm <= 0 || o.cluster <= 0 || o.gemm_tile_m <= 0 || o.gemm_tile_n <= 0 ||
      o.ew_rows <= 0 || o.ew_cols <= 0 || o.ew_tiles <= 0 || o.norm_rows <= 0 ||
      o.gemv_tile_n <= 0 || o.gemv_kstep <= 0 || o.attn_chunk <= 0 || o.attn_tile_q <= 0 ||
      o.argmax_chunk <= 0 || o.argmax_chunk % 8) {
    set_error("mk_compile: every tile size and n_sm must be positive (argmax_chunk a multiple "
              "of 8)");
    return MK_ERR_INVALID_ARG;
  }
  std::vector<TensorRec> ts = tensors_in;
  const int nn = (int)nodes.size();
  plan->node_scratch.assign(nn, -1);
  plan->node_splits.assign(nn, 0);
  plan->node_chunks.assign(nn, 0);
  plan->node_tile_n.assign(nn, 0);
  plan->node_gsplit_slots.assign(nn, 0);
  plan->node_rope.assign(nn, -1);
  std::vector<char> fused(nn, 0);
  for (int ri = 0; ri < nn; ++ri)
    if (rope_fusable(ts, nodes, ri, o)) {
      fused[ri] = 1;
      plan->node_rope[ri - 1] = ri;
    }
  std::vector<std::vector<HInstr>> phases;
  int n_tiles_sem = 0;
  for (int ni = 0; ni < nn; ++ni) {
    const NodeRec& nd = nodes[ni];
    switch (nd.kind) {
      case NK_MATMUL:
        lower_matmul(ts, ni, nd, o, phases, n_tiles_sem, plan,
                     plan->node_rope[ni] >= 0 ? &nodes[plan->node_rope[ni]] : nullptr);
        break;
      case NK_EW: lower_ew(ts, ni, nd, o, phases); break;
      case NK_RMSNORM: lower_rows(ts, ni, nd, o, OP_RMSNORM, phases); break;
      case NK_ROPE:
        if (!fused[ni]) lower_rows(ts, ni, nd, o, OP_ROPE, phases);
        break;
      case NK_ATTN: lower_attention(ts, ni, nd, o, phases, n_tiles_sem, plan); break;
      case NK_ARGMAX: lower_argmax(ts, ni, nd, o, phases, plan); break;
      default: set_error("mk_compile: unknown node kind %d", nd.kind); return MK_ERR_INVALID_ARG;
    }
  }

  if (o.wave_pack) pack_waves(phases, o);

  // Phase 1: flatten, padding every phase to a multiple of the cluster size with Noops.
  std::vector<HInstr> ins;
  std::vector<int> phase_of;
  std::vector<std::pair<int, int>> ranges;
  for (size_t pi = 0; pi < phases.size(); ++pi) {
    const int start = (int)ins.size();
    for (auto& h : phases[pi]) ins.push_back(std::move(h));
    while ((ins.size() - start) % o.cluster) ins.push_back(make(OP_NOOP, 0));
    ranges.push_back({start, (int)ins.size()});
    phase_of.resize(ins.size(), (int)pi);
  }

  // Phase 3: write boxes per base tensor, grouped by phase in phase order.
  struct PhaseWrites {
    int phase;
    std::vector<std::pair<int, Box>> boxes;  // (instruction, box), instruction-ascending
  };
  std::vector<std::vector<PhaseWrites>> wtab(ts.size());
  for (size_t pi = 0; pi < ranges.size(); ++pi) {
    for (int i = ranges[pi].first; i < ranges[pi].second; ++i) {
      for (const Box& w : ins[i].writes) {
        auto& lst = wtab[w.t];
        if (lst.empty() || lst.back().phase != (int)pi) lst.push_back({(int)pi, {}});
        lst.back().boxes.push_back({i, w});
      }
    }
  }
  std::map<std::pair<int, std::vector<int>>, int> keys;
  std::vector<std::vector<int>> members;
  std::vector<int32_t> targets;
  std::vector<int> set;
  for (size_t ci = 0; ci < ins.size(); ++ci) {
    HInstr& c = ins[ci];
    for (const auto& rd : c.reads) {
      const Box& rb = rd.first;
      if (rb.empty()) continue;
      for (const PhaseWrites& pw : wtab[rb.t]) {
        if (pw.phase >= phase_of[ci]) break;
        set.clear();
        for (const auto& ib : pw.boxes)
          if (meets(rb, ib.second) && (set.empty() || set.back() != ib.first))
            set.push_back(ib.first);
        if (set.empty()) continue;
        auto key = std::make_pair(pw.phase, set);
        auto it = keys.find(key);
        int cid;
        if (it == keys.end()) {
          cid = (int)targets.size();
          keys.emplace(key, cid);
          targets.push_back((int32_t)set.size());
          members.push_back(set);
        } else {
          cid = it->second;
        }
        if (rd.second == ROLE_B &&
            (c.rec.op == OP_GEMM || c.rec.op == OP_GEMV || c.rec.op == OP_ATTN_PARTIAL))
          c.rec.flags |= IFLAG_B_DEP;
        bool seen = false;
        for (auto& s : c.src) seen |= (s.first == cid);
        if (!seen) c.src.push_back({cid, (int)set.size()});
      }
    }
  }
  for (size_t cid = 0; cid < members.size(); ++cid)
    for (int p : members[cid]) ins[p].dst.push_back((int)cid);
  const int n_dep = (int)targets.size();

  // Split tiles (GEMV tiles, GEMM split tails per rank) publish through whichever split finishes
  // last: all splits carry split 0's arrivals and share one semaphore, numbered after the
  // dependency counters.
  auto is_split = [](const HInstr& h) {
    return h.rec.op == OP_GEMV || (h.rec.op == OP_GEMM && h.rec.aux1 > 0) ||
           (h.rec.op == OP_ATTN_PARTIAL && h.tile >= 0);
  };
  std::vector<int> first_of_tile(n_tiles_sem, -1);
  for (size_t i = 0; i < ins.size(); ++i)
    if (is_split(ins[i]) && ins[i].rec.k0 == 0) first_of_tile[ins[i].tile] = (int)i;
  for (auto& h : ins) {
    if (!is_split(h)) continue;
    h.dst = ins[first_of_tile[h.tile]].dst;
    h.rec.sem = n_dep + h.tile;
  }

  // Buffer pool ("MegaKittens Internals" §04 phase 2, restated). Transient tensors (plan-owned
  // intermediates) are placed in node order of their writer. A transient takes a pooled buffer of
  // its exact shape and dtype when the writer's first instruction lies at least n_sm
  // instructions (pool_waves times that; one wave by default) past the end (last instruction +
  // 1) of every node that accessed the buffer's current occupant (the one-wave rule: the old
  // accesses sit earlier in every SM's queue); else
  // it gets a new buffer, the first of the equals that qualify being taken. The occupant's own
  // writer counts as an accessor, so a region no reader covered is also finished. Each reuse is
  // one counter, numbered after the dependency counters: every instruction of the accessor nodes
  // arrives on it (a split tile once), and every instruction of the new writer waits for the
  // total before it runs. A node fused into the one before it (a RoPE in its matmul's tiles)
  // has no instructions: its accesses count as accesses of that carrier node.
  {
    const int n_t = (int)tensors_in.size();
    plan->pool_off.assign(ts.size(), -1);
    plan->pool_bytes = 0;
    plan->n_reuse = 0;
    std::vector<int> first(nn, INT32_MAX), last(nn, -1);
    for (size_t i = 0; i < ins.size(); ++i) {
      if (ins[i].rec.op == OP_NOOP) continue;
      const int nd_i = ins[i].rec.node;
      first[nd_i] = std::min(first[nd_i], (int)i);
      last[nd_i] = std::max(last[nd_i], (int)i);
    }
    auto touches = [&](const NodeRec& nd, int base, bool write) {
      std::vector<int> ids;
      if (write) {
        ids = {nd.out, nd.out_k, nd.out_v};
      } else {
        ids = {nd.a, nd.b, nd.b2, nd.bias, nd.res, nd.gamma, nd.ins[0], nd.ins[1]};
      }
      for (int id : ids)
        if (id >= 0 && ts[id].base == base) return true;
      return false;
    };
    struct Occ {
      int tensor;
      std::vector<int> nodes;  // accessor nodes of the occupant
      bool pooled;
    };
    std::vector<Occ> buffers;
    std::vector<int64_t> buf_off, buf_bytes;
    std::vector<int> order;
    std::vector<int> writer(n_t, -1);
    auto carrier = [&](int ni) { return fused[ni] ? ni - 1 : ni; };
    for (int t = 0; t < n_t; ++t) {
      if (!ts[t].transient || ts[t].base != t) continue;
      for (int ni = 0; ni < nn && writer[t] < 0; ++ni)
        if (touches(nodes[ni], t, true)) writer[t] = carrier(ni);
      order.push_back(t);
    }
    std::stable_sort(order.begin(), order.end(), [&](int a, int b) {
      const int wa = writer[a] < 0 ? INT32_MAX : writer[a], wb = writer[b] < 0 ? INT32_MAX : writer[b];
      return wa < wb;
    });
    std::vector<std::pair<std::vector<int>, int>> events;  // (source nodes, writer node)
    for (int t : order) {
      std::vector<int> acc;
      bool ok = writer[t] >= 0;
      for (int ni = 0; ni < nn; ++ni)
        if (touches(nodes[ni], t, false) || touches(nodes[ni], t, true)) {
          const int c = carrier(ni);
          if (std::find(acc.begin(), acc.end(), c) == acc.end()) acc.push_back(c);
          ok = ok && last[c] >= 0;
        }
      const int64_t bytes =
          ((int64_t)ts[t].rows * ts[t].ld * dtype_size(ts[t].dtype) + 1023) & ~(int64_t)1023;
      int chosen = -1;
      if (ok) {
        const int start = first[writer[t]];
        for (size_t bi = 0; bi < buffers.size() && chosen < 0; ++bi) {
          const TensorRec& o_t = ts[buffers[bi].tensor];
          if (!buffers[bi].pooled || o_t.dtype != ts[t].dtype || o_t.rows != ts[t].rows ||
              o_t.cols != ts[t].cols)
            continue;
          bool free = true;
          for (int ni : buffers[bi].nodes)
            free = free && (int64_t)last[ni] + 1 + (int64_t)o.pool_waves * o.n_sm <= start;
          if (free) chosen = (int)bi;
        }
      }
      if (chosen >= 0) {
        events.push_back({buffers[chosen].nodes, writer[t]});
        buffers[chosen] = {t, acc, true};
      } else {
        chosen = (int)buffers.size();
        buffers.push_back({t, acc, ok});
        buf_off.push_back(plan->pool_bytes);
        buf_bytes.push_back(bytes);
        plan->pool_bytes += bytes;
      }
      plan->pool_off[t] = buf_off[chosen];
    }
    for (int t = 0; t < (int)ts.size(); ++t)  // views follow their base
      if (ts[t].transient && ts[t].base != t && plan->pool_off[ts[t].base] >= 0)
        plan->pool_off[t] = plan->pool_off[ts[t].base] +
                            ((ts[t].r0 - ts[ts[t].base].r0) * ts[t].ld + ts[t].c0 -
                             ts[ts[t].base].c0) * dtype_size(ts[t].dtype);
    for (const auto& ev : events) {
      const int cid = (int)targets.size();
      int32_t count = 0;
      std::vector<char> tile_seen(n_tiles_sem, 0);
      for (size_t i = 0; i < ins.size(); ++i) {
        if (ins[i].rec.op == OP_NOOP) continue;
        if (std::find(ev.first.begin(), ev.first.end(), ins[i].rec.node) == ev.first.end())
          continue;
        if (is_split(ins[i])) {
          if (!tile_seen[ins[i].tile]) ++count;
          tile_seen[ins[i].tile] = 1;
        } else {
          ++count;
        }
        ins[i].dst.push_back(cid);
      }
      targets.push_back(count);
      for (size_t i = 0; i < ins.size(); ++i)
        if (ins[i].rec.op != OP_NOOP && ins[i].rec.node == ev.second)
          ins[i].src.push_back({cid, count});
      ++plan->n_reuse;
    }
    if (!events.empty())  // the semaphores follow every dependency counter, reuse ones included
      for (auto& h : ins)
        if (is_split(h)) h.rec.sem = (int)targets.size() + h.tile;
  }

  // Pack.
  plan->instrs.clear();
  plan->src_list.clear();
  plan->dst_list.clear();
  for (auto& h : ins) {
    Instr r = h.rec;
    r.n_src = (int)h.src.size();
    r.src_off = (int)(plan->src_list.size() / 2);
    for (auto& s : h.src) {
      plan->src_list.push_back(s.first);
      plan->src_list.push_back(s.second);
    }
    r.n_dst = (int)h.dst.size();
    r.dst_off = (int)plan->dst_list.size();
    for (int d : h.dst) plan->dst_list.push_back(d);
    plan->instrs.push_back(r);
  }
  plan->targets = targets;
  plan->n_dep = (int)targets.size();
  plan->n_sem = n_tiles_sem;
  plan->n_sm = o.n_sm;
  plan->tensors = ts;
  return MK_OK;
}

}  // namespace mk

using namespace mk;

// ------------------------------------------------------------------ C ABI: graph building

extern "C" const char* mk_last_error(void) { return g_err.c_str(); }
extern "C" int32_t mk_abi_version(void) { return MK_ABI_VERSION; }

extern "C" mk_status mk_graph_create(mk_graph_t* out) {
  if (!out) {
    set_error("mk_graph_create: out is NULL");
    return MK_ERR_INVALID_ARG;
  }
  *out = new (std::nothrow) mk_graph();
  if (!*out) {
    set_error("mk_graph_create: out of host memory");
    return MK_ERR_OOM;
  }
  return MK_OK;
}

extern "C" mk_status mk_graph_destroy(mk_graph_t g) {
  delete g;
  return MK_OK;
}

static bool valid_tensor(const mk_graph* g, int id) {
  return id >= 0 && id < (int)g->tensors.size();
}

extern "C" mk_status mk_add_tensor(mk_graph_t g, void* dev_ptr, int32_t dtype, int32_t rank,
                                   const int64_t* shape, const int64_t* strides, int32_t* id) {
  if (!g || !shape || !id || rank < 1 || rank > 4) {
    set_error("mk_add_tensor: null argument or rank outside 1..4");
    return MK_ERR_INVALID_ARG;
  }
  if (dtype != MK_F16 && dtype != MK_BF16 && dtype != MK_F32 && dtype != MK_I32) {
    set_error("mk_add_tensor: unknown dtype %d", dtype);
    return MK_ERR_INVALID_ARG;
  }
  int64_t st[4];
  int64_t acc = 1;
  for (int i = rank - 1; i >= 0; --i) {
    if (shape[i] < 0) {
      set_error("mk_add_tensor: negative extent");
      return MK_ERR_INVALID_ARG;
    }
    st[i] = strides ? strides[i] : acc;
    acc *= std::max<int64_t>(shape[i], 1);
  }
  if (st[rank - 1] != 1) {
    set_error("mk_add_tensor: the innermost dimension must have stride 1");
    return MK_ERR_UNSUPPORTED;
  }
  for (int i = 0; i + 2 < rank; ++i) {
    if (shape[i] > 1 && st[i] != st[i + 1] * shape[i + 1]) {
      set_error("mk_add_tensor: outer dimensions must be contiguous over each other");
      return MK_ERR_UNSUPPORTED;
    }
  }
  TensorRec t;
  t.ptr = dev_ptr;
  t.dtype = dtype;
  t.cols = shape[rank - 1];
  t.rows = 1;
  for (int i = 0; i + 1 < rank; ++i) t.rows *= shape[i];
  t.ld = rank >= 2 ? st[rank - 2] : t.cols;
  if (t.ld < t.cols) {
    set_error("mk_add_tensor: row stride %lld smaller than the row length %lld",
              (long long)t.ld, (long long)t.cols);
    return MK_ERR_INVALID_ARG;
  }
  t.base = (int)g->tensors.size();
  g->tensors.push_back(t);
  *id = t.base;
  return MK_OK;
}

extern "C" mk_status mk_add_transient(mk_graph_t g, int32_t dtype, int64_t rows, int64_t cols,
                                      int32_t* id) {
  if (!g || !id || rows < 0 || cols < 0) {
    set_error("mk_add_transient: bad graph, id or extents");
    return MK_ERR_INVALID_ARG;
  }
  if (dtype != MK_F16 && dtype != MK_BF16 && dtype != MK_F32 && dtype != MK_I32) {
    set_error("mk_add_transient: unknown dtype %d", dtype);
    return MK_ERR_INVALID_ARG;
  }
  TensorRec t;
  t.dtype = dtype;
  t.rows = rows;
  t.cols = cols;
  const int64_t per16 = 16 / dtype_size(dtype);  // rows start 16-byte aligned
  t.ld = std::max<int64_t>((cols + per16 - 1) / per16 * per16, per16);
  t.base = (int)g->tensors.size();
  t.transient = true;
  *id = t.base;
  g->tensors.push_back(t);
  return MK_OK;
}

extern "C" mk_status mk_add_view(mk_graph_t g, int32_t base, int64_t r0, int64_t c0,
                                 int64_t rows, int64_t cols, int32_t* id) {
  if (!g || !id || !valid_tensor(g, base)) {
    set_error("mk_add_view: bad graph or tensor id");
    return MK_ERR_INVALID_ARG;
  }
  const TensorRec& b = g->tensors[base];
  if (r0 < 0 || c0 < 0 || rows < 0 || cols < 0 || r0 + rows > b.rows || c0 + cols > b.cols) {
    set_error("mk_add_view: window [%lld+%lld, %lld+%lld] outside the %lldx%lld tensor",
              (long long)r0, (long long)rows, (long long)c0, (long long)cols, (long long)b.rows,
              (long long)b.cols);
    return MK_ERR_INVALID_ARG;
  }
  TensorRec v = b;
  v.rows = rows;
  v.cols = cols;
  v.r0 = b.r0 + r0;
  v.c0 = b.c0 + c0;
  v.ptr = b.ptr ? (void*)((char*)b.ptr + (r0 * b.ld + c0) * dtype_size(b.dtype)) : nullptr;
  *id = (int)g->tensors.size();
  g->tensors.push_back(v);
  return MK_OK;
}

static bool same_shape(const mk_graph* g, int a, int64_t rows, int64_t cols) {
  return g->tensors[a].rows == rows && g->tensors[a].cols == cols;
}

extern "C" mk_status mk_add_matmul(mk_graph_t g, int32_t a, int32_t b, int32_t out,
                                   const mk_epilogue* epi, int32_t* node_id) {
  if (!g || !node_id || !valid_tensor(g, a) || !valid_tensor(g, b) || !valid_tensor(g, out)) {
    set_error("mk_add_matmul: bad graph, tensor id or node_id pointer");
    return MK_ERR_INVALID_ARG;
  }
  const TensorRec &A = g->tensors[a], &B = g->tensors[b], &C = g->tensors[out];
  const int64_t m = A.rows, k = A.cols, n = B.cols;
  if (B.rows != k || !same_shape(g, out, m, n)) {
    set_error("mk_add_matmul: shapes A %lldx%lld, B %lldx%lld, out %lldx%lld do not chain",
              (long long)A.rows, (long long)A.cols, (long long)B.rows, (long long)B.cols,
              (long long)C.rows, (long long)C.cols);
    return MK_ERR_INVALID_ARG;
  }
  if (!half_type(A.dtype) || B.dtype != A.dtype || C.dtype != A.dtype) {
    set_error("mk_add_matmul: A, B and out must share one dtype, f16 or bf16");
    return MK_ERR_UNSUPPORTED;
  }
  NodeRec nd;
  nd.kind = NK_MATMUL;
  nd.a = a;
  nd.b = b;
  nd.out = out;
  if (epi) {
    nd.flags = epi->flags;
    nd.eps = epi->eps;
    auto need = [&](uint32_t f, int id, int64_t rows, int64_t cols, const char* what) -> bool {
      if (!(nd.flags & f)) return true;
      if (!valid_tensor(g, id) || !same_shape(g, id, rows, cols) ||
          g->tensors[id].dtype != A.dtype) {
        set_error("mk_add_matmul: %s must be a %lldx%lld tensor of the operands' dtype", what,
                  (long long)rows, (long long)cols);
        return false;
      }
      return true;
    };
    if (!need(MK_EPI_BIAS, epi->bias, m, n, "bias") ||
        !need(MK_EPI_RESIDUAL, epi->residual, m, n, "residual") ||
        !need(MK_EPI_RMSNORM_INPUT, epi->gamma, 1, k, "gamma") ||
        !need(MK_EPI_SILU_MUL, epi->b_up, k, n, "b_up"))
      return MK_ERR_INVALID_ARG;
    if (nd.flags & ~(uint32_t)(MK_EPI_BIAS | MK_EPI_RELU | MK_EPI_RESIDUAL |
                              MK_EPI_RMSNORM_INPUT | MK_EPI_SILU_MUL)) {
      set_error("mk_add_matmul: unknown epilogue flag bits 0x%x", nd.flags);
      return MK_ERR_INVALID_ARG;
    }
    if (nd.flags & MK_EPI_BIAS) nd.bias = epi->bias;
    if (nd.flags & MK_EPI_RESIDUAL) nd.res = epi->residual;
    if (nd.flags & MK_EPI_RMSNORM_INPUT) nd.gamma = epi->gamma;
    if (nd.flags & MK_EPI_SILU_MUL) nd.b2 = epi->b_up;
  }
  *node_id = (int)g->nodes.size();
  g->nodes.push_back(nd);
  return MK_OK;
}

extern "C" mk_status mk_add_elementwise(mk_graph_t g, int32_t op, const int32_t* ins,
                                        int32_t n_in, int32_t out, const mk_ew_params* p,
                                        int32_t* node_id) {
  if (!g || !node_id || !ins || n_in < 1 || n_in > 2 || !valid_tensor(g, out)) {
    set_error("mk_add_elementwise: bad graph, inputs or output");
    return MK_ERR_INVALID_ARG;
  }
  for (int i = 0; i < n_in; ++i)
    if (!valid_tensor(g, ins[i])) {
      set_error("mk_add_elementwise: bad input tensor id %d", ins[i]);
      return MK_ERR_INVALID_ARG;
    }
  const TensorRec& O = g->tensors[out];
  NodeRec nd;
  nd.out = out;
  nd.n_in = n_in;
  nd.ins[0] = ins[0];
  if (n_in > 1) nd.ins[1] = ins[1];
  switch (op) {
    case MK_EW_ADD:
    case MK_EW_SILU_MUL:
    case MK_EW_RELU:
    case MK_EW_COPY: {
      const int want = (op == MK_EW_ADD || op == MK_EW_SILU_MUL) ? 2 : 1;
      if (n_in != want) {
        set_error("mk_add_elementwise: op %d takes %d inputs", op, want);
        return MK_ERR_INVALID_ARG;
      }
      for (int i = 0; i < n_in; ++i)
        if (!same_shape(g, ins[i], O.rows, O.cols) || g->tensors[ins[i]].dtype != O.dtype ||
            O.dtype == MK_I32) {
          set_error("mk_add_elementwise: inputs must match the output's shape and dtype "
                    "(no broadcasting)");
          return MK_ERR_INVALID_ARG;
        }
      nd.kind = NK_EW;
      nd.ewop = op;
      break;
    }
    case MK_EW_RMSNORM: {
      if (!p || n_in != 1 || !same_shape(g, ins[0], O.rows, O.cols) || !half_type(O.dtype) ||
          !valid_tensor(g, p->gamma) || !same_shape(g, p->gamma, 1, O.cols) ||
          g->tensors[ins[0]].dtype != O.dtype || g->tensors[p->gamma].dtype != O.dtype) {
        set_error("mk_add_elementwise: RMSNORM needs x and out of one shape and gamma 1 x cols");
        return MK_ERR_INVALID_ARG;
      }
      nd.kind = NK_RMSNORM;
      nd.gamma = p->gamma;
      nd.eps = p->eps;
      break;
    }
    case MK_EW_ROPE: {
      if (!p || n_in != 1 || p->head_dim <= 0 || p->head_dim % 2 || p->n_q_heads <= 0 ||
          p->n_kv_heads <= 0 || !valid_tensor(g, p->out_k)) {
        set_error("mk_add_elementwise: ROPE needs head counts, an even head_dim and out_k");
        return MK_ERR_INVALID_ARG;
      }
      const int64_t d = p->head_dim, r = g->tensors[ins[0]].rows;
      const int64_t want = (p->n_q_heads + p->n_kv_heads + (p->out_v >= 0 ? p->n_kv_heads : 0)) * d;
      if (g->tensors[ins[0]].cols != want || !same_shape(g, out, r, p->n_q_heads * d) ||
          !same_shape(g, p->out_k, r, p->n_kv_heads * d) ||
          (p->out_v >= 0 && (!valid_tensor(g, p->out_v) ||
                             !same_shape(g, p->out_v, r, p->n_kv_heads * d)))) {
        set_error("mk_add_elementwise: ROPE shapes: x [R x %lld], out [R x Hq*d], out_k/out_v "
                  "[R x Hkv*d]", (long long)want);
        return MK_ERR_INVALID_ARG;
      }
      if (!half_type(g->tensors[ins[0]].dtype)) {
        set_error("mk_add_elementwise: ROPE runs f16 / bf16");
        return MK_ERR_UNSUPPORTED;
      }
      nd.kind = NK_ROPE;
      nd.out_k = p->out_k;
      nd.out_v = p->out_v;
      nd.hq = p->n_q_heads;
      nd.hkv = p->n_kv_heads;
      nd.hd = p->head_dim;
      nd.pos0 = p->pos0;
      nd.theta = p->theta;
      break;
    }
    case MK_EW_ARGMAX: {
      const TensorRec& X = g->tensors[ins[0]];
      if (n_in != 1 || !half_type(X.dtype) || O.dtype != MK_I32 || !same_shape(g, out, X.rows, 1)) {
        set_error("mk_add_elementwise: ARGMAX takes x [R x C] f16 / bf16 and out [R x 1] i32");
        return MK_ERR_INVALID_ARG;
      }
      nd.kind = NK_ARGMAX;
      break;
    }
    default:
      set_error("mk_add_elementwise: unknown op %d", op);
      return MK_ERR_INVALID_ARG;
  }
  *node_id = (int)g->nodes.size();
  g->nodes.push_back(nd);
  return MK_OK;
}

extern "C" mk_status mk_add_attention(mk_graph_t g, int32_t q, int32_t k, int32_t v, int32_t out,
                                      const mk_attn_params* p, int32_t* node_id) {
  if (!g || !p || !node_id || !valid_tensor(g, q) || !valid_tensor(g, k) ||
      !valid_tensor(g, v) || !valid_tensor(g, out)) {
    set_error("mk_add_attention: bad graph, tensor id or params");
    return MK_ERR_INVALID_ARG;
  }
  const int64_t hq = p->n_q_heads, hkv = p->n_kv_heads, d = p->head_dim;
  if (hq <= 0 || hkv <= 0 || d <= 0 || hq % hkv) {
    set_error("mk_add_attention: head counts must be positive and Hq divisible by Hkv");
    return MK_ERR_INVALID_ARG;
  }
  const TensorRec &Q = g->tensors[q], &K = g->tensors[k];
  if (Q.cols != hq * d || K.cols != hkv * d || !same_shape(g, v, K.rows, K.cols) ||
      !same_shape(g, out, Q.rows, Q.cols) || K.rows < 1) {
    set_error("mk_add_attention: q [Tq x Hq*d], k and v [Tk x Hkv*d], out [Tq x Hq*d]");
    return MK_ERR_INVALID_ARG;
  }
  NodeRec nd;
  nd.kind = NK_ATTN;
  nd.a = q;
  nd.b = k;
  nd.b2 = v;
  nd.out = out;
  nd.hq = (int)hq;
  nd.hkv = (int)hkv;
  nd.hd = (int)d;
  nd.causal = p->causal;
  nd.pos0 = p->q_pos0;
  nd.scale = p->scale;
  *node_id = (int)g->nodes.size();
  g->nodes.push_back(nd);
  return MK_OK;
}

extern "C" mk_status mk_default_opts(mk_compile_opts* o) {
  if (!o) {
    set_error("mk_default_opts: NULL");
    return MK_ERR_INVALID_ARG;
  }
  memset(o, 0, sizeof *o);
  o->n_sm = 0;
  o->gemm_tile_m = 128;
  o->gemm_tile_n = 256;
  o->cluster = 1;
  o->ew_rows = 128;
  o->ew_cols = 128;
  o->ew_tiles = 1;
  o->norm_rows = 16;
  o->gemv_max_m = 8;
  o->gemv_tile_n = 256;
  o->gemv_splits = 0;
  o->gemv_kstep = 64;
  o->attn_chunk = 64;
  o->argmax_chunk = 4096;
  o->gemm_group_m = 8;
  o->wave_pack = 1;
  o->row_stage = 1;
  o->pool_waves = 1;
  o->attn_tile_q = 128;
  o->dry_run = 0;
  o->timeout_ms = 2000;
  o->device = -1;
  o->debug_counter = -1;
  o->debug_extra = 0;
  o->snapshot_counters = 0;
  o->trace = 0;
  o->gemm_split_tail = 0;
  o->fuse_rope = 1;
  o->fuse_attn_reduce = 1;
  o->kernel_set = 0;
  o->gemv_pack = 1;
  return MK_OK;
}
