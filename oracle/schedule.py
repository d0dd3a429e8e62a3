"""Lowering of a static op graph into tile instructions, dependency counters and placement.

This is the plain restatement of the compiler's integer work, used to check it bit for bit.
It follows the scheduler of "MegaKittens Internals" §04: phase 1 (count and place: each node
gets a contiguous range, rounded up to the cluster size with Noops), phase 3 (fine-grained
barriers: a consumer's dependency set is the set of producer instructions whose write boxes
meet its read boxes; every distinct (producer, set) pair is one counter whose target is the set
size), phase 2 (the buffer pool, for tensors marked "transient": see ``_pool``), and §05
(instruction i runs on SM i mod S in iteration i div S). Every other buffer is caller-owned, and
no node may write a region an earlier node reads or writes.

Unlike the page, which finds the sets through per-edge GCD unit cells, this module intersects
every read box with every write box of the earlier phases (brute force).

Graph description (plain dicts, shared with the tests):
  tensors: [{"rows": R, "cols": C, "dtype": "f16"|"bf16"|"f32"|"i32", "transient"?: bool}, ...]
  ref      = (tensor_id, r0, c0, rows, cols)      a 2-D window of a tensor
  nodes:   [{"kind": "matmul", "a", "b", "c", "bias"?, "residual"?, "gamma"?, "b2"?, ...},
            {"kind": "ew", "op", "ins": [refs], "out"},
            {"kind": "rmsnorm", "x", "gamma", "out"},
            {"kind": "rope", "x", "out_q", "out_k", "out_v"?, "n_q_heads", "n_kv_heads", "head_dim"},
            {"kind": "attention", "q", "k", "v", "out", "n_q_heads", "n_kv_heads", "head_dim",
             "causal", "q_pos0"},
            {"kind": "argmax", "x", "out"}]

Lowering rules per node (tile sizes come from ``opts``; see ``DEFAULT_OPTS``):
  matmul with M = 0 or N = 0 -> no instructions.
  matmul, M > gemv_max_m  -> GEMM tiles tile_m × tn (tn = tile_n, or tile_n/2 with a second
      weight "b2" for SiLU·mul) in groups of gemm_group_m row tiles (the last group may be
      shorter): group by group, inside a group column by column and row by row within a column
      (gemm_group_m = 1: row-major over (mt, nt)); each tile repeated ``cluster`` times
      (aux0 = rank). Reads A rows×[0,K), B [0,K)×cols (and b2), bias/residual on the tile box;
      writes the tile box (every instruction of a cluster writes the whole cluster tile).
      Split tail (gemm_split_tail = 1; default 0): with T tiles on U = n_sm div cluster units, the last
      R = T mod U tiles fill a fraction of the last wave. When S = min(U div R, ceil(K/64)) >= 2,
      each of those R tiles is split along K: chunk = ceil(ceil(K/64) / S)·64, splits
      ceil(K/chunk); order: tile, then split, then rank; k0/klen = the split's K range, aux0 =
      rank, aux1 = number of splits. A split reads A and B on its K range, bias/residual on the
      tile box; only split 0 carries the output box; every split carries split 0's arrivals (of
      the same rank), because the split that publishes is known only at run time (the last to
      finish; with two splits and no b2, each split finishes half the columns and the later of
      the two publishes). Each (tile, rank) owns one split semaphore.
  matmul, M <= gemv_max_m -> GEMV tiles: column tiles of gemv_tile_n (halved with b2), each
      split along K into S chunks (gemv_splits, or max(1, n_sm div n_col_tiles) when 0); the
      chunk length is ceil(K/S) rounded up to gemv_kstep (at least gemv_kstep) and S is then
      recomputed as ceil(K/chunk). Order: column tile outer, split inner; aux0 = split index, aux1 = S. Split s reads A[:, chunk] (all of A
      with a norm gamma), B[chunk, cols]; only split 0 carries the output box; every split carries
      split 0's counter arrivals, because the last split to finish reduces and publishes the tile.
      Each tile owns one split semaphore, numbered after the dependency counters.
  ew      -> tiles ew_rows × (ew_cols·ew_tiles), row-major; reads each input and writes the
      output on the same box; aux0 = elementwise op code.
  rmsnorm -> one instruction per norm_rows rows (all columns).
  rope    -> one instruction per norm_rows rows; reads all of x's columns, writes out_q, out_k
      (and out_v) on those rows. Fused (fuse_rope = 1): a rope node right after a matmul that
      lowers to GEMV tiles (no b2), whose x is exactly that matmul's output, with head_dim 64 and
      an output width that is a multiple of gemv_tile_n (itself a multiple of 64), emits no
      instructions: split 0 of each GEMV column tile also carries the rotated q / k (and v)
      boxes of its columns. Also fused: a rope node right after a plain matmul (no bias,
      residual, relu, gamma or b2) that lowers to GEMM tiles without a split tail, whose x is
      the left part of that matmul's output window holding exactly the q, k (and, with out_v,
      v) heads, head_dim 64: every GEMM tile instruction also carries the out_q / out_k
      (/ out_v) boxes of its rows and of its columns below that width.
  attention with one query row (decode) -> two phases:
      partial: for kv head g, for chunk c of attn_chunk keys: reads q (the G = Hq/Hkv heads of
        group g), k and v rows of the chunk (columns of head g); writes rows (g·C + c)·G ..+G
        of a per-node fp32 scratch [Hkv·C·G × (d+2)]. n0 = g, k0 = first key, klen = keys,
        aux0 = c, aux1 = C.
      reduce: one per g; reads the group's C·G scratch rows; writes the group's output columns.
      Fused (fuse_attn_reduce = 1, default): no reduce phase; each g owns a split semaphore, the
        partial with c = 0 also carries the group's output box, every partial of g carries its
        arrivals, and the last partial of g to finish combines the group's partials.
  argmax  -> two phases. Partial: per block of norm_rows rows (outer), per chunk c of
      argmax_chunk columns (inner): reads the block's rows of x on the chunk, writes columns
      2c, 2c+1 of those rows of a per-node fp32 scratch [R x 2C]; n0 = first column, klen =
      columns, aux0 = c. Reduce: one per row block; reads the block's scratch rows, writes its
      rows of the output column; aux1 = C.
  attention with several query rows (prefill) -> one instruction per (q tile t of
      attn_tile_q·cluster rows, q head h, rank r < cluster), t descending (longest first), then
      h ascending, then r (aux0 = r); reads q rows of the tile, k and v rows [0, kmax) with
      kmax = min(Tk, q_pos0 + end of tile) when causal; every rank carries the tile's boxes.

Wave packing (wave_pack = 1, default): a run of consecutive phases of one kind, none reading a
region that an earlier phase of the run writes (bounding boxes per tensor), becomes one phase:
GEMM phases without split tails (runs of two or more; cost = klen × number of B operands) or
prefill attention phases (runs of one or more; cost = klen). Its cluster groups (a tile's
instructions) are stably sorted by cost, longest first; each goes to the unit (n_sm div cluster
units) with the least cost so far, the lowest on ties; row r of the run then holds every unit's
r-th group in unit order, Noop groups where a unit has none, trailing Noops dropped.

Flags: B_DEP marks a GEMM, GEMV or attention-partial instruction whose streamed operand (the
weight, or the key/value chunk) has a producer inside the graph, so it cannot be prefetched.

Counters: consumer instructions are visited in index order, their read boxes in order, and for
each the earlier phases in order; a new (phase, set) key takes the next counter id. A consumer's
source list holds each counter once (first occurrence order) with its target; producers list the
counters they arrive on in increasing id order.
"""
import numpy as np

OP_NOOP, OP_GEMM, OP_GEMV, OP_EW, OP_RMSNORM, OP_ROPE, OP_ATTN_PARTIAL, OP_ATTN_REDUCE, \
    OP_ATTN_PREFILL, OP_ARGMAX, OP_ARGMAX_REDUCE = range(11)
EW_CODES = {"add": 0, "relu": 1, "copy": 2, "silu_mul": 3}
FLAG_B_DEP = 1

ROLE_A, ROLE_B, ROLE_E = 0, 1, 2

DEFAULT_OPTS = dict(
    gemm_tile_m=128, gemm_tile_n=256, cluster=1, gemm_split_tail=0, fuse_rope=1,
    fuse_attn_reduce=1,
    ew_rows=128, ew_cols=128, ew_tiles=1,
    norm_rows=16,
    gemv_max_m=8, gemv_tile_n=256, gemv_splits=0, gemv_kstep=64,
    attn_chunk=64, attn_tile_q=128, argmax_chunk=4096, gemm_group_m=8, wave_pack=1,
    pool_waves=1,
)


def cdiv(a, b):
    return -(-a // b)


def _box(ref, r0, r1, c0, c1):
    """Window [r0,r1)×[c0,c1) of a ref, in the base tensor's coordinates."""
    t, br, bc, rows, cols = ref
    r1 = min(r1, rows)
    c1 = min(c1, cols)
    return (t, br + r0, br + r1, bc + c0, bc + c1)


def _full(ref):
    return _box(ref, 0, ref[3], 0, ref[4])


class Instr:
    __slots__ = ("op", "flags", "node", "m0", "n0", "k0", "klen", "aux0", "aux1", "sem",
                 "reads", "writes", "src", "dst", "tile", "sem_adds")

    def __init__(self, op, node, m0=0, n0=0, k0=0, klen=0, aux0=0, aux1=0):
        self.op, self.node = op, node
        self.flags = 0
        self.m0, self.n0, self.k0, self.klen, self.aux0, self.aux1 = m0, n0, k0, klen, aux0, aux1
        self.sem = 0
        self.reads = []      # (box, role)
        self.writes = []     # box
        self.src = []        # (counter, target)
        self.dst = []        # counter ids
        self.tile = None     # GEMV tile ordinal (shares arrivals and semaphore)
        self.sem_adds = 1    # increments of its split semaphore in one run

    def key(self):
        return (self.op, self.flags, self.node, self.m0, self.n0, self.k0, self.klen,
                self.aux0, self.aux1, self.sem)


def _rope_width(r):
    """Columns of its input a rope node reads: the q, k (and, with out_v, v) heads."""
    heads = r["n_q_heads"] + r["n_kv_heads"] + (r["n_kv_heads"] if r.get("out_v") is not None
                                                 else 0)
    return heads * r["head_dim"]


def rope_fusable(nodes, ri, opts):
    """Whether rope node ri folds into the tiles of the matmul right before it: GEMV tiles when
    its input is exactly the matmul's output window, GEMM tiles (a plain matmul, no split tail)
    when its input is the left part of that window holding exactly the heads it reads."""
    r = nodes[ri]
    if not opts["fuse_rope"] or r["kind"] != "rope" or ri == 0:
        return False
    p = nodes[ri - 1]
    if p["kind"] != "matmul" or p.get("b2") is not None:
        return False
    m = p["a"][3]
    if m <= 0 or r["head_dim"] != 64:
        return False
    if m <= opts["gemv_max_m"]:
        return (tuple(r["x"]) == tuple(p["c"]) and opts["gemv_tile_n"] % 64 == 0
                and p["c"][4] % opts["gemv_tile_n"] == 0)
    plain = all(p.get(f) is None for f in ("bias", "residual", "gamma")) and not p.get("relu")
    x, c = r["x"], p["c"]
    return (plain and not opts["gemm_split_tail"] and tuple(x[:4]) == tuple(c[:4])
            and x[4] == _rope_width(r) and x[4] <= c[4])


def _rope_writes(rope, r0, r1, c0, c1):
    """Boxes of the rope outputs that rows [r0, r1) and columns [c0, c1) of its input produce."""
    d = rope["head_dim"]
    qend, kend = rope["n_q_heads"] * d, (rope["n_q_heads"] + rope["n_kv_heads"]) * d
    out = []
    if c0 < qend:
        out.append(_box(rope["out_q"], r0, r1, c0, min(c1, qend)))
    if c1 > qend and c0 < kend:
        out.append(_box(rope["out_k"], r0, r1, max(c0, qend) - qend, min(c1, kend) - qend))
    if rope.get("out_v") is not None and c1 > kend:
        out.append(_box(rope["out_v"], r0, r1, max(c0, kend) - kend, c1 - kend))
    return out


def _lower_matmul(ni, nd, opts, phases, sem_tiles, rope=None):
    a, b, c = nd["a"], nd["b"], nd["c"]
    m, k = a[3], a[4]
    n = c[4]
    b2 = nd.get("b2")
    gamma = nd.get("gamma")
    epi = [(nd[x], x) for x in ("bias", "residual") if nd.get(x) is not None]
    out = []
    if m == 0 or n == 0:
        pass
    elif m <= opts["gemv_max_m"]:
        w = opts["gemv_tile_n"] // 2 if b2 is not None else opts["gemv_tile_n"]
        n_ct = cdiv(n, w)
        s0 = opts["gemv_splits"] if opts["gemv_splits"] > 0 else max(1, opts["n_sm"] // n_ct)
        chunk = max(opts["gemv_kstep"], cdiv(cdiv(k, s0), opts["gemv_kstep"]) * opts["gemv_kstep"])
        s = max(1, cdiv(k, chunk))
        for ct in range(n_ct):
            n0 = ct * w
            tile = len(sem_tiles)
            sem_tiles.append(tile)
            for si in range(s):
                k0 = si * chunk
                kl = min(chunk, k - k0)
                ins = Instr(OP_GEMV, ni, 0, n0, k0, kl, si, s)
                ins.tile = tile
                if gamma is not None:
                    ins.reads.append((_full(a), ROLE_A))
                    ins.reads.append((_full(gamma), ROLE_A))
                else:
                    ins.reads.append((_box(a, 0, m, k0, k0 + kl), ROLE_A))
                ins.reads.append((_box(b, k0, k0 + kl, n0, n0 + w), ROLE_B))
                if b2 is not None:
                    ins.reads.append((_box(b2, k0, k0 + kl, n0, n0 + w), ROLE_B))
                for r, _ in epi:
                    ins.reads.append((_box(r, 0, m, n0, n0 + w), ROLE_E))
                if si == 0:
                    ins.writes.append(_box(c, 0, m, n0, n0 + w))
                    if rope is not None:
                        ins.writes.extend(_rope_writes(rope, 0, m, n0, n0 + w))
                out.append(ins)
    else:
        tm = opts["gemm_tile_m"]
        tn = opts["gemm_tile_n"] // 2 if b2 is not None else opts["gemm_tile_n"]
        cl = opts["cluster"]
        nnt = cdiv(n, tn)
        t_all = cdiv(m, tm) * nnt
        units = opts["n_sm"] // cl
        nks = cdiv(k, 64)
        r_tail = t_all % units if units > 0 else 0
        n_split = min(units // r_tail, nks) if (opts["gemm_split_tail"] and r_tail) else 1
        split_from = t_all - r_tail if n_split >= 2 else t_all
        nmt, gm = cdiv(m, tm), max(1, opts["gemm_group_m"])
        for t in range(t_all):
            g, r = divmod(t, gm * nnt)
            rows_g = min(gm, nmt - g * gm)
            m0, n0 = (g * gm + r % rows_g) * tm, (r // rows_g) * tn
            if t < split_from:
                ranges, base = [(0, k)], None
            else:
                chunk = cdiv(nks, n_split) * 64
                ranges = [(k0, min(chunk, k - k0)) for k0 in range(0, k, chunk)]
                base = len(sem_tiles)
                sem_tiles.extend([base] * cl)
            for si, (k0, kl) in enumerate(ranges):
                for r in range(cl):
                    ins = Instr(OP_GEMM, ni, m0, n0, k0, kl, r, 0 if base is None else len(ranges))
                    if base is not None:
                        ins.tile = base + r
                        # two splits without b2 meet twice at the semaphore (exchange, finish)
                        ins.sem_adds = 2 if (len(ranges) == 2 and b2 is None) else 1
                    ins.reads.append((_box(a, m0, m0 + tm, k0, k0 + kl), ROLE_A))
                    ins.reads.append((_box(b, k0, k0 + kl, n0, n0 + tn), ROLE_B))
                    if b2 is not None:
                        ins.reads.append((_box(b2, k0, k0 + kl, n0, n0 + tn), ROLE_B))
                    for ref, _ in epi:
                        ins.reads.append((_box(ref, m0, m0 + tm, n0, n0 + tn), ROLE_E))
                    if si == 0:
                        ins.writes.append(_box(c, m0, m0 + tm, n0, n0 + tn))
                        if rope is not None:
                            ins.writes.extend(_rope_writes(rope, m0, m0 + tm, n0,
                                                           min(n0 + tn, _rope_width(rope))))
                    out.append(ins)
    phases.append(out)


def _lower_ew(ni, nd, opts, phases):
    o = nd["out"]
    rows, cols = o[3], o[4]
    er, ew = opts["ew_rows"], opts["ew_cols"] * opts["ew_tiles"]
    out = []
    for rt in range(cdiv(rows, er)):
        for ct in range(cdiv(cols, ew)):
            m0, n0 = rt * er, ct * ew
            ins = Instr(OP_EW, ni, m0, n0, 0, 0, EW_CODES[nd["op"]], 0)
            for r in nd["ins"]:
                ins.reads.append((_box(r, m0, m0 + er, n0, n0 + ew), ROLE_E))
            ins.writes.append(_box(o, m0, m0 + er, n0, n0 + ew))
            out.append(ins)
    phases.append(out)


def _lower_rows(ni, nd, opts, phases, op):
    nr = opts["norm_rows"]
    x = nd["x"]
    rows = x[3]
    outs = [nd[k] for k in ("out", "out_q", "out_k", "out_v") if nd.get(k) is not None]
    out = []
    for rt in range(cdiv(rows, nr)):
        m0 = rt * nr
        ins = Instr(op, ni, m0)
        ins.reads.append((_box(x, m0, m0 + nr, 0, x[4]), ROLE_E))
        if nd.get("gamma") is not None:
            ins.reads.append((_full(nd["gamma"]), ROLE_E))
        for o in outs:
            ins.writes.append(_box(o, m0, m0 + nr, 0, o[4]))
        out.append(ins)
    phases.append(out)


def _bounds(ph, reads):
    """Bounding box per tensor of a phase's read (or write) boxes."""
    bb = {}
    for ins in ph:
        boxes = [b for b, _ in ins.reads] if reads else ins.writes
        for (t, r0, r1, c0, c1) in boxes:
            if r0 >= r1 or c0 >= c1:
                continue
            if t in bb:
                u = bb[t]
                bb[t] = (t, min(u[1], r0), max(u[2], r1), min(u[3], c0), max(u[4], c1))
            else:
                bb[t] = (t, r0, r1, c0, c1)
    return bb


def _meets(a, b):
    return (a[0] == b[0] and a[1] < a[2] and a[3] < a[4] and b[1] < b[2] and b[3] < b[4]
            and a[1] < b[2] and b[1] < a[2] and a[3] < b[4] and b[3] < a[4])


def _pack_waves(phases, o):
    cl = o["cluster"]
    units = o["n_sm"] // cl
    if units <= 0:
        return phases

    def kind(ph):
        if len(ph) == 0 or len(ph) % cl:
            return 0
        if all(i.op == OP_GEMM and i.aux1 == 0 for i in ph):
            return 1
        if all(i.op == OP_ATTN_PREFILL for i in ph):
            return 2
        return 0

    out, i = [], 0
    while i < len(phases):
        k0 = kind(phases[i])
        if k0 == 0:
            out.append(phases[i])
            i += 1
            continue
        j = i + 1
        written = _bounds(phases[i], False)
        while j < len(phases) and kind(phases[j]) == k0:
            if any(t in written and _meets(written[t], b)
                   for t, b in _bounds(phases[j], True).items()):
                break
            for t, b in _bounds(phases[j], False).items():
                if t in written:
                    u = written[t]
                    written[t] = (t, min(u[1], b[1]), max(u[2], b[2]), min(u[3], b[3]),
                                  max(u[4], b[4]))
                else:
                    written[t] = b
            j += 1
        if k0 == 1 and j - i < 2:
            out.append(phases[i])
            i += 1
            continue
        groups, cost = [], []
        for ph in phases[i:j]:
            for g in range(0, len(ph), cl):
                grp = ph[g:g + cl]
                groups.append(grp)
                nb = sum(1 for _, role in grp[0].reads if role == ROLE_B)
                cost.append(grp[0].klen * (nb if k0 == 1 else 1))
        order = sorted(range(len(groups)), key=lambda g: -cost[g])   # stable
        load = [0] * units
        queue = [[] for _ in range(units)]
        for g in order:
            u = min(range(units), key=lambda v: (load[v], v))
            load[u] += cost[g]
            queue[u].append(g)
        rows = max(len(q) for q in queue)
        run = []
        for r in range(rows):
            for u in range(units):
                if r < len(queue[u]):
                    run.extend(groups[queue[u][r]])
                else:
                    run.extend(Instr(OP_NOOP, 0) for _ in range(cl))
        while run and run[-1].op == OP_NOOP:
            run.pop()
        out.append(run)
        i = j
    return out


def _lower_argmax(ni, nd, opts, phases, tensors):
    x, o = nd["x"], nd["out"]
    rows, cols = x[3], x[4]
    nr, ch = opts["norm_rows"], opts["argmax_chunk"]
    nc = cdiv(cols, ch)
    scratch_id = len(tensors)
    tensors.append({"rows": rows, "cols": 2 * nc, "dtype": "f32", "internal": True})
    scratch = (scratch_id, 0, 0, rows, 2 * nc)
    part, red = [], []
    for rt in range(cdiv(rows, nr)):
        m0 = rt * nr
        for c in range(nc):
            ins = Instr(OP_ARGMAX, ni, m0, c * ch, 0, min(ch, cols - c * ch), c, 0)
            ins.reads.append((_box(x, m0, m0 + nr, c * ch, c * ch + ch), ROLE_E))
            ins.writes.append(_box(scratch, m0, m0 + nr, 2 * c, 2 * c + 2))
            part.append(ins)
        ins = Instr(OP_ARGMAX_REDUCE, ni, m0, 0, 0, 0, 0, nc)
        ins.reads.append((_box(scratch, m0, m0 + nr, 0, 2 * nc), ROLE_E))
        ins.writes.append(_box(o, m0, m0 + nr, 0, 1))
        red.append(ins)
    phases.append(part)
    phases.append(red)


def _lower_attention(ni, nd, opts, phases, tensors, sem_tiles):
    q, k, v, o = nd["q"], nd["k"], nd["v"], nd["out"]
    hq, hkv, d = nd["n_q_heads"], nd["n_kv_heads"], nd["head_dim"]
    g_sz = hq // hkv
    tq, tk = q[3], k[3]
    if tq == 1:
        ch = opts["attn_chunk"]
        nc = cdiv(tk, ch)
        scratch_id = len(tensors)
        tensors.append({"rows": hkv * nc * g_sz, "cols": d + 2, "dtype": "f32", "internal": True})
        scratch = (scratch_id, 0, 0, hkv * nc * g_sz, d + 2)
        part = []
        fuse = opts["fuse_attn_reduce"]
        for g in range(hkv):
            tile = None
            if fuse:
                tile = len(sem_tiles)
                sem_tiles.append(tile)
            for c in range(nc):
                k0 = c * ch
                kl = min(ch, tk - k0)
                ins = Instr(OP_ATTN_PARTIAL, ni, 0, g, k0, kl, c, nc)
                ins.tile = tile
                ins.reads.append((_box(q, 0, 1, g * g_sz * d, (g + 1) * g_sz * d), ROLE_A))
                ins.reads.append((_box(k, k0, k0 + kl, g * d, (g + 1) * d), ROLE_B))
                ins.reads.append((_box(v, k0, k0 + kl, g * d, (g + 1) * d), ROLE_B))
                r0 = (g * nc + c) * g_sz
                ins.writes.append(_box(scratch, r0, r0 + g_sz, 0, d + 2))
                if fuse and c == 0:
                    ins.writes.append(_box(o, 0, 1, g * g_sz * d, (g + 1) * g_sz * d))
                part.append(ins)
        if fuse:
            phases.append(part)
            return
        red = []
        for g in range(hkv):
            ins = Instr(OP_ATTN_REDUCE, ni, 0, g, 0, 0, 0, nc)
            r0 = g * nc * g_sz
            ins.reads.append((_box(scratch, r0, r0 + nc * g_sz, 0, d + 2), ROLE_E))
            ins.writes.append(_box(o, 0, 1, g * g_sz * d, (g + 1) * g_sz * d))
            red.append(ins)
        phases.append(part)
        phases.append(red)
    else:
        cl = opts["cluster"]
        tt = opts["attn_tile_q"] * cl
        out = []
        for t in reversed(range(cdiv(tq, tt))):
            m0 = t * tt
            kmax = min(tk, nd.get("q_pos0", 0) + m0 + tt) if nd["causal"] else tk
            for h in range(hq):
                g = h // g_sz
                for r in range(cl):
                    ins = Instr(OP_ATTN_PREFILL, ni, m0, h, 0, kmax, r)
                    ins.reads.append((_box(q, m0, m0 + tt, h * d, (h + 1) * d), ROLE_E))
                    ins.reads.append((_box(k, 0, kmax, g * d, (g + 1) * d), ROLE_E))
                    ins.reads.append((_box(v, 0, kmax, g * d, (g + 1) * d), ROLE_E))
                    ins.writes.append(_box(o, m0, m0 + tt, h * d, (h + 1) * d))
                    out.append(ins)
        phases.append(out)


ELT_BYTES = {"f16": 2, "bf16": 2, "f32": 4, "i32": 4}


def _node_refs(nd):
    """(refs the node reads, refs it writes) by the fields of its kind."""
    k = nd["kind"]
    if k == "matmul":
        reads = [nd["a"], nd["b"], nd.get("b2"), nd.get("bias"), nd.get("residual"),
                 nd.get("gamma")]
        writes = [nd["c"]]
    elif k == "ew":
        reads, writes = list(nd["ins"]), [nd["out"]]
    elif k == "rmsnorm":
        reads, writes = [nd["x"], nd["gamma"]], [nd["out"]]
    elif k == "rope":
        reads, writes = [nd["x"]], [nd["out_q"], nd["out_k"], nd.get("out_v")]
    elif k == "attention":
        reads, writes = [nd["q"], nd["k"], nd["v"]], [nd["out"]]
    elif k == "argmax":
        reads, writes = [nd["x"]], [nd["out"]]
    else:
        raise ValueError(k)
    return [r for r in reads if r is not None], [w for w in writes if w is not None]


def transient_bytes(t):
    """Pool bytes of a transient: rows of cols elements padded to 16 bytes (at least 16), the
    whole rounded up to 1 KB."""
    es = ELT_BYTES[t["dtype"]]
    per = 16 // es
    ld = max(cdiv(t["cols"], per) * per, per)
    return cdiv(t["rows"] * ld * es, 1024) * 1024


def _pool(tensors, nodes, instrs, targets, o, split, fused=()):
    """Phase 2 of "MegaKittens Internals" §04, for the transient tensors.

    Transients are visited in the order of the node that writes them. One takes a buffer from
    the pool when its writer's first instruction is at least n_sm instructions (times the
    option pool_waves, 1 by default: the page's one wave) past the end
    (last instruction + 1) of every node that touched the buffer's current occupant, and the
    occupant has the same dtype and shape; otherwise it gets a new buffer at the end of the
    pool. The occupant's writer counts among the nodes that touched it. A node fused into the
    one before it (``fused``: it has no instructions, that node's carry its work) counts as
    that node wherever it touches or writes a transient.

    Each reuse is one new counter: every instruction of the nodes that touched the old occupant
    arrives on it (the splits of one tile once) and every instruction of the new writer waits
    for that count. Returns (byte offset per tensor id or -1, pool bytes, number of reuses);
    ``instrs`` and ``targets`` gain the counters.
    """
    first, last = {}, {}
    for i, ins in enumerate(instrs):
        if ins.op == OP_NOOP:
            continue
        first.setdefault(ins.node, i)
        last[ins.node] = i
    touched = {}
    writer = {}
    for ni, nd in enumerate(nodes):
        ci = ni - 1 if ni in fused else ni      # the node whose instructions do ni's work
        reads, writes = _node_refs(nd)
        for ref in reads + writes:
            touched.setdefault(ref[0], [])
            if ci not in touched[ref[0]]:
                touched[ref[0]].append(ci)
        for ref in writes:
            writer.setdefault(ref[0], ci)
    trans = [t for t, d in enumerate(tensors) if d.get("transient")]
    trans.sort(key=lambda t: writer.get(t, len(nodes)))
    offsets = [-1] * len(tensors)
    buffers = []          # [offset, occupant, nodes that touched it, may be handed on]
    end = 0
    reuses = []           # (nodes that touched the old occupant, new writer)
    for t in trans:
        acc = touched.get(t, [])
        usable = t in writer and all(ni in last for ni in acc)
        chosen = None
        if usable:
            start = first[writer[t]]
            for b in buffers:
                old = tensors[b[1]]
                same = (old["dtype"], old["rows"], old["cols"]) == (
                    tensors[t]["dtype"], tensors[t]["rows"], tensors[t]["cols"])
                gap = o["pool_waves"] * o["n_sm"]
                if b[3] and same and all(start - (last[ni] + 1) >= gap for ni in b[2]):
                    chosen = b
                    break
        if chosen is not None:
            reuses.append((chosen[2], writer[t]))
            chosen[1], chosen[2] = t, acc
        else:
            chosen = [end, t, acc, usable]
            buffers.append(chosen)
            end += transient_bytes(tensors[t])
        offsets[t] = chosen[0]
    for old_nodes, new_writer in reuses:
        cid = len(targets)
        arrivals = set()
        for i, ins in enumerate(instrs):
            if ins.op != OP_NOOP and ins.node in old_nodes:
                arrivals.add(("t", ins.tile) if split(ins) else ("i", i))
                ins.dst.append(cid)
        targets.append(len(arrivals))
        for ins in instrs:
            if ins.op != OP_NOOP and ins.node == new_writer:
                ins.src.append((cid, len(arrivals)))
    return offsets, end, len(reuses)


class Plan:
    """The oracle's schedule: flat instruction list (Noop-padded), counters and placement."""

    def __init__(self, instrs, targets, n_dep, n_sm, sem_count, pool=None):
        self.instrs = instrs
        self.targets = targets          # per dependency counter (reuse counters last)
        self.n_dep = n_dep
        self.n_sem = sem_count
        self.n_sm = n_sm
        # buffer pool: byte offset of every tensor (-1: caller-owned), bytes, reuse events
        self.pool_off, self.pool_bytes, self.n_reuse = pool or ([], 0, 0)

    @property
    def n_instr(self):
        return len(self.instrs)

    @property
    def waves(self):
        return self.n_instr / self.n_sm

    def placement(self, i):
        """(SM, iteration) of instruction i under the static round-robin placement."""
        return i % self.n_sm, i // self.n_sm

    def final_counters(self):
        """Value of every counter after one complete run: deps reach their targets, each split
        semaphore counts its splits' increments (one per split; two for each split of a GEMM
        tile with exactly two splits and no b2, whose splits exchange halves and then finish)."""
        sems = [0] * self.n_sem
        for ins in self.instrs:
            if (ins.op == OP_GEMV or (ins.op == OP_GEMM and ins.aux1 > 0)
                    or (ins.op == OP_ATTN_PARTIAL and ins.tile is not None)):
                sems[ins.sem - self.n_dep] += ins.sem_adds
        return list(self.targets) + sems

    def records(self):
        """Per-instruction fields the compiler must reproduce exactly."""
        return [(ins.key(), tuple(ins.src), tuple(ins.dst)) for ins in self.instrs]


def lower(graph, opts):
    """Lower a graph description into a Plan (see the module docstring for the rules)."""
    o = dict(DEFAULT_OPTS)
    o.update(opts)
    tensors = [dict(t) for t in graph["tensors"]]
    phases = []
    sem_tiles = []
    nodes = graph["nodes"]
    fused = {ri for ri in range(len(nodes)) if rope_fusable(nodes, ri, o)}
    for ni, nd in enumerate(nodes):
        kind = nd["kind"]
        if kind == "matmul":
            _lower_matmul(ni, nd, o, phases, sem_tiles,
                          nodes[ni + 1] if ni + 1 in fused else None)
        elif kind == "ew":
            _lower_ew(ni, nd, o, phases)
        elif kind == "rmsnorm":
            _lower_rows(ni, nd, o, phases, OP_RMSNORM)
        elif kind == "rope":
            if ni not in fused:
                _lower_rows(ni, nd, o, phases, OP_ROPE)
        elif kind == "attention":
            _lower_attention(ni, nd, o, phases, tensors, sem_tiles)
        elif kind == "argmax":
            _lower_argmax(ni, nd, o, phases, tensors)
        else:
            raise ValueError(kind)

    if o["wave_pack"]:
        phases = _pack_waves(phases, o)

    # Phase 1: contiguous ranges, each rounded up to the cluster size with Noops.
    instrs, phase_of, ranges = [], [], []
    for pi, ph in enumerate(phases):
        start = len(instrs)
        instrs.extend(ph)
        pad = (-len(ph)) % o["cluster"]
        instrs.extend(Instr(OP_NOOP, 0) for _ in range(pad))
        ranges.append((start, len(instrs)))
        phase_of.extend([pi] * (len(instrs) - start))

    # Phase 3: dependency sets by brute-force intersection; one counter per (phase, set).
    # For every phase and tensor, the write boxes as arrays (instruction, r0, r1, c0, c1).
    wtab = {}
    for qi, (s0, s1) in enumerate(ranges):
        per = {}
        for p in range(s0, s1):
            for w in instrs[p].writes:
                per.setdefault(w[0], []).append((p, w[1], w[2], w[3], w[4]))
        for t, rows in per.items():
            wtab.setdefault(t, []).append((qi, np.array(rows, dtype=np.int64).reshape(-1, 5)))
    keys = {}
    targets = []
    members = []
    for ci, c in enumerate(instrs):
        seen = set()
        for box, role in c.reads:
            if box[1] >= box[2] or box[3] >= box[4]:
                continue
            for qi, arr in wtab.get(box[0], []):
                if qi >= phase_of[ci]:
                    break
                hit = ((arr[:, 1] < box[2]) & (box[1] < arr[:, 2]) & (arr[:, 3] < box[4])
                       & (box[3] < arr[:, 4]) & (arr[:, 1] < arr[:, 2]) & (arr[:, 3] < arr[:, 4]))
                st = tuple(sorted(set(int(p) for p in arr[hit, 0])))
                if not st:
                    continue
                key = (qi, st)
                if key not in keys:
                    keys[key] = len(targets)
                    targets.append(len(st))
                    members.append(st)
                cid = keys[key]
                if role == ROLE_B and c.op in (OP_GEMM, OP_GEMV, OP_ATTN_PARTIAL):
                    c.flags |= FLAG_B_DEP
                if cid not in seen:
                    seen.add(cid)
                    c.src.append((cid, len(st)))
    for cid, st in enumerate(members):
        for p in st:
            instrs[p].dst.append(cid)
    n_dep = len(targets)

    # Split tiles (GEMV, and GEMM split tails per rank): every split publishes with split 0's
    # arrivals and shares one semaphore.
    def split(ins):
        return (ins.op == OP_GEMV or (ins.op == OP_GEMM and ins.aux1 > 0)
                or (ins.op == OP_ATTN_PARTIAL and ins.tile is not None))

    first = {}
    for ins in instrs:
        if split(ins) and ins.k0 == 0:
            first[ins.tile] = ins
    for ins in instrs:
        if split(ins):
            ins.dst = list(first[ins.tile].dst)

    # Phase 2 after the fact: the pool needs the final instruction order.
    pool = _pool(tensors, nodes, instrs, targets, o, split, fused)
    n_dep = len(targets)
    for ins in instrs:          # semaphores follow every counter, reuse counters included
        if split(ins):
            ins.sem = n_dep + ins.tile
    return Plan(instrs, targets, n_dep, o["n_sm"], len(sem_tiles), pool)


def topologically_valid(plan):
    """Every counter a consumer waits on is fed only by lower-index instructions, and every
    counter's target equals the number of distinct instructions that arrive on it (the splits
    of a GEMV tile, or of a split-tail GEMM tile's rank, count once: whichever finishes last
    arrives). With placement i -> (i mod S, i div S) this is the deadlock-freedom argument of
    "MegaKittens Internals" §11."""
    feeders = {}
    for i, ins in enumerate(plan.instrs):
        split = (ins.op == OP_GEMV or (ins.op == OP_GEMM and ins.aux1 > 0)
                 or (ins.op == OP_ATTN_PARTIAL and ins.tile is not None))
        key = ("t", ins.tile) if split else ("i", i)
        for cid in ins.dst:
            feeders.setdefault(cid, {})
            feeders[cid].setdefault(key, []).append(i)
    for cid, t in enumerate(plan.targets):
        if len(feeders.get(cid, {})) != t:
            return False
    for i, ins in enumerate(plan.instrs):
        for cid, t in ins.src:
            for idxs in feeders[cid].values():
                if max(idxs) >= i:
                    return False
    return True


def levels(plan):
    """Host-side level of each instruction: 0 without sources, else 1 + max level of the
    instructions feeding its counters ("Implementing a Mega Kernel for B300" §7). Used only as
    an independent check of acyclicity."""
    feeders = {}
    for i, ins in enumerate(plan.instrs):
        for cid in ins.dst:
            feeders.setdefault(cid, []).append(i)
    lv = []
    for i, ins in enumerate(plan.instrs):
        best = -1
        for cid, _ in ins.src:
            for p in feeders[cid]:
                best = max(best, lv[p])
        lv.append(best + 1)
    return lv


def waves_text(plan):
    return f"{plan.waves:.2f}"


def as_array(plan):
    """Per-instruction integer fields as an int64 array [N, 10] (op, flags, node, m0, n0, k0,
    klen, aux0, aux1, sem)."""
    return np.array([ins.key() for ins in plan.instrs], dtype=np.int64).reshape(-1, 10)


def count_by_op(plan):
    out = {}
    for ins in plan.instrs:
        out[ins.op] = out.get(ins.op, 0) + 1
    return out
