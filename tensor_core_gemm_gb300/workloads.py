"""The five workloads as graph descriptions plus seeded data, and the builder that turns a
description into a Graph through the C ABI.

A description is plain data (the same dict format the schedule oracle reads):
  tensors: [{"rows", "cols", "dtype"}], ref = (tensor, r0, c0, rows, cols), nodes: [...].
Input distributions follow the workload definitions; "N(0, v)" with v = 1/K or 1/64 or 0.01 is
read as a variance (it keeps GEMM outputs at unit scale), the decoder's "N(0, 0.02)" as a
standard deviation (the usual initialiser range of such models), gamma ~ N(1, 0.02).
"""
import math

import torch

from . import synth
from .api import Graph


def full(t, rows, cols):
    return (t, 0, 0, rows, cols)


class Workload:
    def __init__(self, name, desc, data, flops, hbm_bytes, info):
        self.name = name
        self.desc = desc          # graph description
        self.data = data          # list of torch tensors per description tensor, or None
        self.flops = flops        # algorithmic FLOPs of one run
        self.hbm_bytes = hbm_bytes  # algorithmic bytes of one run (compulsory traffic)
        self.info = info          # workload-specific metadata (ids of inputs/outputs, sizes)


def _mk(tensors, specs, device, seed):
    """Allocate description tensors on `device` (None: descriptions only)."""
    if device is None:
        return None
    out = []
    for i, (t, sp) in enumerate(zip(tensors, specs)):
        kind = sp[0]
        if kind == "normal":
            out.append(synth.normal((t["rows"], t["cols"]), sp[1], t["dtype"], seed + i, device,
                                    mean=sp[2] if len(sp) > 2 else 0.0))
        else:
            out.append(synth.zeros((t["rows"], t["cols"]), t["dtype"], device))
    return out


# ---------------------------------------------------------------------- GEMM workloads

def mlp3(m=1024, h=1024, layers=3, dtype="f16", device=None, seed=0):
    """x = relu(x @ W[i] + b[i]): x [m x h] ~N(0,1), W ~N(0,1/h), b ~N(0,0.01), one node per layer."""
    tensors = [{"rows": m, "cols": h, "dtype": dtype},               # 0 x
               {"rows": layers * h, "cols": h, "dtype": dtype},      # 1 W stacked (K x N each)
               {"rows": layers * m, "cols": h, "dtype": dtype}]      # 2 b stacked
    specs = [("normal", 1.0), ("normal", 1.0 / math.sqrt(h)), ("normal", 0.1)]
    nodes = []
    cur = full(0, m, h)
    outs = []
    for i in range(layers):
        tid = len(tensors)
        tensors.append({"rows": m, "cols": h, "dtype": dtype})
        specs.append(("zeros",))
        out = full(tid, m, h)
        nodes.append({"kind": "matmul", "a": cur, "b": (1, i * h, 0, h, h), "c": out,
                      "bias": (2, i * m, 0, m, h), "relu": True})
        outs.append(tid)
        cur = out
    data = _mk(tensors, specs, device, seed)
    flops = 2.0 * m * h * h * layers
    es = 2
    hbm = es * (m * h + layers * h * h + layers * m * h + layers * m * h)
    return Workload("mlp3", {"tensors": tensors, "nodes": nodes}, data, flops, hbm,
                    {"outputs": outs, "x": 0, "w": 1, "b": 2, "layers": layers})


def gemm(m, n, k, dtype="f16", std=None, device=None, seed=0, b_std=None):
    """C = A @ B, A [m x k], B [k x n] (row-major weight)."""
    sa = std if std is not None else 1.0 / 8.0
    sb = b_std if b_std is not None else sa
    tensors = [{"rows": m, "cols": k, "dtype": dtype}, {"rows": k, "cols": n, "dtype": dtype},
               {"rows": m, "cols": n, "dtype": dtype}]
    specs = [("normal", sa), ("normal", sb), ("zeros",)]
    nodes = [{"kind": "matmul", "a": full(0, m, k), "b": full(1, k, n), "c": full(2, m, n)}]
    data = _mk(tensors, specs, device, seed)
    return Workload("gemm", {"tensors": tensors, "nodes": nodes}, data, 2.0 * m * n * k,
                    2 * (m * k + k * n + m * n), {"a": 0, "b": 1, "c": 2, "m": m, "n": n, "k": k})


def gemm_list(shapes, dtype="f16", device=None, seed=0):
    """Independent GEMMs in one instruction list: shapes = [(m, n, k), ...]; A ~N(0,1),
    W ~N(0, 1/k)."""
    tensors, specs, nodes, groups = [], [], [], []
    flops = 0.0
    hbm = 0
    for (m, n, k) in shapes:
        a, b, c = len(tensors), len(tensors) + 1, len(tensors) + 2
        tensors += [{"rows": m, "cols": k, "dtype": dtype}, {"rows": k, "cols": n, "dtype": dtype},
                    {"rows": m, "cols": n, "dtype": dtype}]
        specs += [("normal", 1.0), ("normal", 1.0 / math.sqrt(k)), ("zeros",)]
        nodes.append({"kind": "matmul", "a": full(a, m, k), "b": full(b, k, n), "c": full(c, m, n)})
        groups.append((a, b, c, m, n, k))
        flops += 2.0 * m * n * k
        hbm += 2 * (m * k + k * n + m * n)
    data = _mk(tensors, specs, device, seed)
    return Workload("gemm_list", {"tensors": tensors, "nodes": nodes}, data, flops, hbm,
                    {"gemms": groups})


LLAMA70B_PREFILL = [(8192, 8192, 8192), (8192, 28672, 8192)]
LLAMA70B_DECODE = [(256, 10240, 8192), (256, 8192, 8192), (256, 28672, 8192), (256, 8192, 28672)]


# ---------------------------------------------------------------------- decoder workloads

class DecoderShape:
    def __init__(self, layers=16, hidden=2048, n_q_heads=32, n_kv_heads=8, head_dim=64,
                 ffn=8192, eps=1e-5, theta=5e5):
        self.layers, self.hidden, self.hq, self.hkv, self.hd, self.ffn = \
            layers, hidden, n_q_heads, n_kv_heads, head_dim, ffn
        self.eps, self.theta = eps, theta

    @property
    def qkv(self):
        return (self.hq + 2 * self.hkv) * self.hd

    def weight_bytes(self):
        d, f = self.hidden, self.ffn
        per = d * self.qkv + self.hq * self.hd * d + 2 * d * f + f * d + 2 * d
        return 2 * per * self.layers


def _decoder_weights(sh, tensors, specs):
    d, f, L = sh.hidden, sh.ffn, sh.layers
    ids = {}
    for name, rows, cols in (("wqkv", L * d, sh.qkv), ("wo", L * sh.hq * sh.hd, d),
                             ("wg", L * d, f), ("wu", L * d, f), ("wd", L * f, d)):
        ids[name] = len(tensors)
        tensors.append({"rows": rows, "cols": cols, "dtype": "bf16"})
        specs.append(("normal", 0.02))
    for name in ("g_attn", "g_mlp"):
        ids[name] = len(tensors)
        tensors.append({"rows": L, "cols": d, "dtype": "bf16"})
        specs.append(("normal", 0.02, 1.0))
    return ids


def decode(sh=None, kv_len=1024, device=None, seed=0, vocab=0):
    """Batch-1 decode of one token at position p = kv_len through every layer; the cache holds
    positions 0..p-1 (~N(0,1)) and gets row p appended; split-KV attention over p+1 keys.
    vocab > 0 adds greedy sampling: final RMSNorm (gamma ~N(1,0.02)) fused into an lm_head GEMV
    (W_lm [hidden x vocab] ~N(0,0.02)) writing bf16 logits, then ARGMAX -> int32 token."""
    sh = sh or DecoderShape()
    d, f, L, hd = sh.hidden, sh.ffn, sh.layers, sh.hd
    kvw = sh.hkv * hd
    cap = kv_len + 1
    p = kv_len
    tensors, specs = [{"rows": 1, "cols": d, "dtype": "bf16"}], [("normal", 1.0)]
    w = _decoder_weights(sh, tensors, specs)

    def add(rows, cols, spec=("zeros",)):
        tensors.append({"rows": rows, "cols": cols, "dtype": "bf16"})
        specs.append(spec)
        return len(tensors) - 1

    kc = add(L * cap, kvw, ("normal", 1.0))
    vc = add(L * cap, kvw, ("normal", 1.0))
    qkv = add(L, sh.qkv)
    qr = add(L, sh.hq * hd)
    att = add(L, sh.hq * hd)
    hh = add(L, d)
    gu = add(L, f)
    xo = add(L, d)
    nodes = []
    x_prev = full(0, 1, d)
    for l in range(L):
        nodes.append({"kind": "matmul", "a": x_prev, "b": (w["wqkv"], l * d, 0, d, sh.qkv),
                      "c": (qkv, l, 0, 1, sh.qkv), "gamma": (w["g_attn"], l, 0, 1, d),
                      "eps": sh.eps})
        nodes.append({"kind": "rope", "x": (qkv, l, 0, 1, sh.qkv), "out_q": (qr, l, 0, 1, sh.hq * hd),
                      "out_k": (kc, l * cap + p, 0, 1, kvw), "out_v": (vc, l * cap + p, 0, 1, kvw),
                      "n_q_heads": sh.hq, "n_kv_heads": sh.hkv, "head_dim": hd, "pos0": p,
                      "theta": sh.theta})
        nodes.append({"kind": "attention", "q": (qr, l, 0, 1, sh.hq * hd),
                      "k": (kc, l * cap, 0, p + 1, kvw), "v": (vc, l * cap, 0, p + 1, kvw),
                      "out": (att, l, 0, 1, sh.hq * hd), "n_q_heads": sh.hq,
                      "n_kv_heads": sh.hkv, "head_dim": hd, "causal": False, "q_pos0": p})
        nodes.append({"kind": "matmul", "a": (att, l, 0, 1, sh.hq * hd),
                      "b": (w["wo"], l * sh.hq * hd, 0, sh.hq * hd, d), "c": (hh, l, 0, 1, d),
                      "residual": x_prev})
        nodes.append({"kind": "matmul", "a": (hh, l, 0, 1, d), "b": (w["wg"], l * d, 0, d, f),
                      "b2": (w["wu"], l * d, 0, d, f), "c": (gu, l, 0, 1, f),
                      "gamma": (w["g_mlp"], l, 0, 1, d), "eps": sh.eps})
        nodes.append({"kind": "matmul", "a": (gu, l, 0, 1, f), "b": (w["wd"], l * f, 0, f, d),
                      "c": (xo, l, 0, 1, d), "residual": (hh, l, 0, 1, d)})
        x_prev = (xo, l, 0, 1, d)
    head = {}
    if vocab > 0:
        head["w_lm"] = add(d, vocab, ("normal", 0.02))
        head["g_f"] = add(1, d, ("normal", 0.02, 1.0))
        head["logits"] = add(1, vocab)
        tensors.append({"rows": 1, "cols": 1, "dtype": "i32"})
        specs.append(("zeros",))
        head["token"] = len(tensors) - 1
        nodes.append({"kind": "matmul", "a": x_prev, "b": full(head["w_lm"], d, vocab),
                      "c": full(head["logits"], 1, vocab), "gamma": full(head["g_f"], 1, d),
                      "eps": sh.eps})
        nodes.append({"kind": "argmax", "x": full(head["logits"], 1, vocab),
                      "out": full(head["token"], 1, 1)})
    data = _mk(tensors, specs, device, seed)
    if data is not None:
        for l in range(L):            # the new token's cache row starts empty
            data[kc][l * cap + p].zero_()
            data[vc][l * cap + p].zero_()
    kv_bytes = 2 * L * 2 * (p + 1) * kvw
    hbm = sh.weight_bytes() + kv_bytes + 2 * d * vocab
    flops = 2.0 * (sh.weight_bytes() / 2) + 4.0 * L * sh.hq * hd * (p + 1) + 2.0 * d * vocab
    info = dict(shape=sh, x=0, w=w, kc=kc, vc=vc, qkv=qkv, qr=qr, att=att, h=hh, gu=gu, out=xo,
                cap=cap, pos=p, vocab=vocab, **head)
    return Workload("decode", {"tensors": tensors, "nodes": nodes}, data, flops, hbm, info)


def prefill(sh=None, tokens=2048, device=None, seed=0):
    """Causal prefill of `tokens` tokens (batch 1) through every layer."""
    sh = sh or DecoderShape()
    d, f, L, hd, T = sh.hidden, sh.ffn, sh.layers, sh.hd, tokens
    tensors, specs = [{"rows": T, "cols": d, "dtype": "bf16"}], [("normal", 1.0)]
    w = _decoder_weights(sh, tensors, specs)

    def add(cols):
        tensors.append({"rows": L * T, "cols": cols, "dtype": "bf16"})
        specs.append(("zeros",))
        return len(tensors) - 1

    xn, qkv, qr, kr, att, hh, hn, gu, xo = (add(d), add(sh.qkv), add(sh.hq * hd), add(sh.hkv * hd),
                                            add(sh.hq * hd), add(d), add(d), add(f), add(d))
    nodes = []
    x_prev = full(0, T, d)
    qk = (sh.hq + sh.hkv) * hd
    for l in range(L):
        r = l * T
        nodes.append({"kind": "rmsnorm", "x": x_prev, "gamma": (w["g_attn"], l, 0, 1, d),
                      "out": (xn, r, 0, T, d), "eps": sh.eps})
        nodes.append({"kind": "matmul", "a": (xn, r, 0, T, d), "b": (w["wqkv"], l * d, 0, d, sh.qkv),
                      "c": (qkv, r, 0, T, sh.qkv)})
        nodes.append({"kind": "rope", "x": (qkv, r, 0, T, qk), "out_q": (qr, r, 0, T, sh.hq * hd),
                      "out_k": (kr, r, 0, T, sh.hkv * hd), "n_q_heads": sh.hq,
                      "n_kv_heads": sh.hkv, "head_dim": hd, "pos0": 0, "theta": sh.theta})
        nodes.append({"kind": "attention", "q": (qr, r, 0, T, sh.hq * hd),
                      "k": (kr, r, 0, T, sh.hkv * hd), "v": (qkv, r, qk, T, sh.hkv * hd),
                      "out": (att, r, 0, T, sh.hq * hd), "n_q_heads": sh.hq,
                      "n_kv_heads": sh.hkv, "head_dim": hd, "causal": True, "q_pos0": 0})
        nodes.append({"kind": "matmul", "a": (att, r, 0, T, sh.hq * hd),
                      "b": (w["wo"], l * sh.hq * hd, 0, sh.hq * hd, d), "c": (hh, r, 0, T, d),
                      "residual": x_prev})
        nodes.append({"kind": "rmsnorm", "x": (hh, r, 0, T, d), "gamma": (w["g_mlp"], l, 0, 1, d),
                      "out": (hn, r, 0, T, d), "eps": sh.eps})
        nodes.append({"kind": "matmul", "a": (hn, r, 0, T, d), "b": (w["wg"], l * d, 0, d, f),
                      "b2": (w["wu"], l * d, 0, d, f), "c": (gu, r, 0, T, f)})
        nodes.append({"kind": "matmul", "a": (gu, r, 0, T, f), "b": (w["wd"], l * f, 0, f, d),
                      "c": (xo, r, 0, T, d), "residual": (hh, r, 0, T, d)})
        x_prev = (xo, r, 0, T, d)
    data = _mk(tensors, specs, device, seed)
    lin = 2.0 * T * (sh.weight_bytes() / 2 - 2 * d * L)
    attn = 4.0 * L * sh.hq * hd * (T * (T + 1) / 2)   # causal: visible (q, k) pairs
    info = dict(shape=sh, x=0, w=w, out=xo, tokens=T, xn=xn, qkv=qkv, qr=qr, kr=kr, att=att,
                h=hh, hn=hn, gu=gu)
    return Workload("prefill", {"tensors": tensors, "nodes": nodes}, data, lin + attn,
                    sh.weight_bytes(), info)


def _is_ref(v):
    return isinstance(v, tuple) and len(v) == 5 and all(isinstance(x, int) for x in v)


def with_transients(wl, stacked, block_rows, keep=()):
    """A copy of workload `wl` in which each tensor id of `stacked` (per-layer row blocks of
    `block_rows` rows stacked in one tensor) becomes one plan-owned transient per block that a
    node touches, except the (tensor, block) pairs in `keep`, which stay in the caller's tensor
    (a graph output). Every other tensor keeps its index and data, so the copy computes the same
    numbers; new tensors are appended (data None) and info["transients"] lists them."""
    tensors = [dict(t) for t in wl.desc["tensors"]]
    new = {}

    def remap(ref):
        t, r0, c0, rows, cols = ref
        if t not in stacked:
            return ref
        blk = r0 // block_rows
        if (t, blk) in keep:
            return ref
        if r0 + rows > (blk + 1) * block_rows:
            raise ValueError(f"ref {ref} spans row blocks of tensor {t}")
        if (t, blk) not in new:
            tensors.append({"rows": block_rows, "cols": tensors[t]["cols"],
                            "dtype": tensors[t]["dtype"], "transient": True})
            new[(t, blk)] = len(tensors) - 1
        return (new[(t, blk)], r0 - blk * block_rows, c0, rows, cols)

    nodes = []
    for nd in wl.desc["nodes"]:
        out = {}
        for k, v in nd.items():
            if _is_ref(v):
                out[k] = remap(v)
            elif isinstance(v, list) and v and all(_is_ref(x) for x in v):
                out[k] = [remap(x) for x in v]
            else:
                out[k] = v
        nodes.append(out)
    data = None
    if wl.data is not None:
        data = list(wl.data) + [None] * (len(tensors) - len(wl.data))
    info = dict(wl.info, transients=sorted(new.values()))
    return Workload(wl.name, {"tensors": tensors, "nodes": nodes}, data, wl.flops, wl.hbm_bytes,
                    info)


def decoder_intermediates(wl):
    """with_transients arguments that make every per-layer intermediate of a decode or
    prefill workload plan-owned, the last layer's output staying the caller's."""
    inf = wl.info
    L = inf["shape"].layers
    if wl.name == "decode":
        ids = [inf[k] for k in ("qkv", "qr", "att", "h", "gu", "out")]
        rows = 1
    else:
        ids = [inf[k] for k in ("xn", "qkv", "qr", "kr", "att", "h", "hn", "gu", "out")]
        rows = inf["tokens"]
    return set(ids), rows, {(inf["out"], L - 1)}


# ---------------------------------------------------------------------- builder

def build_graph(desc, data=None):
    """Register the description's tensors (data: matching torch tensors, or None for a dry run;
    tensors marked "transient" are plan-owned and take no data) and add its nodes. Returns
    (graph, id_of) where id_of(ref) gives the tensor/view id."""
    g = Graph()
    base = []
    for i, t in enumerate(desc["tensors"]):
        if t.get("transient"):
            base.append(g.transient(t["dtype"], t["rows"], t["cols"]))
        elif data is not None:
            base.append(g.tensor(data[i]))
        else:
            dt = t["dtype"]
            base.append(g.tensor(ptr=0, dtype=dt, shape=[t["rows"], t["cols"]], strides=None))
    cache = {}

    def id_of(ref):
        if ref is None:
            return None
        ref = tuple(ref)
        t, r0, c0, rows, cols = ref
        tt = desc["tensors"][t]
        if r0 == 0 and c0 == 0 and rows == tt["rows"] and cols == tt["cols"]:
            return base[t]
        if ref not in cache:
            cache[ref] = g.view(base[t], r0, c0, rows, cols)
        return cache[ref]

    for nd in desc["nodes"]:
        k = nd["kind"]
        if k == "matmul":
            g.matmul(id_of(nd["a"]), id_of(nd["b"]), id_of(nd["c"]), bias=id_of(nd.get("bias")),
                     relu=nd.get("relu", False), residual=id_of(nd.get("residual")),
                     gamma=id_of(nd.get("gamma")), eps=nd.get("eps", 1e-5),
                     b_up=id_of(nd.get("b2")))
        elif k == "ew":
            g.elementwise(nd["op"], [id_of(r) for r in nd["ins"]], id_of(nd["out"]))
        elif k == "rmsnorm":
            g.rmsnorm(id_of(nd["x"]), id_of(nd["gamma"]), id_of(nd["out"]), nd.get("eps", 1e-5))
        elif k == "rope":
            g.rope(id_of(nd["x"]), id_of(nd["out_q"]), id_of(nd["out_k"]),
                   out_v=id_of(nd.get("out_v")), n_q_heads=nd["n_q_heads"],
                   n_kv_heads=nd["n_kv_heads"], head_dim=nd["head_dim"], pos0=nd.get("pos0", 0),
                   theta=nd.get("theta", 5e5))
        elif k == "argmax":
            g.argmax(id_of(nd["x"]), id_of(nd["out"]))
        elif k == "attention":
            g.attention(id_of(nd["q"]), id_of(nd["k"]), id_of(nd["v"]), id_of(nd["out"]),
                        n_q_heads=nd["n_q_heads"], n_kv_heads=nd["n_kv_heads"],
                        head_dim=nd["head_dim"], causal=nd.get("causal", False),
                        q_pos0=nd.get("q_pos0", 0), scale=nd.get("scale", 0.0))
        else:
            raise ValueError(k)
    return g, id_of
