"""GPU parity: the megakernel (through the C ABI) against the oracle, element by element.

Tolerance (floating point): relative Frobenius error <= 5e-3 and per-element
|err| <= 2e-2 * max(1, |ref|). Integer outputs (counters) are compared exactly.
"""
import math
import os
import tempfile

import numpy as np
import pytest
import torch

import _drift
import _graphs
from oracle import models, ops
from oracle import schedule as osched
from oracle.numerics import BF16, F16

from tensor_core_gemm_gb300 import synth, workloads
from tensor_core_gemm_gb300._lib import MK_ERR_TIMEOUT, MkError

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def f32(t):
    return synth.to_numpy_f32(t)


def assert_close(got, ref, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    fro = np.linalg.norm(err) / max(np.linalg.norm(ref), 1e-30)
    bound = 2e-2 * np.maximum(1.0, np.abs(ref))
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    assert fro <= 5e-3, f"{what}: relative Frobenius error {fro:.3e}"
    assert np.all(err <= bound), (f"{what}: element {worst} got {got[worst]} ref {ref[worst]}")


def run(wl, **opts):
    g, id_of = workloads.build_graph(wl.desc, wl.data)
    plan = g.compile(snapshot_counters=1, **opts)
    plan.run()
    plan.check_status()
    torch.cuda.synchronize()
    return plan, id_of


def check_counters(plan, wl, opts):
    opts = {k: v for k, v in opts.items() if k != "snapshot_counters"}
    py = osched.lower(wl.desc, dict(opts, n_sm=plan.stats()["n_sm"]))
    assert plan.counters().tolist() == py.final_counters()


@pytest.fixture(autouse=True)
def _sync():
    yield
    torch.cuda.synchronize()


# ------------------------------------------------------------------ GEMM tiles

@pytest.mark.parametrize("m,n,k,tn,dt", [
    (128, 64, 64, 64, "f16"), (128, 256, 64, 256, "f16"), (128, 256, 128, 256, "f16"),
    (256, 256, 256, 256, "f16"), (256, 256, 256, 128, "bf16"), (300, 392, 200, 256, "f16"),
    (129, 72, 520, 64, "bf16"), (1000, 1024, 777 // 8 * 8, 128, "f16")])
def test_gemm_full_compare(m, n, k, tn, dt):
    wl = workloads.gemm(m, n, k, dtype=dt, device=DEV, seed=m + n + k)
    plan, _ = run(wl, gemm_tile_n=tn)
    ref = ops.matmul(f32(wl.data[0]), f32(wl.data[1]), F16 if dt == "f16" else BF16)
    assert_close(f32(wl.data[2]), ref, f"gemm {m}x{n}x{k}")
    check_counters(plan, wl, dict(gemm_tile_n=tn))


def test_gemm_k_zero_writes_epilogue_of_zero():
    wl = workloads.gemm(200, 64, 0, dtype="f16", device=DEV)
    wl.data[2].fill_(7.0)
    run(wl, gemm_tile_n=64)
    assert torch.count_nonzero(wl.data[2]).item() == 0


def test_gemm_4096_sampled_rows_and_256_cube():
    # the 4096^3 GEMM: 256 seeded random rows checked in full
    wl = workloads.gemm(4096, 4096, 4096, dtype="f16", device=DEV, seed=0)
    run(wl)
    rows = np.sort(torch.randperm(4096, generator=torch.Generator().manual_seed(0))[:256].numpy())
    a = f32(wl.data[0][torch.as_tensor(rows, device=DEV)])
    ref = ops.matmul(a, f32(wl.data[1]), F16)
    assert_close(f32(wl.data[2][torch.as_tensor(rows, device=DEV)]), ref, "4096^3 rows")
    # complete output of a 256^3 instance
    wl = workloads.gemm(256, 256, 256, dtype="f16", device=DEV, seed=0)
    run(wl)
    assert_close(f32(wl.data[2]), ops.matmul(f32(wl.data[0]), f32(wl.data[1]), F16), "256^3")


def test_mlp3_parity_and_identity_pin():
    wl = workloads.mlp3(device=DEV, seed=0)
    plan, _ = run(wl, gemm_tile_n=64)
    x, w, b = f32(wl.data[0]), f32(wl.data[1]).reshape(3, 1024, 1024), \
        f32(wl.data[2]).reshape(3, 1024, 1024)
    refs = models.mlp(x, w, b)
    for i, tid in enumerate(wl.info["outputs"]):
        assert_close(f32(wl.data[tid]), refs[i], f"mlp layer {i}")
    check_counters(plan, wl, dict(gemm_tile_n=64))
    # W = I, b = 0 gives relu(x) exactly
    wl.data[1].copy_(torch.eye(1024, device=DEV, dtype=torch.float16).repeat(3, 1))
    wl.data[2].zero_()
    plan.run()
    plan.check_status()
    relu = torch.relu(wl.data[0])
    for tid in wl.info["outputs"]:
        assert torch.equal(wl.data[tid], relu)


def test_gemm_epilogues_bias_relu_residual_and_silu_mul():
    m, n, k = 256, 256, 320
    a = synth.normal((m, k), 1.0, "bf16", 1, DEV)
    b = synth.normal((k, n), 1 / math.sqrt(k), "bf16", 2, DEV)
    bu = synth.normal((k, n), 1 / math.sqrt(k), "bf16", 3, DEV)
    bias = synth.normal((m, n), 0.5, "bf16", 4, DEV)
    res = synth.normal((m, n), 1.0, "bf16", 5, DEV)
    o1 = torch.zeros((m, n), dtype=torch.bfloat16, device=DEV)
    o2 = torch.zeros((m, n), dtype=torch.bfloat16, device=DEV)
    from tensor_core_gemm_gb300 import Graph
    g = Graph()
    ia, ib, ibu, ibias, ires, i1, i2 = (g.tensor(t) for t in (a, b, bu, bias, res, o1, o2))
    g.matmul(ia, ib, i1, bias=ibias, relu=True, residual=ires)
    g.matmul(ia, ib, i2, b_up=ibu)
    p = g.compile(gemm_tile_n=256)
    p.run()
    p.check_status()
    A, B, BU = f32(a), f32(b), f32(bu)
    assert_close(f32(o1), ops.matmul(A, B, BF16, bias=f32(bias), relu=True, residual=f32(res)),
                 "bias+relu+residual")
    assert_close(f32(o2), ops.matmul_silu_mul(A, B, BU, BF16), "silu_mul")


# ------------------------------------------------------------------ GEMV tiles

@pytest.mark.parametrize("m,n,k,splits,norm,dual,res", [
    (1, 256, 512, 0, False, False, False), (1, 3072, 2048, 0, True, False, False),
    (1, 1024, 2048, 4, True, True, False), (1, 2048, 8192, 0, False, False, True),
    (5, 392, 1000 // 8 * 8, 3, True, False, True), (8, 128, 128, 1, False, True, False)])
def test_gemv(m, n, k, splits, norm, dual, res):
    x = synth.normal((m, k), 1.0, "bf16", 11, DEV)
    w = synth.normal((k, n), 0.02, "bf16", 12, DEV)
    wu = synth.normal((k, n), 0.02, "bf16", 13, DEV)
    gamma = synth.normal((1, k), 0.02, "bf16", 14, DEV, mean=1.0)
    r = synth.normal((m, n), 1.0, "bf16", 15, DEV)
    out = torch.zeros((m, n), dtype=torch.bfloat16, device=DEV)
    from tensor_core_gemm_gb300 import Graph
    g = Graph()
    ix, iw, iwu, ig, ir, io = (g.tensor(t) for t in (x, w, wu, gamma, r, out))
    g.matmul(ix, iw, io, gamma=ig if norm else None, b_up=iwu if dual else None,
             residual=ir if res else None, eps=1e-5)
    p = g.compile(gemv_splits=splits, snapshot_counters=1)
    p.run()
    p.check_status()
    X, W, WU, G, R = f32(x), f32(w), f32(wu), f32(gamma)[0], f32(r)
    if norm:
        ref = ops.matmul_norm_input(X, G, 1e-5, W, BF16, residual=R if res else None,
                                    w_up=WU if dual else None)
    elif dual:
        ref = ops.matmul_silu_mul(X, W, WU, BF16)
    else:
        ref = ops.matmul(X, W, BF16, residual=R if res else None)
    assert_close(f32(out), ref, "gemv")
    # every split semaphore counted every split; every counter reached its target
    st = p.stats()
    ctr = p.counters()
    assert np.all(ctr[st["n_counters"]:] == p.instructions()["aux1"][0])


@pytest.mark.parametrize("m,n,k,dual", [(1, 3072, 2048, False), (5, 392, 1000, False),
                                        (3, 1000, 520, True), (8, 128, 4096, True)])
def test_gemv_packed_weights_bit_identical(m, n, k, dual):
    """GEMV tiles streaming packed weight copies (gemv_pack = 1, one bulk copy per stage) and
    the weights themselves through tensor maps (gemv_pack = 0) fill shared memory with the same
    bytes, so the outputs agree bit for bit; ragged N and K are zero outside the weight."""
    x = synth.normal((m, k), 1.0, "bf16", 31, DEV)
    w = synth.normal((k, n), 0.02, "bf16", 32, DEV)
    wu = synth.normal((k, n), 0.02, "bf16", 33, DEV)
    outs = []
    from tensor_core_gemm_gb300 import Graph
    for pack in (1, 0):
        out = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device=DEV)
        g = Graph()
        ix, iw, iwu, io = (g.tensor(t) for t in (x, w, wu, out))
        g.matmul(ix, iw, io, b_up=iwu if dual else None)
        p = g.compile(gemv_pack=pack)
        assert (p.stats()["packed_bytes"] > 0) == bool(pack)
        p.run()
        p.check_status()
        outs.append(out)
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    ref = (ops.matmul_silu_mul(f32(x), f32(w), f32(wu), BF16) if dual
           else ops.matmul(f32(x), f32(w), BF16))
    assert_close(f32(outs[0]), ref, "packed gemv")


def test_gemv_packed_weights_follow_changes():
    """A packed weight is refreshed by mk_run_host copies into its tensor and by repack()."""
    m, n, k = 2, 512, 1024
    x = synth.normal((m, k), 1.0, "bf16", 41, DEV)
    w = synth.normal((k, n), 0.02, "bf16", 42, DEV)
    out = torch.zeros((m, n), dtype=torch.bfloat16, device=DEV)
    from tensor_core_gemm_gb300 import Graph
    g = Graph()
    ix, iw, io = (g.tensor(t) for t in (x, w, out))
    g.matmul(ix, iw, io)
    p = g.compile()
    assert p.stats()["packed_bytes"] > 0
    w2 = synth.normal((k, n), 0.02, "bf16", 43, DEV)
    # a device-side change followed by repack()
    w.copy_(w2)
    p.repack()
    p.run()
    p.check_status()
    assert_close(f32(out), ops.matmul(f32(x), f32(w2), BF16), "after repack")
    # a host copy into the weight through run_host
    w3 = synth.normal((k, n), 0.02, "bf16", 44, DEV)
    w3_h = w3.cpu().pin_memory()
    s = torch.cuda.Stream()
    p.run_host(inputs=[(iw, w3_h.data_ptr())], stream=s)
    s.synchronize()
    p.check_status()
    assert_close(f32(out), ops.matmul(f32(x), f32(w3), BF16), "after run_host weight copy")


def test_gemv_weight_written_in_graph_is_not_packed():
    """A GEMV whose weight another node writes reads it through its tensor map after the
    producer's tiles (no packed copy)."""
    m, n, k = 1, 256, 256
    x = synth.normal((m, k), 1.0, "bf16", 51, DEV)
    w0 = synth.normal((k, n), 0.02, "bf16", 52, DEV)
    w = torch.zeros((k, n), dtype=torch.bfloat16, device=DEV)
    out = torch.zeros((m, n), dtype=torch.bfloat16, device=DEV)
    from tensor_core_gemm_gb300 import Graph
    g = Graph()
    ix, iw0, iw, io = (g.tensor(t) for t in (x, w0, w, out))
    g.elementwise("relu", [iw0], iw)
    g.matmul(ix, iw, io)
    p = g.compile()
    assert p.stats()["packed_bytes"] == 0
    p.run()
    p.check_status()
    assert_close(f32(out), ops.matmul(f32(x), np.maximum(f32(w0), 0), BF16), "in-graph weight")


# ------------------------------------------------------------------ row / elementwise ops

def test_unfused_mlp_elementwise_tiles():
    import _graphs
    desc = _graphs.mlp_unfused(m=300, h=256, layers=2, dtype="f16")
    data = []
    for i, t in enumerate(desc["tensors"]):
        std = [1 / 16, 1.0, 0.1][i] if i < 3 else 0.0
        data.append(synth.normal((t["rows"], t["cols"]), std, "f16", 20 + i, DEV) if i < 3 else
                    synth.zeros((t["rows"], t["cols"]), "f16", DEV))
    g, _ = workloads.build_graph(desc, data)
    p = g.compile(gemm_tile_n=128, ew_rows=64, ew_cols=64, ew_tiles=2)
    p.run()
    p.check_status()
    x, w, b = f32(data[1]), f32(data[0]).reshape(2, 256, 256), f32(data[2]).reshape(2, 300, 256)
    refs = models.mlp_unfused(x, w, b, F16)
    for l in range(2):
        for j in range(3):
            assert_close(f32(data[3 + 3 * l + j]), refs[l][j], f"layer {l} node {j}")


# Row instructions run three ways: the decode specialisation (rows loaded by the compute
# warpgroup), the general kernel with the rows staged through the operand ring by bulk copies
# (row_stage, where a row fits one 32 KB stage), and the general kernel without staging. The
# three agree bit for bit.
ROW_MODES = [dict(), dict(kernel_set=1), dict(kernel_set=1, row_stage=0)]


def _row_modes(build):
    results = []
    for mode in ROW_MODES:
        g, outs = build()
        p = g.compile(**mode)
        p.run()
        p.check_status()
        torch.cuda.synchronize()
        pads = p.instructions()["pad"]
        results.append(([o.clone() for o in outs], int((pads > 0).sum())))
    for outs, _ in results[1:]:
        for a, b in zip(results[0][0], outs):
            assert torch.equal(a, b)
    return results[0][0], [n for _, n in results]


@pytest.mark.parametrize("t,d,staged", [(67, 2048, True), (16, 16384, True), (3, 20000, False),
                                        (1, 64, True)])
def test_rmsnorm_rows(t, d, staged):
    x = synth.normal((t, d), 1.0, "bf16", 30, DEV)
    gm = synth.normal((1, d), 0.02, "bf16", 31, DEV, mean=1.0)
    from tensor_core_gemm_gb300 import Graph

    def build():
        out = torch.zeros_like(x)
        g = Graph()
        ix, ig, io = g.tensor(x), g.tensor(gm), g.tensor(out)
        g.rmsnorm(ix, ig, io, 1e-5)
        return g, [out]

    (out,), n_staged = _row_modes(build)
    # 16-row instructions: staged in the general kernel where a row fits 32 KB, never in decode
    assert n_staged == [0, -(-t // 16) if staged else 0, 0]
    assert_close(f32(out), ops.rmsnorm(f32(x), f32(gm)[0], 1e-5, BF16), "rmsnorm")


@pytest.mark.parametrize("rows,pos0,with_v", [(1, 1024, True), (40, 0, False), (3, 2045, True)])
def test_rope(rows, pos0, with_v):
    hq, hkv, d = 32, 8, 64
    cols = (hq + hkv + (hkv if with_v else 0)) * d
    x = synth.normal((rows, cols), 1.0, "bf16", 40, DEV)
    from tensor_core_gemm_gb300 import Graph

    def build():
        oq = torch.zeros((rows, hq * d), dtype=torch.bfloat16, device=DEV)
        ok = torch.zeros((rows, hkv * d), dtype=torch.bfloat16, device=DEV)
        ov = torch.zeros((rows, hkv * d), dtype=torch.bfloat16, device=DEV)
        g = Graph()
        ix, iq, ik, iv = g.tensor(x), g.tensor(oq), g.tensor(ok), g.tensor(ov)
        g.rope(ix, iq, ik, out_v=iv if with_v else None, n_q_heads=hq, n_kv_heads=hkv,
               head_dim=d, pos0=pos0, theta=5e5)
        return g, [oq, ok, ov]

    (oq, ok, ov), n_staged = _row_modes(build)
    assert n_staged == [0, -(-rows // 16), 0]
    X = f32(x)
    pos = pos0 + np.arange(rows)
    assert_close(f32(oq), ops.rope(X[:, :hq * d], pos, hq, d, 5e5, BF16), "rope q")
    assert_close(f32(ok), ops.rope(X[:, hq * d:(hq + hkv) * d], pos, hkv, d, 5e5, BF16), "rope k")
    if with_v:
        assert torch.equal(ov, x[:, (hq + hkv) * d:])


# ------------------------------------------------------------------ split-KV attention

@pytest.mark.parametrize("tk,chunk,hq,hkv", [(1025, 64, 32, 8), (70, 16, 8, 2), (1, 64, 4, 4),
                                            (300, 128, 32, 8)])
@pytest.mark.parametrize("fuse", [1, 0])
def test_attention_decode_split_kv(tk, chunk, hq, hkv, fuse):
    d = 64
    q = synth.normal((1, hq * d), 1.0, "bf16", 50, DEV)
    k = synth.normal((tk, hkv * d), 1.0, "bf16", 51, DEV)
    v = synth.normal((tk, hkv * d), 1.0, "bf16", 52, DEV)
    out = torch.zeros((1, hq * d), dtype=torch.bfloat16, device=DEV)
    from tensor_core_gemm_gb300 import Graph
    g = Graph()
    iq, ik, iv, io = g.tensor(q), g.tensor(k), g.tensor(v), g.tensor(out)
    g.attention(iq, ik, iv, io, n_q_heads=hq, n_kv_heads=hkv, head_dim=d, q_pos0=tk - 1)
    p = g.compile(attn_chunk=chunk, fuse_attn_reduce=fuse)
    p.run()
    p.check_status()
    ref = ops.attention(f32(q), f32(k), f32(v), hq, hkv, d, False, tk - 1, 1 / 8, BF16)
    assert_close(f32(out), ref, "split-KV attention")
    assert (p.stats()["per_op"][osched.OP_ATTN_REDUCE] == 0) == bool(fuse)


# ------------------------------------------------------------------ decoder, decode step

def _decode_ref(wl):
    sh = wl.info["shape"]
    L, d, f = sh.layers, sh.hidden, sh.ffn
    D = wl.data
    w = wl.info["w"]
    cap, p = wl.info["cap"], wl.info["pos"]
    wts = models.DecoderWeights(
        f32(D[w["wqkv"]]).reshape(L, d, sh.qkv), f32(D[w["wo"]]).reshape(L, sh.hq * sh.hd, d),
        f32(D[w["wg"]]).reshape(L, d, f), f32(D[w["wu"]]).reshape(L, d, f),
        f32(D[w["wd"]]).reshape(L, f, d), f32(D[w["g_attn"]]), f32(D[w["g_mlp"]]),
        sh.hq, sh.hkv, sh.hd, sh.eps, sh.theta)
    kc = f32(D[wl.info["kc"]]).reshape(L, cap, -1)
    vc = f32(D[wl.info["vc"]]).reshape(L, cap, -1)
    return wts, kc, vc, p


def test_decode_small_decoder():
    sh = workloads.DecoderShape(layers=3, hidden=512, n_q_heads=8, n_kv_heads=2, head_dim=64,
                                ffn=1024)
    wl = workloads.decode(sh, kv_len=200, device=DEV, seed=5)
    x0 = f32(wl.data[0])
    kc0 = f32(wl.data[wl.info["kc"]]).reshape(3, 201, -1).copy()
    vc0 = f32(wl.data[wl.info["vc"]]).reshape(3, 201, -1).copy()
    plan, _ = run(wl)
    wts, _, _, p = _decode_ref(wl)
    per_layer = {}
    ref, kc, vc = models.decode_step(x0, wts, list(kc0), list(vc0), p,
                                     layer_fn=lambda l, dd: per_layer.__setitem__(l, dd))
    out = f32(wl.data[wl.info["out"]])
    for l in range(3):
        assert_close(f32(wl.data[wl.info["qkv"]])[l:l + 1], per_layer[l]["qkv"], f"qkv {l}")
        assert_close(out[l:l + 1], per_layer[l]["x"], f"layer {l} output")
    assert_close(out[-1:], ref, "decode output")
    kcg = f32(wl.data[wl.info["kc"]]).reshape(3, 201, -1)
    for l in range(3):
        assert_close(kcg[l, p], kc[l][p], f"k cache row, layer {l}")
    check_counters(plan, wl, {})


def check_decode_per_node(wl, kc0, vc0):
    """Every node of every layer against the oracle applied to the GPU's own inputs of that node
    (teacher forcing), at full size. End to end, two valid fp32 summation orders of the oracle
    itself drift apart by ~1.4e-2 relative Frobenius over 16 bf16 layers, so the tolerance is
    applied per node, where it is meaningful."""
    sh = wl.info["shape"]
    wts, _, _, p = _decode_ref(wl)
    D = wl.data
    hq, hkv, hd = sh.hq, sh.hkv, sh.hd
    cap = wl.info["cap"]
    qkv, qr, att, hh, gu, xo = (f32(D[wl.info[k]]) for k in ("qkv", "qr", "att", "h", "gu", "out"))
    kc = f32(D[wl.info["kc"]]).reshape(sh.layers, cap, -1)
    vc = f32(D[wl.info["vc"]]).reshape(sh.layers, cap, -1)
    x_prev = f32(D[0])
    for l in range(sh.layers):
        assert_close(qkv[l:l + 1], ops.matmul_norm_input(x_prev, wts.g_attn[l], sh.eps,
                                                         wts.wqkv[l], BF16), f"qkv {l}")
        q_in = qkv[l:l + 1, :hq * hd]
        k_in = qkv[l:l + 1, hq * hd:(hq + hkv) * hd]
        v_in = qkv[l:l + 1, (hq + hkv) * hd:]
        assert_close(qr[l:l + 1], ops.rope(q_in, [p], hq, hd, sh.theta, BF16), f"rope q {l}")
        assert_close(kc[l, p:p + 1], ops.rope(k_in, [p], hkv, hd, sh.theta, BF16), f"rope k {l}")
        assert np.array_equal(vc[l, p:p + 1], v_in), f"v append {l}"
        assert np.array_equal(kc[l, :p], kc0[l, :p]) and np.array_equal(vc[l, :p], vc0[l, :p])
        assert_close(att[l:l + 1], ops.attention(qr[l:l + 1], kc[l, :p + 1], vc[l, :p + 1], hq,
                                                 hkv, hd, False, p, 1 / math.sqrt(hd), BF16),
                     f"attention {l}")
        assert_close(hh[l:l + 1], ops.matmul(att[l:l + 1], wts.wo[l], BF16, residual=x_prev),
                     f"o-proj {l}")
        assert_close(gu[l:l + 1], ops.matmul_norm_input(hh[l:l + 1], wts.g_mlp[l], sh.eps,
                                                        wts.wg[l], BF16, w_up=wts.wu[l]),
                     f"gate/up {l}")
        assert_close(xo[l:l + 1], ops.matmul(gu[l:l + 1], wts.wd[l], BF16,
                                             residual=hh[l:l + 1]), f"down {l}")
        x_prev = xo[l:l + 1]


def test_decode_full_config():
    wl = workloads.decode(device=DEV, seed=0)
    sh = wl.info["shape"]
    cap = wl.info["cap"]
    x0 = f32(wl.data[0])
    kc0 = f32(wl.data[wl.info["kc"]]).reshape(sh.layers, cap, -1).copy()
    vc0 = f32(wl.data[wl.info["vc"]]).reshape(sh.layers, cap, -1).copy()
    plan, _ = run(wl)
    check_counters(plan, wl, {})
    check_decode_per_node(wl, kc0, vc0)
    # End to end: two valid summation orders of the oracle itself drift apart by ~1.4e-2
    # relative Frobenius over 16 bf16 layers (tests/test_oracle_drift.py); the drift is measured
    # here on these very inputs and the GPU held to MARGIN times it.
    wts, _, _, p = _decode_ref(wl)
    drift, ref = _drift.decode_drift(x0, wts, list(kc0), list(vc0), p)
    got = f32(wl.data[wl.info["out"]])[-1:]
    ok, seen = _drift.within_drift(got, ref, drift)
    assert ok, f"16-layer decode: gap {seen} against oracle drift {drift}"


# ------------------------------------------------------------------ runtime behaviour

def test_run_twice_same_result_and_host_path():
    wl = workloads.gemm(256, 512, 384, dtype="f16", device=DEV, seed=9)
    g, id_of = workloads.build_graph(wl.desc, wl.data)
    p = g.compile()
    p.run()
    p.check_status()
    first = wl.data[2].clone()
    wl.data[2].zero_()
    p.run()
    p.check_status()
    assert torch.equal(first, wl.data[2])
    # host buffers: copies in, run, copies out, all on one stream
    a_h = wl.data[0].cpu().pin_memory()
    c_h = torch.zeros((256, 512), dtype=torch.float16).pin_memory()
    wl.data[0].zero_()
    s = torch.cuda.Stream()
    p.run_host(inputs=[(0, a_h.data_ptr())], outputs=[(2, c_h.data_ptr())], stream=s)
    s.synchronize()
    p.check_status()
    assert torch.equal(c_h, first.cpu())


def _pool_check(plan, desc, transients):
    """Counters after the run and pool addresses follow the oracle's pooled schedule."""
    st = plan.stats()
    py = osched.lower(desc, dict(n_sm=st["n_sm"]))
    assert st["pool_bytes"] == py.pool_bytes and st["n_reuse"] == py.n_reuse > 0
    assert plan.counters().tolist() == py.final_counters()
    base = plan.tensor_ptr(transients[0]) - py.pool_off[transients[0]]
    assert [plan.tensor_ptr(t) - base for t in transients] == [py.pool_off[t] for t in transients]


@pytest.mark.parametrize("kind", ["prefill", "decode"])
def test_buffer_pool_decoder_bit_identical(kind):
    # Every per-layer intermediate plan-owned (placed in the pool, buffers handed on under the
    # one-wave rule, reuse counters) computes the same bits as caller-owned intermediates.
    sh = workloads.DecoderShape(layers=6, hidden=256, n_q_heads=4, n_kv_heads=2, head_dim=64,
                                ffn=512)
    if kind == "prefill":
        wl = workloads.prefill(sh, tokens=384, device=DEV, seed=5)
        outs = [wl.info["out"]]
    else:
        wl = workloads.decode(sh, kv_len=100, device=DEV, seed=5, vocab=5000)
        outs = [wl.info["out"], wl.info["logits"], wl.info["token"]]
    L, rows = sh.layers, (384 if kind == "prefill" else 1)
    g, _ = workloads.build_graph(wl.desc, wl.data)
    plain = g.compile()
    plain.run()
    plain.check_status()
    want = [wl.data[t].clone() for t in outs]
    for t in outs:
        wl.data[t].zero_()
    pw = workloads.with_transients(wl, *workloads.decoder_intermediates(wl))
    g2, _ = workloads.build_graph(pw.desc, pw.data)
    pooled = g2.compile(snapshot_counters=1)
    pooled.run()
    pooled.check_status()
    torch.cuda.synchronize()
    for t, w in zip(outs, want):
        if t == wl.info["out"]:   # only the last layer's block is still the caller's
            w, got = w[(L - 1) * rows:], wl.data[t][(L - 1) * rows:]
        else:
            got = wl.data[t]
        assert torch.equal(got, w), t
    _pool_check(pooled, pw.desc, pw.info["transients"])


def test_buffer_pool_mlp_example_host_readback():
    # The MegaKittens MLP (mm -> add(bias) -> relu per layer) with all nine layer outputs
    # plan-owned; the last ReLU's result comes back through mk_run_host from its pool buffer.
    m = h = 1024
    desc_t = _graphs.mlp_unfused(m, h, transient=True)
    desc_p = _graphs.mlp_unfused(m, h)
    data = [synth.normal((3 * h, h), h ** -0.5, "bf16", 1, DEV),
            synth.normal((m, h), 1.0, "bf16", 2, DEV),
            synth.normal((3 * m, h), 0.1, "bf16", 3, DEV)]
    data_p = data + [synth.zeros((m, h), "bf16", DEV) for _ in range(9)]
    g, _ = workloads.build_graph(desc_p, data_p)
    plain = g.compile()
    plain.run()
    plain.check_status()
    g2, _ = workloads.build_graph(desc_t, data + [None] * 9)
    pooled = g2.compile(snapshot_counters=1)
    out_h = torch.zeros((m, h), dtype=torch.bfloat16).pin_memory()
    s = torch.cuda.Stream()
    pooled.run_host(outputs=[(11, out_h.data_ptr())], stream=s)
    s.synchronize()
    pooled.check_status()
    assert torch.equal(out_h, data_p[11].cpu())
    _pool_check(pooled, desc_t, list(range(3, 12)))
    with pytest.raises(MkError, match="transient"):
        pooled.run_host(inputs=[(3, out_h.data_ptr())])


def test_wait_limit_reports_timeout_without_hanging():
    # A counter target nothing can reach: the consumer's wait runs out after timeout_ms and the
    # kernel ends with MK_ERR_TIMEOUT; the context stays usable.
    wl = workloads.mlp3(m=256, h=256, layers=2, device=DEV)
    g, _ = workloads.build_graph(wl.desc, wl.data)
    p = g.compile(debug_counter=0, debug_extra=1, timeout_ms=50, gemm_tile_n=64)
    p.run()
    code, st = p.sync_status()
    assert code == MK_ERR_TIMEOUT and st["counter"] == 0 and st["expected"] == st["observed"] + 1
    ok = workloads.gemm(128, 64, 64, device=DEV)
    run(ok, gemm_tile_n=64)
    assert_close(f32(ok.data[2]), ops.matmul(f32(ok.data[0]), f32(ok.data[1]), F16), "after")


def test_trace_timestamps_are_ordered():
    wl = workloads.mlp3(m=256, h=256, layers=2, device=DEV)
    g, _ = workloads.build_graph(wl.desc, wl.data)
    p = g.compile(trace=1, gemm_tile_n=64)
    p.run()
    p.check_status()
    tr = p.trace().astype(np.int64)
    ins = p.instructions()
    real = ins["op"] != 0
    assert np.all(tr[real, 0] > 0) and np.all(tr[real, 1] > 0)
    assert np.all(tr[real, 2] >= tr[real, 1]) and np.all(tr[real, 3] >= tr[real, 2])
    assert np.all(tr[real, 4] >= tr[real, 3]) and np.all(tr[real, 3] >= tr[real, 0])
    assert np.all(tr[real, 5] == np.arange(len(ins))[real] % p.stats()["n_sm"])
    # GEMM tiles: the accumulator is complete after the sources are seen, before the body ends
    assert np.all(tr[real, 6] >= tr[real, 2]) and np.all(tr[real, 3] >= tr[real, 6])
    assert np.all(tr[:, 7] == 0)
    # the Chrome trace export: one track per SM that ran a tile, one GEMM slice per tile
    import json
    path = os.path.join(tempfile.mkdtemp(), "run.json")
    p.export_trace(path, node_names=["layer 0", "layer 1"])
    ev = json.load(open(path))["traceEvents"]
    tiles = [e for e in ev if e["ph"] == "X" and e["name"] == "gemm"]
    assert len(tiles) == int(real.sum())
    assert {e["tid"] for e in tiles} == set(int(x) for x in tr[real, 5])
    assert all(e["dur"] >= 0 and e["args"]["node_name"].startswith("layer") for e in tiles)


# ------------------------------------------------------------------ CTA pairs (cta_group::2)

PAIR = dict(gemm_tile_m=256, cluster=2)


@pytest.mark.parametrize("m,n,k,tn,dt", [
    (256, 128, 64, 128, "f16"), (256, 256, 256, 256, "f16"), (300, 392, 200, 256, "f16"),
    (129, 72, 520, 128, "bf16"), (1000, 1024, 776, 256, "bf16"), (512, 512, 1024, 128, "f16")])
def test_pair_gemm_full_compare(m, n, k, tn, dt):
    wl = workloads.gemm(m, n, k, dtype=dt, device=DEV, seed=m + n + k + 1)
    opts = dict(PAIR, gemm_tile_n=tn)
    plan, _ = run(wl, **opts)
    ref = ops.matmul(f32(wl.data[0]), f32(wl.data[1]), F16 if dt == "f16" else BF16)
    assert_close(f32(wl.data[2]), ref, f"pair gemm {m}x{n}x{k}")
    check_counters(plan, wl, opts)


def test_pair_gemm_4096_sampled_rows():
    wl = workloads.gemm(4096, 4096, 4096, dtype="f16", device=DEV, seed=0)
    plan, _ = run(wl, **PAIR)
    rows = np.sort(torch.randperm(4096, generator=torch.Generator().manual_seed(1))[:256].numpy())
    a = f32(wl.data[0][torch.as_tensor(rows, device=DEV)])
    ref = ops.matmul(a, f32(wl.data[1]), F16)
    assert_close(f32(wl.data[2][torch.as_tensor(rows, device=DEV)]), ref, "pair 4096^3 rows")
    check_counters(plan, wl, PAIR)


def test_split_tail_gemm_4096_sampled_rows():
    wl = workloads.gemm(4096, 4096, 4096, dtype="f16", device=DEV, seed=0)
    opts = dict(PAIR, gemm_split_tail=1)
    plan, _ = run(wl, **opts)
    rows = np.sort(torch.randperm(4096, generator=torch.Generator().manual_seed(2))[:256].numpy())
    a = f32(wl.data[0][torch.as_tensor(rows, device=DEV)])
    ref = ops.matmul(a, f32(wl.data[1]), F16)
    assert_close(f32(wl.data[2][torch.as_tensor(rows, device=DEV)]), ref, "split tail 4096^3")
    check_counters(plan, wl, opts)


def test_pair_epilogues_and_mixed_graph():
    """Pair GEMMs with bias/ReLU/residual and SiLU·mul epilogues, then a GEMV and a norm in the
    same launch, so the two CTAs of a pair also run unrelated instructions between pair tiles."""
    m, n, k = 384, 512, 320
    a = synth.normal((m, k), 1.0, "bf16", 11, DEV)
    b = synth.normal((k, n), 1 / math.sqrt(k), "bf16", 12, DEV)
    bu = synth.normal((k, n), 1 / math.sqrt(k), "bf16", 13, DEV)
    bias = synth.normal((m, n), 0.5, "bf16", 14, DEV)
    res = synth.normal((m, n), 1.0, "bf16", 15, DEV)
    w2 = synth.normal((n, 768), 1 / math.sqrt(n), "bf16", 16, DEV)
    o1, o2 = (torch.zeros((m, n), dtype=torch.bfloat16, device=DEV) for _ in range(2))
    o3 = torch.zeros((1, 768), dtype=torch.bfloat16, device=DEV)
    from tensor_core_gemm_gb300 import Graph
    g = Graph()
    ia, ib, ibu, ibias, ires, i1, i2, iw2, i3 = (
        g.tensor(t) for t in (a, b, bu, bias, res, o1, o2, w2, o3))
    g.matmul(ia, ib, i1, bias=ibias, relu=True, residual=ires)
    g.matmul(ia, ib, i2, b_up=ibu)
    g.matmul(g.view(i1, 0, 0, 1, n), iw2, i3)
    p = g.compile(gemm_tile_n=256, **PAIR)
    p.run()
    p.check_status()
    A, B, BU = f32(a), f32(b), f32(bu)
    r1 = ops.matmul(A, B, BF16, bias=f32(bias), relu=True, residual=f32(res))
    assert_close(f32(o1), r1, "pair bias+relu+residual")
    assert_close(f32(o2), ops.matmul_silu_mul(A, B, BU, BF16), "pair silu_mul")
    assert_close(f32(o3), ops.matmul(f32(o1)[:1], f32(w2), BF16), "gemv after pair tiles")
    p.run()                                   # a second launch reuses the reset counters
    p.check_status()
    assert_close(f32(o1), r1, "pair second launch")


def test_pair_options_rejected_by_the_kernel_check():
    from tensor_core_gemm_gb300._lib import MkError
    wl = workloads.gemm(256, 256, 256, dtype="f16", device=DEV)
    g, _ = workloads.build_graph(wl.desc, wl.data)
    for bad in (dict(gemm_tile_m=256, cluster=1), dict(gemm_tile_m=128, cluster=2),
                dict(gemm_tile_m=256, cluster=2, gemm_tile_n=64),
                dict(gemm_tile_m=256, cluster=2, n_sm=151)):
        with pytest.raises(MkError):
            g.compile(**bad)


# ------------------------------------------------------------------ causal prefill attention

@pytest.mark.parametrize("pair", [False, True])
@pytest.mark.parametrize("tq,tk,hq,hkv,causal,pos0", [
    (128, 128, 4, 2, True, 0), (200, 200, 8, 2, True, 0), (384, 384, 32, 8, True, 0),
    (130, 300, 4, 4, False, 0), (64, 192, 4, 2, True, 128), (1, 64, 2, 1, True, 0),
    (640, 640, 4, 1, True, 0)])
def test_attention_prefill(tq, tk, hq, hkv, causal, pos0, pair):
    """Causal (and non-causal) prefill attention against the oracle; on CTA pairs a 256-row
    query tile runs as cta_group::2 MMAs with each CTA's softmax on its own 128 rows."""
    if tq == 1:
        pytest.skip("a single query row lowers to split-KV decode tiles")
    d = 64
    q = synth.normal((tq, hq * d), 1.0, "bf16", 60 + tq, DEV)
    k = synth.normal((tk, hkv * d), 1.0, "bf16", 61 + tk, DEV)
    v = synth.normal((tk, hkv * d), 1.0, "bf16", 62, DEV)
    out = torch.zeros((tq, hq * d), dtype=torch.bfloat16, device=DEV)
    from tensor_core_gemm_gb300 import Graph
    g = Graph()
    iq, ik, iv, io = g.tensor(q), g.tensor(k), g.tensor(v), g.tensor(out)
    g.attention(iq, ik, iv, io, n_q_heads=hq, n_kv_heads=hkv, head_dim=d, causal=causal,
                q_pos0=pos0)
    p = g.compile(**(PAIR if pair else {}))
    assert p.stats()["kernel_set"] == 3
    p.run()
    p.check_status()
    ref = ops.attention(f32(q), f32(k), f32(v), hq, hkv, d, causal, pos0, 1 / 8, BF16)
    assert_close(f32(out), ref, f"prefill attention {tq}x{tk}")
    if causal and pos0 == 0:
        # row 0 sees key 0 alone: its output is v_0 of the head's key/value head, exactly
        for h in range(hq):
            gg = h // (hq // hkv)
            assert torch.equal(out[0, h * d:(h + 1) * d], v[0, gg * d:(gg + 1) * d])
    p.run()                                   # a second launch gives the same bytes
    p.check_status()
    again = out.clone()
    p.run()
    p.check_status()
    assert torch.equal(out, again)


# ------------------------------------------------------------------ decoder, causal prefill

def _prefill_weights(wl):
    sh = wl.info["shape"]
    L, d, f = sh.layers, sh.hidden, sh.ffn
    D = wl.data
    w = wl.info["w"]
    return models.DecoderWeights(
        f32(D[w["wqkv"]]).reshape(L, d, sh.qkv), f32(D[w["wo"]]).reshape(L, sh.hq * sh.hd, d),
        f32(D[w["wg"]]).reshape(L, d, f), f32(D[w["wu"]]).reshape(L, d, f),
        f32(D[w["wd"]]).reshape(L, f, d), f32(D[w["g_attn"]]), f32(D[w["g_mlp"]]),
        sh.hq, sh.hkv, sh.hd, sh.eps, sh.theta)


def check_prefill_per_node(wl, rows):
    """Every node of every layer on query rows [0, rows) against the oracle applied to the GPU's
    own inputs of that node (teacher forcing). Row t of every prefill output depends only on
    rows 0..t, so a prefix of the rows is checked exactly by running the oracle on it."""
    sh = wl.info["shape"]
    wts = _prefill_weights(wl)
    D, T = wl.data, wl.info["tokens"]
    hq, hkv, hd = sh.hq, sh.hkv, sh.hd
    L = sh.layers

    def node(key):
        return f32(D[wl.info[key]]).reshape(L, T, -1)[:, :rows]

    xn, qkv, qr, kr, att, hh, hn, gu, xo = (node(k) for k in ("xn", "qkv", "qr", "kr", "att",
                                                               "h", "hn", "gu", "out"))
    pos = np.arange(rows)
    x_prev = f32(D[0])[:rows]
    for l in range(L):
        assert_close(xn[l], ops.rmsnorm(x_prev, wts.g_attn[l], sh.eps, BF16), f"rmsnorm {l}")
        assert_close(qkv[l], ops.matmul(xn[l], wts.wqkv[l], BF16), f"qkv {l}")
        assert_close(qr[l], ops.rope(qkv[l][:, :hq * hd], pos, hq, hd, sh.theta, BF16),
                     f"rope q {l}")
        assert_close(kr[l], ops.rope(qkv[l][:, hq * hd:(hq + hkv) * hd], pos, hkv, hd, sh.theta,
                                     BF16), f"rope k {l}")
        v = qkv[l][:, (hq + hkv) * hd:]
        assert_close(att[l], ops.attention(qr[l], kr[l], v, hq, hkv, hd, True, 0,
                                           1 / math.sqrt(hd), BF16), f"attention {l}")
        assert_close(hh[l], ops.matmul(att[l], wts.wo[l], BF16, residual=x_prev), f"o-proj {l}")
        assert_close(hn[l], ops.rmsnorm(hh[l], wts.g_mlp[l], sh.eps, BF16), f"rmsnorm mlp {l}")
        assert_close(gu[l], ops.matmul_silu_mul(hn[l], wts.wg[l], wts.wu[l], BF16),
                     f"gate/up {l}")
        assert_close(xo[l], ops.matmul(gu[l], wts.wd[l], BF16, residual=hh[l]), f"down {l}")
        x_prev = xo[l]


@pytest.mark.parametrize("pair", [False, True])
def test_prefill_small_decoder(pair):
    """A 2-layer decoder prefill node by node and end to end; on CTA pairs the GEMMs run
    256x256 pair tiles and the causal attention 256-row pair tiles."""
    sh = workloads.DecoderShape(layers=2, hidden=256, n_q_heads=4, n_kv_heads=2, head_dim=64,
                                ffn=512)
    wl = workloads.prefill(sh, tokens=384, device=DEV, seed=7)
    opts = dict(PAIR) if pair else {}
    plan, _ = run(wl, **opts)
    check_counters(plan, wl, opts)
    check_prefill_per_node(wl, 384)
    # end to end against the oracle's own chain
    ref = models.prefill(f32(wl.data[0]), _prefill_weights(wl))
    got = f32(wl.data[wl.info["out"]]).reshape(2, 384, -1)[-1]
    assert_close(got, ref, "prefill output")


@pytest.mark.parametrize("pair", [False, True])
def test_prefill_repeated_runs_report_no_failure(pair):
    """Hand-off races show as a wait that never ends in a few runs out of hundreds: a 4-layer,
    2048-token prefill runs 300 times and the plan's status, which keeps the first failure of
    any run until it is read, stays clean; the last run's output matches the first run's."""
    sh = workloads.DecoderShape(layers=4)
    wl = workloads.prefill(sh, device=DEV, seed=0)
    g, _ = workloads.build_graph(wl.desc, wl.data)
    p = g.compile(**(dict(PAIR) if pair else {}))
    p.run()
    p.check_status()
    out = wl.info["out"]
    first = wl.data[out].clone()
    for _ in range(300):
        p.run()
    p.check_status()
    assert torch.equal(wl.data[out], first)


def test_status_keeps_the_first_failure_until_read():
    """A run that times out, then clean runs: the status still reports the timeout (read once),
    and reads clean afterwards."""
    wl = workloads.mlp3(m=256, h=256, layers=2, device=DEV)
    g, _ = workloads.build_graph(wl.desc, wl.data)
    bad = g.compile(debug_counter=0, debug_extra=1, timeout_ms=50, gemm_tile_n=64)
    bad.run()
    torch.cuda.synchronize()
    # the same plan's status: a clean run of another plan does not touch it; this plan's next
    # runs would time out again, so read it once and check it is cleared
    code, st = bad.sync_status()
    assert code == MK_ERR_TIMEOUT
    code, st = bad.sync_status()
    assert code == 0
    good = g.compile(gemm_tile_n=64)
    good.run()
    good.run()
    good.check_status()


@pytest.mark.parametrize("pair", [False, True])
def test_prefill_full_config_causal_prefix(pair):
    wl = workloads.prefill(device=DEV, seed=0)
    opts = dict(PAIR) if pair else {}
    plan, _ = run(wl, **opts)
    check_counters(plan, wl, opts)
    check_prefill_per_node(wl, 256)
    # End to end over all 16 layers: rows 0..255 of the last layer's output depend only on the
    # first 256 tokens, so the oracle runs the whole decoder on that prefix. Held to MARGIN
    # times the oracle-vs-oracle drift measured on the same prefix (~1.7e-2 after 16 layers,
    # tests/test_oracle_drift.py).
    sh, T = wl.info["shape"], wl.info["tokens"]
    rows = 256
    drift, ref = _drift.prefill_drift(f32(wl.data[0])[:rows], _prefill_weights(wl))
    got = f32(wl.data[wl.info["out"]]).reshape(sh.layers, T, -1)[-1, :rows]
    ok, seen = _drift.within_drift(got, ref, drift)
    assert ok, f"16-layer prefill prefix: gap {seen} against oracle drift {drift}"


# ------------------------------------------------------------------ GEMM split tails

@pytest.mark.parametrize("pair", [False, True])
def test_split_tail_epilogues(pair):
    """Few tiles on many SMs: every tile is a split-tail tile, split along K down to one or two
    k-steps per split; the last split sums the fp32 partials and runs each fused epilogue."""
    m, n, k = (384, 512, 640) if not pair else (512, 512, 1024)
    opts = dict(gemm_tile_m=256, cluster=2, gemm_tile_n=256) if pair else dict(gemm_tile_n=256)
    opts["gemm_split_tail"] = 1
    a = synth.normal((m, k), 1.0, "bf16", 21, DEV)
    b = synth.normal((k, n), 1 / math.sqrt(k), "bf16", 22, DEV)
    bu = synth.normal((k, n), 1 / math.sqrt(k), "bf16", 23, DEV)
    bias = synth.normal((m, n), 0.5, "bf16", 24, DEV)
    res = synth.normal((m, n), 1.0, "bf16", 25, DEV)
    o1, o2, o3 = (torch.zeros((m, n), dtype=torch.bfloat16, device=DEV) for _ in range(3))
    from tensor_core_gemm_gb300 import Graph
    g = Graph()
    ia, ib, ibu, ibias, ires, i1, i2, i3 = (g.tensor(t) for t in (a, b, bu, bias, res, o1, o2, o3))
    g.matmul(ia, ib, i1, bias=ibias, relu=True, residual=ires)
    g.matmul(ia, ib, i2, b_up=ibu)
    g.matmul(ia, ib, i3)
    p = g.compile(**opts)
    ins = p.instructions()
    assert np.any(ins["aux1"][ins["op"] == osched.OP_GEMM] > 1), "no split-tail tiles"
    p.run()
    p.check_status()
    A, B, BU = f32(a), f32(b), f32(bu)
    assert_close(f32(o1), ops.matmul(A, B, BF16, bias=f32(bias), relu=True, residual=f32(res)),
                 "split tail bias+relu+residual")
    assert_close(f32(o2), ops.matmul_silu_mul(A, B, BU, BF16), "split tail silu_mul")
    assert_close(f32(o3), ops.matmul(A, B, BF16), "split tail plain")
    # the partials are summed in split order: repeat launches give the same bytes
    first = o3.clone()
    p.run()
    p.check_status()
    assert torch.equal(o3, first)
    # and the unsplit plan agrees within the tolerance
    o3.zero_()
    g2 = Graph()
    j = [g2.tensor(t) for t in (a, b, o3)]
    g2.matmul(j[0], j[1], j[2])
    p2 = g2.compile(**dict(opts, gemm_split_tail=0))
    p2.run()
    p2.check_status()
    assert_close(f32(o3), f32(first), "split vs unsplit")


@pytest.mark.parametrize("pair", [False, True])
def test_split_tail_two_splits_exchange_halves(pair):
    """A tail of exactly two K splits per tile (n_sm chosen so): each split stores the half of its
    partial the other finishes, both finish their half (bias + ReLU + residual, plain, ragged last
    column tile), the later one publishes; SiLU·mul tiles keep the last-split sum. Counters and
    semaphores end at the oracle's values; a consumer GEMV reads the split tiles' output."""
    full = workloads.full
    m, n, k = (768, 1000, 384) if pair else (384, 1000, 256)
    opts = dict(gemm_tile_m=256, cluster=2, gemm_tile_n=256) if pair else dict(gemm_tile_n=256)
    opts.update(n_sm=16 if pair else 8, gemm_split_tail=1)
    shapes = [(m, k), (k, n), (k, n), (m, n), (m, n), (m, n), (m, n), (m, n), (n, 256), (1, 256)]
    desc = {"tensors": [{"rows": r, "cols": c, "dtype": "bf16"} for r, c in shapes],
            "nodes": [
                {"kind": "matmul", "a": full(0, m, k), "b": full(1, k, n), "c": full(5, m, n),
                 "bias": full(3, m, n), "relu": True, "residual": full(4, m, n)},
                {"kind": "matmul", "a": full(0, m, k), "b": full(1, k, n), "b2": full(2, k, n),
                 "c": full(6, m, n)},
                {"kind": "matmul", "a": full(0, m, k), "b": full(1, k, n), "c": full(7, m, n)},
                {"kind": "matmul", "a": (5, m - 1, 0, 1, n), "b": full(8, n, 256),
                 "c": full(9, 1, 256)}]}
    data = [synth.normal((m, k), 1.0, "bf16", 41, DEV),
            synth.normal((k, n), 1 / math.sqrt(k), "bf16", 42, DEV),
            synth.normal((k, n), 1 / math.sqrt(k), "bf16", 43, DEV),
            synth.normal((m, n), 0.5, "bf16", 44, DEV),
            synth.normal((m, n), 1.0, "bf16", 45, DEV)]
    data += [torch.zeros((m, n), dtype=torch.bfloat16, device=DEV) for _ in range(3)]
    data += [synth.normal((n, 256), 1 / math.sqrt(n), "bf16", 46, DEV),
             torch.zeros((1, 256), dtype=torch.bfloat16, device=DEV)]
    g, _ = workloads.build_graph(desc, data)
    p = g.compile(snapshot_counters=1, **opts)
    ins = p.instructions()
    gem = ins["op"] == osched.OP_GEMM
    assert np.all(np.isin(ins["aux1"][gem], [0, 2])) and np.any(ins["aux1"][gem] == 2)
    p.run()
    p.check_status()
    A, B, BU = f32(data[0]), f32(data[1]), f32(data[2])
    ref1 = ops.matmul(A, B, BF16, bias=f32(data[3]), relu=True, residual=f32(data[4]))
    assert_close(f32(data[5]), ref1, "two splits bias+relu+residual")
    assert_close(f32(data[6]), ops.matmul_silu_mul(A, B, BU, BF16), "two splits silu_mul")
    assert_close(f32(data[7]), ops.matmul(A, B, BF16), "two splits plain")
    assert_close(f32(data[9]), ops.matmul(f32(data[5])[m - 1:], f32(data[8]), BF16),
                 "consumer of split tiles")
    assert p.counters().tolist() == osched.lower(desc, opts).final_counters()
    first = data[7].clone()
    p.run()
    p.check_status()
    assert torch.equal(data[7], first), "the split sum order is fixed"


def test_pair_gemms_interleaved_with_gemvs():
    """Pair GEMM tiles after GEMV tiles in one launch: the two CTAs of a pair arrive with rings
    in different states and resynchronise; consecutive pair tiles stream on without it."""
    from tensor_core_gemm_gb300 import Graph
    shapes = [("gemv", 1, 512, 768), ("gemm", 300, 256, 512), ("gemv", 3, 1024, 512),
              ("gemm", 512, 384, 256), ("gemm", 700, 448, 512), ("gemv", 2, 640, 256)]
    g = Graph()
    data, outs = [], []
    for i, (_, m, k, n) in enumerate(shapes):
        a = synth.normal((m, k), 1.0, "bf16", 80 + i, DEV)
        b = synth.normal((k, n), 1 / math.sqrt(k), "bf16", 90 + i, DEV)
        c = torch.zeros((m, n), dtype=torch.bfloat16, device=DEV)
        data.append((a, b))
        outs.append(c)
        g.matmul(g.tensor(a), g.tensor(b), g.tensor(c))
    p = g.compile(**PAIR)
    for _ in range(2):
        p.run()
        p.check_status()
        for (kind, m, k, n), (a, b), c in zip(shapes, data, outs):
            assert_close(f32(c), ops.matmul(f32(a), f32(b), BF16), f"{kind} {m}x{k}x{n}")


def test_decode_rope_fused_and_unfused_agree():
    """RoPE inside the QKV GEMV tiles (default) and RoPE as its own row instruction give the
    same decode step bit for bit (both rotate the rounded QKV output with the same angle and
    rounding steps)."""
    sh = workloads.DecoderShape(layers=2, hidden=512, n_q_heads=8, n_kv_heads=2, head_dim=64,
                                ffn=1024)
    outs = []
    for fuse in (1, 0):
        wl = workloads.decode(sh, kv_len=130, device=DEV, seed=9)
        plan, _ = run(wl, fuse_rope=fuse)
        assert (plan.stats()["per_op"][osched.OP_ROPE] == 0) == bool(fuse)
        outs.append({k: wl.data[wl.info[k]].clone() for k in ("qr", "kc", "vc", "out")})
    for k in ("qr", "kc", "vc", "out"):
        assert torch.equal(outs[0][k].view(torch.int16), outs[1][k].view(torch.int16)), k


def test_prefill_rope_fused_and_unfused_bit_identical():
    """RoPE inside the QKV GEMM tiles' epilogue (default) and RoPE as row instructions (staged
    16-row blocks, and direct 96-row blocks) rotate the same rounded QKV outputs with the same
    angle steps: q, k and the layer outputs agree bit for bit."""
    sh = workloads.DecoderShape(layers=2, hidden=512, n_q_heads=8, n_kv_heads=2, head_dim=64,
                                ffn=1024)
    outs = []
    for opts in (dict(), dict(fuse_rope=0), dict(fuse_rope=0, norm_rows=96)):
        wl = workloads.prefill(sh, tokens=200, device=DEV, seed=12)
        plan, _ = run(wl, **opts)
        assert (plan.stats()["per_op"][osched.OP_ROPE] == 0) == ("fuse_rope" not in opts)
        outs.append([wl.data[wl.info[k]].clone() for k in ("qr", "kr", "qkv", "out")])
    for other in outs[1:]:
        for name, a, b in zip(("qr", "kr", "qkv", "out"), outs[0], other):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16)), name


@pytest.mark.parametrize("kind", ["decode", "prefill", "prefill_ragged", "prefill_rows96",
                                  "prefill_unfused", "gemm", "gemm_pair", "mlp3"])
def test_kernel_specialisations_bit_identical(kind):
    """The specialisation mk_run picks for a plan and the general kernel (kernel_set = 1) give
    bit-identical outputs; the specialisation is the one the plan statistics name. The prefill
    specialisation's register-resident RMSNorm rows and tabled RoPE angles take the same
    arithmetic in the same order as the general kernel's two-pass loops."""
    sh = workloads.DecoderShape(layers=2, hidden=512, n_q_heads=8, n_kv_heads=2, head_dim=64,
                                ffn=1024)
    pair = dict(gemm_tile_m=256, cluster=2)
    make, opts, want = {
        "decode": (lambda: workloads.decode(sh, kv_len=130, device=DEV, seed=9), {}, 2),
        "prefill": (lambda: workloads.prefill(sh, tokens=320, device=DEV, seed=3), {}, 3),
        # a ragged last row block; row blocks too tall for the shared RoPE angle table
        "prefill_ragged": (lambda: workloads.prefill(sh, tokens=200, device=DEV, seed=6), {}, 3),
        "prefill_rows96": (lambda: workloads.prefill(sh, tokens=320, device=DEV, seed=8),
                           dict(norm_rows=96, fuse_rope=0), 3),
        # RoPE as row instructions (staged blocks) instead of in the QKV tiles
        "prefill_unfused": (lambda: workloads.prefill(sh, tokens=200, device=DEV, seed=6),
                            dict(fuse_rope=0), 3),
        "gemm": (lambda: workloads.gemm(640, 768, 1088, device=DEV, seed=4), {}, 1),
        "gemm_pair": (lambda: workloads.gemm(640, 768, 1088, device=DEV, seed=4), pair, 1),
        "mlp3": (lambda: workloads.mlp3(device=DEV), dict(gemm_tile_n=64), 1),
    }[kind]
    outs = []
    for ks in (0, 1):
        wl = make()
        plan, _ = run(wl, kernel_set=ks, **opts)
        assert plan.stats()["kernel_set"] == (want if ks == 0 else 0)
        outs.append([t.clone() for t in wl.data])
    for i, (a, b) in enumerate(zip(*outs)):
        assert torch.equal(a.view(torch.int16) if a.element_size() == 2 else a,
                           b.view(torch.int16) if b.element_size() == 2 else b), f"tensor {i}"


def test_kernel_set_option_validated():
    g, _ = workloads.build_graph(workloads.gemm(64, 64, 64).desc, None)
    with pytest.raises(Exception, match="kernel_set"):
        g.compile(kernel_set=2)
    with pytest.raises(Exception, match="row_stage"):
        g.compile(row_stage=2)


# ------------------------------------------------------------------ greedy sampling (ARGMAX)

@pytest.mark.parametrize("rows,cols,dt,chunk", [(1, 128256, "bf16", 4096), (37, 10000, "bf16", 1024),
                                               (5, 777, "f16", 64), (3, 4096, "bf16", 4096)])
def test_argmax_rows_exact(rows, cols, dt, chunk):
    """The chosen column is bit-exact against the oracle on the same stored values, including
    planted ties (the lower column wins), NaN entries (skipped) and a row of NaN (-1)."""
    x = synth.normal((rows, cols), 1.0, dt, 61, DEV)
    if rows > 1:
        x[1, cols // 3] = 8.0
        x[1, cols - 1] = 8.0
        x[min(2, rows - 1), :] = float("nan")
    if rows > 3:
        x[3, 0] = float("nan")
        x[3, cols // 2] = 9.0
    out = torch.full((rows, 1), -7, dtype=torch.int32, device=DEV)
    from tensor_core_gemm_gb300 import Graph
    g = Graph()
    ix, io = g.tensor(x), g.tensor(out)
    g.argmax(ix, io)
    p = g.compile(argmax_chunk=chunk, snapshot_counters=1)
    p.run()
    p.check_status()
    want = ops.argmax_rows(f32(x))
    assert out.cpu().numpy().tolist() == want.tolist()


def test_decode_greedy_sampling_head():
    """Final RMSNorm fused into the lm_head GEMV, then ARGMAX: the logits match the oracle's
    head applied to the GPU's last residual row, and the token is exactly the first maximum of
    the GPU's own logits (and the oracle's token where its top two logits are apart)."""
    sh = workloads.DecoderShape(layers=2, hidden=512, n_q_heads=8, n_kv_heads=2, head_dim=64,
                                ffn=1024)
    wl = workloads.decode(sh, kv_len=130, device=DEV, seed=5, vocab=5000)
    plan, _ = run(wl)
    check_counters(plan, wl, {})
    info = wl.info
    x_last = f32(wl.data[info["out"]])[-1:]
    logits_ref, token_ref = models.decode_head(x_last, f32(wl.data[info["g_f"]])[0], f32(wl.data[info["w_lm"]]),
                                               sh.eps)
    logits = f32(wl.data[info["logits"]])
    assert_close(logits, logits_ref, "logits")
    token = int(wl.data[info["token"]].item())
    assert token == int(ops.argmax_rows(logits)[0, 0])
    top = np.sort(logits_ref[0])[-2:]
    if top[1] - top[0] > 2e-2 * max(1.0, abs(top[1])):
        assert token == int(token_ref[0, 0])


# ------------------------------------------------------------------ Llama-70B GEMM lists

@pytest.mark.parametrize("which", ["prefill", "decode"])
def test_llama_gemm_lists_full_size_sampled_rows(which):
    """The Llama-70B linear lists at full size in the benchmark's launch configuration (CTA
    pairs, grouped tile order, wave packing): 64 seeded rows of every GEMM against the oracle."""
    shapes = workloads.LLAMA70B_PREFILL if which == "prefill" else workloads.LLAMA70B_DECODE
    wl = workloads.gemm_list(shapes, device=DEV, seed=0)
    opts = dict(gemm_tile_m=256, cluster=2)
    plan, _ = run(wl, **opts)
    check_counters(plan, wl, opts)
    gen = torch.Generator().manual_seed(11)
    for (a, b, c, m, n, k) in wl.info["gemms"]:
        rows = np.sort(torch.randperm(m, generator=gen)[:64].numpy())
        idx = torch.as_tensor(rows, device=DEV)
        ref = ops.matmul(f32(wl.data[a][idx]), f32(wl.data[b]), F16)
        assert_close(f32(wl.data[c][idx]), ref, f"{which} {m}x{n}x{k}")


def test_tile_order_and_wave_packing_bit_identical():
    """Grouped tile order and wave packing only move tiles between SMs: the outputs of a list of
    independent GEMMs with different K agree bit for bit with row-major, unpacked placement."""
    shapes = [(256, 1024, 512), (300, 768, 2048), (256, 512, 3072), (512, 1280, 1024)]
    outs = []
    for opts in (dict(), dict(wave_pack=0, gemm_group_m=1)):
        wl = workloads.gemm_list(shapes, device=DEV, seed=3)
        run(wl, gemm_tile_m=256, cluster=2, **opts)
        outs.append([wl.data[c].clone() for (_, _, c, _, _, _) in wl.info["gemms"]])
    for x, y in zip(*outs):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
