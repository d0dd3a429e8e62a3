"""Pins of the oracle to facts other than itself (CPU only).

Each test checks an oracle function against something it does not share code with: values the
pages print (tests/golden, cited there), closed forms, brute-force fp64 loops, special cases
that reduce to a textbook or library routine, or invariants of the mathematics.
"""
import math

import numpy as np
import pytest

from conftest import golden_matrix, read_golden
from oracle import models, ops, schedule
from oracle.numerics import BF16, F16, F32, bf16_bits_to_f32, f32_to_bf16_bits, round_to

import _graphs

RNG = np.random.default_rng(1234)


# ----------------------------------------------------------------------------- numerics
def test_bf16_rounding_grid():
    # bf16 keeps 7 mantissa bits: ulp(1) = 2^-7.
    one_plus_half_ulp = np.float32(1 + 2 ** -8)          # exact tie -> even (1.0)
    three_half_ulps = np.float32(1 + 3 * 2 ** -8)        # tie between odd and even -> 1 + 2^-6
    assert round_to(one_plus_half_ulp, BF16) == 1.0
    assert round_to(three_half_ulps, BF16) == np.float32(1 + 2 ** -6)
    assert round_to(np.float32(1 + 2 ** -8 + 2 ** -20), BF16) == np.float32(1 + 2 ** -7)
    assert f32_to_bf16_bits(np.float32(1.0)) == 0x3F80
    assert f32_to_bf16_bits(np.float32(-2.0)) == 0xC000
    assert f32_to_bf16_bits(np.float32(math.pi)) == 0x4049
    big = np.float32((2 - 2 ** -7) * 2.0 ** 127)          # largest finite bf16
    assert round_to(big, BF16) == big
    assert np.isinf(round_to(np.float32(3.4028235e38), BF16))
    tiny = np.float32(2.0 ** -133)                        # smallest bf16 subnormal
    assert round_to(tiny, BF16) == tiny
    assert bf16_bits_to_f32(np.uint16(0x7F80)) == np.inf
    assert np.isnan(round_to(np.float32(np.nan), BF16))


def test_fp16_rounding_grid():
    assert round_to(np.float32(2049.0), F16) == 2048.0    # tie -> even
    assert round_to(np.float32(2051.0), F16) == 2052.0
    assert round_to(np.float32(65504.0), F16) == 65504.0
    assert np.isinf(round_to(np.float32(65520.0), F16))   # tie above max -> inf


# ----------------------------------------------------------------------------- matmul
def test_matmul_epilogue_golden():
    g = read_golden("matmul_epilogue_2x2.txt")
    a, b = golden_matrix(g["A"]), golden_matrix(g["B"])
    np.testing.assert_array_equal(ops.matmul(a, b, F32), golden_matrix(g["plain"]))
    bias = golden_matrix(g["bias"])
    np.testing.assert_array_equal(ops.matmul(a, b, F32, bias=bias, relu=True),
                                  golden_matrix(g["bias_relu"]))
    res = golden_matrix(g["residual"])
    np.testing.assert_array_equal(ops.matmul(a, b, F32, bias=bias, relu=True, residual=res),
                                  golden_matrix(g["bias_relu_residual"]))


def _brute_matmul(a, b):
    m, k = a.shape
    n = b.shape[1]
    c = np.zeros((m, n), np.float64)
    for i in range(m):
        for j in range(n):
            s = 0.0
            for t in range(k):
                s += float(a[i, t]) * float(b[t, j])
            c[i, j] = s
    return c


def test_matmul_brute_force():
    a = round_to(RNG.standard_normal((7, 13)), F16)
    b = round_to(RNG.standard_normal((13, 5)), F16)
    bias = round_to(RNG.standard_normal((7, 5)), F16)
    res = round_to(RNG.standard_normal((7, 5)), F16)
    ref = np.maximum(_brute_matmul(a, b) + bias, 0.0) + res
    got = ops.matmul(a, b, F32, bias=bias, relu=True, residual=res)
    np.testing.assert_allclose(got, ref, rtol=1e-5, atol=1e-5)
    # one rounding to fp16 at the end
    np.testing.assert_array_equal(ops.matmul(a, b, F16, bias=bias, relu=True, residual=res),
                                  round_to(got, F16))


def test_mlp_identity_weights_gives_relu():
    # spec invariant: W = I and b = 0 gives relu(x) exactly.
    x = round_to(RNG.standard_normal((64, 64)), F16)
    w = np.stack([np.eye(64, dtype=np.float32)] * 3)
    b = np.zeros((3, 64, 64), np.float32)
    outs = models.mlp(x, w, b)
    np.testing.assert_array_equal(outs[0], np.maximum(x, 0))
    np.testing.assert_array_equal(outs[-1], np.maximum(x, 0))


def test_mlp_fused_matches_unfused_within_rounding():
    x = round_to(RNG.standard_normal((32, 48)), F16)
    w = round_to(RNG.standard_normal((3, 48, 48)) / np.sqrt(48), F16)
    b = round_to(0.1 * RNG.standard_normal((3, 32, 48)), F16)
    fused = models.mlp(x, w, b)[-1]
    unfused = models.mlp_unfused(x, w, b, F16)[-1][2]
    assert np.max(np.abs(fused - unfused)) < 2e-2 * max(1.0, np.max(np.abs(fused)))


def test_silu_mul_with_identity_up():
    # SiLU·mul of the gate product with an identity up-projection is silu(A·Wg) ⊙ A.
    a = round_to(RNG.standard_normal((16, 16)), BF16)
    wg = round_to(RNG.standard_normal((16, 16)) / 4, BF16)
    got = ops.matmul_silu_mul(a, wg, np.eye(16, dtype=np.float32), BF16)
    z = a.astype(np.float64) @ wg.astype(np.float64)
    ref = z / (1.0 + np.exp(-z)) * a          # up product with W_up = I is A itself
    np.testing.assert_allclose(got, round_to(ref.astype(np.float32), BF16), rtol=1e-2, atol=1e-2)
    assert abs(float(ops.silu(np.float32(1.0))) - 1.0 / (1.0 + math.exp(-1.0))) < 1e-7
    assert float(ops.silu(np.float32(0.0))) == 0.0


# ----------------------------------------------------------------------------- rmsnorm
def test_rmsnorm_golden():
    g = read_golden("rmsnorm_small.txt")
    x = golden_matrix(g["x"])
    gamma = golden_matrix(g["gamma"]).reshape(-1)
    y = ops.rmsnorm(x, gamma, float(g["eps"]), F32)
    np.testing.assert_allclose(y, golden_matrix(g["y"]), rtol=1e-6)


def test_rmsnorm_constant_row_and_scale_invariance():
    c, eps = 3.0, 1e-5
    gamma = round_to(1 + 0.02 * RNG.standard_normal(8), BF16)
    y = ops.rmsnorm(np.full((1, 8), c, np.float32), gamma, eps, F32)
    np.testing.assert_allclose(y[0], gamma * c / math.sqrt(c * c + eps), rtol=1e-6)
    x = RNG.standard_normal((4, 32)).astype(np.float32)
    np.testing.assert_allclose(ops.rmsnorm(x, np.ones(32), 0.0, F32),
                               ops.rmsnorm(7.5 * x, np.ones(32), 0.0, F32), rtol=1e-5)


def test_norm_input_gemv_matches_fp64():
    x = round_to(RNG.standard_normal((1, 64)), BF16)
    gamma = round_to(1 + 0.02 * RNG.standard_normal(64), BF16)
    w = round_to(0.1 * RNG.standard_normal((64, 24)), BF16)
    res = round_to(RNG.standard_normal((1, 24)), BF16)
    x64 = x.astype(np.float64)
    xn = x64 / np.sqrt(np.mean(x64 ** 2) + 1e-5) * gamma
    ref = xn @ w + res
    got = ops.matmul_norm_input(x, gamma, 1e-5, w, F32, residual=res)
    np.testing.assert_allclose(got, ref, rtol=1e-5, atol=1e-5)


# ----------------------------------------------------------------------------- rope
def test_rope_is_complex_rotation():
    # Pairs (i, i+h) form the complex number x_i + j·x_{i+h}; rope multiplies it by
    # exp(j·p·theta^(-2i/d)). Checked with numpy complex arithmetic.
    d, heads, theta = 8, 3, 5e5
    pos = np.array([0, 1, 17, 1024])
    x = RNG.standard_normal((4, heads * d)).astype(np.float32)
    got = ops.rope(x, pos, heads, d, theta, F32)
    h = d // 2
    for t in range(4):
        for hd in range(heads):
            seg = x[t, hd * d:(hd + 1) * d].astype(np.float64)
            z = seg[:h] + 1j * seg[h:]
            rot = z * np.exp(1j * pos[t] * theta ** (-2.0 * np.arange(h) / d))
            np.testing.assert_allclose(got[t, hd * d:hd * d + h], rot.real, rtol=1e-5, atol=1e-5)
            np.testing.assert_allclose(got[t, hd * d + h:(hd + 1) * d], rot.imag, rtol=1e-5,
                                       atol=1e-5)
    # position 0 is the identity, exactly
    np.testing.assert_array_equal(got[0], x[0])


def test_rope_head_dim_2_closed_form():
    x = np.array([[1.0, 0.0]], np.float32)
    y = ops.rope(x, [1], 1, 2, 5e5, F32)
    np.testing.assert_allclose(y[0], [math.cos(1.0), math.sin(1.0)], rtol=1e-6)


# ----------------------------------------------------------------------------- attention
def _brute_attention(q, k, v, hq, hkv, d, causal, q_pos0):
    tq, tk = q.shape[0], k.shape[0]
    out = np.zeros((tq, hq * d))
    for h in range(hq):
        g = h // (hq // hkv)
        for i in range(tq):
            s = []
            for j in range(tk):
                if causal and j > q_pos0 + i:
                    continue
                s.append((j, sum(float(q[i, h * d + e]) * float(k[j, g * d + e])
                                 for e in range(d)) / math.sqrt(d)))
            mx = max(x for _, x in s)
            w = [(j, math.exp(x - mx)) for j, x in s]
            tot = sum(x for _, x in w)
            for e in range(d):
                out[i, h * d + e] = sum(p * float(v[j, g * d + e]) for j, p in w) / tot
    return out


@pytest.mark.parametrize("causal", [False, True])
def test_attention_brute_force(causal):
    hq, hkv, d, t = 4, 2, 8, 6
    q = round_to(RNG.standard_normal((t, hq * d)), BF16)
    k = round_to(RNG.standard_normal((t, hkv * d)), BF16)
    v = round_to(RNG.standard_normal((t, hkv * d)), BF16)
    got = ops.attention(q, k, v, hq, hkv, d, causal, 0, 1 / math.sqrt(d), F32)
    np.testing.assert_allclose(got, _brute_attention(q, k, v, hq, hkv, d, causal, 0),
                               rtol=2e-5, atol=2e-5)


def test_attention_special_cases():
    hq, hkv, d, t = 4, 1, 16, 9
    q = round_to(RNG.standard_normal((t, hq * d)), BF16)
    k = round_to(RNG.standard_normal((t, hkv * d)), BF16)
    v = round_to(RNG.standard_normal((t, hkv * d)), BF16)
    o = ops.attention(q, k, v, hq, hkv, d, True, 0, 1 / 4, BF16)
    # causal row 0 sees only key 0: output equals v_0 (rounded), for every head
    for h in range(hq):
        np.testing.assert_array_equal(o[0, h * d:(h + 1) * d], v[0])
    # zero query: uniform weights over the visible keys -> running mean of v
    o0 = ops.attention(np.zeros_like(q), k, v, hq, hkv, d, True, 0, 1 / 4, F32)
    for i in range(t):
        np.testing.assert_allclose(o0[i, :d], v[:i + 1].mean(axis=0), rtol=1e-5, atol=1e-6)
    # GQA with identical kv heads equals MHA
    k2 = np.concatenate([k, k], axis=1)
    v2 = np.concatenate([v, v], axis=1)
    np.testing.assert_array_equal(ops.attention(q, k2, v2, hq, 2, d, True, 0, 0.25, F32),
                                  ops.attention(q, k, v, hq, 1, d, True, 0, 0.25, F32))


def test_softmax_rows_sum_to_one():
    s = (5 * RNG.standard_normal((10, 37))).astype(np.float32)
    p = ops.softmax_rows(s)
    np.testing.assert_allclose(p.sum(axis=1), 1.0, rtol=1e-6)


@pytest.mark.parametrize("splits", [1, 2, 3, 8, 17])
def test_split_kv_reduce_equals_unsplit(splits):
    hq, hkv, d, tk = 8, 2, 16, 70
    q = round_to(RNG.standard_normal((1, hq * d)), BF16)
    k = round_to(RNG.standard_normal((tk, hkv * d)), BF16)
    v = round_to(RNG.standard_normal((tk, hkv * d)), BF16)
    edges = np.linspace(0, tk, splits + 1).round().astype(int)
    chunks = [(int(a), int(b)) for a, b in zip(edges[:-1], edges[1:])]
    m, l, o = ops.attention_partial(q, k, v, hq, hkv, d, chunks, 1 / 4)
    got = ops.attention_reduce(m, l, o, F32)
    ref = ops.attention(q, k, v, hq, hkv, d, False, tk - 1, 1 / 4, F32)
    np.testing.assert_allclose(got, ref, rtol=1e-5, atol=1e-6)
    if splits == 1:
        np.testing.assert_allclose(got.reshape(hq, d), o[:, 0] / l[:, 0:1], rtol=1e-6)


# ----------------------------------------------------------------------------- decoder
def _tiny_decoder(layers=2, dm=32, hq=4, hkv=2, d=8, f=48, seed=0):
    rng = np.random.default_rng(seed)
    w = lambda *s: round_to(0.2 * rng.standard_normal(s), BF16)
    qkv_cols = (hq + 2 * hkv) * d
    return models.DecoderWeights(
        wqkv=w(layers, dm, qkv_cols), wo=w(layers, hq * d, dm), wg=w(layers, dm, f),
        wu=w(layers, dm, f), wd=w(layers, f, dm),
        g_attn=round_to(1 + 0.02 * rng.standard_normal((layers, dm)), BF16),
        g_mlp=round_to(1 + 0.02 * rng.standard_normal((layers, dm)), BF16),
        n_q_heads=hq, n_kv_heads=hkv, head_dim=d, eps=1e-5, theta=5e5)


def test_prefill_is_causal_in_rows():
    wts = _tiny_decoder()
    x = round_to(RNG.standard_normal((12, 32)), BF16)
    full = models.prefill(x, wts)
    pref = models.prefill(x[:5], wts)
    np.testing.assert_array_equal(full[:5], pref)


def test_decode_step_continues_prefill():
    # Decoding token p with the cache built by prefilling tokens 0..p-1 reproduces prefill's
    # row p (the two differ only in where the norm output is rounded).
    wts = _tiny_decoder()
    t = 7
    x = round_to(RNG.standard_normal((t + 1, 32)), BF16)
    caches = {}

    def grab(l, d):
        caches[l] = d

    full = models.prefill(x, wts, layer_fn=grab)
    kcs, vcs = [], []
    hq, hkv, d = 4, 2, 8
    for l in range(wts.n_layers):
        kc = np.zeros((t + 1, hkv * d), np.float32)
        vc = np.zeros((t + 1, hkv * d), np.float32)
        kc[:t] = caches[l]["k_r"][:t]
        vc[:t] = caches[l]["qkv"][:t, (hq + hkv) * d:]
        kcs.append(kc)
        vcs.append(vc)
    out, _, _ = models.decode_step(x[t:t + 1], wts, kcs, vcs, t)
    err = np.abs(out - full[t:t + 1])
    assert np.max(err) <= 2e-2 * max(1.0, float(np.max(np.abs(full[t]))))


def _zero_query_zero_gate(wts):
    """The tiny decoder with W_q = 0 (every score 0: causal softmax weighs the visible keys
    equally), W_gate = 0 (silu(0) = 0: the MLP adds exactly 0) and W_o = I (h = a + x)."""
    hq, d = wts.n_q_heads, wts.head_dim
    for l in range(wts.n_layers):
        wts.wqkv[l][:, :hq * d] = 0.0
        wts.wg[l][:] = 0.0
        wts.wo[l][:] = np.eye(hq * d, wts.wo[l].shape[1])
    return wts


def _prefix_means(v, hq, hkv, d, first=0):
    """Row i, query head h: the mean of v rows first..i of kv head h // (hq / hkv), in fp64."""
    t = v.shape[0]
    g = hq // hkv
    out = np.zeros((t - first, hq * d))
    for i in range(first, t):
        for h in range(hq):
            kvh = h // g
            out[i - first, h * d:(h + 1) * d] = v[:i + 1, kvh * d:(kvh + 1) * d].astype(
                np.float64).mean(axis=0)
    return out


def test_prefill_closed_form_with_zero_query_and_gate():
    # Pins the decoder composition (head grouping, causal mask, W_o and residual wiring, the
    # MLP's zero path) against prefix means of v computed here, not by the attention routine.
    wts = _zero_query_zero_gate(_tiny_decoder(layers=2))
    hq, hkv, d = 4, 2, 8
    x = round_to(RNG.standard_normal((9, 32)), BF16)
    seen = {}
    out = models.prefill(x, wts, layer_fn=lambda l, dd: seen.setdefault(l, dd))
    x_in = x
    for l in range(2):
        s = seen[l]
        np.testing.assert_array_equal(s["q_r"], 0.0)
        v = s["qkv"][:, (hq + hkv) * d:]
        a_ref = round_to(_prefix_means(v, hq, hkv, d), BF16)
        np.testing.assert_allclose(s["a"], a_ref, rtol=2.0 ** -7, atol=1e-30)
        np.testing.assert_allclose(s["h"], round_to(s["a"].astype(np.float64) + x_in, BF16),
                                   rtol=0, atol=0)
        np.testing.assert_array_equal(s["gu"], 0.0)
        np.testing.assert_array_equal(s["x"], s["h"])
        x_in = s["x"]
    np.testing.assert_array_equal(out, x_in)


def test_decode_closed_form_with_zero_query_and_gate():
    # The decode step attends to every cache row plus the appended one with equal weight.
    wts = _zero_query_zero_gate(_tiny_decoder(layers=2))
    hq, hkv, d = 4, 2, 8
    p = 6
    x = round_to(RNG.standard_normal((1, 32)), BF16)
    kcs = [round_to(RNG.standard_normal((p + 1, hkv * d)), BF16) for _ in range(2)]
    vcs = [round_to(RNG.standard_normal((p + 1, hkv * d)), BF16) for _ in range(2)]
    seen = {}
    out, kc, vc = models.decode_step(x, wts, kcs, vcs, p,
                                     layer_fn=lambda l, dd: seen.setdefault(l, dd))
    x_in = x
    for l in range(2):
        s = seen[l]
        v_new = s["qkv"][:, (hq + hkv) * d:]
        np.testing.assert_array_equal(vc[l][p], v_new[0])          # appended value row
        np.testing.assert_array_equal(kc[l][p], s["k_r"][0])       # appended rotated key
        np.testing.assert_array_equal(vc[l][:p], vcs[l][:p])       # earlier rows untouched
        a_ref = round_to(_prefix_means(vc[l][:p + 1], hq, hkv, d, first=p), BF16)
        np.testing.assert_allclose(s["a"], a_ref, rtol=2.0 ** -7, atol=1e-30)
        np.testing.assert_allclose(s["h"], round_to(s["a"].astype(np.float64) + x_in, BF16),
                                   rtol=0, atol=0)
        np.testing.assert_array_equal(s["x"], s["h"])
        x_in = s["x"]
    np.testing.assert_array_equal(out, x_in)


# ----------------------------------------------------------------------------- schedule
def test_p3_worked_schedule():
    g = read_golden("p3_mlp_schedule.txt")
    plan = schedule.lower(_graphs.mlp_unfused(), _graphs.P3_OPTS)
    assert plan.n_instr == int(g["instructions"])
    assert f"{plan.waves:.2f}" == g["waves"]
    assert plan.n_dep == int(g["input_barriers"])
    per = int(g["instructions_per_layer"])
    # barriers created while visiting each layer's consumers
    created = []
    seen = set()
    for lyr in range(3):
        new = set()
        for ins in plan.instrs[lyr * per:(lyr + 1) * per]:
            for cid, _ in ins.src:
                if cid not in seen:
                    new.add(cid)
        seen |= new
        created.append(len(new))
    assert created == [int(g["input_barriers_layer1"]), int(g["input_barriers_layer2"]),
                       int(g["input_barriers_layer3"])]
    # mm -> add counters have target 2 (the pair's duplicate instructions)
    add1 = plan.instrs[16]
    assert add1.op == schedule.OP_EW and add1.src == [(add1.src[0][0], 2)]
    assert int(g["gemm_counter_target"]) == 2
    lo, hi = int(g["layer2_gemm_rowblock0_first"]), int(g["layer2_gemm_rowblock0_last"])
    for i in range(lo, hi + 1):
        ins = plan.instrs[i]
        assert ins.op == schedule.OP_GEMM and ins.m0 == 0
        assert len(ins.src) == 1
        cid, tgt = ins.src[0]
        assert tgt == int(g["layer2_gemm_rowblock0_waits_on_relu_instructions"])
        feeders = [j for j, p in enumerate(plan.instrs) if cid in p.dst]
        assert all(48 <= j < 80 and plan.instrs[j].m0 < 512 for j in feeders)
    assert plan.instrs[hi + 1].m0 == 512
    assert plan.instrs[int(g["layer3_add_first"])].op == schedule.OP_EW
    assert plan.instrs[int(g["layer3_add_first"]) - 1].op == schedule.OP_GEMM
    assert plan.instrs[int(g["layer3_relu_first"])].aux0 == schedule.EW_CODES["relu"]
    assert plan.instrs[int(g["layer3_relu_first"]) - 1].aux0 == schedule.EW_CODES["add"]
    assert plan.instrs[int(g["layer1_add_last_plus_one"])].aux0 == schedule.EW_CODES["relu"]
    assert schedule.topologically_valid(plan)
    assert plan.final_counters() == plan.targets


def test_p3_buffer_pool_matches_page():
    g = read_golden("p3_mlp_schedule.txt")
    desc = _graphs.mlp_unfused(transient=True)
    plan = schedule.lower(desc, _graphs.P3_OPTS)
    assert plan.n_dep == int(g["pool_total_barriers"])
    assert plan.n_reuse == int(g["pool_reuse_barriers"])
    # every caller-owned tensor is a slot, and each distinct pool buffer is one more
    slots = sum(1 for o in plan.pool_off[:3] if o < 0) + len(set(plan.pool_off[3:12]))
    assert slots == int(g["pool_tensor_slots"])
    mm1, add1, relu3, add3 = 3, 4, 11, 10  # tensor ids: layer 1 mm and add, layer 3 add and relu
    assert plan.pool_off[relu3] == plan.pool_off[mm1]
    assert plan.pool_off[add3] not in [plan.pool_off[t] for t in range(3, 10)]
    node_first = {}
    node_end = {}
    for i, ins in enumerate(plan.instrs):
        node_first.setdefault(ins.node, i)
        node_end[ins.node] = i + 1
    assert node_end[1] == int(g["pool_layer1_add_end"])
    assert node_first[8] == int(g["pool_final_relu_start"])
    assert node_first[7] == int(g["pool_layer3_add_start"])
    # the reuse counter: every instruction of layer 1's mm and add arrives, every instruction of
    # the final ReLU waits for that count (the pair's duplicate GEMM instructions both arrive)
    cid = plan.n_dep - 1
    feeders = [i for i, ins in enumerate(plan.instrs) if cid in ins.dst]
    assert feeders == list(range(0, int(g["pool_layer1_add_end"])))
    waiters = [i for i, ins in enumerate(plan.instrs) if (cid, len(feeders)) in ins.src]
    assert waiters == list(range(int(g["pool_final_relu_start"]), 240))
    assert schedule.topologically_valid(plan)
    assert plan.final_counters() == plan.targets


@pytest.mark.parametrize("n_sm,final_relu,layer3_add", [
    (148, True, False), (160, True, False), (161, False, False), (128, False, True),
    (129, True, False)])
def test_pool_one_wave_threshold(n_sm, final_relu, layer3_add):
    # start - end >= #SMs, with the end exclusive: the page's final ReLU (208) against layer 1's
    # add (ends at 48) qualifies up to 160 SMs, layer 3's add (176) up to 128. The lowering of
    # this chain does not depend on n_sm, so only the threshold moves.
    plan = schedule.lower(_graphs.mlp_unfused(transient=True), dict(_graphs.P3_OPTS, n_sm=n_sm))
    assert (plan.pool_off[11] == plan.pool_off[3]) == final_relu
    assert (plan.pool_off[10] == plan.pool_off[3]) == layer3_add
    if layer3_add:
        # T3's buffer now holds layer 3's add; the final ReLU takes layer 1's add buffer, whose
        # readers (layer 1's add and ReLU) end at 80: 208 - 80 = 128
        assert plan.pool_off[11] == plan.pool_off[4]
        assert plan.n_reuse == 2
    assert schedule.topologically_valid(plan)


def test_schedule_levels_are_acyclic_and_placement():
    plan = schedule.lower(_graphs.mlp_unfused(), _graphs.P3_OPTS)
    lv = schedule.levels(plan)
    # 9 dependent nodes in a chain -> 9 levels
    assert max(lv) == 8
    assert plan.placement(239) == (239 % 148, 1)
    assert plan.placement(147) == (147, 0)


def test_schedule_brute_force_matches_naive_pairs():
    # The vectorised intersection equals a plain double loop over instruction pairs.
    plan = schedule.lower(_graphs.mlp_unfused(m=256, h=384, layers=2),
                          dict(n_sm=7, gemm_tile_m=128, gemm_tile_n=128, ew_rows=64,
                               ew_cols=128))
    def meets(a, b):
        return (a[0] == b[0] and a[1] < b[2] and b[1] < a[2] and a[3] < b[4] and b[3] < a[4])
    node_first = {}
    for i, ins in enumerate(plan.instrs):
        node_first.setdefault(ins.node, i)
    for ci, c in enumerate(plan.instrs):
        want = set()
        for box, _ in c.reads:
            for pi in range(node_first[c.node]):
                if any(meets(box, w) for w in plan.instrs[pi].writes):
                    want.add(pi)
        got = set()
        for cid, _ in c.src:
            got |= {j for j, p in enumerate(plan.instrs) if cid in p.dst}
        assert got == want


def test_argmax_rows_first_maximum_nan_and_empty_rows():
    """Greedy sampling: the first column of the row maximum; NaN ignored; no number -> -1.
    Checked against a plain scan and hand-placed cases (ties, -inf only, all NaN)."""
    rng = np.random.default_rng(3)
    x = rng.standard_normal((7, 37)).astype(np.float32)
    x[1, [5, 20]] = 9.0                      # tie: the lower column wins
    x[2, :] = np.nan
    x[2, 30] = -np.inf                       # the only number is -inf
    x[3, :] = np.nan                         # no number at all
    x[4, 0] = np.nan
    x[4, 7] = 50.0
    x[5, :] = 0.0                            # all equal: column 0
    x[6, :] = np.float32(np.finfo(np.float32).max)
    x[6, 36] = np.inf                        # +inf beats every finite value
    got = ops.argmax_rows(x).ravel().tolist()
    want = []
    for row in x:
        best = -1
        for j, v in enumerate(row):
            if v != v:
                continue
            if best < 0 or v > row[best]:
                best = j
        want.append(best)
    assert got == want
    assert got[1] == 5 and got[2] == 30 and got[3] == -1 and got[4] == 7 and got[5] == 0
    assert got[6] == 36


def test_argmax_on_rounded_logits_decides_on_the_stored_values():
    """Two logits that differ in fp32 but round to one bf16 value tie after rounding: the
    decision is taken on the stored (rounded) values, so the lower column wins."""
    a = np.float32(1.0)
    b = np.nextafter(a, np.float32(2.0))     # fp32 neighbour, same bf16
    x = round_to(np.array([[0.5, a, b, 0.25]], dtype=np.float32), BF16)
    assert x[0, 1] == x[0, 2]
    assert ops.argmax_rows(x)[0, 0] == 1
