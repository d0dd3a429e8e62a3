"""Pins of the oracle's decoder compositions by an fp64 brute force written here.

The decoder layer ("Implementing a Mega Kernel for B300" §1, "Build the graph": norm -> QKV ->
RoPE -> attention -> O + residual -> norm -> gate/up SiLU·mul -> down + residual) is restated
below with explicit loops in fp64, calling nothing from ``oracle.ops``. Node outputs are
rounded to bf16 at the same places as the graph stores them (torch's bf16 cast, round to
nearest even), so the oracle's ``models.prefill`` and ``models.decode_step`` must agree with it
to within fp32-vs-fp64 accumulation.

Each plausible wiring mistake (the two norm weights swapped, the MLP norm taken over x instead
of h, the residual of x instead of h, k and v exchanged, the wrong query-to-key/value head
grouping, RoPE left off k, a causal mask shifted by one, gate and up exchanged) is planted in
the brute force, on the CPU, and must then fail the same comparison: the pin has the power to
see each of them.
"""
import math

import numpy as np
import pytest
import torch

from oracle import models

D, HQ, HKV, HD, F = 64, 4, 2, 16, 96   # hidden, query heads, key/value heads, head dim, MLP
EPS, THETA = 1e-5, 5e5
MUTATIONS = ["gamma_swap", "mlp_norm_of_x", "mlp_residual_x", "attn_residual_missing",
             "kv_swapped", "gqa_modulo", "rope_k_missing", "causal_shift", "gate_up_swapped"]


def bf16(x):
    """Round an fp64 array to the nearest bf16 value (ties to even), returned as fp64."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float64)).to(torch.float32)
    return t.to(torch.bfloat16).to(torch.float64).numpy()


def dot(a, b):
    """fp64 matrix product by explicit sums: out[i, j] = sum_k a[i, k] * b[k, j]."""
    n, kk = a.shape
    m = b.shape[1]
    out = np.zeros((n, m))
    for i in range(n):
        for k in range(kk):
            if a[i, k] != 0.0:
                out[i] += a[i, k] * b[k]
    return out


def rms_normalise(x, gamma):
    """Each row divided by sqrt(mean of its squares + eps), times gamma per column."""
    out = np.empty_like(x)
    for r in range(x.shape[0]):
        ms = sum(v * v for v in x[r]) / x.shape[1]
        out[r] = x[r] / math.sqrt(ms + EPS) * gamma
    return out


def rotate(row, pos, n_heads):
    """Rotary embedding of one row at position pos: in every head, the pair (i, i + HD/2) is
    turned by the angle pos * THETA^(-2i/HD) (a plane rotation of the pair)."""
    out = np.empty_like(row)
    half = HD // 2
    for h in range(n_heads):
        for i in range(half):
            a = pos * THETA ** (-2.0 * i / HD)
            x1, x2 = row[h * HD + i], row[h * HD + i + half]
            out[h * HD + i] = x1 * math.cos(a) - x2 * math.sin(a)
            out[h * HD + i + half] = x2 * math.cos(a) + x1 * math.sin(a)
    return out


def attend(q_row, keys, values, visible, mutate):
    """One query row over key rows `keys` (visible[j] says whether key j takes part): per query
    head, softmax of q·k / sqrt(HD) over the visible keys, times the values."""
    out = np.zeros(HQ * HD)
    for h in range(HQ):
        g = h % HKV if mutate == "gqa_modulo" else h // (HQ // HKV)
        q = q_row[h * HD:(h + 1) * HD]
        s = [sum(q[e] * keys[j][g * HD + e] for e in range(HD)) / math.sqrt(HD)
             for j in range(len(keys)) if visible[j]]
        vis = [j for j in range(len(keys)) if visible[j]]
        mx = max(s)
        w = [math.exp(v - mx) for v in s]
        tot = sum(w)
        for wj, j in zip(w, vis):
            out[h * HD:(h + 1) * HD] += wj / tot * values[j][g * HD:(g + 1) * HD]
    return out


def silu(z):
    return z / (1.0 + np.exp(-z))


def brute_layer(x, pos, lw, k_prev, v_prev, prefill, mutate=None):
    """One decoder layer over rows x (positions pos) in fp64.

    prefill: the rows attend causally to each other (a separate RMSNorm node writes the
    normalised rows, rounded). Decode (one row): the normalised row stays unrounded inside the
    fused GEMV; the row's rotated key and its value are appended after k_prev / v_prev and the
    row attends to every key. Returns the layer output and the (keys, values) it attended to.
    """
    g_attn, g_mlp = (lw["g_mlp"], lw["g_attn"]) if mutate == "gamma_swap" else (lw["g_attn"],
                                                                                lw["g_mlp"])
    xn = rms_normalise(x, g_attn)
    if prefill:
        xn = bf16(xn)
    qkv = bf16(dot(xn, lw["wqkv"]))
    nq, nk = HQ * HD, HKV * HD
    q, k, v = qkv[:, :nq], qkv[:, nq:nq + nk], qkv[:, nq + nk:]
    if mutate == "kv_swapped":
        k, v = v, k
    q_r = bf16(np.stack([rotate(q[t], pos[t], HQ) for t in range(len(pos))]))
    k_r = k if mutate == "rope_k_missing" else bf16(
        np.stack([rotate(k[t], pos[t], HKV) for t in range(len(pos))]))
    keys = list(k_prev) + list(k_r)
    values = list(v_prev) + list(v)
    att = []
    for t in range(len(pos)):
        limit = pos[t] + (1 if mutate == "causal_shift" else 0)
        visible = [j <= limit for j in range(len(keys))] if prefill else [True] * len(keys)
        att.append(attend(q_r[t], keys, values, visible, mutate))
    att = bf16(np.stack(att))
    o = dot(att, lw["wo"])
    h = bf16(o if mutate == "attn_residual_missing" else o + x)
    hsrc = x if mutate == "mlp_norm_of_x" else h
    hn = rms_normalise(hsrc, g_mlp)
    if prefill:
        hn = bf16(hn)
    gate, up = dot(hn, lw["wg"]), dot(hn, lw["wu"])
    if mutate == "gate_up_swapped":
        gate, up = up, gate
    gu = bf16(silu(gate) * up)
    res = x if mutate == "mlp_residual_x" else h
    out = bf16(dot(gu, lw["wd"]) + res)
    return out, np.stack(keys), np.stack(values)


def _weights(rng, layers):
    """bf16-valued weights with scales that keep every branch of the layer O(1): the attention
    and MLP contributions are as large as the residual stream, and the two norm weights differ
    everywhere (so a mix-up of any of them changes the output by O(1))."""
    def w(*shape, std):
        return bf16(rng.standard_normal(shape) * std)

    return [dict(wqkv=w(D, (HQ + 2 * HKV) * HD, std=1 / math.sqrt(D)),
                 wo=w(HQ * HD, D, std=1.0 / math.sqrt(HQ * HD)),
                 wg=w(D, F, std=1.0 / math.sqrt(D)), wu=w(D, F, std=1.0 / math.sqrt(D)),
                 wd=w(F, D, std=1.0 / math.sqrt(F)),
                 g_attn=bf16(1.0 + 0.5 * rng.standard_normal(D)),
                 g_mlp=bf16(0.8 * rng.standard_normal(D)))
            for _ in range(layers)]


def _oracle_weights(lws):
    st = lambda key: np.stack([lw[key] for lw in lws]).astype(np.float32)
    return models.DecoderWeights(st("wqkv"), st("wo"), st("wg"), st("wu"), st("wd"),
                                 st("g_attn"), st("g_mlp"), HQ, HKV, HD, EPS, THETA)


def rel_err(got, ref):
    return np.linalg.norm(np.asarray(got, np.float64) - ref) / np.linalg.norm(ref)


def within_tolerance(got, ref):
    """The parity tolerance: relative Frobenius <= 5e-3 and |err| <= 2e-2 * max(1, |ref|)."""
    got = np.asarray(got, np.float64)
    return (rel_err(got, ref) <= 5e-3 and
            bool(np.all(np.abs(got - ref) <= 2e-2 * np.maximum(1.0, np.abs(ref)))))


LAYERS, T_PREFILL, KV_PREV = 2, 7, 9


def _prefill_case(seed, mutate=None):
    rng = np.random.default_rng(seed)
    lws = _weights(rng, LAYERS)
    x = bf16(rng.standard_normal((T_PREFILL, D)))
    pos = list(range(T_PREFILL))
    ref = x
    for lw in lws:
        ref, _, _ = brute_layer(ref, pos, lw, [], [], prefill=True, mutate=mutate)
    got = models.prefill(x.astype(np.float32), _oracle_weights(lws))
    return got, ref


def _decode_case(seed, mutate=None):
    rng = np.random.default_rng(seed)
    lws = _weights(rng, LAYERS)
    x = bf16(rng.standard_normal((1, D)))
    cap = KV_PREV + 1
    kc = [np.zeros((cap, HKV * HD)) for _ in range(LAYERS)]
    vc = [np.zeros((cap, HKV * HD)) for _ in range(LAYERS)]
    for l in range(LAYERS):
        kc[l][:KV_PREV] = bf16(rng.standard_normal((KV_PREV, HKV * HD)))
        vc[l][:KV_PREV] = bf16(rng.standard_normal((KV_PREV, HKV * HD)))
    ref = x
    ref_k, ref_v = [], []
    for l, lw in enumerate(lws):
        ref, keys, values = brute_layer(ref, [KV_PREV], lw, kc[l][:KV_PREV], vc[l][:KV_PREV],
                                        prefill=False, mutate=mutate)
        ref_k.append(keys[-1])
        ref_v.append(values[-1])
    got, kc_o, vc_o = models.decode_step(x.astype(np.float32), _oracle_weights(lws),
                                         [c.astype(np.float32) for c in kc],
                                         [c.astype(np.float32) for c in vc], KV_PREV)
    return got, ref, (kc_o, vc_o, ref_k, ref_v)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_prefill_layers_match_fp64_brute_force(seed):
    got, ref = _prefill_case(seed)
    assert within_tolerance(got, ref), rel_err(got, ref)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_decode_layers_match_fp64_brute_force(seed):
    got, ref, (kc_o, vc_o, ref_k, ref_v) = _decode_case(seed)
    assert within_tolerance(got, ref), rel_err(got, ref)
    for l in range(LAYERS):   # the appended cache rows: rotated key, plain value
        assert within_tolerance(kc_o[l][KV_PREV], ref_k[l])
        assert np.array_equal(vc_o[l][KV_PREV], ref_v[l].astype(np.float32))


@pytest.mark.parametrize("mutate", MUTATIONS)
def test_planted_wiring_mistakes_fail_the_prefill_pin(mutate):
    got, ref = _prefill_case(0, mutate)
    assert not within_tolerance(got, ref)
    assert rel_err(got, ref) > 5e-2   # ten times the tolerance: far outside, not marginal


@pytest.mark.parametrize("mutate", [m for m in MUTATIONS if m != "causal_shift"])
def test_planted_wiring_mistakes_fail_the_decode_pin(mutate):
    # the decode row sees every key, so the causal mask has nothing to shift there
    got, ref, _ = _decode_case(0, mutate)
    assert not within_tolerance(got, ref)
    assert rel_err(got, ref) > 5e-2
