"""How far two valid fp32 evaluations of the same decoder drift apart after many bf16 layers.

The decoder is equivariant under relabelling its hidden and MLP features: with a permutation
P of the hidden columns and Q of the MLP columns, the network whose x, gammas and weights are
permuted (Wqkv rows by P; Wo columns by P; Wg, Wu rows by P and columns by Q; Wd rows by Q and
columns by P) computes exactly the permuted output in real arithmetic. In fp32 every
contraction over a relabelled dimension sums its terms in another order, so running the oracle
on both labellings gives two results that are equally valid; their gap after L layers, where
bf16 roundings of the node outputs amplify order differences, is the spread any implementation
with a different summation order can show. Test helper only (calls the oracle, no GPU).
"""
import numpy as np

from oracle import models
from tensor_core_gemm_gb300 import synth

# An implementation is held to this multiple of the oracle-vs-oracle drift end to end.
MARGIN = 2.0


def relabel(wts, perm_d, perm_f):
    """The decoder weights with hidden features relabelled by perm_d and MLP features by
    perm_f (new feature i is old feature perm[i]); attention features keep their labels."""
    def rows_cols(w, pr, pc):
        out = np.empty_like(w)
        for layer in range(w.shape[0]):
            m = w[layer] if pr is None else np.take(w[layer], pr, axis=0)
            out[layer] = m if pc is None else np.take(m, pc, axis=1)
        return out

    return models.DecoderWeights(
        rows_cols(wts.wqkv, perm_d, None), rows_cols(wts.wo, None, perm_d),
        rows_cols(wts.wg, perm_d, perm_f), rows_cols(wts.wu, perm_d, perm_f),
        rows_cols(wts.wd, perm_f, perm_d),
        np.ascontiguousarray(wts.g_attn[:, perm_d]), np.ascontiguousarray(wts.g_mlp[:, perm_d]),
        wts.n_q_heads, wts.n_kv_heads, wts.head_dim, wts.eps, wts.theta)


def _perms(wts, seed):
    rng = np.random.default_rng(seed)
    return rng.permutation(wts.wqkv.shape[1]), rng.permutation(wts.wg.shape[2])


def gap(got, ref):
    """(relative Frobenius error, largest element error) of got against ref."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    return (float(np.linalg.norm(got - ref) / np.linalg.norm(ref)),
            float(np.max(np.abs(got - ref))))


def decoder_weights(wl):
    """The oracle's weights of a decode or prefill workload (exact fp32 values)."""
    sh = wl.info["shape"]
    L, d, f = sh.layers, sh.hidden, sh.ffn
    D, w = wl.data, wl.info["w"]
    f32 = synth.to_numpy_f32
    return models.DecoderWeights(
        f32(D[w["wqkv"]]).reshape(L, d, sh.qkv), f32(D[w["wo"]]).reshape(L, sh.hq * sh.hd, d),
        f32(D[w["wg"]]).reshape(L, d, f), f32(D[w["wu"]]).reshape(L, d, f),
        f32(D[w["wd"]]).reshape(L, f, d), f32(D[w["g_attn"]]), f32(D[w["g_mlp"]]),
        sh.hq, sh.hkv, sh.hd, sh.eps, sh.theta)


def decode_drift(x, wts, kc, vc, pos, ref=None, seed=1):
    """gap() between models.decode_step on a relabelled copy (mapped back) and on the given
    labelling (`ref`, its output, when already computed). Returns (gap, ref)."""
    if ref is None:
        ref, _, _ = models.decode_step(x, wts, kc, vc, pos)
    pd, pf = _perms(wts, seed)
    alt, _, _ = models.decode_step(np.ascontiguousarray(x[:, pd]), relabel(wts, pd, pf), kc, vc,
                                   pos)
    back = np.empty_like(alt)
    back[:, pd] = alt
    return gap(back, ref), ref


def prefill_drift(x, wts, ref=None, seed=1):
    """The same for models.prefill on the rows x."""
    if ref is None:
        ref = models.prefill(x, wts)
    pd, pf = _perms(wts, seed)
    alt = models.prefill(np.ascontiguousarray(x[:, pd]), relabel(wts, pd, pf))
    back = np.empty_like(alt)
    back[:, pd] = alt
    return gap(back, ref), ref


def within_drift(got, ref, drift, margin=MARGIN):
    """got is within `margin` times the oracle-vs-oracle drift of ref, in relative Frobenius
    error and in the largest element error."""
    fro, mx = gap(got, ref)
    return fro <= margin * drift[0] and mx <= margin * drift[1], (fro, mx)
