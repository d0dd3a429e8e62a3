"""The five workloads, composed from ``ops`` at the granularity of the graph's nodes.

Every function takes fp32 arrays of quantised values (see ``numerics.to_f32``) and returns the
graph's output(s) as fp32 arrays of values in the storage dtype. Each node output is rounded
once, exactly as ``ops`` does, so intermediate buffers match what the GPU graph stores.
"""
import numpy as np

from . import ops
from .numerics import BF16, F16


def mlp(x, w, b, out_dtype=F16):
    """3-layer MLP x = relu(x @ W[i] + b[i]), i = 0..L-1, bias a full matrix per layer.

    "MegaKittens Internals" §02: the worked example traced from ``x = relu(x @ W[i] + b[i])``
    with W (3, 1024, 1024), x (1024, 1024), b (3, 1024, 1024). One fused node per layer
    (matmul + bias + ReLU epilogue), so each layer output is rounded once.
    Returns the list of per-layer outputs [h1, h2, h3].
    """
    outs = []
    h = x
    for i in range(w.shape[0]):
        h = ops.matmul(h, w[i], out_dtype, bias=b[i], relu=True)
        outs.append(h)
    return outs


def mlp_unfused(x, w, b, out_dtype):
    """The same MLP as three nodes per layer (mm, add, relu), each output rounded.

    The aten graph of "MegaKittens Internals" §02 (mm -> add -> relu).
    """
    outs = []
    h = x
    for i in range(w.shape[0]):
        mm = ops.matmul(h, w[i], out_dtype)
        ad = ops.elementwise("add", [mm, b[i]], out_dtype)
        h = ops.elementwise("relu", [ad], out_dtype)
        outs.append((mm, ad, h))
    return outs


def gemm(a, b, out_dtype=F16):
    """C = A @ B, fp32 accumulate, rounded once ("Hand-writing a Blackwell GEMM", intro)."""
    return ops.matmul(a, b, out_dtype)


def gemm_rows(a, b, rows, out_dtype=F16):
    """Selected rows of C = A @ B (row r of C depends only on row r of A)."""
    return ops.matmul(a[rows], b, out_dtype)


class DecoderWeights:
    """Per-layer weights of the Llama-style decoder (row-major K×N matrices, as in x @ W).

    wqkv [L, D, (Hq + 2·Hkv)·d] with columns [q | k | v]; wo [L, Hq·d, D]; wg, wu [L, D, F];
    wd [L, F, D]; g_attn, g_mlp [L, D]. All bf16 values held as fp32.
    """

    def __init__(self, wqkv, wo, wg, wu, wd, g_attn, g_mlp, n_q_heads, n_kv_heads, head_dim,
                 eps, theta):
        self.wqkv, self.wo, self.wg, self.wu, self.wd = wqkv, wo, wg, wu, wd
        self.g_attn, self.g_mlp = g_attn, g_mlp
        self.n_q_heads, self.n_kv_heads, self.head_dim = n_q_heads, n_kv_heads, head_dim
        self.eps, self.theta = eps, theta

    @property
    def n_layers(self):
        return len(self.wqkv)


def decode_step(x, wts, k_cache, v_cache, pos, layer_fn=None):
    """One batch-1 decode token through every layer ("Implementing a Mega Kernel for B300" §1).

    Per layer l, with D the hidden size and p = ``pos`` the new token's position:
      1. qkv = GEMV(x, Wqkv, RMS_NORM_INPUT gamma_attn)                  -> bf16 [1 × 3072]
      2. q = rope(q, p), k = rope(k, p); K[l][p] = k, V[l][p] = v (ATTENTION_APPEND)
      3. a = attention(q, K[l][0..p], V[l][0..p])   (split-KV partial + combine on the GPU)
      4. h = GEMV(a, Wo) + x                          (ADD_RESIDUAL)
      5. gu = silu(ĥ Wg) ⊙ (ĥ Wu) with ĥ = rmsnorm(h) (RMS_NORM_INPUT + SILU_MUL)
      6. x = GEMV(gu, Wd) + h                         (ADD_RESIDUAL)
    k_cache / v_cache: lists of fp32 arrays [cap × Hkv·d] holding positions 0..pos-1; rows
    ``pos`` are written (copies are returned, the inputs are not modified).
    No final norm, lm_head or sampling: the output is the residual stream after the last layer.
    ``layer_fn(l, dict)`` receives each layer's intermediates (for checks).
    """
    hq, hkv, d = wts.n_q_heads, wts.n_kv_heads, wts.head_dim
    kc = [c.copy() for c in k_cache]
    vc = [c.copy() for c in v_cache]
    for l in range(wts.n_layers):
        qkv = ops.matmul_norm_input(x, wts.g_attn[l], wts.eps, wts.wqkv[l], BF16)
        q = qkv[:, :hq * d]
        k = qkv[:, hq * d:(hq + hkv) * d]
        v = qkv[:, (hq + hkv) * d:]
        q_r = ops.rope(q, [pos], hq, d, wts.theta, BF16)
        k_r = ops.rope(k, [pos], hkv, d, wts.theta, BF16)
        kc[l][pos] = k_r[0]
        vc[l][pos] = v[0]
        a = ops.attention(q_r, kc[l][:pos + 1], vc[l][:pos + 1], hq, hkv, d, causal=False,
                          q_pos0=pos, scale=1.0 / np.sqrt(d), out_dtype=BF16)
        h = ops.matmul(a, wts.wo[l], BF16, residual=x)
        gu = ops.matmul_norm_input(h, wts.g_mlp[l], wts.eps, wts.wg[l], BF16, w_up=wts.wu[l])
        x_new = ops.matmul(gu, wts.wd[l], BF16, residual=h)
        if layer_fn is not None:
            layer_fn(l, dict(qkv=qkv, q_r=q_r, k_r=k_r, a=a, h=h, gu=gu, x=x_new))
        x = x_new
    return x, kc, vc


def decode_head(x, g_final, w_lm, eps):
    """Greedy sampling after the last layer: logits = GEMV(x, W_lm, RMS_NORM_INPUT g_final)
    rounded to bf16, token = the first column holding the largest logit
    ("Implementing a Mega Kernel for B300" §8: final norm, lm_head, SAMPLE)."""
    logits = ops.matmul_norm_input(x, g_final, eps, w_lm, BF16)
    return logits, ops.argmax_rows(logits)


def prefill(x, wts, layer_fn=None):
    """Causal prefill of T tokens (positions 0..T-1) through every layer, batch 1.

    Per layer: x̂ = rmsnorm(x); qkv = x̂ Wqkv; q, k = rope(q, k); a = causal attention;
    h = a Wo + x; ĥ = rmsnorm(h); gu = silu(ĥ Wg) ⊙ (ĥ Wu); x = gu Wd + h. Every node output
    is rounded to bf16. Row t of every output depends only on rows 0..t of the input, so a
    prefix of the rows can be checked by running this function on that prefix.
    """
    hq, hkv, d = wts.n_q_heads, wts.n_kv_heads, wts.head_dim
    t = x.shape[0]
    pos = np.arange(t)
    for l in range(wts.n_layers):
        xn = ops.rmsnorm(x, wts.g_attn[l], wts.eps, BF16)
        qkv = ops.matmul(xn, wts.wqkv[l], BF16)
        q = qkv[:, :hq * d]
        k = qkv[:, hq * d:(hq + hkv) * d]
        v = qkv[:, (hq + hkv) * d:]
        q_r = ops.rope(q, pos, hq, d, wts.theta, BF16)
        k_r = ops.rope(k, pos, hkv, d, wts.theta, BF16)
        a = ops.attention(q_r, k_r, v, hq, hkv, d, causal=True, q_pos0=0,
                          scale=1.0 / np.sqrt(d), out_dtype=BF16)
        h = ops.matmul(a, wts.wo[l], BF16, residual=x)
        hn = ops.rmsnorm(h, wts.g_mlp[l], wts.eps, BF16)
        gu = ops.matmul_silu_mul(hn, wts.wg[l], wts.wu[l], BF16)
        x_new = ops.matmul(gu, wts.wd[l], BF16, residual=h)
        if layer_fn is not None:
            layer_fn(l, dict(xn=xn, qkv=qkv, q_r=q_r, k_r=k_r, a=a, h=h, hn=hn, gu=gu, x=x_new))
        x = x_new
    return x
