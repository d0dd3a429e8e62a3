"""One function per graph operation, each the plain definition, computed in fp32 with numpy.

Inputs are fp32 arrays holding values already quantised to their storage dtype (see
``numerics``); each function rounds its result to ``out_dtype`` exactly once, at the end, which
is the node-output rounding rule. A library matmul serves as the contraction step; nothing is
blocked, fused or reordered beyond the definition written in each docstring.

Citations name the page and section the definition follows:
  [GEMM]  "Hand-writing a Blackwell GEMM: 164 to 1400 TFLOP/s"
  [MK]    "MegaKittens Internals"
  [B300]  "Implementing a Mega Kernel for B300"
  [CUTE]  "Beating torch.compile with Megakernels in CuTe DSL [Part 1]"
  [TL]    "Designing High-Performance GPU Kernels with TileLang ..."
"""
import numpy as np

from .numerics import round_to


def _f32(x):
    return np.asarray(x, dtype=np.float32)


def matmul(a, b, out_dtype, bias=None, relu=False, residual=None):
    """C = A·B with fp32 accumulation, then the fused epilogue, then one rounding.

    A is [M×K], B is [K×N] (row-major weight, as ``aten.mm(x, W[i])`` in [MK] §02). The epilogue
    order is: + bias[m,n] (a full M×N matrix: the elementwise ops do not broadcast, [MK] §12),
    ReLU, + residual[m,n] ([B300] §2 "ADD_RESIDUAL"). The 3-layer MLP x = relu(x@W[i] + b[i]) of
    [MK] §02 is matmul(..., bias=b[i], relu=True).

    Pinned by: identity weights with zero bias give relu(x) exactly; brute-force fp64 triple
    loops on tiny shapes; a hand-computed 2×2 case (tests/golden/matmul_2x2.txt).
    """
    acc = _f32(a) @ _f32(b)
    if bias is not None:
        acc = acc + _f32(bias)
    if relu:
        acc = np.maximum(acc, np.float32(0.0))
    if residual is not None:
        acc = acc + _f32(residual)
    return round_to(acc, out_dtype)


def silu(z):
    """silu(z) = z / (1 + e^{-z}) = z·sigmoid(z) (the SwiGLU gate of [CUTE] "Model Architecture")."""
    z = _f32(z)
    return z / (np.float32(1.0) + np.exp(-z))


def rms_scale(x, eps):
    """Per-row 1/sqrt(mean_k x_k^2 + eps) in fp32 (the RMSNorm statistic)."""
    x = _f32(x)
    ms = np.mean(x * x, axis=-1, keepdims=True, dtype=np.float32)
    return (np.float32(1.0) / np.sqrt(ms + np.float32(eps))).astype(np.float32)


def rmsnorm(x, gamma, eps, out_dtype):
    """y = x / sqrt(mean(x^2) + eps) · gamma, one rounding at the end.

    [CUTE] "Shared Memory Layout / RMSNorm" (row-parallel norm) and [MK] §12 "RMSNorm" (gamma read
    per column). eps is the graph's value; [MK] §16 notes a kernel that ignored it, which this
    definition does not copy. Pinned by: a constant row c gives gamma·c/sqrt(c^2+eps); scaling a
    row by s>0 leaves the output unchanged when eps=0 (tests).
    """
    x = _f32(x)
    y = x * rms_scale(x, eps) * _f32(gamma).reshape(1, -1)
    return round_to(y, out_dtype)


def matmul_norm_input(x, gamma, eps, w, out_dtype, residual=None, w_up=None):
    """The GEMV node with the RMS_NORM_INPUT flag: y = (x·rstd(x)·gamma)·W (+ residual).

    [B300] §2 "Lower each op into tasks": RMS-norm is a flag on the GEMV that consumes it, "so a
    single GEMV does norm -> dot -> residual in one pass". The normalised row is not rounded
    to storage before the dot (it never leaves the task); the node output is rounded once.
    With ``w_up`` the SILU_MUL flag applies: y = silu(x̂·W)·(x̂·W_up).

    Pinned by: gamma = 1 and a row already of unit RMS (eps -> 0) reduces to plain matmul;
    equals matmul(rmsnorm(x) without rounding, W) computed in fp64 (tests).
    """
    xn = _f32(x) * rms_scale(x, eps) * _f32(gamma).reshape(1, -1)
    if w_up is not None:
        g = xn @ _f32(w)
        u = xn @ _f32(w_up)
        y = silu(g) * u
    else:
        y = xn @ _f32(w)
    if residual is not None:
        y = y + _f32(residual)
    return round_to(y, out_dtype)


def matmul_silu_mul(a, w_gate, w_up, out_dtype):
    """y = silu(A·W_gate) ⊙ (A·W_up), both products accumulated in fp32, rounded once.

    The SILU_MUL epilogue of [B300] §2 (bit0 of the task flags) applied to the gate/up pair of
    a SwiGLU MLP ([CUTE] "Model Architecture"). Gate and up are separate K×N weights.
    Pinned by: W_up = I and square shapes give silu(A·W_gate) rounded (tests).
    """
    g = _f32(a) @ _f32(w_gate)
    u = _f32(a) @ _f32(w_up)
    return round_to(silu(g) * u, out_dtype)


def elementwise(op, ins, out_dtype):
    """Same-shape elementwise tiles, no broadcasting ([MK] §12 "ElementwiseUnary and Binary").

    op: "add" (a + b), "relu" (max(a, 0)), "copy" (a), "silu_mul" (silu(a)·b).
    """
    if op == "add":
        y = _f32(ins[0]) + _f32(ins[1])
    elif op == "relu":
        y = np.maximum(_f32(ins[0]), np.float32(0.0))
    elif op == "copy":
        y = _f32(ins[0])
    elif op == "silu_mul":
        y = silu(ins[0]) * _f32(ins[1])
    else:
        raise ValueError(op)
    return round_to(y, out_dtype)


def rope_angles(positions, head_dim, theta):
    """angle[p, i] = p · theta^(-2i/head_dim) for i < head_dim/2, in fp64.

    Rotary embedding as applied by [B300] §8 ATTENTION_APPEND ("RoPE-append current k,v"); the
    pages give no formula, so this is the standard rotary definition with the pairing below.
    """
    i = np.arange(head_dim // 2, dtype=np.float64)
    inv_freq = theta ** (-2.0 * i / head_dim)
    return np.asarray(positions, dtype=np.float64).reshape(-1, 1) * inv_freq.reshape(1, -1)


def rope(x, positions, n_heads, head_dim, theta, out_dtype):
    """Rotate each head's pairs (i, i + head_dim/2) by angle[p, i] ("rotate_half" pairing).

    x: [T × n_heads·head_dim], row t at position positions[t]. For each head:
      y[i]        = x[i]·cos - x[i+h]·sin
      y[i + h]    = x[i+h]·cos + x[i]·sin,   h = head_dim/2.
    Parity unpinned beyond: position 0 is the identity; rotation preserves each pair's norm;
    rotating by p then by -p returns x (tests).
    """
    x = _f32(x)
    t = x.shape[0]
    ang = rope_angles(positions, head_dim, theta)                 # [T, h] fp64
    cos = np.cos(ang).astype(np.float32)[:, None, :]
    sin = np.sin(ang).astype(np.float32)[:, None, :]
    xh = x.reshape(t, n_heads, head_dim)
    h = head_dim // 2
    x1, x2 = xh[..., :h], xh[..., h:]
    y = np.concatenate([x1 * cos - x2 * sin, x2 * cos + x1 * sin], axis=-1)
    return round_to(y.reshape(t, n_heads * head_dim), out_dtype)


def softmax_rows(s):
    """Row softmax: exp(s - max) / sum(exp(s - max)) ([TL] §5 "REDUCTIONS — row-wise softmax").

    A row that is entirely -inf (no visible key) is not produced by any graph here.
    """
    s = _f32(s)
    m = np.max(s, axis=-1, keepdims=True)
    p = np.exp(s - m)
    return p / np.sum(p, axis=-1, keepdims=True, dtype=np.float32)


def attention(q, k, v, n_q_heads, n_kv_heads, head_dim, causal, q_pos0, scale, out_dtype):
    """O = softmax(Q·K^T·scale [+ causal mask]) · V per head, grouped-query heads.

    q: [Tq × Hq·d], k, v: [Tk × Hkv·d]; query row i sits at position q_pos0 + i and key row j at
    position j. With ``causal`` a key is visible iff j <= q_pos0 + i ([TL] §6 FlashAttention:
    the mask keeps q_idx >= k_idx; [MK] §14 "Causal"). Query head h reads kv head
    h // (Hq/Hkv). scale is 1/sqrt(d) unless given.
    Pinned by: causal row 0 equals v_0; identical kv heads equal plain MHA; a single key gives
    that key's value; rows of the probability matrix sum to 1 (tests).
    """
    q, k, v = _f32(q), _f32(k), _f32(v)
    tq, tk = q.shape[0], k.shape[0]
    group = n_q_heads // n_kv_heads
    out = np.empty((tq, n_q_heads * head_dim), dtype=np.float32)
    if causal:
        qpos = q_pos0 + np.arange(tq).reshape(-1, 1)
        visible = np.arange(tk).reshape(1, -1) <= qpos
    for h in range(n_q_heads):
        g = h // group
        qh = q[:, h * head_dim:(h + 1) * head_dim]
        kh = k[:, g * head_dim:(g + 1) * head_dim]
        vh = v[:, g * head_dim:(g + 1) * head_dim]
        s = (qh @ kh.T) * np.float32(scale)
        if causal:
            s = np.where(visible, s, np.float32(-np.inf))
        out[:, h * head_dim:(h + 1) * head_dim] = softmax_rows(s) @ vh
    return round_to(out, out_dtype)


def attention_partial(q, k, v, n_q_heads, n_kv_heads, head_dim, chunks, scale):
    """Split-KV partials ([B300] §2 "ATTENTION_PARTIAL ... online-softmax over one KV chunk -> (m,l,o)").

    For one query row (decode, every cached key visible), per query head h and key chunk c
    (a half-open row range of k/v):
        s_j = q_h·k_j·scale,  m = max_j s_j,  l = sum_j e^{s_j - m},  o = sum_j e^{s_j - m} v_j.
    Returns fp32 arrays m[H, C], l[H, C], o[H, C, d] (o unnormalised).
    """
    q, k, v = _f32(q).reshape(-1), _f32(k), _f32(v)
    group = n_q_heads // n_kv_heads
    nc = len(chunks)
    m = np.empty((n_q_heads, nc), np.float32)
    l = np.empty((n_q_heads, nc), np.float32)
    o = np.empty((n_q_heads, nc, head_dim), np.float32)
    for h in range(n_q_heads):
        g = h // group
        qh = q[h * head_dim:(h + 1) * head_dim]
        for c, (j0, j1) in enumerate(chunks):
            kh = k[j0:j1, g * head_dim:(g + 1) * head_dim]
            vh = v[j0:j1, g * head_dim:(g + 1) * head_dim]
            s = (kh @ qh) * np.float32(scale)
            m[h, c] = np.max(s)
            p = np.exp(s - m[h, c])
            l[h, c] = np.sum(p, dtype=np.float32)
            o[h, c] = p @ vh
    return m, l, o


def attention_reduce(m, l, o, out_dtype):
    """LSE merge of split-KV partials ([B300] §2 "ATTENTION_COMBINE ... LSE-merge of the partials").

        M = max_c m_c,  L = sum_c l_c e^{m_c - M},  O = sum_c o_c e^{m_c - M} / L.
    Returns the [1 × H·d] row rounded to out_dtype.
    Pinned by: the merge of any split equals unsplit softmax attention (tests, splits
    {1, 2, 3, 8, 17}); a single chunk gives o/l.
    """
    mm = np.max(m, axis=1, keepdims=True)
    w = np.exp(m - mm)                                   # [H, C]
    big_l = np.sum(l * w, axis=1, dtype=np.float32)      # [H]
    big_o = np.sum(o * w[:, :, None], axis=1, dtype=np.float32) / big_l[:, None]
    return round_to(big_o.reshape(1, -1), out_dtype)


def argmax_rows(x):
    """Greedy sampling: per row the first column holding the row's largest value ([B300] §8
    SAMPLE, the argmax of the logits). NaN entries take no part; a row without a number gives -1.
    Returns int32 [rows × 1]. Pinned by brute force and planted ties (tests).
    """
    x = _f32(x)
    out = np.full((x.shape[0], 1), -1, dtype=np.int32)
    for r in range(x.shape[0]):
        cols = np.nonzero(~np.isnan(x[r]))[0]
        if cols.size:
            out[r, 0] = cols[np.argmax(x[r, cols])]   # np.argmax: the first maximum
    return out
