"""Seeded random graphs: the host compiler's plan equals the oracle schedule, field by field.

Each graph is a chain over one activation: matmuls (GEMM shapes and GEMV shapes, with bias,
ReLU, residual, RMSNorm-input and SiLU·mul epilogues), elementwise ops and RMSNorm rows, with
random widths (multiples of 8), random placement options, and a random subset of the
intermediates declared plan-owned (the buffer pool). CPU only (dry-run plans)."""
import numpy as np
import pytest

from test_host_compiler import assert_same_plan


def _random_graph(rng):
    m = int(rng.choice([1, 3, 8, 64, 128, 200, 384]))
    width = int(rng.choice([64, 128, 256, 320]))
    tensors = [{"rows": m, "cols": width, "dtype": "bf16"}]
    nodes = []
    cur = (0, 0, 0, m, width)

    def new(rows, cols, transient=False):
        tensors.append({"rows": rows, "cols": cols, "dtype": "bf16", "transient": transient})
        return (len(tensors) - 1, 0, 0, rows, cols)

    long_rows = bool(rng.random() < 0.4)   # long same-shape runs: buffers can be handed on
    n_nodes = int(rng.integers(6, 12)) if long_rows else int(rng.integers(2, 7))
    for i in range(n_nodes):
        last = i == n_nodes - 1
        trans = (not last) and bool(rng.random() < (0.8 if long_rows else 0.5))
        kinds = ["ew", "ew", "rmsnorm", "matmul"] if long_rows else ["matmul", "matmul", "ew", "rmsnorm"]
        kind = rng.choice(kinds)
        k = cur[4]
        if kind == "matmul":
            n = int(rng.choice([64, 128, 256, 384, 512]))
            nd = {"kind": "matmul", "a": cur, "b": new(k, n)}
            if rng.random() < 0.3:
                nd["bias"] = new(m, n)
            if rng.random() < 0.3:
                nd["relu"] = True
            if rng.random() < 0.3:
                nd["residual"] = new(m, n)
            if m <= 8 and rng.random() < 0.4:
                nd["gamma"] = new(1, k)
            if rng.random() < 0.25 and not nd.get("relu") and "bias" not in nd:
                nd["b2"] = new(k, n)
            nd["c"] = new(m, n, trans)
            nodes.append(nd)
            cur = nd["c"]
        elif kind == "ew":
            op = str(rng.choice(["relu", "copy", "add"]))
            ins = [cur] if op != "add" else [cur, new(m, k)]
            out = new(m, k, trans)
            nodes.append({"kind": "ew", "op": op, "ins": ins, "out": out})
            cur = out
        else:
            out = new(m, k, trans)
            nodes.append({"kind": "rmsnorm", "x": cur, "gamma": new(1, k), "out": out})
            cur = out
    return {"tensors": tensors, "nodes": nodes}


def _random_opts(rng):
    cluster = int(rng.choice([1, 1, 2]))
    o = dict(n_sm=int(rng.choice([2, 3, 4, 7, 16, 37, 152])) * (2 if cluster == 2 else 1),
             cluster=cluster,
             gemm_tile_m=128 * cluster,
             gemm_tile_n=int(rng.choice([128, 256])) if cluster == 2 else int(rng.choice([64, 128, 256])),
             wave_pack=int(rng.integers(0, 2)),
             gemm_group_m=int(rng.choice([1, 2, 8])),
             pool_waves=int(rng.choice([1, 2])),
             ew_rows=int(rng.choice([32, 128])),
             norm_rows=int(rng.choice([4, 16])),
             gemm_split_tail=int(rng.integers(0, 2)),
             gemv_splits=int(rng.choice([0, 0, 1, 3])))
    return o


@pytest.mark.parametrize("seed", range(300))
def test_random_plan_matches_oracle(seed):
    rng = np.random.default_rng(1000 + seed)
    desc = _random_graph(rng)
    opts = _random_opts(rng)
    assert_same_plan(desc, opts)


@pytest.mark.parametrize("seed", range(60))
def test_random_decoder_plan_matches_oracle(seed):
    # Decoder graphs (split-KV decode with optional sampling head, causal prefill) of random
    # shapes: attention lowering (key chunks, prefill query tiles, GQA ratios, ragged token
    # counts), the RoPE and combine fusions, wave packing of attention phases and pooled
    # intermediates, against the oracle schedule.
    from tensor_core_gemm_gb300 import workloads
    rng = np.random.default_rng(5000 + seed)
    hkv = int(rng.choice([1, 2, 4]))
    hq = hkv * int(rng.choice([1, 2, 4]))
    sh = workloads.DecoderShape(layers=int(rng.integers(1, 4)), hidden=int(rng.choice([128, 256])),
                                n_q_heads=hq, n_kv_heads=hkv, head_dim=64,
                                ffn=int(rng.choice([256, 512])))
    if rng.random() < 0.5:
        wl = workloads.decode(sh, kv_len=int(rng.choice([1, 17, 100, 300])),
                              vocab=int(rng.choice([0, 0, 1000])))
    else:
        wl = workloads.prefill(sh, tokens=int(rng.choice([64, 130, 256, 384])))
    if rng.random() < 0.4:
        wl = workloads.with_transients(wl, *workloads.decoder_intermediates(wl))
    opts = dict(n_sm=int(rng.choice([8, 37, 152])), attn_chunk=int(rng.choice([16, 64])),
                fuse_rope=int(rng.integers(0, 2)), fuse_attn_reduce=int(rng.integers(0, 2)),
                wave_pack=int(rng.integers(0, 2)), gemm_group_m=int(rng.choice([1, 8])),
                gemv_splits=int(rng.choice([0, 2])), norm_rows=int(rng.choice([4, 16])))
    assert_same_plan(wl.desc, opts)
