"""Neutral graph descriptions used by the schedule tests (plain data, no arithmetic)."""


def mlp_unfused(m=1024, h=1024, layers=3, dtype="bf16", transient=False):
    """The aten graph of the MegaKittens MLP example: per layer mm -> add(bias) -> relu.

    Tensors: 0 = W [layers·h × h] (stacked K×N weights), 1 = x [m × h], 2 = b [layers·m × h],
    then per layer mm, add, relu outputs (plan-owned transients when ``transient``).
    """
    tensors = [{"rows": layers * h, "cols": h, "dtype": dtype},
               {"rows": m, "cols": h, "dtype": dtype},
               {"rows": layers * m, "cols": h, "dtype": dtype}]
    nodes = []
    cur = (1, 0, 0, m, h)
    for i in range(layers):
        ids = []
        for _ in range(3):
            ids.append(len(tensors))
            tensors.append({"rows": m, "cols": h, "dtype": dtype, "transient": transient})
        mm, ad, rl = [(t, 0, 0, m, h) for t in ids]
        nodes.append({"kind": "matmul", "a": cur, "b": (0, i * h, 0, h, h), "c": mm})
        nodes.append({"kind": "ew", "op": "add", "ins": [mm, (2, i * m, 0, m, h)], "out": ad})
        nodes.append({"kind": "ew", "op": "relu", "ins": [ad], "out": rl})
        cur = rl
    return {"tensors": tensors, "nodes": nodes}


P3_OPTS = dict(n_sm=148, gemm_tile_m=512, gemm_tile_n=256, cluster=2, gemm_split_tail=0,
               gemm_group_m=1,
               ew_rows=128, ew_cols=128, ew_tiles=2)
