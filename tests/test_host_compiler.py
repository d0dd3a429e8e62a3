"""The C-ABI library on the CPU: exports, validation, and the compiler's integer output
(instruction list, counters, targets, arrivals, placement) bit-exact against the oracle's
schedule, computed independently by brute-force box intersection."""
import ctypes as C
import os
import re

import numpy as np
import pytest

import _graphs
from oracle import schedule as osched

mk = pytest.importorskip("tensor_core_gemm_gb300")
from tensor_core_gemm_gb300 import _lib, workloads  # noqa: E402
from tensor_core_gemm_gb300._lib import MkError  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

FIELDS = ["op", "flags", "node", "m0", "n0", "k0", "klen", "aux0", "aux1", "sem"]


@pytest.fixture(scope="module", autouse=True)
def built():
    if not os.path.exists(_lib.LIB_PATH):
        from tensor_core_gemm_gb300 import build
        build.build()


def test_library_exports_every_declared_symbol():
    with open(os.path.join(ROOT, "include", "mk.h")) as f:
        header = f.read()
    declared = set(re.findall(r"^\s*(?:mk_status|const char\*|int32_t)\s+(mk_\w+)\s*\(", header,
                              re.M))
    assert declared == set(_lib.EXPORTS)
    lib = C.CDLL(_lib.LIB_PATH)
    for name in declared:
        assert hasattr(lib, name), name
    assert _lib.load().mk_abi_version() == 2


def _dry(desc, **opts):
    g, _ = workloads.build_graph(desc, None)
    return g.compile(dry_run=1, **opts)


def assert_same_plan(desc, opts):
    """Compiler output == oracle schedule, field by field and list by list."""
    py = osched.lower(desc, opts)
    c = _dry(desc, **opts)
    st = c.stats()
    assert st["n_instr"] == py.n_instr
    assert st["n_counters"] == py.n_dep
    assert st["n_sems"] == py.n_sem
    assert abs(st["waves"] - py.waves) < 1e-12
    ins = c.instructions()
    want = osched.as_array(py)
    got = np.stack([ins[f].astype(np.int64) for f in FIELDS], axis=1)
    bad = np.nonzero(np.any(want != got, axis=1))[0]
    assert bad.size == 0, f"first differing instruction {bad[:5]}: {want[bad[0]]} vs {got[bad[0]]}"
    src = c.src_list()
    dst = c.dst_list()
    want_src = [pair for i in py.instrs for pair in i.src]
    want_dst = [d for i in py.instrs for d in i.dst]
    assert [tuple(x) for x in src.tolist()] == want_src
    assert dst.tolist() == want_dst
    assert ins["n_src"].tolist() == [len(i.src) for i in py.instrs]
    assert ins["n_dst"].tolist() == [len(i.dst) for i in py.instrs]
    assert ins["src_off"].tolist() == list(np.cumsum([0] + [len(i.src) for i in py.instrs])[:-1])
    assert ins["dst_off"].tolist() == list(np.cumsum([0] + [len(i.dst) for i in py.instrs])[:-1])
    assert c.counter_targets().tolist() == py.targets
    assert st["pool_bytes"] == py.pool_bytes and st["n_reuse"] == py.n_reuse
    assert osched.topologically_valid(py)
    return py, c


def test_p3_mlp_plan_matches_oracle_and_page():
    py, c = assert_same_plan(_graphs.mlp_unfused(), _graphs.P3_OPTS)
    st = c.stats()
    assert st["n_instr"] == 240 and st["n_counters"] == 124 and f"{st['waves']:.2f}" == "1.62"


@pytest.mark.parametrize("m,n,k,tn", [(1024, 1024, 1024, 256), (300, 392, 200, 256),
                                      (128, 64, 64, 64), (4096, 4096, 4096, 256),
                                      (257, 136, 0, 128)])
def test_gemm_plans(m, n, k, tn):
    assert_same_plan(workloads.gemm(m, n, k).desc, dict(n_sm=152, gemm_tile_n=tn))


@pytest.mark.parametrize("m,n,k,tn", [(4096, 4096, 4096, 256), (300, 392, 200, 128),
                                      (129, 72, 520, 128)])
def test_pair_gemm_plans(m, n, k, tn):
    """CTA-pair tiles: 256 x tn, two instructions per tile on an even/odd SM pair."""
    opts = dict(n_sm=152, gemm_tile_n=tn, gemm_tile_m=256, cluster=2, gemm_split_tail=0)
    py, c = assert_same_plan(workloads.gemm(m, n, k).desc, opts)
    ins = c.instructions()
    gem = np.nonzero(ins["op"] == osched.OP_GEMM)[0]
    assert gem.size == 2 * (-(-m // 256)) * (-(-n // tn))
    assert np.all(gem[0::2] % 2 == 0) and np.all(gem[1::2] == gem[0::2] + 1)
    assert np.all(ins["aux0"][gem[0::2]] == 0) and np.all(ins["aux0"][gem[1::2]] == 1)


@pytest.mark.parametrize("m,n,k,tm,tn,cl", [(4096, 4096, 4096, 256, 256, 2),
                                            (4096, 4096, 4096, 128, 256, 1),
                                            (1000, 1024, 776, 128, 128, 1),
                                            (600, 640, 200, 256, 128, 2)])
def test_split_tail_plans(m, n, k, tm, tn, cl):
    """The last, partly filled wave of GEMM tiles is split along K: the plan equals the
    oracle's, the splits of a tile cover K exactly once per rank in order, split 0 alone carries
    the output box, and every split of a (tile, rank) shares split 0's arrivals and semaphore."""
    opts = dict(n_sm=152, gemm_tile_m=tm, gemm_tile_n=tn, cluster=cl, gemm_split_tail=1)
    py, c = assert_same_plan(workloads.gemm(m, n, k).desc, opts)
    tiles = -(-m // tm) * -(-n // tn)
    units = 152 // cl
    r_tail = tiles % units
    ins = c.instructions()
    gem = ins[ins["op"] == osched.OP_GEMM]
    split = gem[gem["aux1"] > 0]
    n_split = min(units // r_tail, -(-k // 64)) if r_tail else 1
    if n_split < 2:
        assert split.size == 0
        return
    nr = int(split["aux1"][0])
    assert split.size == r_tail * nr * cl
    assert gem.size == (tiles - r_tail) * cl + split.size
    for t in range(r_tail):
        blk = split[t * nr * cl:(t + 1) * nr * cl]
        assert len(set(zip(blk["m0"], blk["n0"]))) == 1
        for r in range(cl):
            mine = blk[blk["aux0"] == r]
            assert list(mine["split"]) == list(range(nr))
            assert mine["k0"][0] == 0 and (mine["k0"] + mine["klen"])[-1] == k
            assert np.all(mine["k0"][1:] == (mine["k0"] + mine["klen"])[:-1])
            assert len(set(mine["sem"])) == 1
            assert np.all(mine["slot"] == mine["slot"][0])
    fin = py.final_counters()
    sem_vals = fin[py.n_dep:]
    # two splits meet twice (exchange of halves, then finish); more splits once each
    assert sem_vals.count(4 if nr == 2 else nr) == r_tail * cl


def test_mlp3_plan():
    py, c = assert_same_plan(workloads.mlp3().desc, dict(n_sm=152, gemm_tile_n=64))
    # layer-2 tiles wait on exactly the 16 layer-1 tiles of their 128-row block
    l2 = [i for i in py.instrs if i.node == 1]
    assert all(len(i.src) == 1 and i.src[0][1] == 16 for i in l2)


def test_gemm_list_plans():
    assert_same_plan(workloads.gemm_list(workloads.LLAMA70B_DECODE).desc, dict(n_sm=152))
    assert_same_plan(workloads.gemm_list(workloads.LLAMA70B_PREFILL).desc, dict(n_sm=148))


def test_decode_plan_full_size():
    py, c = assert_same_plan(workloads.decode().desc, dict(n_sm=152))
    per_op = c.stats()["per_op"]
    # RoPE runs inside the QKV GEMV tiles and the split-KV combine inside the last partial of
    # each key/value head (both fused by default), or as separate instructions
    assert per_op[osched.OP_ROPE] == 0 and per_op[osched.OP_ATTN_REDUCE] == 0
    py0, c0 = assert_same_plan(workloads.decode().desc,
                               dict(n_sm=152, fuse_rope=0, fuse_attn_reduce=0))
    assert c0.stats()["per_op"][osched.OP_ROPE] == 16
    assert c0.stats()["per_op"][osched.OP_ATTN_REDUCE] == 16 * 8
    # fused partials: every partial of a head shares one semaphore, which counts all of them
    parts = [i for i in py.instrs if i.op == osched.OP_ATTN_PARTIAL]
    assert len({i.sem for i in parts}) == 16 * 8
    fin = py.final_counters()[py.n_dep:]
    assert fin.count(17) == 16 * 8
    # the fused QKV tiles carry the rotated q / k and the appended v boxes
    qkv_tiles = [i for i in py.instrs if i.op == osched.OP_GEMV and i.node == 0 and i.k0 == 0]
    assert sum(len(i.writes) for i in qkv_tiles) == 12 + 8 + 2 + 2
    assert per_op[osched.OP_ATTN_PARTIAL] == 16 * 8 * 17   # 1025 keys in chunks of 64


def test_prefill_plan_small():
    sh = workloads.DecoderShape(layers=2, hidden=256, n_q_heads=4, n_kv_heads=2, head_dim=64,
                                ffn=512)
    assert_same_plan(workloads.prefill(sh, tokens=384).desc, dict(n_sm=37))
    # on CTA pairs: 256-row GEMM and attention tiles, one instruction per rank
    py, c = assert_same_plan(workloads.prefill(sh, tokens=384).desc,
                             dict(n_sm=38, gemm_tile_m=256, cluster=2))
    ins = c.instructions()
    att = ins[ins["op"] == osched.OP_ATTN_PREFILL]
    assert len(att) == 2 * 2 * 4 * 2 and sorted(set(att["m0"])) == [0, 256]  # layers, tiles, heads, ranks
    assert np.all(att["aux0"][0::2] == 0) and np.all(att["aux0"][1::2] == 1)


@pytest.mark.slow
def test_prefill_plan_full_size():
    assert_same_plan(workloads.prefill(tokens=2048).desc, dict(n_sm=152))


def test_gemv_split_and_unfused_elementwise_plans():
    assert_same_plan(workloads.gemm(1, 3072, 2048, dtype="bf16").desc, dict(n_sm=152))
    assert_same_plan(workloads.gemm(3, 1000, 520, dtype="bf16").desc,
                     dict(n_sm=20, gemv_splits=3))
    assert_same_plan(_graphs.mlp_unfused(m=300, h=256, layers=2, dtype="f16"),
                     dict(n_sm=16, ew_rows=64, ew_cols=64, ew_tiles=2, gemm_tile_n=128))


@pytest.mark.parametrize("gm", [1, 2, 3, 8])
def test_grouped_gemm_tile_order(gm):
    """Tiles go group by group of gm row tiles, column by column inside a group, row by row
    within a column (the last group shorter), bit-exact with the oracle for every group size."""
    desc = workloads.gemm(5 * 128, 3 * 256, 192).desc
    py, c = assert_same_plan(desc, dict(n_sm=8, gemm_group_m=gm))
    order = [(i.m0 // 128, i.n0 // 256) for i in py.instrs if i.op == osched.OP_GEMM]
    want = []
    for g0 in range(0, 5, gm):
        rows = list(range(g0, min(5, g0 + gm)))
        for nt in range(3):
            want += [(mt, nt) for mt in rows]
    assert order == want


def test_wave_packing_of_independent_gemms():
    """Independent GEMM nodes are placed as one run, longest K first on the least loaded CTA
    pair: the same tiles as without packing, each pair's total K within the longest-first bound
    (average + one tile), the list mirrored bit for bit by the oracle; equal costs keep the
    order."""
    desc = workloads.gemm_list(workloads.LLAMA70B_DECODE).desc
    opts = dict(n_sm=152, gemm_tile_m=256, cluster=2)
    packed, _ = assert_same_plan(desc, dict(opts, wave_pack=1))
    plain, _ = assert_same_plan(desc, dict(opts, wave_pack=0))
    tiles = lambda py: sorted(i.key() for i in py.instrs if i.op == osched.OP_GEMM)
    assert tiles(packed) == tiles(plain)
    load = {}
    for idx, ins in enumerate(packed.instrs):
        if ins.op == osched.OP_GEMM and ins.aux0 == 0:
            load[(idx % 152) // 2] = load.get((idx % 152) // 2, 0) + ins.klen
    loads = [load.get(u, 0) for u in range(76)]
    assert max(loads) <= sum(loads) / 76 + 28672
    plain_load = {}
    for idx, ins in enumerate(plain.instrs):
        if ins.op == osched.OP_GEMM and ins.aux0 == 0:
            plain_load[(idx % 152) // 2] = plain_load.get((idx % 152) // 2, 0) + ins.klen
    assert max(loads) < max(plain_load.values())
    # equal K everywhere: the packed list is the plain one
    pre = workloads.gemm_list(workloads.LLAMA70B_PREFILL).desc
    a, _ = assert_same_plan(pre, dict(opts, wave_pack=1))
    b, _ = assert_same_plan(pre, dict(opts, wave_pack=0))
    assert [i.key() for i in a.instrs] == [i.key() for i in b.instrs]


def test_argmax_plans():
    """ARGMAX lowers to chunk partials and one reduce per row block, bit-exact with the oracle
    (ragged rows and chunks; the decode head after the last layer)."""
    desc = {"tensors": [{"rows": 37, "cols": 10000, "dtype": "bf16"},
                        {"rows": 37, "cols": 1, "dtype": "i32"}],
            "nodes": [{"kind": "argmax", "x": (0, 0, 0, 37, 10000), "out": (1, 0, 0, 37, 1)}]}
    py, c = assert_same_plan(desc, dict(n_sm=16, argmax_chunk=1024))
    assert c.stats()["per_op"][osched.OP_ARGMAX] == 3 * 10
    assert c.stats()["per_op"][osched.OP_ARGMAX_REDUCE] == 3
    sh = workloads.DecoderShape(layers=2, hidden=256, n_q_heads=4, n_kv_heads=2, head_dim=64,
                                ffn=512)
    assert_same_plan(workloads.decode(sh, kv_len=100, vocab=5000).desc, dict(n_sm=40))
    assert_same_plan(workloads.decode(vocab=128256).desc, dict(n_sm=152))


def test_final_counter_values_definition():
    py = osched.lower(workloads.gemm(1, 512, 1024, dtype="bf16").desc, dict(n_sm=8))
    fin = py.final_counters()
    assert fin[py.n_dep:] == [py.instrs[0].aux1] * py.n_sem


# ------------------------------------------------------------------ validation

def test_shape_and_id_errors():
    g = mk.Graph()
    a = g.tensor(ptr=0, dtype="f16", shape=[64, 32])
    b = g.tensor(ptr=0, dtype="f16", shape=[16, 64])
    c = g.tensor(ptr=0, dtype="f16", shape=[64, 64])
    with pytest.raises(MkError) as e:
        g.matmul(a, b, c)
    assert e.value.code == _lib.MK_ERR_INVALID_ARG
    with pytest.raises(MkError):
        g.view(a, 60, 0, 8, 32)
    with pytest.raises(MkError):
        g.matmul(a, 99, c)
    bf = g.tensor(ptr=0, dtype="bf16", shape=[32, 64])
    with pytest.raises(MkError) as e:
        g.matmul(a, bf, c)
    assert e.value.code == _lib.MK_ERR_UNSUPPORTED
    with pytest.raises(MkError):
        g.elementwise("add", [a], c)


def test_hazards_rejected():
    g = mk.Graph()
    x = g.tensor(ptr=0, dtype="f16", shape=[128, 128])
    w = g.tensor(ptr=0, dtype="f16", shape=[128, 128])
    g.matmul(x, w, x)                     # in place: writes what it reads
    with pytest.raises(MkError) as e:
        g.compile(dry_run=1, n_sm=4)
    assert e.value.code == _lib.MK_ERR_HAZARD
    g = mk.Graph()
    x = g.tensor(ptr=0, dtype="f16", shape=[128, 128])
    w = g.tensor(ptr=0, dtype="f16", shape=[128, 128])
    y = g.tensor(ptr=0, dtype="f16", shape=[128, 128])
    g.matmul(x, w, y)
    g.elementwise("relu", [x], y)         # second writer of y
    with pytest.raises(MkError) as e:
        g.compile(dry_run=1, n_sm=4)
    assert e.value.code == _lib.MK_ERR_HAZARD


def test_dry_run_requires_n_sm_and_run_rejects_dry_plans():
    g, _ = workloads.build_graph(workloads.gemm(128, 128, 64).desc, None)
    with pytest.raises(MkError):
        g.compile(dry_run=1)
    p = g.compile(dry_run=1, n_sm=4)
    with pytest.raises(MkError):
        p.run()


def test_empty_graph_and_empty_matmul():
    g = mk.Graph()
    p = g.compile(dry_run=1, n_sm=8)
    assert p.stats()["n_instr"] == 0
    for m, n, k in [(0, 64, 64), (64, 0, 64), (1, 0, 128)]:
        d = workloads.gemm(m, n, k, dtype="bf16").desc
        assert_same_plan(d, dict(n_sm=8))
        assert _dry(d, n_sm=8).stats()["n_instr"] == 0
    # K = 0: one instruction per tile whose output is the epilogue of zero
    for m in (1, 200):
        py, c = assert_same_plan(workloads.gemm(m, 64, 0, dtype="bf16").desc, dict(n_sm=8))
        assert c.stats()["n_instr"] == 1 + (m > 128)


# ------------------------------------------------------------------ kernel specialisation

def _mixed_gemv_gemm(h=256):
    """One GEMV-sized product (1 row) and one GEMM-sized product (256 rows) sharing a weight."""
    t = [{"rows": h, "cols": h, "dtype": "bf16"}, {"rows": 1, "cols": h, "dtype": "bf16"},
         {"rows": 1, "cols": h, "dtype": "bf16"}, {"rows": 256, "cols": h, "dtype": "bf16"},
         {"rows": 256, "cols": h, "dtype": "bf16"}]
    w = (0, 0, 0, h, h)
    return {"tensors": t, "nodes": [
        {"kind": "matmul", "a": (1, 0, 0, 1, h), "b": w, "c": (2, 0, 0, 1, h)},
        {"kind": "matmul", "a": (3, 0, 0, 256, h), "b": w, "c": (4, 0, 0, 256, h)}]}


def test_kernel_specialisation_choice():
    """mk_run launches the smallest specialisation whose instruction kinds cover the plan:
    0 general, 1 GEMM tiles only, 2 decode (GEMV, split-KV attention, rows), 3 prefill (GEMM,
    prefill attention, rows); CTA-pair kernels exist for the GEMM-only, prefill and general
    sets."""
    sh = workloads.DecoderShape(layers=2, hidden=256, n_q_heads=4, n_kv_heads=2, head_dim=64,
                                ffn=512)
    pair = dict(gemm_tile_m=256, cluster=2)
    unf = _graphs.mlp_unfused(m=300, h=256, layers=2, dtype="f16")
    cases = [
        (workloads.gemm(512, 512, 256).desc, dict(n_sm=8), 1),
        (workloads.gemm(512, 512, 256).desc, dict(n_sm=8, **pair), 1),
        (workloads.mlp3().desc, dict(n_sm=152, gemm_tile_n=64), 1),
        (workloads.gemm(1, 3072, 2048, dtype="bf16").desc, dict(n_sm=152), 2),
        (workloads.decode(sh, kv_len=200).desc, dict(n_sm=40), 2),
        (workloads.decode(sh, kv_len=200).desc, dict(n_sm=40, fuse_rope=0, fuse_attn_reduce=0), 2),
        (workloads.prefill(sh, tokens=384).desc, dict(n_sm=37), 3),
        (unf, dict(n_sm=16, gemm_tile_n=128), 3),
        (unf, dict(n_sm=16, **pair), 3),  # GEMM + rows on pairs: the prefill pair kernel
        (workloads.prefill(sh, tokens=384).desc, dict(n_sm=38, **pair), 3),
        (workloads.decode(sh, kv_len=200).desc, dict(n_sm=40, **pair), 0),
        (_mixed_gemv_gemm(), dict(n_sm=16), 0),
        (workloads.gemm(512, 512, 256).desc, dict(n_sm=8, kernel_set=1), 0),
        (workloads.decode(sh, kv_len=200).desc, dict(n_sm=40, kernel_set=1), 0),
    ]
    for desc, opts, want in cases:
        assert _dry(desc, **opts).stats()["kernel_set"] == want, (opts, want)


# ----------------------------------------------------------------------------- buffer pool
_SMALL = dict(layers=6, hidden=256, n_q_heads=4, n_kv_heads=2, head_dim=64, ffn=512)


def test_p3_mlp_pool_plan_matches_oracle_and_page():
    py, c = assert_same_plan(_graphs.mlp_unfused(transient=True), _graphs.P3_OPTS)
    st = c.stats()
    assert st["n_counters"] == 125 and st["n_reuse"] == 1 and st["n_instr"] == 240
    assert st["pool_bytes"] == 8 * 1024 * 1024 * 2   # eight 1024 x 1024 bf16 buffers


@pytest.mark.parametrize("kind,n_sm", [("prefill", 37), ("decode", 40), ("decode", 8),
                                       ("decode_full", 152)])
def test_pooled_decoder_plans_match_oracle(kind, n_sm):
    sh = workloads.DecoderShape(**_SMALL)
    wl = {"prefill": lambda: workloads.prefill(sh, tokens=384),
          "decode": lambda: workloads.decode(sh, kv_len=100, vocab=5000),
          "decode_full": lambda: workloads.decode(vocab=128256)}[kind]()
    pw = workloads.with_transients(wl, *workloads.decoder_intermediates(wl))
    py, c = assert_same_plan(pw.desc, dict(n_sm=n_sm))
    summed = sum(osched.transient_bytes(pw.desc["tensors"][t]) for t in pw.info["transients"])
    assert py.n_reuse > 0 and py.pool_bytes < summed
    # plain and pooled plans run the same instructions; only the counter lists grow
    plain = osched.lower(wl.desc, dict(n_sm=n_sm))
    assert np.array_equal(osched.as_array(plain)[:, :9], osched.as_array(py)[:, :9])
    assert py.n_dep == plain.n_dep + py.n_reuse


@pytest.mark.parametrize("waves", [2, 5])
def test_pool_reuse_distance_option(waves):
    sh = workloads.DecoderShape(**_SMALL)
    wl = workloads.prefill(sh, tokens=384)
    pw = workloads.with_transients(wl, *workloads.decoder_intermediates(wl))
    py, c = assert_same_plan(pw.desc, dict(n_sm=37, pool_waves=waves))
    one = osched.lower(pw.desc, dict(n_sm=37))
    # a longer reuse distance hands fewer buffers on and keeps a larger pool
    assert py.n_reuse <= one.n_reuse and py.pool_bytes >= one.pool_bytes
    assert py.n_reuse < one.n_reuse or py.pool_bytes > one.pool_bytes or waves == 1


def test_pool_waves_validated():
    g, _ = workloads.build_graph(workloads.gemm(128, 128, 64).desc, None)
    with pytest.raises(MkError, match="pool_waves"):
        g.compile(dry_run=1, n_sm=4, pool_waves=0)


def test_pool_footprint_llama_prefill():
    wl = workloads.prefill(tokens=2048)
    pw = workloads.with_transients(wl, *workloads.decoder_intermediates(wl))
    c = _dry(pw.desc, n_sm=152)
    summed = sum(osched.transient_bytes(pw.desc["tensors"][t]) for t in pw.info["transients"])
    assert c.stats()["pool_bytes"] * 10 < summed


def test_transient_validation():
    g = workloads.Graph()
    t = g.transient("bf16", 128, 64)
    o = g.tensor(ptr=0x200000, dtype="bf16", shape=[128, 64])
    g.elementwise("relu", [t], o)                     # read before any node writes it
    with pytest.raises(MkError, match="before a node writes"):
        g.compile(dry_run=1, n_sm=4)
    g = workloads.Graph()
    a = g.tensor(ptr=0x1000, dtype="bf16", shape=[128, 64])
    t = g.transient("bf16", 128, 64)
    top, bot = g.view(t, 0, 0, 64, 64), g.view(t, 64, 0, 64, 64)
    g.elementwise("relu", [g.view(a, 0, 0, 64, 64)], top)
    g.elementwise("relu", [g.view(a, 64, 0, 64, 64)], bot)   # a second writer
    with pytest.raises(MkError, match="one writer"):
        g.compile(dry_run=1, n_sm=4)
    with pytest.raises(MkError, match="unknown dtype"):
        workloads.Graph().transient(7, 4, 4)


def test_transient_addresses_in_dry_plans():
    g = workloads.Graph()
    a = g.tensor(ptr=0x1000, dtype="bf16", shape=[128, 64])
    t = g.transient("bf16", 128, 44)     # 44 columns: rows padded to 48 elements (96 bytes)
    o = g.tensor(ptr=0x200000, dtype="bf16", shape=[128, 44])
    g.elementwise("relu", [g.view(a, 0, 0, 128, 44)], t)
    g.elementwise("relu", [t], o)
    p = g.compile(dry_run=1, n_sm=4)
    assert p.tensor_ptr(a) == 0x1000 and p.tensor_ptr(t) == 0
    assert p.stats()["pool_bytes"] == (128 * 48 * 2 + 1023) // 1024 * 1024


def test_every_entry_point_rejects_null_handles():
    # Each call validates its handles and pointers before any device work and returns an error
    # code (never a crash); destroying NULL is a no-op.
    lib = _lib.load()
    P = C.c_void_p
    bad = _lib.MK_ERR_INVALID_ARG
    i32 = C.c_int32()
    st = _lib.Stats()
    ds = _lib.DeviceStatus()
    buf = (C.c_int32 * 4)()
    assert lib.mk_graph_create(None) == bad
    assert lib.mk_graph_destroy(None) == _lib.MK_OK
    assert lib.mk_plan_destroy(None) == _lib.MK_OK
    shape = (C.c_int64 * 2)(4, 8)
    assert lib.mk_add_tensor(None, P(0x1000), _lib.MK_BF16, 2, shape, None, C.byref(i32)) == bad
    assert lib.mk_add_view(None, 0, 0, 0, 1, 1, C.byref(i32)) == bad
    assert lib.mk_add_transient(None, _lib.MK_BF16, 4, 8, C.byref(i32)) == bad
    assert lib.mk_add_matmul(None, 0, 1, 2, None, C.byref(i32)) == bad
    assert lib.mk_add_elementwise(None, _lib.EW_RELU, buf, 1, 0, None, C.byref(i32)) == bad
    assert lib.mk_add_attention(None, 0, 1, 2, 3, None, C.byref(i32)) == bad
    assert lib.mk_compile(None, None, C.byref(P())) == bad
    assert lib.mk_run(None, None) == bad
    assert lib.mk_run_host(None, None, 0, None) == bad
    assert lib.mk_sync_status(None, C.byref(ds)) == bad
    assert lib.mk_plan_repack(None, None) == bad
    assert lib.mk_plan_stats(None, C.byref(st)) == bad
    assert lib.mk_plan_tensor_ptr(None, 0, C.byref(P())) == bad
    assert lib.mk_get_instructions(None, buf, 16) == bad
    assert lib.mk_get_src_list(None, buf, 4) == bad
    assert lib.mk_get_dst_list(None, buf, 4) == bad
    assert lib.mk_get_counter_targets(None, buf, 4) == bad
    assert lib.mk_get_counters(None, buf, 4) == bad
    assert lib.mk_get_trace(None, (C.c_uint64 * 8)(), 8) == bad
    assert lib.mk_default_opts(None) == bad
    # the allocation-free GEMV checks its arguments before looking for a device
    assert lib.mk_gemv_noalloc(None, None, None, 1, 256, 64, _lib.MK_BF16, None, None) == bad
    assert lib.mk_gemv_noalloc(None, None, None, 9, 256, 64, _lib.MK_BF16, None, None) == \
        _lib.MK_ERR_UNSUPPORTED
    assert lib.mk_last_error()  # the last failure left a message


def test_dry_plan_getters_check_buffer_sizes():
    g, _ = workloads.build_graph(workloads.mlp3(m=256, h=256).desc, None)
    p = g.compile(dry_run=1, n_sm=4, gemm_tile_n=64)
    n = p.stats()["n_instr"]
    from tensor_core_gemm_gb300.api import INSTR_DTYPE
    small = np.zeros(max(1, n - 1), dtype=INSTR_DTYPE)
    with pytest.raises(MkError):
        _lib.check(p._lib.mk_get_instructions(p._h, small.ctypes.data_as(C.c_void_p),
                                              small.nbytes))
    targets = p.counter_targets()
    assert len(targets) > 1
    with pytest.raises(MkError):
        buf = np.zeros(1, dtype=np.int32)
        _lib.check(p._lib.mk_get_counter_targets(p._h, buf.ctypes.data_as(C.POINTER(C.c_int32)),
                                                 max(0, len(targets) - 1)))
