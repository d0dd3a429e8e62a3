"""The allocation-free GEMV entry point (mk_gemv_noalloc) against the oracle and the compiled
plan.

Some callers cannot allocate device memory when they need a product: a serving loop whose
device memory an up-front pool owns, code running inside that pool's callbacks, or a
latency-bound path where cudaMalloc / cudaFree would synchronise the device. mk_gemv_noalloc
keeps its run state in a fixed device array inside the library instead. This test calls it
through the C ABI, twice in a row per shape and back to back with shapes whose split counts
differ, and checks every result element by element against the CPU oracle's matmul on the same
quantised inputs, within the parity tolerance of the other GPU tests (and against
mk_compile + mk_run), and runs it inside a stream capture. It sits in a file of its own that pytest collects last.
"""
import ctypes as C

import numpy as np
import pytest
import torch

from oracle import ops
from oracle.numerics import BF16, F16
from tensor_core_gemm_gb300 import Graph, _lib, synth

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _close(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(got - ref)
    assert np.linalg.norm(err) <= 5e-3 * max(np.linalg.norm(ref), 1e-30)
    assert np.all(err <= 2e-2 * np.maximum(1.0, np.abs(ref)))


def _inputs(m, n, k, dt, seed=101):
    if k == 0:   # an empty product: real (unread) buffers, since the call refuses NULL inputs
        x = synth.normal((m, 8), 1.0, dt, seed, DEV)
        w = synth.normal((8, n), 0.02, dt, seed + 1, DEV)
        return x, w, np.zeros((m, n), np.float32)
    x = synth.normal((m, k), 1.0, dt, seed, DEV)
    w = synth.normal((k, n), 0.02, dt, seed + 1, DEV)
    ref = ops.matmul(synth.to_numpy_f32(x), synth.to_numpy_f32(w), BF16 if dt == "bf16" else F16)
    return x, w, ref


def _call(lib, x, w, out, m, n, k, dt, status=None):
    code = _lib.MK_BF16 if dt == "bf16" else _lib.MK_F16
    return lib.mk_gemv_noalloc(C.c_void_p(x.data_ptr()), C.c_void_p(w.data_ptr()),
                               C.c_void_p(out.data_ptr()), m, n, k, code,
                               C.c_void_p(torch.cuda.current_stream().cuda_stream),
                               C.byref(status) if status is not None else None)


@pytest.mark.parametrize("m,n,k,dt", [(1, 3072, 2048, "bf16"), (4, 1000, 520, "bf16"),
                                      (8, 256, 4096, "f16"), (1, 2048, 8192, "bf16"),
                                      (3, 8, 64, "bf16"), (2, 264, 0, "f16")])
def test_noalloc_gemv_matches_oracle_and_compiled_plan(m, n, k, dt):
    lib = _lib.load()
    x, w, ref = _inputs(m, n, k, dt)
    plan_out = None
    if k > 0:
        plan_out = torch.zeros((m, n), dtype=x.dtype, device=DEV)
        g = Graph()
        ix, iw, io = g.tensor(x), g.tensor(w), g.tensor(plan_out)
        g.matmul(ix, iw, io)
        plan = g.compile()
        plan.run()
        plan.check_status()
    for call in range(2):
        out = torch.full((m, n), 3.0, dtype=x.dtype, device=DEV)
        st = _lib.DeviceStatus()
        rc = _call(lib, x, w, out, m, n, k, dt, st)
        assert rc == _lib.MK_OK, lib.mk_last_error().decode()
        assert st.code == 0
        got = synth.to_numpy_f32(out)
        _close(got, ref)
        if plan_out is not None:
            _close(got, synth.to_numpy_f32(plan_out))


def test_noalloc_back_to_back_calls_with_different_split_counts():
    # three calls queued on one stream before a single synchronisation, with 12 column tiles x
    # 11 K splits, 8 tiles x 16 splits and 1 tile x 3 splits (the split counts of 152 SMs)
    lib = _lib.load()
    shapes = [(1, 3072, 2048, "bf16"), (2, 2048, 2048, "bf16"), (1, 128, 192, "f16")]
    cases = []
    for i, (m, n, k, dt) in enumerate(shapes):
        x, w, ref = _inputs(m, n, k, dt, seed=200 + 10 * i)
        out = torch.full((m, n), -7.0, dtype=x.dtype, device=DEV)
        assert _call(lib, x, w, out, m, n, k, dt) == _lib.MK_OK, lib.mk_last_error().decode()
        cases.append((out, ref))
    torch.cuda.synchronize()
    for out, ref in cases:
        _close(synth.to_numpy_f32(out), ref)
    st = _lib.DeviceStatus()   # the status of the last run, read with a synchronising call
    m, n, k, dt = shapes[0]
    x, w, ref = _inputs(m, n, k, dt, seed=200)
    out = torch.empty((m, n), dtype=x.dtype, device=DEV)
    assert _call(lib, x, w, out, m, n, k, dt, st) == _lib.MK_OK and st.code == 0
    _close(synth.to_numpy_f32(out), ref)


def test_noalloc_rejects_sizes_beyond_its_fixed_scratch():
    lib = _lib.load()
    x = torch.zeros((1, 64), dtype=torch.bfloat16, device=DEV)
    w = torch.zeros((64, 8), dtype=torch.bfloat16, device=DEV)
    o = torch.zeros((1, 8), dtype=torch.bfloat16, device=DEV)
    p = [C.c_void_p(t.data_ptr()) for t in (x, w, o)]
    rc = lib.mk_gemv_noalloc(*p, 1, 262144 + 8, 64, _lib.MK_BF16, None, None)
    assert rc == _lib.MK_ERR_UNSUPPORTED and b"maximum" in lib.mk_last_error()
    rc = lib.mk_gemv_noalloc(*p, 9, 8, 64, _lib.MK_BF16, None, None)
    assert rc == _lib.MK_ERR_UNSUPPORTED


def test_noalloc_inside_a_stream_capture():
    # a status-reading call is refused on a capturing stream (it would synchronise); a call
    # without status becomes graph nodes that replay on whatever the captured buffers hold
    lib = _lib.load()
    m, n, k, dt = 2, 512, 1024, "bf16"
    x, w, ref = _inputs(m, n, k, dt, seed=300)
    out = torch.zeros((m, n), dtype=x.dtype, device=DEV)
    assert _call(lib, x, w, out, m, n, k, dt) == _lib.MK_OK   # per-device set-up, uncaptured
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        refused = _call(lib, x, w, out, m, n, k, dt, _lib.DeviceStatus())
        refused_msg = lib.mk_last_error()
        captured = _call(lib, x, w, out, m, n, k, dt)
    assert refused == _lib.MK_ERR_UNSUPPORTED and b"capturing" in refused_msg
    assert captured == _lib.MK_OK, lib.mk_last_error().decode()
    for seed in (300, 310):
        x2, w2, ref = _inputs(m, n, k, dt, seed=seed)
        x.copy_(x2)   # new contents at the captured addresses (w through its tensor map)
        w.copy_(w2)
        out.fill_(5.0)
        graph.replay()
        torch.cuda.synchronize()
        _close(synth.to_numpy_f32(out), ref)
