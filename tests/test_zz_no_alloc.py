"""The allocation-free GEMV entry point (mk_gemv_noalloc) against the compiled-plan path.

Callers that cannot allocate device memory when they need a product (an up-front memory pool
owns the device, or cudaMalloc would synchronise a latency-bound path) use mk_gemv_noalloc,
whose run state lives in a fixed device array inside the library. This test calls it through
the C ABI twice in a row per shape and checks each result against mk_compile + mk_run on the
same inputs, within the parity tolerance of the other GPU tests. It sits in a file of its own
that pytest collects last.
"""
import ctypes as C

import numpy as np
import pytest
import torch

from tensor_core_gemm_gb300 import Graph, _lib, synth

pytestmark = pytest.mark.gpu


def _close(got, ref):
    got = got.float().cpu().numpy().astype(np.float64)
    ref = ref.float().cpu().numpy().astype(np.float64)
    err = np.abs(got - ref)
    assert np.linalg.norm(err) <= 5e-3 * max(np.linalg.norm(ref), 1e-30)
    assert np.all(err <= 2e-2 * np.maximum(1.0, np.abs(ref)))


@pytest.mark.parametrize("m,n,k,dt", [(1, 3072, 2048, "bf16"), (4, 1000, 520, "bf16"),
                                      (8, 256, 4096, "f16"), (1, 2048, 8192, "bf16")])
def test_noalloc_gemv_matches_compiled_plan(m, n, k, dt):
    dev = "cuda:0"
    lib = _lib.load()
    x = synth.normal((m, k), 1.0, dt, 101, dev)
    w = synth.normal((k, n), 0.02, dt, 102, dev)
    ref = torch.zeros((m, n), dtype=x.dtype, device=dev)
    g = Graph()
    ix, iw, io = g.tensor(x), g.tensor(w), g.tensor(ref)
    g.matmul(ix, iw, io)
    plan = g.compile()
    plan.run()
    plan.check_status()
    code = _lib.MK_BF16 if dt == "bf16" else _lib.MK_F16
    for call in range(2):
        out = torch.full((m, n), 3.0, dtype=x.dtype, device=dev)
        st = _lib.DeviceStatus()
        rc = lib.mk_gemv_noalloc(C.c_void_p(x.data_ptr()), C.c_void_p(w.data_ptr()),
                                 C.c_void_p(out.data_ptr()), m, n, k, code,
                                 C.c_void_p(torch.cuda.current_stream().cuda_stream),
                                 C.byref(st))
        assert rc == _lib.MK_OK, lib.mk_last_error().decode()
        assert st.code == 0
        _close(out, ref)


def test_noalloc_rejects_sizes_beyond_its_fixed_scratch():
    lib = _lib.load()
    x = torch.zeros((1, 64), dtype=torch.bfloat16, device="cuda:0")
    w = torch.zeros((64, 8), dtype=torch.bfloat16, device="cuda:0")
    o = torch.zeros((1, 8), dtype=torch.bfloat16, device="cuda:0")
    p = [C.c_void_p(t.data_ptr()) for t in (x, w, o)]
    rc = lib.mk_gemv_noalloc(*p, 1, 262144 + 8, 64, _lib.MK_BF16, None, None)
    assert rc == _lib.MK_ERR_UNSUPPORTED and b"maximum" in lib.mk_last_error()
    rc = lib.mk_gemv_noalloc(*p, 9, 8, 64, _lib.MK_BF16, None, None)
    assert rc == _lib.MK_ERR_UNSUPPORTED
