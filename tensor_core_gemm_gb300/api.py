"""Python face of the C ABI: Graph (build) and Plan (compile once, run many times).

Marshalling only: every step of the hot path runs inside libmk.so and its kernel. Tensors are
registered by device pointer (torch tensors are accepted for convenience; the caller keeps
them alive for the plan's lifetime).
"""
import ctypes as C

import numpy as np

from . import _lib
from ._lib import check

INSTR_DTYPE = np.dtype([
    ("op", "<u2"), ("flags", "<u2"), ("node", "<i4"), ("m0", "<i4"), ("n0", "<i4"),
    ("k0", "<i4"), ("klen", "<i4"), ("aux0", "<i4"), ("aux1", "<i4"), ("sem", "<i4"),
    ("n_src", "<i4"), ("src_off", "<i4"), ("n_dst", "<i4"), ("dst_off", "<i4"),
    ("slot", "<i4"), ("split", "<i4"), ("pad", "<i4"),
])
assert INSTR_DTYPE.itemsize == 64

_DT = {"f16": _lib.MK_F16, "bf16": _lib.MK_BF16, "f32": _lib.MK_F32, "i32": _lib.MK_I32}


def _torch_dtype_code(t):
    import torch
    return {torch.float16: _lib.MK_F16, torch.bfloat16: _lib.MK_BF16,
            torch.float32: _lib.MK_F32, torch.int32: _lib.MK_I32}[t.dtype]


def _stream_handle(stream):
    if stream is None:
        return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


class Graph:
    def __init__(self):
        self._lib = _lib.load()
        self._h = C.c_void_p()
        check(self._lib.mk_graph_create(C.byref(self._h)))
        self._keep = []

    def __del__(self):
        if getattr(self, "_h", None) and self._h.value:
            self._lib.mk_graph_destroy(self._h)
            self._h = C.c_void_p()

    def tensor(self, t=None, *, ptr=0, dtype=None, shape=None, strides=None):
        """Register a torch tensor, or raw (ptr, dtype 'f16'|'bf16'|'f32'|'i32', shape,
        strides)."""
        if t is not None:
            ptr = t.data_ptr()
            dtype = _torch_dtype_code(t)
            shape = list(t.shape)
            strides = list(t.stride())
            self._keep.append(t)
        else:
            dtype = _DT[dtype] if isinstance(dtype, str) else dtype
        rank = len(shape)
        sh = (C.c_int64 * rank)(*shape)
        st = (C.c_int64 * rank)(*strides) if strides is not None else None
        tid = C.c_int32()
        check(self._lib.mk_add_tensor(self._h, C.c_void_p(ptr or None), dtype, rank, sh, st,
                                      C.byref(tid)))
        return tid.value

    def transient(self, dtype, rows, cols):
        """A plan-owned rows x cols intermediate ('f16'|'bf16'|'f32'|'i32'): one node writes
        it, later nodes read it, and mk_compile places it in the plan's buffer pool."""
        dtype = _DT[dtype] if isinstance(dtype, str) else dtype
        tid = C.c_int32()
        check(self._lib.mk_add_transient(self._h, dtype, rows, cols, C.byref(tid)))
        return tid.value

    def view(self, base, r0, c0, rows, cols):
        vid = C.c_int32()
        check(self._lib.mk_add_view(self._h, base, r0, c0, rows, cols, C.byref(vid)))
        return vid.value

    def matmul(self, a, b, out, *, bias=None, relu=False, residual=None, gamma=None, eps=1e-5,
               b_up=None):
        e = _lib.Epilogue(0, -1, -1, -1, -1, float(eps))
        if bias is not None:
            e.flags |= _lib.EPI_BIAS
            e.bias = bias
        if relu:
            e.flags |= _lib.EPI_RELU
        if residual is not None:
            e.flags |= _lib.EPI_RESIDUAL
            e.residual = residual
        if gamma is not None:
            e.flags |= _lib.EPI_RMSNORM_INPUT
            e.gamma = gamma
        if b_up is not None:
            e.flags |= _lib.EPI_SILU_MUL
            e.b_up = b_up
        nid = C.c_int32()
        check(self._lib.mk_add_matmul(self._h, a, b, out, C.byref(e), C.byref(nid)))
        return nid.value

    def _ew(self, op, ins, out, params=None):
        arr = (C.c_int32 * len(ins))(*ins)
        nid = C.c_int32()
        check(self._lib.mk_add_elementwise(self._h, op, arr, len(ins), out,
                                           C.byref(params) if params is not None else None,
                                           C.byref(nid)))
        return nid.value

    def elementwise(self, op, ins, out):
        code = {"add": _lib.EW_ADD, "relu": _lib.EW_RELU, "copy": _lib.EW_COPY,
                "silu_mul": _lib.EW_SILU_MUL}[op]
        return self._ew(code, list(ins), out)

    def rmsnorm(self, x, gamma, out, eps=1e-5):
        p = _lib.EwParams(float(eps), gamma, 0, 0, 0, 0, 0.0, -1, -1)
        return self._ew(_lib.EW_RMSNORM, [x], out, p)

    def rope(self, x, out_q, out_k, *, out_v=None, n_q_heads, n_kv_heads, head_dim, pos0=0,
             theta=5e5):
        p = _lib.EwParams(0.0, -1, n_q_heads, n_kv_heads, head_dim, pos0, float(theta), out_k,
                          -1 if out_v is None else out_v)
        return self._ew(_lib.EW_ROPE, [x], out_q, p)

    def argmax(self, x, out):
        """out [R x 1] int32 = per row of x the first column holding its largest value."""
        return self._ew(_lib.EW_ARGMAX, [x], out)

    def attention(self, q, k, v, out, *, n_q_heads, n_kv_heads, head_dim, causal=False,
                  q_pos0=0, scale=0.0):
        p = _lib.AttnParams(n_q_heads, n_kv_heads, head_dim, int(causal), q_pos0, float(scale))
        nid = C.c_int32()
        check(self._lib.mk_add_attention(self._h, q, k, v, out, C.byref(p), C.byref(nid)))
        return nid.value

    def compile(self, **opts):
        o = _lib.CompileOpts()
        check(self._lib.mk_default_opts(C.byref(o)))
        for k, v in opts.items():
            if not hasattr(o, k):
                raise TypeError(f"unknown compile option {k}")
            setattr(o, k, int(v))
        h = C.c_void_p()
        check(self._lib.mk_compile(self._h, C.byref(o), C.byref(h)))
        return Plan(self._lib, h, list(self._keep))


class Plan:
    def __init__(self, lib, handle, keep):
        self._lib = lib
        self._h = handle
        self._keep = keep

    def __del__(self):
        if getattr(self, "_h", None) and self._h.value:
            self._lib.mk_plan_destroy(self._h)
            self._h = C.c_void_p()

    def run(self, stream=None):
        """Enqueue one run (counter reset + one persistent launch) on `stream`."""
        check(self._lib.mk_run(self._h, _stream_handle(stream)))

    def repack(self, stream=None):
        """Refresh the plan's packed copies of GEMV weights after changing such a weight in
        device memory (runs mk_plan_repack on `stream`)."""
        check(self._lib.mk_plan_repack(self._h, _stream_handle(stream)))

    def run_host(self, inputs=(), outputs=(), stream=None):
        """inputs/outputs: lists of (tensor_id, host pointer); host->device copies, the run and
        device->host copies are all enqueued on `stream`."""
        copies = [(t, p, 1) for t, p in inputs] + [(t, p, 0) for t, p in outputs]
        arr = (_lib.HostCopy * max(1, len(copies)))()
        for i, (t, p, d) in enumerate(copies):
            arr[i] = _lib.HostCopy(t, p, d)
        check(self._lib.mk_run_host(self._h, arr, len(copies), _stream_handle(stream)))

    def sync_status(self):
        st = _lib.DeviceStatus()
        code = self._lib.mk_sync_status(self._h, C.byref(st))
        return code, {f: getattr(st, f) for f, _ in _lib.DeviceStatus._fields_}

    def check_status(self):
        code, st = self.sync_status()
        if code != _lib.MK_OK:
            raise _lib.MkError(code, self._lib.mk_last_error().decode(errors="replace"))
        return st

    def tensor_ptr(self, tensor):
        """Device address of a tensor in this plan (a transient's place in the buffer pool)."""
        p = C.c_void_p()
        check(self._lib.mk_plan_tensor_ptr(self._h, tensor, C.byref(p)))
        return p.value or 0

    def stats(self):
        s = _lib.Stats()
        check(self._lib.mk_plan_stats(self._h, C.byref(s)))
        d = {f: getattr(s, f) for f, _ in _lib.Stats._fields_ if f != "per_op"}
        d["per_op"] = list(s.per_op)
        return d

    def instructions(self):
        n = self.stats()["n_instr"]
        buf = np.zeros(n, dtype=INSTR_DTYPE)
        check(self._lib.mk_get_instructions(self._h, buf.ctypes.data_as(C.c_void_p), buf.nbytes))
        return buf

    def _ints(self, fn, n):
        buf = np.zeros(max(1, n), dtype=np.int32)
        check(fn(self._h, buf.ctypes.data_as(C.POINTER(C.c_int32)), n))
        return buf[:n]

    def src_list(self):
        return self._ints(self._lib.mk_get_src_list, 2 * self.stats()["n_src"]).reshape(-1, 2)

    def dst_list(self):
        return self._ints(self._lib.mk_get_dst_list, self.stats()["n_dst"])

    def counter_targets(self):
        return self._ints(self._lib.mk_get_counter_targets, self.stats()["n_counters"])

    def trace(self):
        """Per-instruction [t_descriptor, t_sources_ready (scheduler), t_sources_seen (compute),
        t_body_end, t_published, sm, t_accumulated (GEMM / GEMV), 0] (ns) of the last run."""
        n = self.stats()["n_instr"]
        buf = np.zeros(max(1, 8 * n), dtype=np.uint64)
        check(self._lib.mk_get_trace(self._h, buf.ctypes.data_as(C.POINTER(C.c_uint64)), 8 * n))
        return buf[:8 * n].reshape(-1, 8)

    def export_trace(self, path, node_names=None):
        """Write the last run's per-instruction timeline (plan compiled with trace=1) as a
        Chrome trace-event JSON file, one track per SM (see trace.py); returns the event count."""
        from .trace import write_chrome_trace
        return write_chrome_trace(path, self.trace(), self.instructions(), node_names)

    def counters(self):
        s = self.stats()
        return self._ints(self._lib.mk_get_counters, s["n_counters"] + s["n_sems"])
