"""ctypes declarations of libmk.so (include/mk.h). Argument marshalling only."""
import ctypes as C
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmk.so")

MK_OK, MK_ERR_INVALID_ARG, MK_ERR_UNSUPPORTED, MK_ERR_HAZARD, MK_ERR_OOM, MK_ERR_CUDA, \
    MK_ERR_TIMEOUT, MK_ERR_DEVICE_CHECK = range(8)
MK_F16, MK_BF16, MK_F32, MK_I32 = 0, 1, 2, 3
EPI_BIAS, EPI_RELU, EPI_RESIDUAL, EPI_RMSNORM_INPUT, EPI_SILU_MUL = 1, 2, 4, 8, 16
EW_ADD, EW_RELU, EW_COPY, EW_SILU_MUL, EW_RMSNORM, EW_ROPE, EW_ARGMAX = 0, 1, 2, 3, 16, 17, 18

EXPORTS = [
    "mk_graph_create", "mk_graph_destroy", "mk_add_tensor", "mk_add_view", "mk_add_matmul",
    "mk_add_elementwise", "mk_add_attention", "mk_default_opts", "mk_compile", "mk_run",
    "mk_run_host", "mk_sync_status", "mk_plan_destroy", "mk_plan_stats", "mk_get_instructions",
    "mk_get_src_list", "mk_get_dst_list", "mk_get_counter_targets", "mk_get_counters",
    "mk_last_error", "mk_abi_version", "mk_gemv_noalloc", "mk_get_trace", "mk_plan_repack",
    "mk_add_transient", "mk_plan_tensor_ptr",
]


class Epilogue(C.Structure):
    _fields_ = [("flags", C.c_uint32), ("bias", C.c_int32), ("residual", C.c_int32),
                ("gamma", C.c_int32), ("b_up", C.c_int32), ("eps", C.c_float)]


class EwParams(C.Structure):
    _fields_ = [("eps", C.c_float), ("gamma", C.c_int32), ("n_q_heads", C.c_int32),
                ("n_kv_heads", C.c_int32), ("head_dim", C.c_int32), ("pos0", C.c_int32),
                ("theta", C.c_float), ("out_k", C.c_int32), ("out_v", C.c_int32)]


class AttnParams(C.Structure):
    _fields_ = [("n_q_heads", C.c_int32), ("n_kv_heads", C.c_int32), ("head_dim", C.c_int32),
                ("causal", C.c_int32), ("q_pos0", C.c_int32), ("scale", C.c_float)]


class CompileOpts(C.Structure):
    _fields_ = [(n, C.c_int32) for n in (
        "n_sm", "gemm_tile_m", "gemm_tile_n", "cluster", "ew_rows", "ew_cols", "ew_tiles",
        "norm_rows", "gemv_max_m", "gemv_tile_n", "gemv_splits", "gemv_kstep", "attn_chunk",
        "attn_tile_q", "dry_run", "timeout_ms", "device", "debug_counter", "debug_extra",
        "snapshot_counters", "trace", "gemm_split_tail", "fuse_rope",
        "fuse_attn_reduce", "kernel_set", "gemv_pack", "argmax_chunk", "gemm_group_m",
        "wave_pack", "row_stage", "pool_waves")]


class HostCopy(C.Structure):
    _fields_ = [("tensor", C.c_int32), ("host", C.c_void_p), ("to_device", C.c_int32)]


class DeviceStatus(C.Structure):
    _fields_ = [(n, C.c_int32) for n in (
        "code", "instr", "counter", "observed", "expected", "sm", "role", "where")]


class Stats(C.Structure):
    _fields_ = [("n_instr", C.c_int64), ("n_counters", C.c_int64), ("n_sems", C.c_int64),
                ("n_sm", C.c_int64), ("n_iter", C.c_int64), ("waves", C.c_double),
                ("n_src", C.c_int64), ("n_dst", C.c_int64), ("per_op", C.c_int64 * 16),
                ("smem_bytes", C.c_int64), ("scratch_bytes", C.c_int64),
                ("kernel_set", C.c_int64), ("packed_bytes", C.c_int64),
                ("pool_bytes", C.c_int64), ("n_reuse", C.c_int64)]


_lib = None


def load():
    """Load libmk.so from the package directory; raise if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libmk.so is not built ({LIB_PATH}); run "
                           "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = C.CDLL(LIB_PATH)
    P, I32, I64, VP = C.c_void_p, C.c_int32, C.c_int64, C.c_void_p
    PI32 = C.POINTER(C.c_int32)
    sig = {
        "mk_graph_create": [C.POINTER(P)],
        "mk_graph_destroy": [P],
        "mk_add_tensor": [P, VP, I32, I32, C.POINTER(I64), C.POINTER(I64), PI32],
        "mk_add_view": [P, I32, I64, I64, I64, I64, PI32],
        "mk_add_transient": [P, I32, I64, I64, PI32],
        "mk_plan_tensor_ptr": [P, I32, C.POINTER(VP)],
        "mk_add_matmul": [P, I32, I32, I32, C.POINTER(Epilogue), PI32],
        "mk_add_elementwise": [P, I32, PI32, I32, I32, C.POINTER(EwParams), PI32],
        "mk_add_attention": [P, I32, I32, I32, I32, C.POINTER(AttnParams), PI32],
        "mk_default_opts": [C.POINTER(CompileOpts)],
        "mk_compile": [P, C.POINTER(CompileOpts), C.POINTER(P)],
        "mk_run": [P, VP],
        "mk_run_host": [P, C.POINTER(HostCopy), I32, VP],
        "mk_sync_status": [P, C.POINTER(DeviceStatus)],
        "mk_plan_repack": [P, VP],
        "mk_plan_destroy": [P],
        "mk_plan_stats": [P, C.POINTER(Stats)],
        "mk_get_instructions": [P, VP, C.c_size_t],
        "mk_get_src_list": [P, PI32, C.c_size_t],
        "mk_get_dst_list": [P, PI32, C.c_size_t],
        "mk_get_counter_targets": [P, PI32, C.c_size_t],
        "mk_get_counters": [P, PI32, C.c_size_t],
        "mk_get_trace": [P, C.POINTER(C.c_uint64), C.c_size_t],
        "mk_gemv_noalloc": [VP, VP, VP, I32, I32, I32, I32, VP, C.POINTER(DeviceStatus)],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = C.c_int32
    lib.mk_last_error.argtypes = []
    lib.mk_last_error.restype = C.c_char_p
    lib.mk_abi_version.argtypes = []
    lib.mk_abi_version.restype = C.c_int32
    _lib = lib
    return lib


class MkError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"mk error {code}: {msg}")
        self.code = code


def check(code):
    if code != MK_OK:
        raise MkError(code, load().mk_last_error().decode(errors="replace"))
    return code
