"""Storage formats: IEEE fp16 and bfloat16, held as fp32 arrays of exactly representable values.

Every buffer in a graph has a storage dtype (fp16 for the GEMM workloads, bf16 for the decoder
ones). The oracle computes in fp32 and rounds to the storage dtype, round-to-nearest-even, at
each node output ("Hand-writing a Blackwell GEMM", "How I measured": fp16 in, fp32 accumulate,
fp16 out). bf16 is not a numpy dtype, so its values travel as uint16 bit patterns.

Pinned by tests/test_oracle_pins.py: exact values of the bf16/fp16 grids (1 + 2^-8 ties, the
largest finite values, overflow to inf, subnormals) that follow from the IEEE definitions.
"""
import numpy as np

F16 = "f16"
BF16 = "bf16"
F32 = "f32"


def bf16_bits_to_f32(bits):
    """Widen bf16 bit patterns (uint16) to fp32: the bf16 pattern is the top half of the fp32 one."""
    b = np.asarray(bits).astype(np.uint16).astype(np.uint32)
    return (b << np.uint32(16)).view(np.float32)


def f32_to_bf16_bits(x):
    """Round fp32 to bf16 (nearest, ties to even) and return the uint16 bit patterns.

    Dropping the low 16 bits after adding 0x7FFF plus the lowest kept bit is round-half-to-even
    on the magnitude; the carry walks into the exponent exactly as IEEE rounding does, which
    also turns values above the largest finite bf16 into infinity. NaNs map to a quiet NaN.
    """
    x = np.asarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)
    nan = np.isnan(x)
    if np.any(nan):
        r = np.where(nan, np.uint16(0x7FC0), r)
    return r


def round_to(x, dtype):
    """Round an fp32 array to the storage dtype and return it widened back to fp32."""
    x = np.asarray(x, dtype=np.float32)
    if dtype == F32:
        return x.copy()
    if dtype == F16:
        with np.errstate(over="ignore"):
            return x.astype(np.float16).astype(np.float32)
    if dtype == BF16:
        return bf16_bits_to_f32(f32_to_bf16_bits(x))
    raise ValueError(f"unknown dtype {dtype!r}")


def to_f32(arr, dtype):
    """Interpret stored data (numpy float16 array, or uint16/int16 bf16 bits) as fp32 values."""
    arr = np.asarray(arr)
    if dtype == F16:
        return arr.astype(np.float32)
    if dtype == BF16:
        if arr.dtype in (np.uint16, np.int16):
            return bf16_bits_to_f32(arr.view(np.uint16))
        return round_to(arr.astype(np.float32), BF16)
    if dtype == F32:
        return arr.astype(np.float32)
    raise ValueError(f"unknown dtype {dtype!r}")
