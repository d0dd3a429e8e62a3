"""Seeded synthetic inputs (shared by the GPU path, the tests and the benchmark).

Holds no arithmetic of the method: only draws from torch's generator and quantises to the
storage dtype (round-to-nearest-even, torch's cast). Every tensor has its own seed so inputs do
not depend on creation order across workloads.
"""
import torch

DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32,
          "i32": torch.int32}


def normal(shape, std, dtype, seed, device="cpu", mean=0.0):
    """N(mean, std^2) samples, drawn in fp32 with a fresh generator seeded by `seed`."""
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(int(seed))
    x = torch.randn(tuple(shape), generator=g, device=dev, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    if mean != 0.0:
        x.add_(mean)
    return x.to(DTYPES[dtype] if isinstance(dtype, str) else dtype)


def zeros(shape, dtype, device="cpu"):
    return torch.zeros(tuple(shape), dtype=DTYPES[dtype] if isinstance(dtype, str) else dtype,
                       device=device)


def to_numpy_f32(t):
    """Exact fp32 values of a fp16/bf16/fp32 tensor, as a numpy array (for the oracle)."""
    return t.detach().to(device="cpu", dtype=torch.float32).numpy()
