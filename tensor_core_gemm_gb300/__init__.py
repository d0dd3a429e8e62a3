"""GB300-native persistent megakernel: a static op graph compiled into tile instructions and run
as one sm_103a kernel launch (C ABI in include/mk.h, library libmk.so built in-tree).

Importing the package does not load the library; ``Graph`` loads it on first use and raises
if it has not been built.
"""
from .api import INSTR_DTYPE, Graph, Plan  # noqa: F401

OPS = {0: "noop", 1: "gemm", 2: "gemv", 3: "ew", 4: "rmsnorm", 5: "rope", 6: "attn_partial",
       7: "attn_reduce", 8: "attn_prefill", 9: "argmax", 10: "argmax_reduce"}
