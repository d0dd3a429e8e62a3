"""Oracle: a plain, slow, obviously correct CPU restatement of what the megakernel computes.

TEST INFRASTRUCTURE ONLY. Nothing on the product path imports, calls or links this package;
only the tests, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference``
legs of ``bench.py`` use it. It shares no code with ``tensor_core_gemm_gb300`` (neither imports
the other); inputs reach it as numpy arrays produced by the seeded generators.

Modules
-------
numerics   fp16 / bf16 round-to-nearest-even on fp32 arrays (the storage formats of every buffer).
ops        one function per graph operation, each the textbook definition in fp32.
models     the five workloads composed from ``ops`` at the granularity of the graph's nodes.
schedule   the lowering of a graph into tile instructions, dependency counters and the static
           per-SM placement, computed by brute-force box intersection.

Precision: fp32 arithmetic over the fp16/bf16-quantised inputs, rounding (RNE) to the declared
storage dtype at every node output; fp64 is used only by the self-checks in the tests.

Parity status per function is recorded in each function's docstring ("pinned by" / "parity
unpinned").
"""
