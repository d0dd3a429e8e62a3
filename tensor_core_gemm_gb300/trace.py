"""Per-instruction timelines of a run as a Chrome trace-event file (loads in Perfetto or
chrome://tracing).

A plan compiled with ``trace=1`` records, per instruction, globaltimer stamps (ns) of: the
descriptor reaching the compute warpgroup, the scheduler seeing every source counter at its
target, the compute warpgroup seeing that, the accumulator completing (GEMM / GEMV), the body
ending, and the release of the instruction's counters, plus the SM that ran it. Each SM becomes
one track; each instruction gives up to three slices on it:

  wait     descriptor -> sources ready    (the dependency wait: producers on other SMs)
  <op>     sources seen -> body end       (the instruction's own work; args name the node)
  publish  body end -> counters released  (stores drained, release increments)

Host-side only: this module reads the arrays ``Plan.trace()`` and ``Plan.instructions()``
return and writes JSON; it launches nothing.
"""
import json

import numpy as np

OP_NAMES = {0: "noop", 1: "gemm", 2: "gemv", 3: "ew", 4: "rmsnorm", 5: "rope",
            6: "attn_partial", 7: "attn_reduce", 8: "attn_prefill", 9: "argmax",
            10: "argmax_reduce"}

# trace words (kTraceWords = 8 per instruction)
T_DESC, T_READY, T_SEEN, T_END, T_PUB, T_SM, T_ACC = range(7)


def chrome_events(trace, instrs, node_names=None):
    """Trace-event dicts for one run.

    trace: uint64 [n_instr x 8] from Plan.trace(); instrs: the INSTR_DTYPE records from
    Plan.instructions() (fields op, node, m0, n0, k0, klen). Instructions that did not run
    (no-ops, or stamps left at zero) are skipped. Times are in microseconds from the earliest
    stamp of the run."""
    tr = np.asarray(trace, dtype=np.int64).reshape(-1, 8)
    if len(tr) != len(instrs):
        raise ValueError(f"{len(tr)} trace rows for {len(instrs)} instructions")
    ran = (instrs["op"] != 0) & (tr[:, T_DESC] > 0) & (tr[:, T_PUB] > 0)
    if not ran.any():
        return []
    t0 = int(tr[ran][:, [T_DESC, T_READY, T_SEEN]].min())
    us = lambda t: (int(t) - t0) / 1000.0  # noqa: E731
    events = []
    for sm in sorted(set(int(x) for x in tr[ran, T_SM])):
        events.append({"ph": "M", "name": "thread_name", "pid": 0, "tid": sm,
                       "args": {"name": f"SM {sm}"}})
    for i in np.nonzero(ran)[0]:
        r, ins = tr[i], instrs[i]
        op = OP_NAMES.get(int(ins["op"]), str(int(ins["op"])))
        node = int(ins["node"])
        args = {"instr": int(i), "node": node, "m0": int(ins["m0"]), "n0": int(ins["n0"]),
                "k0": int(ins["k0"]), "klen": int(ins["klen"])}
        if node_names is not None and node < len(node_names):
            args["node_name"] = node_names[node]
        if r[T_ACC] > 0:
            args["accumulated_us"] = us(r[T_ACC])
        sm = int(r[T_SM])
        ready = max(int(r[T_READY]), int(r[T_DESC]))
        slices = [("wait", r[T_DESC], ready, "wait"),
                  (op, max(int(r[T_SEEN]), ready), r[T_END], "op"),
                  ("publish", r[T_END], r[T_PUB], "publish")]
        for name, a, b, cat in slices:
            if a <= 0 or b <= a:
                continue
            events.append({"ph": "X", "name": name, "cat": cat, "pid": 0, "tid": sm,
                           "ts": us(a), "dur": (int(b) - int(a)) / 1000.0, "args": args})
    return events


def write_chrome_trace(path, trace, instrs, node_names=None):
    """Write the run's timeline to `path` (JSON object format); returns the event count."""
    ev = chrome_events(trace, instrs, node_names)
    with open(path, "w") as f:
        json.dump({"traceEvents": ev, "displayTimeUnit": "ns"}, f)
    return len(ev)
