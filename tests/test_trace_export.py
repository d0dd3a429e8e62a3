"""The Chrome trace export of per-instruction timestamps (host only, synthetic stamps)."""
import json

import numpy as np
import pytest

from tensor_core_gemm_gb300.api import INSTR_DTYPE
from tensor_core_gemm_gb300.trace import chrome_events, write_chrome_trace


def _run(n=5):
    ins = np.zeros(n, dtype=INSTR_DTYPE)
    ins["op"] = [1, 1, 0, 2, 8][:n]
    ins["node"] = [0, 0, 0, 1, 2][:n]
    ins["n0"] = [0, 256, 0, 512, 3][:n]
    tr = np.zeros((n, 8), dtype=np.uint64)
    base = 1_000_000
    # desc, ready, seen, end, pub, sm, acc, 0  (ns)
    rows = [(0, 500, 600, 4000, 4500, 0, 3000),
            (100, 700, 800, 5000, 5200, 1, 4200),
            (0, 0, 0, 0, 0, 2, 0),                 # a no-op
            (4600, 6000, 6100, 9000, 9900, 0, 8000),
            (5300, 5250, 5400, 7000, 7100, 1, 0)]  # ready stamped before the descriptor
    for i, r in enumerate(rows[:n]):
        if ins["op"][i] == 0:
            continue
        tr[i, :7] = [x if j == 5 or (j == 6 and x == 0) else base + x for j, x in enumerate(r)]
    return tr, ins


def test_events_per_instruction_and_track():
    tr, ins = _run()
    ev = chrome_events(tr, ins, node_names=["qkv", "o", "attn"])
    names = [e["args"]["name"] for e in ev if e["ph"] == "M"]
    assert names == ["SM 0", "SM 1"]
    x = [e for e in ev if e["ph"] == "X"]
    # the no-op is skipped; 4 instructions x 3 slices, less the empty wait of instruction 4
    assert len(x) == 11
    first = [e for e in x if e["args"]["instr"] == 0]
    assert [e["name"] for e in first] == ["wait", "gemm", "publish"]
    assert first[0]["ts"] == 0.0 and first[0]["dur"] == 0.5
    assert first[1]["ts"] == 0.6 and first[1]["dur"] == pytest.approx(3.4)
    assert first[2]["dur"] == 0.5 and first[1]["args"]["accumulated_us"] == 3.0
    assert first[1]["args"]["node_name"] == "qkv"
    gemv = [e for e in x if e["args"]["instr"] == 3]
    assert gemv[1]["name"] == "gemv" and gemv[1]["tid"] == 0 and gemv[1]["args"]["n0"] == 512
    late = [e for e in x if e["args"]["instr"] == 4]
    assert [e["name"] for e in late] == ["attn_prefill", "publish"]
    assert all(e["dur"] >= 0 for e in x)


def test_written_file_is_json(tmp_path):
    tr, ins = _run()
    path = tmp_path / "t.json"
    n = write_chrome_trace(str(path), tr, ins)
    doc = json.loads(path.read_text())
    assert len(doc["traceEvents"]) == n == 13


def test_mismatched_lengths_and_empty_runs():
    tr, ins = _run()
    with pytest.raises(ValueError):
        chrome_events(tr[:3], ins)
    assert chrome_events(np.zeros_like(tr), ins) == []
