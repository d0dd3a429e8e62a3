"""Host logic of bench.py on CPU: the replica path's aggregation over ranks (world size 2 over
gloo), the reference arm's rank-0-only line, and the profiled-traffic lookup."""
import json
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_worker(rank, world, port, out_dir):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # each replica timed a different mean step; the job is as slow as the slowest one
    ms = bench.max_over_ranks(1.5 + rank, world, "cpu")
    dist.barrier()
    res = {"ms": ms, "tflops": bench.job_value(10.0 / ms, "TFLOP/s", world),
           "latency": bench.job_value(ms * 1e3, "us/token", world)}
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump(res, f)
    dist.destroy_process_group()


def test_replicas_aggregate_over_two_gloo_ranks(tmp_path):
    import torch.multiprocessing as mp
    world = 2
    mp.spawn(_rank_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    got = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for g in got:
        assert g["ms"] == 2.5                      # max over ranks
        assert g["tflops"] == pytest.approx(2 * 10.0 / 2.5)   # units of both ranks / max time
        assert g["latency"] == 2500.0              # a latency is not summed


def test_single_rank_aggregation_is_identity():
    assert bench.max_over_ranks(3.25, 1, "cpu") == 3.25
    assert bench.job_value(7.0, "TFLOP/s", 1) == 7.0
    assert bench.job_value(7.0, "us/token", 4) == 7.0


class _Args:
    config = "gemm4096"
    steps = 2
    warmup = 3


def test_reference_arm_prints_on_rank_zero_only(monkeypatch, capsys):
    calls = []

    def fake_sample(name, seconds_budget=15.0):
        calls.append(name)
        return 0.5 + 0.1 * len(calls), "fake sample"

    monkeypatch.setattr(bench, "oracle_sample", fake_sample)
    bench.run_reference(_Args(), 2, 1)
    assert capsys.readouterr().out == "" and calls == []
    bench.run_reference(_Args(), 2, 0)
    line = json.loads(capsys.readouterr().out.strip())
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert len(calls) == 5                          # warm-up steps are run but not timed
    assert line["value"] == pytest.approx((0.9 + 1.0) / 2)
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"],
                           "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_profiled_traffic_follows_the_kernel_source(tmp_path, monkeypatch):
    # a summary captured on the current kernel source gives its traffic; one captured on other
    # source, or none at all, gives no traffic (the bench line then reports null)
    prof = tmp_path / "profiles"
    prof.mkdir()
    sha = bench.kernel_source_sha()
    (prof / "megakernel_decode.md").write_text(
        f"kernel_source_sha: {sha}\n\ndram_bytes_per_launch: 1996604568\n")
    (prof / "megakernel_gemm4096.md").write_text(
        "kernel_source_sha: 0000000000000000\n\ndram_bytes_per_launch: 123\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_sha", lambda: sha)
    assert bench.profiled_traffic("decode") == 1996604568
    assert bench.profiled_traffic("gemm4096") is None
    assert bench.profiled_traffic("prefill") is None
