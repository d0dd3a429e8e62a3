"""Benchmark of the persistent megakernel (one JSON line on rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl mk|reference] [--config NAME]
                    [--only]

Default workload: the single fp16 GEMM C = A @ B, M = N = K = 4096 (A, B ~N(0, 1/64)), one
megakernel launch per step; its figures are the line's top-level keys. The default run then
measures the rest of the suite the same way in the same process (batch-1 decode of the
16-layer decoder in us/token and HBM GB/s, its 2048-token causal prefill, the Llama-70B prefill
and decode linear lists, the 3-layer MLP) and nests each record under "configs". Other
workloads alone (--config, or --only for the GEMM alone): mlp3, llama_prefill, llama_decode,
decode, prefill, and decode_sample (decode followed by greedy sampling over a 128256-token
vocabulary).

Timing: W untimed warm-up runs, then K runs, each bracketed by CUDA events on the launch stream
with a 256 MB L2 flush (a device write larger than the 129 MB L2) before each run, outside the
events; barrier + synchronize on both sides of the timed region; max over ranks. `e2e` times
the same workload through mk_run_host: pinned host inputs copied in, the run, the output copied
back, every step. With N > 1 every rank runs an independent replica (the path does not shard):
value = the units all ranks processed / the slowest rank's time.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

CORES = len(os.sched_getaffinity(0))
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, str(CORES))

import numpy as np  # noqa: E402

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


# ------------------------------------------------------------------ workloads

CONFIGS = {
    "gemm4096": "single fp16 GEMM C=A@B, M=N=K=4096, A,B ~N(0,1/64), fp32 accumulate, fp16 out",
    "mlp3": "3-layer MLP x=relu(x@W[i]+b[i]), x fp16 1024x1024, W 3x1024x1024, b 3x1024x1024",
    "llama_prefill": "Llama-3-70B prefill linears M=8192 (N,K)=(8192,8192),(28672,8192) fp16",
    "llama_decode": "Llama-3-70B decode linears M=256 (N,K)=(10240,8192),(8192,8192),"
                    "(28672,8192),(8192,28672) fp16",
    "decode": "batch-1 decode, 16-layer decoder hidden 2048, 32/8 heads x 64, MLP 8192, "
              "KV 1024, bf16",
    "prefill": "causal prefill 2048 tokens, 16-layer decoder hidden 2048, bf16",
    "decode_sample": "batch-1 decode as 'decode', then final RMSNorm + lm_head GEMV over a "
                     "synthetic 128256-token vocabulary + greedy ARGMAX, bf16 (int32 token)",
}


def make_workload(name, device):
    from tensor_core_gemm_gb300 import workloads as W
    pair = {"gemm_tile_m": 256, "cluster": 2}   # 256 x 256 tiles on CTA pairs
    if name == "gemm4096":
        # 256 pair tiles on 76 pairs: the quarter-full last wave's tiles split along K
        return (W.gemm(4096, 4096, 4096, dtype="f16", device=device, seed=0),
                dict(pair, gemm_split_tail=1))
    if name == "mlp3":
        return W.mlp3(device=device, seed=0), {"gemm_tile_n": 64}
    if name == "llama_prefill":
        return W.gemm_list(W.LLAMA70B_PREFILL, device=device, seed=0), dict(pair)
    if name == "llama_decode":
        return W.gemm_list(W.LLAMA70B_DECODE, device=device, seed=0), dict(pair)
    if name == "decode":
        return W.decode(device=device, seed=0), {}
    if name == "decode_sample":
        return W.decode(device=device, seed=0, vocab=128256), {}
    if name == "prefill":
        return W.prefill(device=device, seed=0), {}
    raise ValueError(name)


def metric_of(name):
    if name in ("decode", "decode_sample"):
        return "batch-1 decode latency", "us/token", False
    return "megakernel TFLOP/s", "TFLOP/s", True


def binding_roof(wl, peaks):
    """The roof a run of `wl` meets first: the tensor pipe when its FLOPs take longer at the
    measured tensor peak than its compulsory bytes at the measured HBM bandwidth, else HBM
    (the Llama decode linears, M = 256, sit below the ridge point of this chip)."""
    t_tensor = wl.flops / (float(peaks["bf16_tflops"]) * 1e12)
    t_hbm = wl.hbm_bytes / (float(peaks["hbm_gbs"]) * 1e9)
    return "tensor" if t_tensor >= t_hbm else "hbm"


def io_tensors(wl):
    """(inputs, outputs) description-tensor ids copied by the end-to-end path."""
    n = wl.name
    if n == "gemm":
        return [wl.info["a"], wl.info["b"]], [wl.info["c"]]
    if n == "gemm_list":
        ins = [x for g in wl.info["gemms"] for x in g[:2]]
        return ins, [g[2] for g in wl.info["gemms"]]
    if n == "mlp3":
        return [wl.info["x"], wl.info["w"], wl.info["b"]], [wl.info["outputs"][-1]]
    if n == "decode":
        out = wl.info["token"] if wl.info.get("vocab") else wl.info["out"]
        return [wl.info["x"]], [out]
    if n == "prefill":
        return [wl.info["x"]], [wl.info["out"]]
    raise ValueError(n)


def value_of(wl, ms, name):
    if name in ("decode", "decode_sample"):
        return ms * 1e3
    return wl.flops / (ms * 1e-3) / 1e12


KERNEL_SETS = ("general", "gemm", "decode", "prefill")  # specialisation mk_run launches


def kernel_source_sha():
    import hashlib
    h = hashlib.sha256()
    for f in ("mk_megakernel.cuh", "mk_ptx.cuh", "mk_types.h", "mk_kernel.cu",
              "mk_kernel_gemm.cu", "mk_kernel_decode.cu", "mk_kernel_prefill.cu"):
        with open(os.path.join(ROOT, "tensor_core_gemm_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(config):
    """DRAM bytes per launch from the committed ncu summary of this workload, or None when
    there is none or the kernel source changed since it was captured."""
    path = os.path.join(ROOT, "profiles", f"megakernel_{config}.md")
    if not os.path.exists(path):
        return None
    sha, traffic = None, None
    with open(path) as f:
        for line in f:
            if line.startswith("kernel_source_sha:"):
                sha = line.split()[1]
            elif line.startswith("dram_bytes_per_launch:"):
                traffic = int(line.split()[1])
    return traffic if sha == kernel_source_sha() else None


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.th.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ oracle (CPU) timing

def oracle_sample(name, seconds_budget=15.0):
    """Time the oracle on a bounded sample of the workload on this host's cores.
    Returns (value in the workload's unit, description of the sample)."""
    from oracle import models, ops
    from oracle.numerics import BF16, F16
    rng = np.random.default_rng(0)

    def f16(shape, std):
        return (rng.standard_normal(shape, dtype=np.float32) * std).astype(np.float16).astype(
            np.float32)

    if name in ("gemm4096", "llama_prefill", "llama_decode"):
        shapes = {"gemm4096": [(4096, 4096, 4096)],
                  "llama_prefill": [(8192, 8192, 8192), (8192, 28672, 8192)],
                  "llama_decode": [(256, 10240, 8192), (256, 8192, 8192), (256, 28672, 8192),
                                   (256, 8192, 28672)]}[name]
        rows = 64
        flops, t = 0.0, 0.0
        for (m, n, k) in shapes:
            a = f16((rows, k), 1 / 8)
            b = f16((k, n), 1 / 8)
            t0 = time.perf_counter()
            ops.matmul(a, b, F16)
            t += time.perf_counter() - t0
            flops += 2.0 * rows * n * k
        return flops / t / 1e12, f"{rows} rows of each GEMM ({len(shapes)} GEMMs)"
    if name == "mlp3":
        x = f16((1024, 1024), 1.0)
        w = f16((3, 1024, 1024), 1 / 32)
        b = f16((3, 1024, 1024), 0.1)
        t0 = time.perf_counter()
        models.mlp(x, w, b)
        t = time.perf_counter() - t0
        return 2.0 * 3 * 1024 ** 3 / t / 1e12, "the full 3-layer MLP"
    if name in ("decode", "decode_sample"):
        # two layers of the decoder, scaled to 16 (the layers are identical in cost)
        from tensor_core_gemm_gb300 import workloads as W
        sh = W.DecoderShape(layers=2)
        d, f = sh.hidden, sh.ffn
        bf = lambda *s: (rng.standard_normal(s, dtype=np.float32) * 0.02)
        wts = models.DecoderWeights(bf(2, d, sh.qkv), bf(2, d, d), bf(2, d, f), bf(2, d, f),
                                    bf(2, f, d), 1 + bf(2, d), 1 + bf(2, d), sh.hq, sh.hkv,
                                    sh.hd, sh.eps, sh.theta)
        kc = [rng.standard_normal((1025, 512), dtype=np.float32) for _ in range(2)]
        vc = [rng.standard_normal((1025, 512), dtype=np.float32) for _ in range(2)]
        x = rng.standard_normal((1, d), dtype=np.float32)
        t0 = time.perf_counter()
        x, _, _ = models.decode_step(x, wts, kc, vc, 1024)
        t = (time.perf_counter() - t0) * 8
        if name == "decode":
            return t * 1e6, "2 of 16 decoder layers, time x8"
        w_lm = bf(d, 128256)
        t0 = time.perf_counter()
        models.decode_head(x, 1 + bf(d), w_lm, sh.eps)
        t += time.perf_counter() - t0
        return t * 1e6, "2 of 16 decoder layers, time x8, plus the full sampling head"
    if name == "prefill":
        from tensor_core_gemm_gb300 import workloads as W
        sh = W.DecoderShape(layers=1)
        d, f = sh.hidden, sh.ffn
        bf = lambda *s: (rng.standard_normal(s, dtype=np.float32) * 0.02)
        wts = models.DecoderWeights(bf(1, d, sh.qkv), bf(1, d, d), bf(1, d, f), bf(1, d, f),
                                    bf(1, f, d), 1 + bf(1, d), 1 + bf(1, d), sh.hq, sh.hkv,
                                    sh.hd, sh.eps, sh.theta)
        t_ = 256
        x = rng.standard_normal((t_, d), dtype=np.float32)
        t0 = time.perf_counter()
        models.prefill(x, wts)
        t = time.perf_counter() - t0
        fl = 2.0 * t_ * (d * sh.qkv + d * d + 3 * d * f) + 4.0 * sh.hq * sh.hd * t_ * (t_ + 1) / 2
        return fl / t / 1e12, f"1 layer, causal prefix of {t_} tokens"
    raise ValueError(name)


# ------------------------------------------------------------------ main

def max_over_ranks(x, world, device):
    """Largest value of x over the ranks of the process group (x itself on one rank)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.item()


def job_value(per_rank, unit, world):
    """Whole-job value of N replicas timed by the slowest one: throughput adds over the
    replicas; a per-token latency stays the slowest replica's."""
    return per_rank * world if unit == "TFLOP/s" else per_rank


def run_reference(args, world, rank):
    """The oracle, as it stands, timed on this host's cores (the reference arm)."""
    if rank != 0:
        return
    metric, unit, hib = metric_of(args.config)
    vals = []
    sample = ""
    for i in range(args.warmup + args.steps):
        v, sample = oracle_sample(args.config)
        if i >= args.warmup:
            vals.append(v)
    value = statistics.mean(vals)
    ms = (value / 1e3) if unit == "us/token" else None
    line = {
        "impl": "reference", "metric": metric, "value": value, "unit": unit, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": hib, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32 (fp16/bf16-quantised inputs)", "data": "synthetic",
        "config": {"workload": CONFIGS[args.config], "sample": sample},
        "cpu_baseline": {"value": value, "unit": unit, "cores": CORES, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# The default run times the headline workload, then every other workload of the suite, each
# measured the same way in the same process; their records nest under "configs".
SUITE = ("decode", "prefill", "llama_prefill", "llama_decode", "mlp3")


def measure(name, args, world, rank, local, dev, barrier, opt_overrides=()):
    """One workload through the megakernel: W warm-up runs, K timed runs (CUDA events on the
    launch stream, L2 flushed before each), the end-to-end runs through host buffers, clocks
    sampled during the timed region, and (rank 0, one GPU) the oracle on a bounded sample.
    Returns the JSON record (without the run-level keys n_gpus / steps / warmup)."""
    import torch
    from tensor_core_gemm_gb300 import workloads as W

    wl, opts = make_workload(name, dev)
    for kv in opt_overrides:
        k, v = kv.split("=", 1)
        opts[k] = int(v)
    g, id_of = W.build_graph(wl.desc, wl.data)
    plan = g.compile(**opts)
    stream = torch.cuda.current_stream()
    flush = torch.empty(64 * 1024 * 1024, dtype=torch.int32, device=dev)   # 256 MB > L2

    for _ in range(args.warmup):
        plan.run(stream)
    plan.check_status()
    torch.cuda.synchronize()

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.5)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush.fill_(i)
        starts[i].record(stream)
        plan.run(stream)
        ends[i].record(stream)
    torch.cuda.synchronize()
    barrier()
    clock_info = clocks.stop()
    plan.check_status()
    times = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms = max_over_ranks(statistics.mean(times), world, dev)

    # End to end through the C ABI with host buffers (pinned), copies inside the timed region.
    ins, outs = io_tensors(wl)

    def ref_of(t):
        return id_of((t, 0, 0, wl.desc["tensors"][t]["rows"], wl.desc["tensors"][t]["cols"]))

    host_in = [(ref_of(t), wl.data[t].cpu().pin_memory()) for t in ins]
    host_out = [(ref_of(t), torch.empty_like(wl.data[t], device="cpu").pin_memory())
                for t in outs]
    h2d = sum(h.numel() * h.element_size() for _, h in host_in)
    d2h = sum(h.numel() * h.element_size() for _, h in host_out)
    e_in = [(tid, h.data_ptr()) for tid, h in host_in]
    e_out = [(tid, h.data_ptr()) for tid, h in host_out]
    for _ in range(2):
        plan.run_host(e_in, e_out, stream)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    e0.record(stream)
    for _ in range(args.steps):
        plan.run_host(e_in, e_out, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    plan.check_status()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, dev)

    metric, unit, hib = metric_of(name)
    value = job_value(value_of(wl, ms, name), unit, world)
    e2e_value = job_value(value_of(wl, e2e_ms, name), unit, world)
    peaks, peak_src = load_peaks()
    bound = binding_roof(wl, peaks)
    # fp16 and bf16 have the same dense tensor rate
    roofs = {"tensor": (wl.flops / (ms * 1e-3) / 1e12, float(peaks["bf16_tflops"]), "TFLOP/s"),
             "hbm": (wl.hbm_bytes / (ms * 1e-3) / 1e9, float(peaks["hbm_gbs"]), "GB/s")}
    achieved, peak, runit = roofs[bound]
    other = "hbm" if bound == "tensor" else "tensor"
    secondary = {"bound": other, "achieved": roofs[other][0], "peak": roofs[other][1],
                 "unit": roofs[other][2], "frac": roofs[other][0] / roofs[other][1]}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, sample = oracle_sample(name)
        cpu = {"value": v, "unit": unit, "cores": CORES, "kind": "oracle", "sample": sample}

    st = plan.stats()
    dtype = "bf16" if name in ("decode", "prefill", "decode_sample") else "f16"
    rec = {
        "metric": metric, "value": value, "unit": unit, "ms_per_step": ms,
        "higher_is_better": hib, "scaling": "weak", "vs_baseline": None, "dtype": dtype,
        "data": "synthetic",
        "config": {"workload": CONFIGS[name],
                   "l2": "flushed before every timed run (256 MB device write)",
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "instructions": st["n_instr"], "waves_per_sm": round(st["waves"], 3),
                   "kernel_set": KERNEL_SETS[st["kernel_set"]], "compile_opts": opts},
        "roofline": {"bound": bound, "achieved": achieved, "peak": peak, "unit": runit,
                     "frac": achieved / peak, "traffic": profiled_traffic(name),
                     "peak_source": f"{peak_src} "
                                    f"({'bf16_tflops' if bound == 'tensor' else 'hbm_gbs'})",
                     "secondary": secondary},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": unit, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": args.steps,
        "clocks": clock_info,
    }
    if unit == "us/token":   # the decode metric's other half: HBM GB/s of the token
        rec["hbm_gbs"] = roofs["hbm"][0]
    del plan, g, wl, flush, host_in, host_out
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return rec


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="mk", choices=["mk", "reference"])
    ap.add_argument("--config", default="gemm4096", choices=sorted(CONFIGS))
    ap.add_argument("--only", action="store_true",
                    help="time the named workload alone (the default run adds the others)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--opt", action="append", default=[], metavar="KEY=INT",
                    help="override a compile option of the workload, e.g. --opt cluster=2")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, world, rank)
        return

    import torch
    import torch.distributed as dist
    from tensor_core_gemm_gb300 import _lib

    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device(dev))

    def barrier():
        if world > 1:
            dist.barrier()

    _lib.load()
    rec = measure(args.config, args, world, rank, local, dev, barrier, args.opt)
    line = {"metric": rec["metric"], "value": rec["value"], "unit": rec["unit"],
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup}
    line.update({k: v for k, v in rec.items() if k not in line})
    if args.config == "gemm4096" and not args.only and not args.opt:
        line["configs"] = {}
        for name in SUITE:
            try:
                line["configs"][name] = measure(name, args, world, rank, local, dev, barrier)
            except Exception as e:  # a failure of one workload leaves the others' records
                line["configs"][name] = {"error": f"{type(e).__name__}: {e}"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
