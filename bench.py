"""Benchmark of the KLA scan on the headline workload (one JSON line).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl kla|reference]

A step is one kla_forward over the headline workload — B=8, H=16, T=4096,
d_k=d_v=64, bf16 inputs/outputs, fp32 state — with inputs resident in HBM.
The inputs (403 MB) exceed the 135 MB L2, so no flush is needed between
steps. Under torchrun every rank runs its own independent batch (weak
scaling; no collective on the data path) and rank 0 reports the whole-job
throughput over the slowest rank's time.

``--impl reference`` times the fp64 CPU oracle (the stand-in reference arm,
on this host's cores) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KLA scan tokens/s (B·H·T/s) at H=16,d=64,T=4096 bf16; % of roofline"
FLOPS_PER_ELEMENT_STEP = 13  # algorithmic count of the printed recursion
WORKLOAD = "headline"
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic_headline.json")
KERNEL_SOURCES = [os.path.join(ROOT, "bayesian_filtering_linear_gb300", "csrc", f)
                  for f in ("kla_scan.cu", "kla_common.cuh", "kla_device.cuh")]


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        h.update(open(f, "rb").read())
    return h.hexdigest()[:16]


def measured_peaks() -> dict:
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        return {}


def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x: float, world: int) -> float:
    """Max of a host float over all ranks (timing only; not on the data path)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"kla_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self) -> dict:
        rows = []
        try:
            for line in open(self.path):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9 and parts[1].isdigit():
                    rows.append(parts)
        except OSError:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        busy = [r for r in rows if float(r[3] or 0) > 300.0] or rows
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({n for r in busy for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(float(r[1]) for r in busy), "sm_max_mhz": float(busy[0][2]),
                "reasons": reasons, "samples": len(busy)}


def cpu_oracle_sample(heads: int, tokens: int, nthreads: int) -> tuple[float, dict]:
    """Time the fp64 oracle, as it stands, on `heads` heads × `tokens` tokens of
    the headline recipe. Returns (tokens/s, description)."""
    import oracle
    from bayesian_filtering_linear_gb300.inputs import WORKLOADS, make_inputs
    w = WORKLOADS[WORKLOAD]
    x = make_inputs(1, heads, tokens, w.dk, w.dv, io=w.io, seed=w.seed)
    oracle.build()
    t0 = time.perf_counter()
    oracle.forward(x["q"], x["k"], x["v"], x["lam_v"], x["a"], x["pbar"], x["lam0"], x["eta0"],
                   nthreads=nthreads, want_scales=False)
    dt = time.perf_counter() - t0
    used = min(nthreads, heads)
    return heads * tokens / dt, {"kind": "oracle", "cores": used,
                                 "sample": f"{heads} heads x {tokens} tokens of the headline recipe "
                                           f"(d_k=d_v=64, bf16-rounded inputs), fp64 C++ loop, {used} threads"}


def run_reference(args, world, rank):
    """Reference arm: the CPU oracle on bounded samples, timed per step."""
    if rank != 0:
        return
    heads, tokens = 16, 256
    nthreads = min(os.cpu_count() or 1, heads)
    import oracle
    from bayesian_filtering_linear_gb300.inputs import WORKLOADS, make_inputs
    w = WORKLOADS[WORKLOAD]
    x = make_inputs(1, heads, tokens, w.dk, w.dv, io=w.io, seed=w.seed)
    oracle.build()
    run = lambda: oracle.forward(x["q"], x["k"], x["v"], x["lam_v"], x["a"], x["pbar"], x["lam0"], x["eta0"],
                                 nthreads=nthreads, want_scales=False)
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    dt = time.perf_counter() - t0
    value = heads * tokens * args.steps / dt
    sample = f"each step: {heads} heads x {tokens} tokens of the headline recipe, fp64 C++ oracle"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "headline B8 H16 T4096 dk64 dv64 bf16 I/O (sampled)", "B": 8, "H": 16, "T": 4096,
                   "dk": 64, "dv": 64, "io": "bf16"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": nthreads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def run_kla(args, world, rank, local):
    import torch
    from bayesian_filtering_linear_gb300 import kla
    from bayesian_filtering_linear_gb300.inputs import WORKLOADS, make_workload
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = WORKLOADS[WORKLOAD]
    x = make_workload(w, device=dev)
    x = {n: t for n, t in x.items()}
    if rank:  # independent batch per rank
        from bayesian_filtering_linear_gb300.inputs import make_inputs
        x = make_inputs(w.B, w.H, w.T, w.dk, w.dv, io=w.io, seed=w.seed + 1000 * rank, device=dev)
    plan = kla.plan(w.B, w.H, w.T, w.dk, w.dv, w.io)
    ws = torch.empty(plan["workspace_bytes"], dtype=torch.uint8, device=dev) if plan["workspace_bytes"] else None
    y = torch.empty((w.B, w.H, w.T, w.dv), dtype=x["q"].dtype, device=dev)
    lamT = torch.empty_like(x["lam0"])
    etaT = torch.empty_like(x["eta0"])
    stream = torch.cuda.current_stream(dev)

    def step():
        kla.forward(x["q"], x["k"], x["v"], x["lam_v"], x["a"], x["pbar"], x["lam0"], x["eta0"],
                    y=y, lamT=lamT, etaT=etaT, workspace=ws, stream=stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with ClockSampler(local) as clocks:
        barrier(world)
        torch.cuda.synchronize()
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for i in range(args.steps):
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
        end.record(stream)
        torch.cuda.synchronize()
        barrier(world)
    total_ms = start.elapsed_time(end)
    per_launch_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    total_ms = max_over_ranks(total_ms, world)
    ms_per_step = total_ms / args.steps
    tokens = w.B * w.H * w.T
    value = tokens * world / (ms_per_step * 1e-3)

    # ---- end to end through host buffers: H2D of the inputs, the call, D2H of
    # the outputs, every step, inside the timed region ------------------------
    names = ("q", "k", "v", "lam_v", "a", "pbar", "lam0", "eta0")
    host = {n: x[n].cpu().pin_memory() for n in names}
    devb = {n: torch.empty_like(x[n]) for n in names}
    y_h = torch.empty(y.shape, dtype=y.dtype).pin_memory()
    l_h = torch.empty(lamT.shape, dtype=lamT.dtype).pin_memory()
    e_h = torch.empty(etaT.shape, dtype=etaT.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = sum(t.numel() * t.element_size() for t in (y_h, l_h, e_h))
    e2e_steps = max(5, min(args.steps, 50))

    def e2e_step():
        for n in names:
            devb[n].copy_(host[n], non_blocking=True)
        kla.forward(devb["q"], devb["k"], devb["v"], devb["lam_v"], devb["a"], devb["pbar"], devb["lam0"],
                    devb["eta0"], y=y, lamT=lamT, etaT=etaT, workspace=ws, stream=stream)
        y_h.copy_(y, non_blocking=True)
        l_h.copy_(lamT, non_blocking=True)
        e_h.copy_(etaT, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    barrier(world)
    s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s2.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e2.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(s2.elapsed_time(e2) / e2e_steps, world)
    barrier(world)
    if rank != 0:
        return

    peaks = measured_peaks()
    sm_mhz = float(peaks.get("sm_max_mhz", 2070.0))
    nsm = torch.cuda.get_device_properties(dev).multi_processor_count
    peak_tflops = nsm * 128 * 2 * sm_mhz * 1e6 / 1e12
    flops = FLOPS_PER_ELEMENT_STEP * tokens * w.dk * w.dv
    achieved = flops / (per_launch_ms * 1e-3) / 1e12
    traffic = None
    try:
        rec = json.load(open(TRAFFIC_FILE))
        if rec.get("source_hash") == kernel_source_hash() and rec.get("plan") == plan:
            traffic = rec["dram_bytes_per_launch"]
    except (OSError, ValueError, KeyError):
        pass
    cpu_value, cpu_desc = cpu_oracle_sample(32, 4096, os.cpu_count() or 1)
    launches_per_step = 1 if plan["strategy"] == "sequential" else 3
    print(json.dumps({
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": "headline B8 H16 T4096 dk64 dv64 bf16 I/O, fp32 state", "B": w.B, "H": w.H,
                   "T": w.T, "dk": w.dk, "dv": w.dv, "io": w.io, "strategy": plan["strategy"],
                   "chunk_len": plan["chunk_len"], "cols_per_block": plan["cols_per_block"],
                   "rows_per_lane": plan["rows_per_lane"],
                   "l2": "inputs (403 MB) larger than L2; no flush", "parallelism": f"{world} independent batches"},
        "roofline": {"bound": "alu", "achieved": achieved, "peak": peak_tflops, "unit": "TFLOP/s",
                     "frac": achieved / peak_tflops, "traffic": traffic,
                     "kernel": "kla_scan_kernel", "kernel_ms": per_launch_ms,
                     "peak_basis": f"{nsm} SMs x 128 fp32 lanes x 2 flop x {sm_mhz:.0f} MHz (max SM clock)",
                     "flops_per_launch": flops},
        "cpu_baseline": {"value": cpu_value, "unit": "tokens/s", **cpu_desc},
        "e2e": {"value": tokens * world / (e2e_ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks.summary(),
    }), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("kla", "reference"), default="kla")
    args = ap.parse_args(argv)
    world, rank, local = dist_info()
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "kla" else "gloo"
        if backend == "nccl":
            import torch
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    try:
        if args.impl == "reference":
            run_reference(args, world, rank)
        else:
            run_kla(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
