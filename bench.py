"""Benchmark of the KLA scan (one JSON line).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl kla|reference]
                    [--workload headline|medium|long|tiny|decode]
                    [--pass forward|backward|conv|conv_backward]

By default a step is one kla_forward over the headline workload — B=8, H=16,
T=4096, d_k=d_v=64, bf16 inputs/outputs, fp32 state — with inputs resident
in HBM. The inputs (403 MB) exceed the 135 MB L2, so no flush is needed
between steps. The other workloads print the same line for their own
configuration: medium (B4 H8 T2048 d64 fp32; its 120 MB of inputs fit in L2,
so L2 is flushed between steps), long (B1 H16 T65536 d128 bf16), tiny
(B1 H1 T256 d16 fp32, launch-bound) and decode (one kla_step over B256 H16
d64 fp32 per step, state from a 1024-token prefix; HBM-bound). Under
torchrun every rank runs its own independent batch (weak scaling; no
collective on the data path) and rank 0 reports the whole-job throughput over
the slowest rank's time.

``--pass backward`` times kla_backward instead (gradients of every input for a
random dL/dy and dL/dλ_T, dL/dη_T) on the same forward workloads.
``--pass conv`` times the block's causal convolution with SiLU on the
workload's q, k and v streams (kla_conv, width 4, one launch each);
``--pass conv_backward`` its backward (kla_conv_backward).

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

METRICS = {
    "headline": "KLA scan tokens/s (B·H·T/s) at H=16,d=64,T=4096 bf16; % of roofline",
    "medium": "KLA scan tokens/s (B·H·T/s) at B=4,H=8,d=64,T=2048 fp32; % of roofline",
    "long": "KLA scan tokens/s (B·H·T/s) at H=16,d=128,T=65536 bf16; % of roofline",
    "tiny": "KLA scan tokens/s (B·H·T/s) at B=1,H=1,d=16,T=256 fp32",
    "decode": "KLA decode step tokens/s (B·H per step) at B=256,H=16,d=64 fp32; % of HBM roofline",
}
DESCRIPTIONS = {
    "headline": "headline B8 H16 T4096 dk64 dv64 bf16 I/O, fp32 state",
    "medium": "medium B4 H8 T2048 dk64 dv64 fp32 I/O",
    "long": "long context B1 H16 T65536 dk128 dv128 bf16 I/O, fp32 state, a=sigmoid(N(4,1))",
    "tiny": "tiny B1 H1 T256 dk16 dv16 fp32 I/O",
    "decode": "decode kla_step B256 H16 dk64 dv64 fp32, state from a 1024-token kla_forward prefix",
}
CONV_NAMES = {"conv": "causal convolution + SiLU", "conv_backward": "backward of the causal convolution"}


def metric_for(wname: str, pass_: str) -> str:
    """The metric string of a workload and pass (the same for both arms)."""
    if pass_ == "backward":
        return METRICS[wname].replace("KLA scan tokens/s", "KLA backward tokens/s")
    if pass_ in CONV_NAMES:
        return METRICS[wname].replace("KLA scan tokens/s", f"KLA block {CONV_NAMES[pass_]} of q, k, v: tokens/s")
    return METRICS[wname]


# Algorithmic flops per element-step of the printed recursion (FMA = 2, each
# reciprocal or division = 1): c = k²Λ^v (1), a² + p̄λ (2), its reciprocal (1),
# λr + c (2), a·r (1), kΛ^v v (1), fη + b (2), η/λ (1), y += qμ (2).
FLOPS_PER_ELEMENT_STEP = 13
# Backward: the checkpointing forward (13) plus the adjoint step as written in
# kla_backward.cu with the forward quantities it needs recomputed (48).
BWD_FLOPS_PER_ELEMENT_STEP = 13 + 48
ORACLE_FLAGS = "g++ -O2 -std=c++17 -fno-fast-math -ffp-contract=off, std::thread over heads"
DECODE_GRAPH_STEPS = 8       # decode token steps per captured CUDA graph
L2_FLUSH_BYTES = 256 << 20   # written between steps when a workload's inputs fit in L2
TRAFFIC_FILES = {"headline": os.path.join(ROOT, "profiles", "traffic_headline.json")}
KERNEL_SOURCES = [os.path.join(ROOT, "bayesian_filtering_linear_gb300", "csrc", f)
                  for f in ("kla_scan_kernel.cuh", "kla_scan_inst_y.cu", "kla_scan.cu", "kla_common.cuh",
                            "kla_device.cuh")]


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


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else platform)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu model")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def cpu_oracle_variants(wname: str, nthreads: int) -> dict:
    """The oracle's other timed builds on the same recipe, as it stands: fp64
    on one thread (a sample of heads) and the fp32 build of the same loop on
    all threads. Returns {name: {value, unit, cores, sample}}."""
    import oracle
    from bayesian_filtering_linear_gb300.inputs import WORKLOADS, make_inputs
    w = WORKLOADS[wname]
    out = {}
    if wname == "decode":
        return out
    heads_all = w.B * w.H
    for name, prec, threads, heads in (("fp64_1_thread", "f64", 1, min(heads_all, 4)),
                                       ("fp32_all_threads", "f32", nthreads, heads_all)):
        x = make_inputs(1, heads, w.T, w.dk, w.dv, io=w.io, seed=w.seed, a_logit_mean=w.a_logit_mean)
        t0 = time.perf_counter()
        oracle.forward(x["q"], x["k"], x["v"], x["lam_v"], x["a"], x["pbar"], x["lam0"], x["eta0"],
                       precision=prec, nthreads=threads, want_scales=False)
        dt = time.perf_counter() - t0
        used = min(threads, heads)
        out[name] = {"value": heads * w.T / dt, "unit": "tokens/s", "cores": used,
                     "sample": f"{heads} heads x {w.T} tokens of the {wname} recipe, {prec} C++ loop, {used} threads"}
    return out


def cpu_oracle_sample(wname: str, nthreads: int) -> tuple[float, dict]:
    """Time the fp64 oracle, as it stands, on a bounded sample of a workload's
    recipe (same shapes per head, fresh draws): whole heads of the forward
    workloads, or 64 single-token steps over all heads for decode. Returns
    (tokens/s, description); the description also carries the CPU model, the
    compiler flags and the other builds' rates (cpu_oracle_variants)."""
    import oracle
    from bayesian_filtering_linear_gb300.inputs import WORKLOADS, make_inputs
    w = WORKLOADS[wname]
    oracle.build()
    if wname == "decode":
        heads, steps = w.B * w.H, 64
        x = make_inputs(1, heads, 1, w.dk, w.dv, io=w.io, seed=w.seed, random_state=True)
        lam, eta = x["lam0"], x["eta0"]
        t0 = time.perf_counter()
        for _ in range(steps):
            r = oracle.forward(x["q"], x["k"], x["v"], x["lam_v"], x["a"], x["pbar"], lam, eta,
                               nthreads=nthreads, want_scales=False)
            lam, eta = r["lamT"], r["etaT"]
        dt = time.perf_counter() - t0
        used = min(nthreads, heads)
        return heads * steps / dt, {
            "kind": "oracle", "cores": used, "cpu_model": cpu_model(), "compiler": ORACLE_FLAGS,
            "sample": f"{steps} single-token steps over {heads} heads (d_k=d_v={w.dk}), fp64 C++ loop, "
                      f"{used} threads, state converted to fp32 between steps"}
    heads = w.B * w.H
    tokens = w.T
    x = make_inputs(1, heads, tokens, w.dk, w.dv, io=w.io, seed=w.seed, a_logit_mean=w.a_logit_mean)
    t0 = time.perf_counter()
    oracle.forward(x["q"], x["k"], x["v"], x["lam_v"], x["a"], x["pbar"], x["lam0"], x["eta0"],
                   nthreads=nthreads, want_scales=False)
    dt = time.perf_counter() - t0
    used = min(nthreads, heads)
    return heads * tokens / dt, {
        "kind": "oracle", "cores": used,
        "sample": f"all {heads} heads x {tokens} tokens of the {wname} recipe (d_k={w.dk}, d_v={w.dv}, "
                  f"{w.io}-rounded inputs), fp64 C++ loop, {used} threads",
        "cpu_model": cpu_model(), "compiler": ORACLE_FLAGS,
        "other_builds": cpu_oracle_variants(wname, nthreads)}


def run_reference(args, world, rank):
    """Reference arm: the CPU oracle on bounded samples of the workload, timed
    per step (rank 0 only)."""
    if rank != 0:
        return
    import oracle
    from bayesian_filtering_linear_gb300.inputs import WORKLOADS, make_inputs
    wname = args.workload
    w = WORKLOADS[wname]
    heads = 16
    tokens = 1 if wname == "decode" else max(1, min(w.T, (256 * 64 * 64) // (w.dk * w.dv)))
    nthreads = min(os.cpu_count() or 1, heads)
    x = make_inputs(1, heads, tokens, w.dk, w.dv, io=w.io, seed=w.seed, a_logit_mean=w.a_logit_mean,
                    random_state=wname == "decode")
    oracle.build()
    kind = "fp64 C++ oracle"
    if args.pass_ == "backward":
        import numpy as np
        gy = np.random.default_rng(0).standard_normal((1, heads, tokens, w.dv)).astype(np.float32)
        run = lambda: oracle.backward(x["q"], x["k"], x["v"], x["lam_v"], x["a"], x["pbar"], x["lam0"], x["eta0"], gy,
                                      nthreads=nthreads, want_scales=False)
        kind = "fp64 C++ reverse-mode oracle"
    elif args.pass_ in CONV_NAMES:
        from bayesian_filtering_linear_gb300.inputs import make_conv_inputs
        from oracle import conv as C
        streams = [{k: v.double().numpy() for k, v in make_conv_inputs(1, heads, tokens, d, CONV_TAPS, io=w.io,
                                                                         seed=i).items()}
                   for i, d in enumerate((w.dk, w.dk, w.dv))]
        if args.pass_ == "conv":
            run = lambda: [C.conv(p["x"], p["weight"], p["bias"]) for p in streams]
        else:
            run = lambda: [C.conv_backward(p["x"], p["weight"], p["bias"], None, p["gy"]) for p in streams]
        nthreads = 1
        kind = "fp64 numpy oracle of q, k and v's convolutions"
    else:
        run = lambda: oracle.forward(x["q"], x["k"], x["v"], x["lam_v"], x["a"], x["pbar"], x["lam0"], x["eta0"],
                                     nthreads=nthreads, want_scales=False)
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    dt = time.perf_counter() - t0
    value = heads * tokens * args.steps / dt
    sample = f"each step: {heads} heads x {tokens} tokens of the {wname} recipe, {kind}"
    print(json.dumps({
        "impl": "reference", "metric": metric_for(wname, args.pass_), "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": DESCRIPTIONS[wname] + " (sampled)", "B": w.B, "H": w.H, "T": w.T,
                   "dk": w.dk, "dv": w.dv, "io": w.io},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": nthreads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def timed_steps(step, args, world, local, stream, flush=None):
    """Warm up, then time exactly args.steps calls of `step` with CUDA events on
    `stream` (barrier + synchronize on both sides), sampling clocks meanwhile.
    Returns (total ms over the slowest rank, mean per-launch ms, clocks).
    With `flush`, it runs between steps, outside the per-launch events."""
    import torch
    for _ in range(max(args.warmup, 3)):
        step()
        if flush:
            flush()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with ClockSampler(local) as clocks:
        barrier(world)
        torch.cuda.synchronize()
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for i in range(args.steps):
            if flush:
                flush()
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
        end.record(stream)
        torch.cuda.synchronize()
        barrier(world)
    per_launch_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    total_ms = max_over_ranks(start.elapsed_time(end), world)
    return total_ms, max_over_ranks(per_launch_ms, world), clocks


E2E_BUFFERS = 2
E2E_OVERLAP = ("every step copies its own inputs in from pinned host memory and its results out; with two "
               "buffer sets the copies run on their own streams and overlap the neighbouring steps' compute")


def packed_inputs(tensors: dict, device, nbuf: int):
    """One pinned host byte buffer holding `tensors` back to back (each at a
    16-byte aligned offset), `nbuf` device byte buffers of the same layout,
    and per buffer the tensors as views into it, so that a step's inputs move
    in one host-to-device copy. Returns (host, device buffers, views, bytes)."""
    import torch
    offs, total = {}, 0
    for n, t in tensors.items():
        offs[n] = total
        total += -(-t.numel() * t.element_size() // 16) * 16
    host = torch.empty(total, dtype=torch.uint8).pin_memory()
    for n, t in tensors.items():
        raw = t.detach().contiguous().reshape(-1).cpu().view(torch.uint8)
        host[offs[n]:offs[n] + raw.numel()].copy_(raw)
    flats = [torch.empty(total, dtype=torch.uint8, device=device) for _ in range(nbuf)]

    def views(flat):
        return {n: flat[offs[n]:offs[n] + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
                for n, t in tensors.items()}
    return host, flats, [views(f) for f in flats], total


def pipelined_e2e(copy_in, compute, copy_out, args, world, stream, nbuf=E2E_BUFFERS) -> float:
    """Mean ms of an end-to-end step, slowest rank, with `nbuf` sets of device
    buffers: step i copies its inputs into set i % nbuf on one stream,
    computes on `stream` and copies its results out on a third stream, so the
    copy engines work on neighbouring steps while the GPU computes. Each
    callback gets (buffer index, stream) and must enqueue its work there."""
    import torch
    s_in, s_out = torch.cuda.Stream(device=stream.device), torch.cuda.Stream(device=stream.device)
    ev_in = [torch.cuda.Event() for _ in range(nbuf)]
    ev_comp = [torch.cuda.Event() for _ in range(nbuf)]
    ev_out = [torch.cuda.Event() for _ in range(nbuf)]
    used = [False] * nbuf

    def one(i):
        b = i % nbuf
        if used[b]:
            s_in.wait_event(ev_comp[b])  # the last compute on set b has read its inputs
        with torch.cuda.stream(s_in):
            copy_in(b, s_in)
        ev_in[b].record(s_in)
        stream.wait_event(ev_in[b])
        if used[b]:
            stream.wait_event(ev_out[b])  # set b's previous results are out
        with torch.cuda.stream(stream):
            compute(b, stream)
        ev_comp[b].record(stream)
        s_out.wait_event(ev_comp[b])
        with torch.cuda.stream(s_out):
            copy_out(b, s_out)
        ev_out[b].record(s_out)
        used[b] = True

    steps = max(5, min(args.steps, 50))
    for i in range(2 * nbuf):
        one(i)
    torch.cuda.synchronize()
    barrier(world)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(s_in)
    for i in range(steps):
        one(i)
    stream.wait_event(ev_out[(steps - 1) % nbuf])
    e.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(s.elapsed_time(e) / steps, world)
    barrier(world)
    return ms


def run_kla(args, world, rank, local):
    import torch
    from bayesian_filtering_linear_gb300 import kla
    from bayesian_filtering_linear_gb300.inputs import WORKLOADS, make_workload, make_inputs
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wname = args.workload
    w = WORKLOADS[wname]
    if args.T:
        import dataclasses
        w = dataclasses.replace(w, T=args.T)
    if rank == 0:
        x = make_workload(w, device=dev)
    else:  # independent batch per rank
        x = make_inputs(w.B, w.H, w.T, w.dk, w.dv, io=w.io, seed=w.seed + 1000 * rank,
                        a_logit_mean=w.a_logit_mean, device=dev)
    stream = torch.cuda.current_stream(dev)
    names = ("q", "k", "v", "lam_v", "a", "pbar", "lam0", "eta0")
    if wname == "decode":
        return run_kla_decode(args, world, rank, local, w, x, stream)
    if args.pass_ == "backward":
        return run_kla_backward(args, world, rank, local, w, x, stream)
    if args.pass_ in ("conv", "conv_backward"):
        return run_conv(args, world, rank, local, w, stream, backward=args.pass_ == "conv_backward")

    fwd_opt = {"strategy": args.strategy, "chunk_len": args.chunk_len, "coef_pass": args.coef_pass}
    plan = kla.plan(w.B, w.H, w.T, w.dk, w.dv, w.io, **fwd_opt)
    ws = torch.empty(plan["workspace_bytes"], dtype=torch.uint8, device=dev) if plan["workspace_bytes"] else None
    y = torch.empty((w.B, w.H, w.T, w.dv), dtype=x["q"].dtype, device=dev)
    lamT = torch.empty_like(x["lam0"])
    etaT = torch.empty_like(x["eta0"])
    in_bytes = sum(x[n].numel() * x[n].element_size() for n in names)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = None
    if in_bytes < 2 * l2:
        scratch = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        flush = lambda: scratch.fill_(1.0)

    def step():
        kla.forward(x["q"], x["k"], x["v"], x["lam_v"], x["a"], x["pbar"], x["lam0"], x["eta0"],
                    y=y, lamT=lamT, etaT=etaT, workspace=ws, stream=stream, **fwd_opt)

    total_ms, per_launch_ms, clocks = timed_steps(step, args, world, local, stream, flush)
    # With a flush between steps the step time is the launch time (events
    # around each forward); otherwise the whole timed region over K steps.
    ms_per_step = per_launch_ms if flush else total_ms / args.steps
    tokens = w.B * w.H * w.T
    value = tokens * world / (ms_per_step * 1e-3)

    # ---- end to end through host buffers: H2D of the inputs, the call, D2H of
    # the outputs, every step, inside the timed region ------------------------
    nb = E2E_BUFFERS
    host, flat, devb, h2d = packed_inputs({n: x[n] for n in names}, dev, nb)
    outs = [(torch.empty_like(y), torch.empty_like(lamT), torch.empty_like(etaT)) for _ in range(nb)]
    outs_h = [tuple(torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in o) for o in outs]
    d2h = sum(t.numel() * t.element_size() for t in outs_h[0])

    def copy_in(b, s):  # the step's eight inputs, packed: one copy
        flat[b].copy_(host, non_blocking=True)

    def compute(b, s):
        d, (yb, lb, eb) = devb[b], outs[b]
        kla.forward(d["q"], d["k"], d["v"], d["lam_v"], d["a"], d["pbar"], d["lam0"], d["eta0"],
                    y=yb, lamT=lb, etaT=eb, workspace=ws, stream=s, **fwd_opt)

    def copy_out(b, s):
        for t_h, t in zip(outs_h[b], outs[b]):
            t_h.copy_(t, non_blocking=True)

    e2e_ms = pipelined_e2e(copy_in, compute, copy_out, args, world, stream)
    if rank != 0:
        return

    peaks = measured_peaks()
    sm_mhz = float(peaks.get("sm_max_mhz", 2070.0))
    nsm = torch.cuda.get_device_properties(dev).multi_processor_count
    peak_tflops = nsm * 128 * 2 * sm_mhz * 1e6 / 1e12
    element_steps = tokens * w.dk * w.dv
    flops = FLOPS_PER_ELEMENT_STEP * element_steps
    achieved = flops / (per_launch_ms * 1e-3) / 1e12
    traffic = None
    try:
        rec = json.load(open(TRAFFIC_FILES[wname]))
        if rec.get("source_hash") == kernel_source_hash() and rec.get("plan") == plan:
            traffic = rec["dram_bytes_per_launch"]
    except (KeyError, OSError, ValueError):
        pass
    cpu_value, cpu_desc = cpu_oracle_sample(wname, os.cpu_count() or 1)
    launches_per_step = (2 if plan["coef_pass"] else 1) if plan["strategy"] == "sequential" else 3
    l2_note = (f"inputs ({in_bytes / 1e6:.0f} MB) fit in L2: {L2_FLUSH_BYTES >> 20} MB written between steps, "
               "step time from per-launch events" if flush else
               f"inputs ({in_bytes / 1e6:.0f} MB) larger than L2; no flush")
    print(json.dumps({
        "metric": METRICS[wname], "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "io_dtype": w.io, "data": "synthetic",
        "config": {"workload": DESCRIPTIONS[wname] + (f" (T overridden to {w.T})" if args.T else ""),
                   "B": w.B, "H": w.H,
                   "T": w.T, "dk": w.dk, "dv": w.dv, "io": w.io, "strategy": plan["strategy"],
                   "chunk_len": plan["chunk_len"], "cols_per_block": plan["cols_per_block"],
                   "rows_per_lane": plan["rows_per_lane"], "coef_pass": plan["coef_pass"],
                   "l2": l2_note, "parallelism": f"{world} independent batches"},
        "roofline": {"bound": "alu", "achieved": achieved, "peak": peak_tflops, "unit": "TFLOP/s",
                     "frac": achieved / peak_tflops, "traffic": traffic,
                     "kernel": ("whole pass: kla_coef_kernel + kla_scan_kernel" if plan["coef_pass"] else
                                "kla_scan_kernel") if plan["strategy"] == "sequential" else "whole chunked pass",
                     "kernel_ms": per_launch_ms,
                     "peak_basis": f"{nsm} SMs x 128 fp32 lanes x 2 flop x {sm_mhz:.0f} MHz (max SM clock)",
                     "flops_per_launch": flops},
        # The hardware-honest bound of the element-step: max(FP32 lane-ops / 128,
        # MUFU ops / 16) SM-clocks; 9 lane-ops and 1 reciprocal per element-step
        # make the MUFU term the larger, 16 element-steps per SM-clock.
        "hw_bound": {"unit": "element-steps/s", "achieved": element_steps / (per_launch_ms * 1e-3),
                     "peak": 16 * nsm * sm_mhz * 1e6,
                     "frac": element_steps / (per_launch_ms * 1e-3) / (16 * nsm * sm_mhz * 1e6),
                     "basis": "max(9 FP32 lane-ops / 128, 1 MUFU reciprocal / 16) SM-clocks per element-step"},
        "cpu_baseline": {"value": cpu_value, "unit": "tokens/s", **cpu_desc},
        "e2e": {"value": tokens * world / (e2e_ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "overlap": E2E_OVERLAP},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks.summary(),
    }), flush=True)


def run_kla_decode(args, world, rank, local, w, x, stream):
    """Decode: one kla_step over all B·H heads per step, the fp32 state
    (λ, η) resident in HBM and updated in place; state from a kla_forward over
    the first 1024 tokens, then the remaining tokens' inputs are fed in turn
    (cycling when the run is longer)."""
    import torch
    from bayesian_filtering_linear_gb300 import kla
    from bayesian_filtering_linear_gb300.inputs import DECODE_PREFIX
    dev = x["q"].device
    per_tok = ("q", "k", "v", "lam_v", "a", "pbar")
    pre = {n: x[n][:, :, :DECODE_PREFIX].contiguous() for n in per_tok}
    _, lam, eta = kla.forward(*(pre[n] for n in per_tok), x["lam0"], x["eta0"])
    del pre
    n_steps = w.T - DECODE_PREFIX
    toks = [{n: x[n][:, :, DECODE_PREFIX + s].contiguous() for n in per_tok} for s in range(n_steps)]
    y = torch.empty((w.B, w.H, w.dv), dtype=x["q"].dtype, device=dev)
    it = [0]

    def eager_step():
        t = toks[it[0] % n_steps]
        it[0] += 1
        kla.step(t["q"], t["k"], t["v"], t["lam_v"], t["a"], t["pbar"], lam, eta, y=y, stream=stream)

    # A decode loop is replayed from a CUDA graph, as a server runs it: one
    # graph holds DECODE_GRAPH_STEPS consecutive token steps (each its own
    # inputs and y), so the timed launches carry no per-call host time. The
    # eager per-step time (one kla_step call from Python) is reported beside.
    ys_g = [torch.empty_like(y) for _ in range(DECODE_GRAPH_STEPS)]
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream(device=dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        kla.step(*(toks[0][n] for n in per_tok), lam, eta, y=ys_g[0])  # first-launch work outside the capture
        with torch.cuda.graph(graph, stream=side):
            for g in range(DECODE_GRAPH_STEPS):
                t = toks[g % n_steps]
                kla.step(*(t[n] for n in per_tok), lam, eta, y=ys_g[g])
    stream.wait_stream(side)
    torch.cuda.synchronize()

    total_ms, per_launch_ms, clocks = timed_steps(graph.replay, args, world, local, stream)
    ms_per_step = total_ms / (args.steps * DECODE_GRAPH_STEPS)
    per_launch_ms /= DECODE_GRAPH_STEPS
    eager_total_ms, _, _ = timed_steps(eager_step, args, world, local, stream)
    eager_ms_per_step = eager_total_ms / args.steps
    heads = w.B * w.H
    value = heads * world / (ms_per_step * 1e-3)

    # A token's six inputs sit back to back in one pinned host buffer and one
    # device buffer per set (the tensors kla.step gets are views into it), so
    # a step makes one host-to-device copy instead of six: at ~50 µs per step
    # the per-call host time of the copies is a large part of the step.
    sizes = [toks[0][n].numel() for n in per_tok]
    offs = [sum(sizes[:i]) for i in range(len(sizes))]
    io_dt = toks[0]["q"].dtype
    host = []
    for t in toks[:8]:
        hb = torch.empty(sum(sizes), dtype=io_dt).pin_memory()
        for n, o, sz in zip(per_tok, offs, sizes):
            hb[o:o + sz].copy_(t[n].reshape(-1).cpu())
        host.append(hb)
    nb = E2E_BUFFERS
    flat = [torch.empty(sum(sizes), dtype=io_dt, device=dev) for _ in range(nb)]
    devb = [{n: flat[b][o:o + sz].view(toks[0][n].shape) for n, o, sz in zip(per_tok, offs, sizes)}
            for b in range(nb)]
    ys = [torch.empty_like(y) for _ in range(nb)]
    ys_h = [torch.empty(y.shape, dtype=y.dtype).pin_memory() for _ in range(nb)]
    h2d = host[0].numel() * host[0].element_size()
    d2h = ys_h[0].numel() * ys_h[0].element_size()
    ie = [0]

    def copy_in(b, s):
        h = host[ie[0] % len(host)]
        ie[0] += 1
        flat[b].copy_(h, non_blocking=True)

    def compute(b, s):  # the state is updated in place, so steps stay in order on `stream`
        d = devb[b]
        kla.step(d["q"], d["k"], d["v"], d["lam_v"], d["a"], d["pbar"], lam, eta, y=ys[b], stream=s)

    def copy_out(b, s):
        ys_h[b].copy_(ys[b], non_blocking=True)

    e2e_ms = pipelined_e2e(copy_in, compute, copy_out, args, world, stream)
    if rank != 0:
        return
    peaks = measured_peaks()
    hbm = float(peaks.get("hbm_gbs", 6800.0))
    io_size = x["q"].element_size()
    bytes_per_step = 16 * heads * w.dk * w.dv + heads * (4 * w.dk + 3 * w.dv) * io_size
    achieved = bytes_per_step / (per_launch_ms * 1e-3) / 1e9
    cpu_value, cpu_desc = cpu_oracle_sample("decode", os.cpu_count() or 1)
    print(json.dumps({
        "metric": METRICS["decode"], "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps * DECODE_GRAPH_STEPS, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "eager_ms_per_step": eager_ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": DESCRIPTIONS["decode"], "B": w.B, "H": w.H, "dk": w.dk, "dv": w.dv, "io": w.io,
                   "l2": f"state ({16 * heads * w.dk * w.dv / 1e6:.0f} MB read and written per step) larger "
                         "than L2; no flush",
                   "parallelism": f"{world} independent batches",
                   "timing": f"{args.steps} replays of a CUDA graph of {DECODE_GRAPH_STEPS} kla_step calls"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                     "traffic": None, "kernel": "kla_step_kernel", "kernel_ms": per_launch_ms,
                     "peak_basis": "measured copy bandwidth (MEASURED_PEAKS.json hbm_gbs)",
                     "bytes_per_launch": bytes_per_step},
        "cpu_baseline": {"value": cpu_value, "unit": "tokens/s", **cpu_desc},
        "e2e": {"value": heads * world / (e2e_ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "overlap": E2E_OVERLAP},
        "gpu_launches": args.steps * DECODE_GRAPH_STEPS,
        "clocks": clocks.summary(),
    }), flush=True)


def run_kla_backward(args, world, rank, local, w, x, stream):
    """One kla_backward per step: gradients of every input for a fixed random
    dL/dy and dL/dλ_T, dL/dη_T, inputs resident in HBM."""
    import torch
    from bayesian_filtering_linear_gb300 import kla
    dev = x["q"].device
    g = torch.Generator(device=dev)
    g.manual_seed(7 + rank)
    gy = torch.randn(w.B, w.H, w.T, w.dv, generator=g, device=dev).to(x["q"].dtype)
    gl = torch.randn(w.B, w.H, w.dk, w.dv, generator=g, device=dev)
    ge = torch.randn(w.B, w.H, w.dk, w.dv, generator=g, device=dev)
    ws = torch.empty(max(16, kla.LIB.kla_backward_workspace_size(w.B, w.H, w.T, w.dk, w.dv)), dtype=torch.uint8,
                     device=dev)
    names = ("q", "k", "v", "lam_v", "a", "pbar", "lam0", "eta0")

    def step():
        kla.backward(*(x[n] for n in names), gy=gy, glamT=gl, getaT=ge, workspace=ws, stream=stream)

    total_ms, per_launch_ms, clocks = timed_steps(step, args, world, local, stream)
    ms_per_step = total_ms / args.steps
    tokens = w.B * w.H * w.T
    value = tokens * world / (ms_per_step * 1e-3)

    nb = E2E_BUFFERS
    host, flat, devb, h2d = packed_inputs(dict({n: x[n] for n in names}, gy=gy, gl=gl, ge=ge), dev, nb)
    sample = kla.backward(*(x[n] for n in names), gy=gy, glamT=gl, getaT=ge, workspace=ws, stream=stream)
    outs_h = [{n: torch.empty(t.shape, dtype=t.dtype).pin_memory() for n, t in sample.items()} for _ in range(nb)]
    d2h = sum(t.numel() * t.element_size() for t in outs_h[0].values())
    results = [None] * nb

    def copy_in(b, s):
        flat[b].copy_(host, non_blocking=True)  # inputs and upstream gradients, packed: one copy

    def compute(b, s):  # the gradients are allocated on `s` (the current stream here)
        d = devb[b]
        results[b] = kla.backward(*(d[n] for n in names), gy=d["gy"], glamT=d["gl"], getaT=d["ge"], workspace=ws,
                                  stream=s)

    def copy_out(b, s):
        for n, t in results[b].items():
            t.record_stream(s)  # read on the copy stream: not reused before the copy is done
            outs_h[b][n].copy_(t, non_blocking=True)

    e2e_ms = pipelined_e2e(copy_in, compute, copy_out, args, world, stream)
    if rank != 0:
        return
    ckpt_bytes = (-(-w.T // 16) + 1) * 2 * w.B * w.H * w.dk * w.dv * 4
    peaks = measured_peaks()
    sm_mhz = float(peaks.get("sm_max_mhz", 2070.0))
    nsm = torch.cuda.get_device_properties(dev).multi_processor_count
    peak_tflops = nsm * 128 * 2 * sm_mhz * 1e6 / 1e12
    flops = BWD_FLOPS_PER_ELEMENT_STEP * tokens * w.dk * w.dv
    achieved = flops / (per_launch_ms * 1e-3) / 1e12
    cpu_value, cpu_desc = cpu_oracle_backward_sample(w, os.cpu_count() or 1)
    print(json.dumps({
        "metric": metric_for(w.name, "backward"), "value": value,
        "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": DESCRIPTIONS[w.name] + "; backward pass", "B": w.B, "H": w.H, "T": w.T, "dk": w.dk,
                   "dv": w.dv, "io": w.io, "workspace_bytes": ws.numel(),
                   "l2": "inputs larger than L2; no flush", "parallelism": f"{world} independent batches"},
        "roofline": {"bound": "alu", "achieved": achieved, "peak": peak_tflops, "unit": "TFLOP/s",
                     "frac": achieved / peak_tflops, "traffic": None,
                     "kernel": "kla_backward (checkpointing scan + kla_bwd_kernel)", "kernel_ms": per_launch_ms,
                     "peak_basis": f"{nsm} SMs x 128 fp32 lanes x 2 flop x {sm_mhz:.0f} MHz (max SM clock)",
                     "flops_per_launch": flops},
        "cpu_baseline": {"value": cpu_value, "unit": "tokens/s", **cpu_desc},
        "e2e": {"value": tokens * world / (e2e_ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "overlap": E2E_OVERLAP},
        # checkpointing scan + reverse kernel, + the row-sum pass when the
        # workspace holds more than the checkpoints (columns split over blocks)
        "gpu_launches": (2 + int(ws.numel() > ckpt_bytes)) * args.steps,
        "clocks": clocks.summary(),
    }), flush=True)


CONV_TAPS = 4  # width of the block's causal convolution (the KLA summary gives none; 4 as in Mamba-style blocks)


def run_conv(args, world, rank, local, w, stream, backward: bool):
    """The block's convolution prologue on the workload's streams: q, k and v
    (``[B,H,T,d]``) each through kla_conv with its own taps, bias and SiLU
    (three launches per step), or through kla_conv_backward (gradients of the
    input, taps and bias). HBM-bound: reported against the measured copy
    bandwidth."""
    import torch
    from bayesian_filtering_linear_gb300 import kla
    from bayesian_filtering_linear_gb300.inputs import make_conv_inputs
    dev = torch.device("cuda", local)
    W = CONV_TAPS
    dims = {"q": w.dk, "k": w.dk, "v": w.dv}
    s = {n: make_conv_inputs(w.B, w.H, w.T, d, W, io=w.io, seed=w.seed + 100 * i + 1000 * rank, device=dev)
         for i, (n, d) in enumerate(dims.items())}
    ys = {n: torch.empty_like(s[n]["x"]) for n in dims}
    wos = {n: torch.empty_like(s[n]["window"]) for n in dims}  # window after the last token
    ws = {}
    if backward:
        for n, d in dims.items():
            ws[n] = torch.empty(max(16, kla.LIB.kla_conv_backward_workspace_size(w.B, w.H, w.T, d, W)),
                                dtype=torch.uint8, device=dev)

    def run_one(n, src, out, s_):
        if backward:
            return kla.conv_backward(src["x"], src["weight"], src["bias"], None, gy=src["gy"], window_grad=False,
                                     workspace=ws[n], stream=s_)
        return kla.conv(src["x"], src["weight"], src["bias"], None, y=out, window_out=wos[n] if out is not None else None,
                        stream=s_)

    def step():
        for n in dims:
            run_one(n, s[n], ys[n], stream)

    in_bytes = sum(s[n]["x"].numel() * s[n]["x"].element_size() for n in dims)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = None
    if in_bytes * (3 if backward else 2) < 2 * l2:
        scratch = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        flush = lambda: scratch.fill_(1.0)
    # The step's three launches are replayed from a CUDA graph (as a layer
    # inside a captured model step runs them), so the timed region carries no
    # per-call host time; the eager step time is reported beside.
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream(device=dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        step_on = lambda: [run_one(n, s[n], ys[n], side) for n in dims]
        step_on()  # first-launch work outside the capture
        with torch.cuda.graph(graph, stream=side):
            step_on()
    stream.wait_stream(side)
    torch.cuda.synchronize()
    total_ms, per_launch_ms, clocks = timed_steps(graph.replay, args, world, local, stream, flush)
    ms_per_step = per_launch_ms if flush else total_ms / args.steps
    eager_total_ms, eager_launch_ms, _ = timed_steps(step, args, world, local, stream, flush)
    eager_ms_per_step = eager_launch_ms if flush else eager_total_ms / args.steps
    tokens = w.B * w.H * w.T
    value = tokens * world / (ms_per_step * 1e-3)

    # end to end: the streams (and gy) in from pinned host memory, the results out
    keys = ("x", "gy") if backward else ("x",)
    host = {n: {k: s[n][k].cpu().pin_memory() for k in keys} for n in dims}
    nb = E2E_BUFFERS
    devb = [{n: {k: torch.empty_like(s[n][k]) for k in keys} for n in dims} for _ in range(nb)]
    results = [None] * nb
    sample = {n: run_one(n, s[n], ys[n], stream) for n in dims}
    flat = lambda r: list(r.values()) if isinstance(r, dict) else [r[0]]
    outs_h = [{n: [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in flat(sample[n])] for n in dims}
              for _ in range(nb)]
    h2d = sum(t.numel() * t.element_size() for n in dims for t in host[n].values())
    d2h = sum(t.numel() * t.element_size() for n in dims for t in outs_h[0][n])

    def copy_in(b, s_):
        for n in dims:
            for k in keys:
                devb[b][n][k].copy_(host[n][k], non_blocking=True)

    def compute(b, s_):
        results[b] = {n: run_one(n, dict(s[n], **devb[b][n]), None, s_) for n in dims}

    def copy_out(b, s_):
        for n in dims:
            for t_h, t in zip(outs_h[b][n], flat(results[b][n])):
                t.record_stream(s_)
                t_h.copy_(t, non_blocking=True)

    e2e_ms = pipelined_e2e(copy_in, compute, copy_out, args, world, stream)
    if rank != 0:
        return
    esz = s["q"]["x"].element_size()
    # algorithmic bytes: every stream element read once (and gy) and its output written once; taps and bias
    elems = sum(w.B * w.H * w.T * d for d in dims.values())
    params = sum(w.H * d * (W + 1) * 4 for d in dims.values())
    alg_bytes = elems * esz * (3 if backward else 2) + params * (2 if backward else 1)
    peaks = measured_peaks()
    peak_gbs = float(peaks.get("hbm_gbs", 6800.0))
    achieved = alg_bytes / (per_launch_ms * 1e-3) / 1e9
    cpu_value, cpu_desc = cpu_oracle_conv_sample(w, W, backward)
    name = CONV_NAMES["conv_backward" if backward else "conv"]
    print(json.dumps({
        "metric": metric_for(w.name, "conv_backward" if backward else "conv"),
        "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_per_step, "eager_ms_per_step": eager_ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "io_dtype": w.io, "data": "synthetic",
        "config": {"workload": DESCRIPTIONS[w.name] + f"; {name} of q, k and v (width {W}, own taps each)",
                   "timing": "replays of a CUDA graph of the step's launches",
                   "B": w.B, "H": w.H, "T": w.T, "dk": w.dk, "dv": w.dv, "io": w.io, "taps": W,
                   "l2": (f"streams fit in L2: {L2_FLUSH_BYTES >> 20} MB written between steps" if flush
                          else "streams larger than L2; no flush"),
                   "parallelism": f"{world} independent batches"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak_gbs, "unit": "GB/s",
                     "frac": achieved / peak_gbs, "traffic": None,
                     "kernel": "kla_conv_bwd_kernel + finish" if backward else "kla_conv_kernel",
                     "kernel_ms": per_launch_ms, "launches_per_step": 6 if backward else 3,
                     "peak_basis": "measured copy bandwidth", "bytes_per_step": alg_bytes},
        "cpu_baseline": {"value": cpu_value, "unit": "tokens/s", **cpu_desc},
        "e2e": {"value": tokens * world / (e2e_ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "overlap": E2E_OVERLAP},
        "gpu_launches": (6 if backward else 3) * args.steps,
        "clocks": clocks.summary(),
    }), flush=True)


def cpu_oracle_conv_sample(w, W: int, backward: bool) -> tuple[float, dict]:
    """The fp64 numpy oracle of the convolution, as it stands, on 16 heads × up
    to 1024 tokens of q, k and v of the workload. Returns (tokens/s, description)."""
    from bayesian_filtering_linear_gb300.inputs import make_conv_inputs
    from oracle import conv as C
    heads, tokens = min(16, w.B * w.H), min(w.T, 1024)
    t_total = 0.0
    for i, d in enumerate((w.dk, w.dk, w.dv)):
        p = {k: v.double().numpy() for k, v in make_conv_inputs(1, heads, tokens, d, W, io=w.io, seed=i).items()}
        t0 = time.perf_counter()
        if backward:
            C.conv_backward(p["x"], p["weight"][:heads], p["bias"][:heads], None, p["gy"])
        else:
            C.conv(p["x"], p["weight"][:heads], p["bias"][:heads])
        t_total += time.perf_counter() - t0
    return heads * tokens / t_total, {"kind": "oracle", "cores": 1,
                                      "sample": f"{heads} heads x {tokens} tokens of q, k and v of the {w.name} "
                                                f"recipe, fp64 numpy oracle (one thread)"}


def cpu_oracle_backward_sample(w, nthreads: int) -> tuple[float, dict]:
    """The fp64 oracle's backward, as it stands, on 16 heads of the recipe
    (up to 1024 tokens). Returns (tokens/s, description)."""
    import numpy as np
    import oracle
    from bayesian_filtering_linear_gb300.inputs import make_inputs
    heads, tokens = min(16, w.B * w.H), min(w.T, 1024)
    x = make_inputs(1, heads, tokens, w.dk, w.dv, io=w.io, seed=w.seed, a_logit_mean=w.a_logit_mean)
    gy = np.random.default_rng(0).standard_normal((1, heads, tokens, w.dv)).astype(np.float32)
    oracle.build()
    t0 = time.perf_counter()
    oracle.backward(x["q"], x["k"], x["v"], x["lam_v"], x["a"], x["pbar"], x["lam0"], x["eta0"], gy,
                    nthreads=nthreads, want_scales=False)
    dt = time.perf_counter() - t0
    used = min(nthreads, heads)
    return heads * tokens / dt, {"kind": "oracle", "cores": used,
                                 "sample": f"{heads} heads x {tokens} tokens of the {w.name} recipe, fp64 C++ "
                                           f"reverse-mode loop, {used} threads"}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("kla", "reference"), default="kla")
    ap.add_argument("--workload", choices=tuple(METRICS), default="headline")
    ap.add_argument("--pass", dest="pass_", choices=("forward", "backward", "conv", "conv_backward"),
                    default="forward")
    ap.add_argument("--T", type=int, default=0,
                    help="override the workload's sequence length (for profiling a smaller case of its shape)")
    ap.add_argument("--strategy", choices=("auto", "sequential", "chunked"), default="auto",
                    help="force the forward's strategy (default: the planner's choice)")
    ap.add_argument("--chunk-len", dest="chunk_len", type=int, default=0,
                    help="tokens per chunk with --strategy chunked (0: the planner's choice)")
    ap.add_argument("--coef-pass", dest="coef_pass", choices=("auto", "off", "on"), default="auto",
                    help="the sequential plan's coefficient pass (kla_coef_pass; default: the planner's choice)")
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
