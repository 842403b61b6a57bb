"""The entry points are stream-ordered and allocation-free given their
buffers, so they can be captured in a CUDA graph and replayed: a captured
kla_forward (both strategies) and a captured run of kla_step calls reproduce
the eager results exactly (same kernels, same inputs)."""
import pytest
import torch

from bayesian_filtering_linear_gb300 import kla
from bayesian_filtering_linear_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu

NAMES = ("q", "k", "v", "lam_v", "a", "pbar")


@pytest.mark.parametrize("strategy,chunk_len", [("sequential", 0), ("chunked", 64)], ids=str)
def test_captured_forward_replays_exactly(strategy, chunk_len):
    x = {n: t.cuda() for n, t in make_inputs(2, 4, 300, 64, 64, io="bf16", seed=4, random_state=True).items()}
    info = kla.plan(2, 4, 300, 64, 64, "bf16", strategy, chunk_len)
    ws = torch.empty(max(16, info["workspace_bytes"]), dtype=torch.uint8, device="cuda")
    y = torch.empty(2, 4, 300, 64, dtype=torch.bfloat16, device="cuda")
    lamT, etaT = torch.empty_like(x["lam0"]), torch.empty_like(x["eta0"])
    run = lambda: kla.forward(*(x[n] for n in NAMES), x["lam0"], x["eta0"], y=y, lamT=lamT, etaT=etaT,
                              workspace=ws, strategy=strategy, chunk_len=chunk_len)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        run()  # warm-up outside the capture (first-launch attributes)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    want = (y.clone(), lamT.clone(), etaT.clone())
    y.zero_(); lamT.zero_(); etaT.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run()
    g.replay()
    torch.cuda.synchronize()
    for got, ref in zip((y, lamT, etaT), want):
        assert torch.equal(got, ref)


def test_captured_decode_steps_replay_exactly():
    T = 24
    x = {n: t.cuda() for n, t in make_inputs(4, 2, T, 64, 32, io="f32", seed=6, random_state=True).items()}
    toks = [{n: x[n][:, :, t].contiguous() for n in NAMES} for t in range(T)]
    lam, eta = x["lam0"].clone(), x["eta0"].clone()
    ys = [torch.empty(4, 2, 32, device="cuda") for _ in range(T)]

    def steps():
        for t in range(T):
            kla.step(*(toks[t][n] for n in NAMES), lam, eta, y=ys[t])

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        steps()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    want = [y.clone() for y in ys] + [lam.clone(), eta.clone()]
    lam.copy_(x["lam0"]); eta.copy_(x["eta0"])
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        steps()
    lam.copy_(x["lam0"]); eta.copy_(x["eta0"])  # capture ran nothing; start from the same state
    g.replay()
    torch.cuda.synchronize()
    for got, ref in zip(ys + [lam, eta], want):
        assert torch.equal(got, ref)


def test_captured_conv_decode_and_backward_replay_exactly():
    """The block's causal convolution fed one token per call with the window
    updated in place (a decode loop), then its backward, captured once and
    replayed: the same bits as the eager calls."""
    from bayesian_filtering_linear_gb300.inputs import make_conv_inputs
    B, H, T, D, W = 2, 4, 12, 64, 4
    p = {k: v.cuda() for k, v in make_conv_inputs(B, H, T, D, W, io="bf16", seed=8).items()}
    toks = [p["x"][:, :, t:t + 1].contiguous() for t in range(T)]
    win = p["window"].clone()
    ys = [torch.empty(B, H, 1, D, dtype=torch.bfloat16, device="cuda") for _ in range(T)]
    ws = torch.empty(max(16, kla.LIB.kla_conv_backward_workspace_size(B, H, T, D, W)), dtype=torch.uint8,
                     device="cuda")
    grads = {}

    def run():
        for t in range(T):
            kla.conv(toks[t], p["weight"], p["bias"], win, y=ys[t], update_window=True)
        grads.update(kla.conv_backward(p["x"], p["weight"], p["bias"], p["window"], gy=p["gy"],
                                       gwindow_out=p["gwindow_out"], workspace=ws))

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        run()  # warm-up outside the capture (first-launch attributes)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    want = [y.clone() for y in ys] + [win.clone()] + [grads[k].clone() for k in sorted(grads)]
    win.copy_(p["window"])
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run()
    for y in ys:
        y.zero_()
    g.replay()
    torch.cuda.synchronize()
    got = [y for y in ys] + [win] + [grads[k] for k in sorted(grads)]
    for a, b in zip(got, want):
        assert torch.equal(a, b)
