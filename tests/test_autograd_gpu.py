"""The autograd wrappers (kla.scan, kla.causal_conv) give the gradients of
the entry points they wrap: loss.backward() through them equals the direct
kla_backward / kla_conv_backward calls on the same inputs (up to the order of
the backward's cross-warp sums, which is not fixed), and a whole block —
three convolutions feeding the scan — trains through them. The entry points
themselves are checked against the oracle elsewhere."""
import pytest
import torch

from bayesian_filtering_linear_gb300 import kla
from bayesian_filtering_linear_gb300.inputs import make_conv_inputs, make_inputs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
NAMES = ("q", "k", "v", "lam_v", "a", "pbar", "lam0", "eta0")


def close(a, b, tol=1e-6):
    scale = max(float(b.abs().max()), 1e-30)
    return float((a.double() - b.double()).abs().max()) <= tol * scale


def test_scan_autograd_matches_the_backward_entry_point():
    x = {n: t.to(DEV) for n, t in make_inputs(2, 2, 80, 32, 32, io="f32", seed=21, random_state=True).items()}
    g = torch.Generator().manual_seed(1)
    gy = torch.randn(2, 2, 80, 32, generator=g).to(DEV)
    gl, ge = torch.randn(2, 2, 32, 32, generator=g).to(DEV), torch.randn(2, 2, 32, 32, generator=g).to(DEV)
    leaves = {n: x[n].clone().requires_grad_(True) for n in NAMES}
    y, lamT, etaT = kla.scan(*(leaves[n] for n in NAMES))
    ((y * gy).sum() + (lamT * gl).sum() + (etaT * ge).sum()).backward()
    direct = kla.backward(*(x[n] for n in NAMES), gy=gy, glamT=gl, getaT=ge)
    torch.cuda.synchronize()
    for n, key in (("q", "gq"), ("k", "gk"), ("v", "gv"), ("lam_v", "glam_v"), ("a", "ga"), ("pbar", "gpbar"),
                   ("lam0", "glam0"), ("eta0", "geta0")):
        assert close(leaves[n].grad, direct[key]), n


def test_conv_autograd_matches_the_backward_entry_point():
    p = {k: v.to(DEV) for k, v in make_conv_inputs(2, 3, 70, 16, 4, io="f32", seed=22).items()}
    leaves = {n: p[n].clone().requires_grad_(True) for n in ("x", "weight", "bias", "window")}
    y, wout = kla.causal_conv(leaves["x"], leaves["weight"], leaves["bias"], leaves["window"])
    ((y * p["gy"]).sum() + (wout * p["gwindow_out"]).sum()).backward()
    direct = kla.conv_backward(p["x"], p["weight"], p["bias"], p["window"], gy=p["gy"], gwindow_out=p["gwindow_out"])
    torch.cuda.synchronize()
    for n, key in (("x", "gx"), ("weight", "gweight"), ("bias", "gbias"), ("window", "gwindow")):
        assert torch.equal(leaves[n].grad, direct[key]), n  # the convolution's backward is deterministic


def test_block_trains_through_autograd():
    """x_q, x_k, x_v → causal conv + SiLU → scan → loss: the gradients of the
    stream inputs and of every tap equal the chain of direct calls, and one
    gradient step lowers the loss."""
    B, H, T, dk, dv, W = 1, 2, 64, 16, 16, 4
    base = {k: v.to(DEV) for k, v in make_inputs(B, H, T, dk, dv, io="f32", seed=23).items()}
    streams = {n: {k: v.to(DEV) for k, v in make_conv_inputs(B, H, T, dk if n != "v" else dv, W, io="f32",
                                                              seed=70 + i).items()}
               for i, n in enumerate(("q", "k", "v"))}
    for n in streams:
        streams[n]["weight"] *= 0.5
    target = torch.randn(B, H, T, dv, generator=torch.Generator().manual_seed(5)).to(DEV)

    def loss_of(params):
        qkv = {n: kla.causal_conv(streams[n]["x"], params[n], streams[n]["bias"])[0] for n in streams}
        y, _, _ = kla.scan(qkv["q"], qkv["k"], qkv["v"], base["lam_v"], base["a"], base["pbar"])
        return ((y - target) ** 2).mean()

    params = {n: streams[n]["weight"].clone().requires_grad_(True) for n in streams}
    loss = loss_of(params)
    loss.backward()
    # the same gradients from the chain of direct calls
    qkv = {n: kla.conv(streams[n]["x"], streams[n]["weight"], streams[n]["bias"])[0] for n in streams}
    y, _, _ = kla.forward(qkv["q"], qkv["k"], qkv["v"], base["lam_v"], base["a"], base["pbar"])
    gy = (2.0 / y.numel()) * (y - target)
    sg = kla.backward(qkv["q"], qkv["k"], qkv["v"], base["lam_v"], base["a"], base["pbar"], gy=gy,
                      state_grads=False)
    for n in streams:
        cg = kla.conv_backward(streams[n]["x"], streams[n]["weight"], streams[n]["bias"], gy=sg["g" + n])
        assert close(params[n].grad, cg["gweight"], 1e-5), n
    with torch.no_grad():
        stepped = {n: params[n] - 0.5 * params[n].grad for n in params}
        assert float(loss_of(stepped)) < float(loss)
