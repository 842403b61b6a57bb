"""Pins for the oracle's causal convolution (oracle/conv.py), each from
something other than the oracle itself:

* torch's own depthwise ``conv1d`` (a library routine: cross-correlation over
  a left-padded input) and ``silu`` give the same outputs;
* the impulse response is the taps, in the stated order, and nothing before
  the impulse moves (causality);
* SiLU identities: SiLU(u) − SiLU(−u) = u, SiLU(0) = 0, SiLU' against central
  differences of SiLU;
* cutting a sequence anywhere (or feeding it one token at a time) and carrying
  the window gives the same outputs and final window as one pass;
* the backward equals central finite differences of the fp64 forward, and for
  the plain convolution the adjoint identity ⟨gy, J·dx⟩ = ⟨Jᵀ·gy, dx⟩ holds;
* each planted mistake (reversed taps, window one token early, SiLU' without
  its u·(1 − σ) term, a tap's gradient paired with the input one token off)
  breaks one of these.

Source of the operation: "Technische Samenvatting: Kalman Linear Attention
(KLA)", Methodologie §4 (Architectuur): 1-D causal convolutions and SiLU
activations in the Mamba-like block around the scan.
"""
import numpy as np
import pytest
import torch

from oracle import conv as C


def problem(seed, B=2, H=3, T=11, D=4, W=4):
    rng = np.random.default_rng(seed)
    return {"x": rng.standard_normal((B, H, T, D)), "weight": rng.standard_normal((H, D, W)) / np.sqrt(W),
            "bias": rng.standard_normal((H, D)) / 2, "window": rng.standard_normal((B, H, W - 1, D)),
            "gy": rng.standard_normal((B, H, T, D)), "gwindow_out": rng.standard_normal((B, H, W - 1, D))}


def torch_conv(x, weight, bias, window, activation):
    """The same layer through torch.nn.functional.conv1d (fp64, CPU)."""
    B, H, T, D = x.shape
    W = weight.shape[-1]
    xe = np.concatenate([window if window is not None else np.zeros((B, H, W - 1, D)), x], axis=2)
    inp = torch.from_numpy(xe).permute(0, 1, 3, 2).reshape(B, H * D, T + W - 1)
    wt = torch.from_numpy(weight).reshape(H * D, 1, W)
    bt = None if bias is None else torch.from_numpy(bias).reshape(H * D)
    out = torch.nn.functional.conv1d(inp, wt, bt, padding=0, groups=H * D)  # valid: T outputs
    if activation:
        out = torch.nn.functional.silu(out)
    return out.reshape(B, H, D, T).permute(0, 1, 3, 2).numpy()


@pytest.mark.parametrize("W,T,D", [(4, 11, 4), (1, 5, 8), (2, 1, 4), (3, 2, 4), (8, 13, 4)])
@pytest.mark.parametrize("with_bias,with_window,activation", [(True, True, True), (False, False, True),
                                                              (True, False, False), (False, True, False)])
def test_matches_torch_conv1d(W, T, D, with_bias, with_window, activation):
    p = problem(1, T=T, D=D, W=W)
    bias = p["bias"] if with_bias else None
    window = p["window"] if with_window else None
    y, _ = C.conv(p["x"], p["weight"], bias, window, activation)
    want = torch_conv(p["x"], p["weight"], bias, window, activation)
    assert np.abs(y - want).max() <= 1e-13 * max(1.0, np.abs(want).max())


def test_torch_pin_catches_reversed_taps():
    p = problem(2)
    y, _ = C.conv(p["x"], p["weight"], p["bias"], p["window"], True, _mutant=1)
    want = torch_conv(p["x"], p["weight"], p["bias"], p["window"], True)
    assert np.abs(y - want).max() > 1e-3


def test_impulse_response_is_the_taps_in_order():
    B, H, T, D, W = 1, 2, 12, 3, 4
    rng = np.random.default_rng(3)
    weight = rng.standard_normal((H, D, W))
    bias = rng.standard_normal((H, D))
    t0, h0, d0 = 5, 1, 2
    x = np.zeros((B, H, T, D))
    x[0, h0, t0, d0] = 1.0
    u = C.preactivation(x, weight)
    want = np.zeros_like(u)
    for k in range(W):
        want[0, h0, t0 + (W - 1) - k, d0] = weight[h0, d0, k]  # tap W-1 is the current token
    assert np.array_equal(u, want)
    assert not u[0, :, :t0, :].any()  # causal: nothing before the impulse
    # the bias is added to every token of its channel
    ub = C.preactivation(x, weight, bias)
    assert np.allclose(ub - bias[None, :, None, :], want, rtol=0, atol=1e-15)
    # a mistake in the tap order moves the response
    assert not np.array_equal(C.preactivation(x, weight, _mutant=1), want)


def test_silu_identities():
    u = np.linspace(-30.0, 30.0, 601)
    assert C.silu(np.array(0.0)) == 0.0
    assert np.allclose(C.silu(u) - C.silu(-u), u, rtol=0, atol=1e-13)
    h = 1e-6
    fd = (C.silu(u + h) - C.silu(u - h)) / (2 * h)
    assert np.abs(C.dsilu(u) - fd).max() < 1e-8
    assert np.abs(C.dsilu(u, _mutant=3) - fd).max() > 0.1


@pytest.mark.parametrize("cuts", [[5], [1, 2, 3], [0, 11], list(range(1, 11))])
def test_streaming_with_the_window_equals_one_pass(cuts):
    p = problem(4)
    y_all, win_all = C.conv(p["x"], p["weight"], p["bias"], p["window"])
    win, ys = p["window"], []
    bounds = [0] + cuts + [p["x"].shape[2]]
    for t0, t1 in zip(bounds[:-1], bounds[1:]):
        y, win = C.conv(p["x"][:, :, t0:t1], p["weight"], p["bias"], win)
        ys.append(y)
    assert np.array_equal(np.concatenate(ys, axis=2), y_all)
    assert np.array_equal(win, win_all)


def test_streaming_pin_catches_a_late_window():
    p = problem(5)
    y_all, _ = C.conv(p["x"], p["weight"], p["bias"], p["window"], _mutant=2)
    y1, win = C.conv(p["x"][:, :, :6], p["weight"], p["bias"], p["window"], _mutant=2)
    y2, _ = C.conv(p["x"][:, :, 6:], p["weight"], p["bias"], win, _mutant=2)
    assert np.abs(np.concatenate([y1, y2], axis=2) - y_all).max() > 1e-3


def test_window_out_is_the_last_inputs():
    p = problem(6, T=2, W=5)  # T < W-1: part of the window out comes from the window in
    _, win = C.conv(p["x"], p["weight"], p["bias"], p["window"])
    assert np.array_equal(win[:, :, :2], p["window"][:, :, 2:])
    assert np.array_equal(win[:, :, 2:], p["x"])


def _loss(p, activation):
    y, win = C.conv(p["x"], p["weight"], p["bias"], p["window"], activation)
    return (y * p["gy"]).sum() + (win * p["gwindow_out"]).sum()


def _fd(p, name, activation):
    base = p[name]
    out = np.zeros_like(base)
    for idx in np.ndindex(base.shape):
        h = 1e-6 * max(1.0, abs(base[idx]))
        pp, pm = dict(p), dict(p)
        pp[name], pm[name] = base.copy(), base.copy()
        pp[name][idx] += h
        pm[name][idx] -= h
        out[idx] = (_loss(pp, activation) - _loss(pm, activation)) / (2 * h)
    return out


GRAD_OF = {"x": "gx", "weight": "gweight", "bias": "gbias", "window": "gwindow"}


@pytest.mark.parametrize("activation", [True, False])
@pytest.mark.parametrize("T,W", [(7, 4), (2, 4), (5, 1), (6, 2)])
def test_backward_matches_finite_differences(activation, T, W):
    p = problem(7, B=2, H=2, T=T, D=2, W=W)
    g = C.conv_backward(p["x"], p["weight"], p["bias"], p["window"], p["gy"], p["gwindow_out"], activation)
    for name, gname in GRAD_OF.items():
        want = _fd(p, name, activation)
        assert g[gname].shape == want.shape
        if want.size == 0:  # W = 1: no window
            continue
        assert np.abs(g[gname] - want).max() <= 1e-7 * max(1.0, np.abs(want).max()), name


@pytest.mark.parametrize("mutant,name", [(3, "x"), (4, "weight")])
def test_planted_backward_mistakes_are_caught(mutant, name):
    p = problem(8, B=2, H=2, T=7, D=2, W=3)
    g = C.conv_backward(p["x"], p["weight"], p["bias"], p["window"], p["gy"], p["gwindow_out"], True,
                        _mutant=mutant)
    want = _fd(p, name, True)
    assert np.abs(g[GRAD_OF[name]] - want).max() > 1e-3 * np.abs(want).max()


def test_adjoint_identity_of_the_plain_convolution():
    p = problem(9, B=3, H=2, T=9, D=5, W=4)
    rng = np.random.default_rng(10)
    dx = rng.standard_normal(p["x"].shape)
    dwin = rng.standard_normal(p["window"].shape)
    # J·(dx, dwin): the convolution is linear in (x, window) without bias and activation
    jy, jwin = C.conv(dx, p["weight"], None, dwin, activation=False)
    g = C.conv_backward(p["x"], p["weight"], None, p["window"], p["gy"], p["gwindow_out"], activation=False)
    lhs = (p["gy"] * jy).sum() + (p["gwindow_out"] * jwin).sum()
    rhs = (g["gx"] * dx).sum() + (g["gwindow"] * dwin).sum()
    assert abs(lhs - rhs) <= 1e-12 * max(1.0, abs(lhs))
