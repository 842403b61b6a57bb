"""Property-based checks of the oracles (hypothesis; CPU only): on randomly
drawn small problems anywhere in the model's domain — a ∈ (0, 1], p̄ ≥ 0,
Λ^v ≥ 0 (zeros included), any k, q, v, λ0 > 0 — the fp64 scan equals the
exact-rational information form, keeps its invariants, is linear in q and
restarts exactly from its own final state; the causal convolution is causal,
linear without bias and activation, streams exactly, and its backward is the
adjoint of the forward.

Source: "Technische Samenvatting: Kalman Linear Attention (KLA)",
Methodologie §1–§2 (the filter), §4 (the block's causal convolution).
"""
import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

import oracle  # noqa: E402
from oracle import conv as C  # noqa: E402
from oracle import exact  # noqa: E402

SETTINGS = settings(max_examples=30, deadline=None, derandomize=True)


@st.composite
def problems(draw, max_T=6, max_d=3):
    T = draw(st.integers(1, max_T))
    dk = draw(st.integers(1, max_d))
    dv = draw(st.integers(1, max_d))
    seed = draw(st.integers(0, 2**31 - 1))
    rng = np.random.default_rng(seed)
    zero_some = draw(st.booleans())

    def maybe_zero(x):
        if zero_some:
            x[rng.random(x.shape) < 0.25] = 0.0
        return x

    return {
        "q": rng.uniform(-3, 3, (1, 1, T, dk)), "k": maybe_zero(rng.uniform(-3, 3, (1, 1, T, dk))),
        "v": rng.uniform(-3, 3, (1, 1, T, dv)), "lam_v": maybe_zero(rng.uniform(0, 4, (1, 1, T, dv))),
        "a": rng.uniform(0.05, 1.0, (1, 1, T, dk)), "pbar": maybe_zero(rng.uniform(0, 4, (1, 1, T, dk))),
        "lam0": rng.uniform(0.1, 10, (1, 1, dk, dv)), "eta0": rng.uniform(-3, 3, (1, 1, dk, dv)),
    }


ORDER = ("q", "k", "v", "lam_v", "a", "pbar", "lam0", "eta0")


def run(x, **kw):
    return oracle.forward64(*(x[n] for n in ORDER), want_scales=True, **kw)


@SETTINGS
@given(problems())
def test_fp64_scan_equals_the_exact_information_form(x):
    out = run(x)
    ys, lams, etas = exact.information_form_exact(*(x[n][0, 0] for n in ORDER))
    y_ex = np.array([[float(e) for e in row] for row in ys])
    lam_ex = np.array([[float(e) for e in row] for row in lams[-1]])
    eta_ex = np.array([[float(e) for e in row] for row in etas[-1]])
    assert np.all(np.abs(out["y"][0, 0] - y_ex) <= 1e-11 * (out["y_scale"][0, 0] + 1e-300))
    assert np.all(np.abs(out["lamT"][0, 0] - lam_ex) <= 1e-11 * lam_ex)
    assert np.all(np.abs(out["etaT"][0, 0] - eta_ex) <= 1e-11 * (out["eta_scale"][0, 0] + 1e-300))


@SETTINGS
@given(problems())
def test_invariants_of_the_final_precision(x):
    out = run(x)
    lam = out["lamT"][0, 0]
    c = x["k"][0, 0, -1][:, None] ** 2 * x["lam_v"][0, 0, -1][None, :]
    pb = x["pbar"][0, 0, -1][:, None]
    assert np.all(lam > 0)
    assert np.all(lam >= c * (1 - 1e-12))
    ok = pb > 0
    bound = np.where(ok, 1.0 / np.where(ok, pb, 1.0) + c, np.inf)
    assert np.all(lam <= bound * (1 + 1e-12))


@SETTINGS
@given(problems(), st.floats(-2, 2), st.floats(-2, 2))
def test_readout_is_linear_in_q(x, alpha, beta):
    x2 = dict(x, q=np.random.default_rng(1).uniform(-3, 3, x["q"].shape))
    mix = dict(x, q=alpha * x["q"] + beta * x2["q"])
    y1, y2, ym = run(x)["y"], run(x2)["y"], run(mix)
    want = alpha * y1 + beta * y2
    assert np.all(np.abs(ym["y"] - want) <= 1e-12 * (np.abs(alpha) * run(x)["y_scale"] +
                                                   np.abs(beta) * run(x2)["y_scale"] + ym["y_scale"] + 1e-300))


@SETTINGS
@given(problems(max_T=8), st.data())
def test_restarting_from_the_final_state_equals_one_pass(x, data):
    T = x["q"].shape[2]
    t1 = data.draw(st.integers(0, T))
    full = run(x)
    first = run({n: (x[n][:, :, :t1] if n not in ("lam0", "eta0") else x[n]) for n in ORDER})
    rest = {n: x[n][:, :, t1:] for n in ORDER if n not in ("lam0", "eta0")}
    second = run(dict(rest, lam0=first["lamT"], eta0=first["etaT"]))
    assert np.allclose(np.concatenate([first["y"], second["y"]], axis=2), full["y"], rtol=0,
                       atol=1e-12 * (full["y_scale"].max() + 1e-300))
    assert np.allclose(second["lamT"], full["lamT"], rtol=1e-12, atol=0)


@st.composite
def conv_problems(draw):
    B, H = draw(st.integers(1, 2)), draw(st.integers(1, 2))
    T, D, W = draw(st.integers(0, 9)), draw(st.integers(1, 3)), draw(st.integers(1, 5))
    rng = np.random.default_rng(draw(st.integers(0, 2**31 - 1)))
    return {"x": rng.standard_normal((B, H, T, D)), "weight": rng.standard_normal((H, D, W)),
            "bias": rng.standard_normal((H, D)), "window": rng.standard_normal((B, H, W - 1, D))}


@SETTINGS
@given(conv_problems(), st.data())
def test_convolution_is_causal(p, data):
    T = p["x"].shape[2]
    if T == 0:
        return
    t0 = data.draw(st.integers(0, T - 1))
    y, _ = C.conv(p["x"], p["weight"], p["bias"], p["window"])
    x2 = p["x"].copy()
    x2[:, :, t0:] += 1.0
    y2, _ = C.conv(x2, p["weight"], p["bias"], p["window"])
    assert np.array_equal(y2[:, :, :t0], y[:, :, :t0])


@SETTINGS
@given(conv_problems(), st.floats(-2, 2))
def test_plain_convolution_is_linear(p, alpha):
    x2 = np.random.default_rng(2).standard_normal(p["x"].shape)
    y1, _ = C.conv(p["x"], p["weight"], None, None, activation=False)
    y2, _ = C.conv(x2, p["weight"], None, None, activation=False)
    ym, _ = C.conv(alpha * p["x"] + x2, p["weight"], None, None, activation=False)
    scale = C.preactivation(np.abs(alpha * p["x"]) + np.abs(x2), np.abs(p["weight"]))
    assert np.all(np.abs(ym - (alpha * y1 + y2)) <= 1e-13 * (scale + 1e-300))


@SETTINGS
@given(conv_problems(), st.data())
def test_convolution_streams_exactly(p, data):
    T = p["x"].shape[2]
    t1 = data.draw(st.integers(0, T))
    y, win = C.conv(p["x"], p["weight"], p["bias"], p["window"])
    ya, wa = C.conv(p["x"][:, :, :t1], p["weight"], p["bias"], p["window"])
    yb, wb = C.conv(p["x"][:, :, t1:], p["weight"], p["bias"], wa)
    assert np.array_equal(np.concatenate([ya, yb], axis=2), y)
    assert np.array_equal(wb, win)


@SETTINGS
@given(conv_problems())
def test_convolution_backward_is_the_adjoint(p):
    rng = np.random.default_rng(3)
    dx, dwin = rng.standard_normal(p["x"].shape), rng.standard_normal(p["window"].shape)
    gy, gwo = rng.standard_normal(p["x"].shape), rng.standard_normal(p["window"].shape)
    jy, jw = C.conv(dx, p["weight"], None, dwin, activation=False)
    g = C.conv_backward(p["x"], p["weight"], None, p["window"], gy, gwo, activation=False)
    lhs = (gy * jy).sum() + (gwo * jw).sum()
    rhs = (g["gx"] * dx).sum() + (g["gwindow"] * dwin).sum()
    assert abs(lhs - rhs) <= 1e-12 * (1 + abs(lhs) + np.abs(gy).sum() + np.abs(gwo).sum())
