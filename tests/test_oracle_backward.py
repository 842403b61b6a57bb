"""Pins of the oracle's backward (reverse-mode derivative of the scan).

The pages define only the forward scan ("Technische Samenvatting: Kalman
Linear Attention (KLA)", Methodologie §1–§2); the gradient is its exact
derivative. The pin is numerical differentiation of the fp64 forward oracle
(itself pinned in test_oracle_pins.py): central differences of
L = Σ dy·y + Σ dλ_T·λ_T + Σ dη_T·η_T with respect to every input entry must
match the backward to ~1e-6 (the finite-difference truncation and rounding
error at h ≈ 1e-6 is far below that). Planted mistakes in the backward fail it.
"""
import numpy as np
import pytest

import oracle

ORDER = ("q", "k", "v", "lam_v", "a", "pbar", "lam0", "eta0")
GRAD = {"q": "dq", "k": "dk", "v": "dv", "lam_v": "dlam_v", "a": "da", "pbar": "dpbar", "lam0": "dlam0",
        "eta0": "deta0"}


def problem(B=1, H=2, T=7, dk=3, dv=2, seed=0, state=True):
    rng = np.random.default_rng(seed)
    r = lambda *s: rng.standard_normal(s)
    sp = lambda x: np.log1p(np.exp(x))
    x = {"q": r(B, H, T, dk) / 2, "k": r(B, H, T, dk) / 2, "v": r(B, H, T, dv), "lam_v": sp(r(B, H, T, dv)),
         "a": 1 / (1 + np.exp(-r(B, H, T, dk) - 2)), "pbar": sp(r(B, H, T, dk) - 2),
         "lam0": 0.5 + sp(r(B, H, dk, dv)) if state else np.ones((B, H, dk, dv)),
         "eta0": r(B, H, dk, dv) if state else np.zeros((B, H, dk, dv))}
    up = {"dy": r(B, H, T, dv), "dlamT": r(B, H, dk, dv), "detaT": r(B, H, dk, dv)}
    return x, up


def loss(x, up):
    f = oracle.forward64(*(x[n] for n in ORDER))
    total = (f["y"] * up["dy"]).sum()
    if up.get("dlamT") is not None:
        total += (f["lamT"] * up["dlamT"]).sum()
    if up.get("detaT") is not None:
        total += (f["etaT"] * up["detaT"]).sum()
    return total


def finite_differences(x, up, name):
    base = x[name]
    fd = np.zeros_like(base)
    for idx in np.ndindex(base.shape):
        h = 1e-6 * max(1.0, abs(base[idx]))
        xp, xm = dict(x), dict(x)
        xp[name] = base.copy()
        xm[name] = base.copy()
        xp[name][idx] += h
        xm[name][idx] -= h
        fd[idx] = (loss(xp, up) - loss(xm, up)) / (2 * h)
    return fd


def rel_err(got, want):
    return float(np.abs(got - want).max() / max(np.abs(want).max(), 1e-300))


@pytest.mark.parametrize("name", ORDER)
def test_backward_matches_finite_differences(name):
    x, up = problem()
    g = oracle.backward64(*(x[n] for n in ORDER), up["dy"], up["dlamT"], up["detaT"])
    assert rel_err(g[GRAD[name]], finite_differences(x, up, name)) < 1e-6


def test_backward_without_state_gradients_matches_finite_differences():
    # dλ_T = dη_T = 0 and the default start (λ0 = 1, η0 = 0), a longer sequence
    x, up = problem(B=1, H=1, T=20, dk=2, dv=3, seed=5, state=False)
    up["dlamT"] = up["detaT"] = None
    g = oracle.backward64(*(x[n] for n in ORDER), up["dy"])
    for name in ("a", "pbar", "k", "lam_v"):
        assert rel_err(g[GRAD[name]], finite_differences(x, up, name)) < 1e-6, name


@pytest.mark.parametrize("mutant", [7, 8, 9])
def test_planted_backward_mistakes_fail_the_pin(mutant):
    x, up = problem(seed=2)
    g = oracle.backward64(*(x[n] for n in ORDER), up["dy"], up["dlamT"], up["detaT"], _mutant=mutant)
    worst = max(rel_err(g[GRAD[n]], finite_differences(x, up, n)) for n in ("a", "pbar", "k", "lam0"))
    assert worst > 1e-3


def test_float_and_double_input_paths_agree_and_scales_bound_the_gradients():
    x, up = problem(B=2, H=2, T=33, dk=4, dv=4, seed=7)
    x32 = {n: t.astype(np.float32) for n, t in x.items()}
    up32 = {n: t.astype(np.float32) for n, t in up.items()}
    g = oracle.backward(*(x32[n] for n in ORDER), up32["dy"], up32["dlamT"], up32["detaT"])
    g64 = oracle.backward64(*(x32[n].astype(np.float64) for n in ORDER),
                            *(up32[n].astype(np.float64) for n in ("dy", "dlamT", "detaT")))
    for n in oracle.GRAD_NAMES:
        np.testing.assert_array_equal(g[n], g64[n])
        assert np.all(np.abs(g[n]) <= g[n + "_scale"] * (1 + 1e-12) + 1e-300), n


def test_backward_selected_heads_match_the_full_batch():
    x, up = problem(B=2, H=3, T=9, dk=2, dv=2, seed=11)
    x32 = {n: t.astype(np.float32) for n, t in x.items()}
    full = oracle.backward(*(x32[n] for n in ORDER), up["dy"].astype(np.float32))
    part = oracle.backward(*(x32[n] for n in ORDER), up["dy"].astype(np.float32), heads=[1, 4])
    for n in oracle.GRAD_NAMES:
        flat = full[n].reshape((6,) + full[n].shape[2:])
        np.testing.assert_array_equal(part[n][:, 0], flat[[1, 4]])
