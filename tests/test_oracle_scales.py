"""Pins of the oracle's condition scales (no GPU).

Every GPU parity test divides its error by a condition scale that the oracle
returns beside the result: for y, Σ_i |q_i| μ̂_ij with μ̂ the mean recursion
run on absolute values; for η_T, μ̂/P; for each gradient, the reverse-mode
recursion with every term in absolute value. A mistake that inflated these
scales would loosen every parity check without failing one, so they are
pinned here against what the mathematics fixes.

Where every term that the scale takes in absolute value is already
non-negative, the scale and the magnitude of the value are the same sum of
the same terms in the same order, so they are equal bit for bit:

* forward — q, k, v > 0, Λ^v > 0, 0 < a, η0 ≥ 0: every term of the mean
  recursion (a·μ, k·Λ^v·v) and of the readout (q·μ) is ≥ 0, so
  y_scale == y and eta_scale == η_T;
* backward, the mean adjoint — the same inputs and dL/dy ≥ 0, dL/dη_T ≥ 0:
  the adjoint of μ only ever adds q·dy ≥ 0 and multiplies by w, a > 0, so
  |dq|, |dv|, |dη0| equal their scales;
* backward, the variance adjoint — with Λ^v = 0 (nothing observed: c = b = 0,
  w = 1), v = 0 and dL/dλ_T ≤ 0, dL/dη_T = 0, the adjoint of P stays ≥ 0 and
  the terms of da, dp̄, dλ0 and dΛ^v each keep one sign;
* backward, dk — one token (T = 1) with v = 0, dL/dλ_T ≤ 0 and dL/dη_T = 0:
  dk = 2kΛ^v·c̄ with c̄ = −w̄P⁻w² ≤ 0, a single signed term.

Together these fix all eight gradient scales and both forward scales, and
planted mistakes that inflate one of them (a copy of the oracle built with
one change) must break an equality. On random inputs the scales bound the
values from above.

The filter: "Technische Samenvatting: Kalman Linear Attention (KLA)"
(gist.science/nl/paper/2602.10743), Methodologie §1–§2; the gradient is the
exact reverse-mode derivative of that scan.
"""
import numpy as np
import pytest

import oracle

ORDER = ("q", "k", "v", "lam_v", "a", "pbar", "lam0", "eta0")
GRADS = ("dq", "dk", "da", "dpbar", "dv", "dlam_v", "dlam0", "deta0")


def positive_problem(B=2, H=2, T=24, dk=4, dv=3, seed=0):
    """Inputs on which every term of the forward mean recursion is ≥ 0."""
    rng = np.random.default_rng(seed)
    r = lambda *s: rng.standard_normal(s).astype(np.float32)
    sp = lambda x: np.log1p(np.exp(x)).astype(np.float32)
    return {"q": np.abs(r(B, H, T, dk)) + 0.01, "k": np.abs(r(B, H, T, dk)) + 0.01,
            "v": np.abs(r(B, H, T, dv)) + 0.01, "lam_v": sp(r(B, H, T, dv)),
            "a": (1 / (1 + np.exp(-r(B, H, T, dk) - 2))).astype(np.float32), "pbar": sp(r(B, H, T, dk) - 2),
            "lam0": (0.5 + sp(r(B, H, dk, dv))).astype(np.float32), "eta0": np.abs(r(B, H, dk, dv))}


def fwd(x, mutant=0):
    return oracle.forward(*(x[n] for n in ORDER), _mutant=mutant)


def bwd(x, dy, dlamT, detaT, mutant=0):
    return oracle.backward(*(x[n] for n in ORDER), dy, dlamT, detaT, _mutant=mutant)


def forward_equalities(mutant=0):
    x = positive_problem()
    o = fwd(x, mutant)
    return {"y": np.array_equal(o["y_scale"], o["y"]), "eta": np.array_equal(o["eta_scale"], o["etaT"])}


def backward_equalities(mutant=0):
    """Which gradient scales equal |gradient| exactly on the sign-definite
    problems described in the module docstring."""
    rng = np.random.default_rng(1)
    ok = {}
    # the mean adjoint: positive forward, dy ≥ 0, dη_T ≥ 0 (dλ_T arbitrary)
    x = positive_problem(seed=2)
    B, H, T, dk = x["q"].shape
    dv = x["v"].shape[-1]
    dy = np.abs(rng.standard_normal((B, H, T, dv))).astype(np.float32)
    dl = rng.standard_normal((B, H, dk, dv)).astype(np.float32)
    de = np.abs(rng.standard_normal((B, H, dk, dv))).astype(np.float32)
    g = bwd(x, dy, dl, de, mutant)
    for n in ("dq", "dv", "deta0"):
        ok[n] = np.array_equal(np.abs(g[n]), g[n + "_scale"])
    # the variance adjoint: nothing observed (Λ^v = 0), v = 0, dλ_T ≤ 0, dη_T = 0
    x = positive_problem(seed=3)
    x["lam_v"][:] = 0.0
    x["v"][:] = 0.0
    g = bwd(x, dy, -np.abs(dl), np.zeros_like(de), mutant)
    for n in ("da", "dpbar", "dlam0", "dlam_v"):
        ok[n] = np.array_equal(np.abs(g[n]), g[n + "_scale"])
    # dk: one token, v = 0, dλ_T ≤ 0, dη_T = 0
    x = positive_problem(T=1, seed=4)
    x["v"][:] = 0.0
    g = bwd(x, dy[:, :, :1], -np.abs(dl), np.zeros_like(de), mutant)
    ok["dk"] = np.array_equal(np.abs(g["dk"]), g["dk_scale"])
    assert np.any(g["dk"] != 0)
    return ok


def test_forward_scales_equal_the_values_when_every_term_is_non_negative():
    assert all(forward_equalities().values()), forward_equalities()


def test_backward_scales_equal_the_gradients_on_sign_definite_problems():
    eq = backward_equalities()
    assert sorted(eq) == sorted(GRADS)
    assert all(eq.values()), eq


def test_scales_bound_the_values_on_random_inputs():
    rng = np.random.default_rng(5)
    B, H, T, dk, dv = 2, 3, 40, 8, 8
    x = {"q": rng.standard_normal((B, H, T, dk)), "k": rng.standard_normal((B, H, T, dk)),
         "v": rng.standard_normal((B, H, T, dv)), "lam_v": np.log1p(np.exp(rng.standard_normal((B, H, T, dv)))),
         "a": 1 / (1 + np.exp(-rng.standard_normal((B, H, T, dk)) - 2)),
         "pbar": np.log1p(np.exp(rng.standard_normal((B, H, T, dk)) - 2)),
         "lam0": 0.5 + np.log1p(np.exp(rng.standard_normal((B, H, dk, dv)))),
         "eta0": rng.standard_normal((B, H, dk, dv))}
    x = {n: t.astype(np.float32) for n, t in x.items()}
    o = fwd(x)
    assert np.all(np.abs(o["y"]) <= o["y_scale"] * (1 + 1e-12))
    assert np.all(np.abs(o["etaT"]) <= o["eta_scale"] * (1 + 1e-12))
    # the scale is a sum of the same magnitudes, so cancellation shows up as
    # scale > |value| somewhere on random signs
    assert np.any(o["y_scale"] > 1.5 * np.abs(o["y"]))


# Planted inflated scales (oracle/kla_oracle.cpp, KLA_ORACLE_MUTANT):
FORWARD_SCALE_MUTANTS = {11: "|q| counted twice in y_scale", 12: "|k Λ^v v| counted twice in the mean's scale"}
BACKWARD_SCALE_MUTANTS = {13: "dq scale doubled", 14: "carried variance adjoint counted twice in the scale",
                          15: "scale of the observation-precision adjoint doubled"}


@pytest.mark.parametrize("mutant", sorted(FORWARD_SCALE_MUTANTS))
def test_inflated_forward_scale_breaks_the_equality(mutant):
    eq = forward_equalities(mutant)
    assert not all(eq.values()), FORWARD_SCALE_MUTANTS[mutant]
    # and the results themselves are unchanged: only the scale is wrong
    x = positive_problem()
    good, bad = fwd(x), fwd(x, mutant)
    for n in ("y", "lamT", "etaT"):
        np.testing.assert_array_equal(good[n], bad[n])


@pytest.mark.parametrize("mutant", sorted(BACKWARD_SCALE_MUTANTS))
def test_inflated_backward_scale_breaks_an_equality(mutant):
    eq = backward_equalities(mutant)
    assert not all(eq.values()), BACKWARD_SCALE_MUTANTS[mutant]
