"""Pins for the CPU oracle (no GPU): the fp64 variance-form loop in
``oracle/kla_oracle.cpp`` checked against things that do not depend on it —
a hand-worked example of the printed recursion, exact rational arithmetic of
the information form, dense Gaussian conditioning of the whole chain, closed
forms and invariants.

Source of the model: "Technische Samenvatting: Kalman Linear Attention (KLA)"
(gist.science/nl/paper/2602.10743), Methodologie §1 (OU prior, observation
model, posterior-mean readout) and §2 (Möbius precision recursion,
associativity, affine mean recursion).
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from oracle import exact
from bayesian_filtering_linear_gb300.inputs import make_inputs, WORKLOADS, make_workload

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _np(t):
    return t.to(torch.float32).numpy()


def _small(T, dk, dv, seed, random_state=True, a_logit_mean=2.0):
    return {n: _np(t) for n, t in make_inputs(1, 1, T, dk, dv, io="f32", seed=seed,
                                              a_logit_mean=a_logit_mean,
                                              random_state=random_state).items()}


def _run(x, **kw):
    return oracle.forward(x["q"], x["k"], x["v"], x["lam_v"], x["a"], x["pbar"],
                          x.get("lam0"), x.get("eta0"), **kw)


def test_golden_hand_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "hand_two_tokens.json")))
    inp = g["inputs"]
    ys, lams, etas = exact.information_form_exact(inp["q"], inp["k"], inp["v"], inp["lam_v"],
                                                  inp["a"], inp["pbar"])
    exp = g["expected"]
    assert [l[0][0] for l in lams] == [Fraction(s) for s in exp["lam"]]
    assert [e[0][0] for e in etas] == [Fraction(s) for s in exp["eta"]]
    assert [y[0] for y in ys] == [Fraction(s) for s in exp["y"]]
    shp = lambda key: np.array(inp[key], np.float32).reshape(1, 1, 2, 1)
    out = oracle.forward(shp("q"), shp("k"), shp("v"), shp("lam_v"), shp("a"), shp("pbar"))
    assert np.allclose(out["y"].ravel(), [float(Fraction(s)) for s in exp["y"]], rtol=1e-15, atol=0)
    assert out["lamT"].ravel()[0] == pytest.approx(8.0, rel=1e-15)
    assert out["etaT"].ravel()[0] == pytest.approx(8.0, rel=1e-15)


@pytest.mark.parametrize("seed,T,dk,dv", [(11, 12, 2, 3), (12, 16, 3, 2), (13, 9, 4, 4)])
def test_oracle_matches_exact_rational_information_form(seed, T, dk, dv):
    x = _small(T, dk, dv, seed)
    out = _run(x)
    ys, lams, etas = exact.information_form_exact(x["q"][0, 0], x["k"][0, 0], x["v"][0, 0], x["lam_v"][0, 0],
                                                  x["a"][0, 0], x["pbar"][0, 0], x["lam0"][0, 0], x["eta0"][0, 0])
    y_ex = np.array([[float(e) for e in row] for row in ys])
    lam_ex = np.array([[float(e) for e in row] for row in lams[-1]])
    eta_ex = np.array([[float(e) for e in row] for row in etas[-1]])
    assert np.max(np.abs(out["y"][0, 0] - y_ex) / out["y_scale"][0, 0]) < 1e-13
    assert np.max(np.abs(out["lamT"][0, 0] - lam_ex) / lam_ex) < 1e-13
    assert np.max(np.abs(out["etaT"][0, 0] - eta_ex) / out["eta_scale"][0, 0]) < 1e-13
    assert out["violations"] == 0


@pytest.mark.parametrize("seed", [21, 22, 23])
def test_oracle_matches_dense_gaussian_conditioning(seed):
    """A one-hot q makes y[t, j] the posterior mean of element (i, j) after
    token t, which dense conditioning of the joint chain gives independently."""
    T, dk, dv = 24, 3, 2
    x = _small(T, dk, dv, seed)
    for i in range(dk):
        xi = dict(x)
        xi["q"] = np.zeros_like(x["q"])
        xi["q"][..., i] = 1.0
        out = _run(xi)
        for j in range(dv):
            lam_d, mu_d = exact.dense_filter_marginals(
                x["a"][0, 0, :, i], x["pbar"][0, 0, :, i], x["k"][0, 0, :, i],
                x["lam_v"][0, 0, :, j], x["v"][0, 0, :, j],
                float(x["lam0"][0, 0, i, j]), float(x["eta0"][0, 0, i, j]))
            assert np.allclose(out["y"][0, 0, :, j], mu_d, rtol=1e-9, atol=1e-11)
            assert out["lamT"][0, 0, i, j] == pytest.approx(lam_d[-1], rel=1e-10)
            assert out["etaT"][0, 0, i, j] == pytest.approx(lam_d[-1] * mu_d[-1], rel=1e-9, abs=1e-11)


def test_closed_form_no_forgetting_is_recursive_least_squares():
    """a = 1, p̄ = 0: λ_T = λ0 + Σ k²Λ^v and η_T = η0 + Σ kΛ^v v."""
    x = _small(200, 4, 3, 31)
    x["a"][:] = 1.0
    x["pbar"][:] = 0.0
    out = _run(x)
    k, L, v = x["k"][0, 0].astype(np.float64), x["lam_v"][0, 0].astype(np.float64), x["v"][0, 0].astype(np.float64)
    lam_cf = x["lam0"][0, 0] + np.einsum("ti,tj->ij", k * k, L)
    eta_cf = x["eta0"][0, 0] + np.einsum("ti,tj->ij", k, L * v)
    assert np.allclose(out["lamT"][0, 0], lam_cf, rtol=1e-12)
    assert np.allclose(out["etaT"][0, 0], eta_cf, rtol=1e-10, atol=1e-12)


def test_closed_form_constant_coefficients_reach_riccati_fixed_point():
    T = 3000
    a, pbar, k, L = 0.9, 0.05, 0.7, 1.3
    sh = (1, 1, T, 1)
    x = {"q": np.ones(sh, np.float32), "k": np.full(sh, k, np.float32), "v": np.zeros(sh, np.float32),
         "lam_v": np.full(sh, L, np.float32), "a": np.full(sh, a, np.float32),
         "pbar": np.full(sh, pbar, np.float32)}
    out = _run(x)
    f = lambda z: float(np.float32(z))
    lam_star = exact.riccati_fixed_point(f(a), f(pbar), f(k) * f(k) * f(L))
    assert out["lamT"].ravel()[0] == pytest.approx(lam_star, rel=1e-12)


def test_closed_form_no_observations_relax_to_stationary_ou_prior():
    """Λ^v = 0: λ_t → (1 − a²)/p̄ and the mean decays as μ_T = a^T μ0."""
    T = 400
    a, pbar = np.float32(0.95), np.float32(0.02)
    sh = (1, 1, T, 1)
    x = {"q": np.ones(sh, np.float32), "k": np.full(sh, 0.3, np.float32), "v": np.ones(sh, np.float32),
         "lam_v": np.zeros(sh, np.float32), "a": np.full(sh, a, np.float32),
         "pbar": np.full(sh, pbar, np.float32),
         "lam0": np.full((1, 1, 1, 1), 5.0, np.float32), "eta0": np.full((1, 1, 1, 1), 10.0, np.float32)}
    out = _run(x)
    a64, p64 = float(a), float(pbar)
    assert out["lamT"].ravel()[0] == pytest.approx((1 - a64 * a64) / p64, rel=1e-12)
    mu_T = out["etaT"].ravel()[0] / out["lamT"].ravel()[0]
    assert mu_T == pytest.approx(a64 ** T * 2.0, rel=1e-12)
    assert out["y"].ravel()[-1] == pytest.approx(mu_T, rel=1e-12)


def test_mobius_composition_is_associative_and_matches_sequential():
    x = _small(10, 1, 1, 41)
    lam0 = Fraction(float(x["lam0"].ravel()[0]))
    mats, lam = [], lam0
    for t in range(10):
        a, p, kk, L = (Fraction(float(x[n][0, 0, t, 0])) for n in ("a", "pbar", "k", "lam_v"))
        al, be, ga, de = exact.mobius_coefficients(a, p, kk * kk * L)
        mats.append([[al, be], [ga, de]])
        lam = exact.apply_mobius(mats[-1], lam)
    assert exact.apply_mobius(exact.compose_mobius(mats), lam0) == lam
    left = exact.compose_mobius([exact.compose_mobius(mats[:4]), exact.compose_mobius(mats[4:])])
    assert exact.apply_mobius(left, lam0) == lam
    out = _run(x)
    assert out["lamT"].ravel()[0] == pytest.approx(float(lam), rel=1e-13)


def test_invariants_hold_on_the_tiny_workload():
    x = {n: _np(t) for n, t in make_workload("tiny").items()}
    out = _run(x)
    assert out["violations"] == 0
    assert np.all(out["lamT"] > 0)
    last_c = (x["k"][0, 0, -1][:, None] ** 2) * x["lam_v"][0, 0, -1][None, :]
    assert np.all(out["lamT"][0, 0] >= last_c * (1 - 1e-12))
    bound = 1.0 / x["pbar"][0, 0, -1][:, None] + last_c
    assert np.all(out["lamT"][0, 0] <= bound * (1 + 1e-12))


def test_readout_is_linear_in_q_and_state_scales_with_v():
    x = _small(64, 4, 4, 51, random_state=False)
    rng = np.random.default_rng(5)
    # dyadic q rows so that q1 + q2 is exact in fp32
    q1 = (rng.integers(-64, 64, x["q"].shape) / 64.0).astype(np.float32)
    q2 = (rng.integers(-64, 64, x["q"].shape) / 64.0).astype(np.float32)
    o1, o2 = _run(dict(x, q=q1)), _run(dict(x, q=q2))
    o12 = _run(dict(x, q=q1 + q2))
    scale = o1["y_scale"] + o2["y_scale"]
    assert np.max(np.abs(o12["y"] - o1["y"] - o2["y"]) / scale) < 1e-13
    o = _run(x)
    o4 = _run(dict(x, v=x["v"] * 4.0))
    assert np.allclose(o4["etaT"], 4 * o["etaT"], rtol=1e-12, atol=1e-14)
    assert np.allclose(o4["y"], 4 * o["y"], rtol=1e-12, atol=1e-14)
    assert np.array_equal(o4["lamT"], o["lamT"])


def test_permuting_rows_permutes_state_and_keeps_readout():
    x = _small(50, 6, 3, 61)
    perm = np.array([3, 0, 5, 1, 4, 2])
    xp = dict(x)
    for n in ("q", "k", "a", "pbar"):
        xp[n] = np.ascontiguousarray(x[n][..., perm])
    for n in ("lam0", "eta0"):
        xp[n] = np.ascontiguousarray(x[n][:, :, perm, :])
    o, op = _run(x), _run(xp)
    assert np.array_equal(op["lamT"], o["lamT"][:, :, perm, :])
    assert np.array_equal(op["etaT"], o["etaT"][:, :, perm, :])
    assert np.allclose(op["y"], o["y"], rtol=0, atol=1e-13 * np.max(o["y_scale"]))


def test_heads_are_independent_and_thread_count_does_not_matter():
    x = {n: _np(t) for n, t in make_inputs(2, 3, 40, 16, 16, io="f32", seed=71, random_state=True).items()}
    full = _run(x, nthreads=4)
    one = _run(x, nthreads=1)
    for key in ("y", "lamT", "etaT"):
        assert np.array_equal(full[key], one[key])
    sub = _run(x, heads=[4, 1])
    assert np.array_equal(sub["y"][0, 0], full["y"][1, 1])
    assert np.array_equal(sub["lamT"][1, 0], full["lamT"][0, 1])


def test_fp32_build_tracks_fp64():
    x = {n: _np(t) for n, t in make_workload("tiny").items()}
    o64 = _run(x)
    o32 = _run(x, precision="f32")
    assert np.max(np.abs(o32["y"] - o64["y"]) / o64["y_scale"]) < 1e-5
    assert np.max(np.abs(o32["lamT"] - o64["lamT"]) / o64["lamT"]) < 1e-5


def test_workload_recipe_shapes_and_ranges():
    w = WORKLOADS["tiny"]
    x = make_workload(w)
    assert x["q"].shape == (1, 1, 256, 16) and x["v"].shape == (1, 1, 256, 16)
    assert float(x["a"].min()) > 0 and float(x["a"].max()) < 1
    assert float(x["pbar"].min()) > 0 and float(x["lam_v"].min()) > 0
    assert abs(float(x["q"].std()) - 0.25) < 0.02
    y = make_workload(w)
    assert all(torch.equal(x[n], y[n]) for n in x)


MUTANTS = {1: "dropped p̄ in the predict", 2: "a instead of a² in the predict",
           3: "k instead of k² in the observation precision", 4: "prior mean read out",
           5: "Λ^v missing from the information term", 6: "prior variance in the mean update"}


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_pins_catch_planted_mistakes(mutant):
    """Each planted mistake in a copy of the oracle must fail the exact-rational
    pin or the dense-conditioning pin (the sensitivity of the pins)."""
    T, dk, dv = 12, 2, 3
    x = _small(T, dk, dv, 81)
    ys, lams, etas = exact.information_form_exact(x["q"][0, 0], x["k"][0, 0], x["v"][0, 0], x["lam_v"][0, 0],
                                                  x["a"][0, 0], x["pbar"][0, 0], x["lam0"][0, 0], x["eta0"][0, 0])
    y_ex = np.array([[float(e) for e in row] for row in ys])
    lam_ex = np.array([[float(e) for e in row] for row in lams[-1]])
    good = _run(x)
    bad = _run(x, _mutant=mutant)
    err = lambda o: max(np.max(np.abs(o["y"][0, 0] - y_ex) / good["y_scale"][0, 0]),
                        np.max(np.abs(o["lamT"][0, 0] - lam_ex) / lam_ex))
    assert err(good) < 1e-13
    assert err(bad) > 1e-6, MUTANTS[mutant]
