"""Pins for the oracle's variance readout y_var[t, j] = Σ_i q_{t,i}² P_{t,i,j},
the per-token belief uncertainty of the layer ("Technische Samenvatting:
Kalman Linear Attention (KLA)", Belangrijkste Bijdragen item 3: the layer
produces an explicit belief-state uncertainty). P is each element's posterior
variance after token t; two independent statements of it pin the readout.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import exact
from bayesian_filtering_linear_gb300.inputs import make_inputs


def _small(T, dk, dv, seed):
    return {n: t.to(torch.float32).numpy() for n, t in make_inputs(1, 1, T, dk, dv, io="f32", seed=seed,
                                                                    random_state=True).items()}


def _run(x, mutant=0):
    return oracle.forward(x["q"], x["k"], x["v"], x["lam_v"], x["a"], x["pbar"], x["lam0"], x["eta0"],
                          want_var=True, _mutant=mutant)


def rls_closed_form(x):
    """a = 1, p̄ = 0: P_t = 1 / (λ0 + Σ_{s≤t} k_s² Λ^v_s) element-wise, so
    y_var[t, j] = Σ_i q_{t,i}² / (λ0_ij + Σ_{s≤t} k_{s,i}² Λ^v_{s,j})."""
    q, k, L = (x[n][0, 0].astype(np.float64) for n in ("q", "k", "lam_v"))
    lam0 = x["lam0"][0, 0].astype(np.float64)
    prec = lam0[None] + np.cumsum(k[:, :, None] ** 2 * L[:, None, :], axis=0)  # [T, dk, dv]
    return np.einsum("ti,tij->tj", q ** 2, 1.0 / prec)


@pytest.mark.parametrize("seed", [1, 2])
def test_variance_readout_without_forgetting_is_the_least_squares_closed_form(seed):
    x = _small(150, 4, 3, seed)
    x["a"][:] = 1.0
    x["pbar"][:] = 0.0
    out = _run(x)
    np.testing.assert_allclose(out["y_var"][0, 0], rls_closed_form(x), rtol=1e-12, atol=0)


def test_variance_readout_matches_dense_gaussian_conditioning():
    """A one-hot q makes y_var[t, j] the posterior variance of element (i, j)
    after token t, which dense conditioning of the joint chain gives."""
    T, dk, dv = 20, 3, 2
    x = _small(T, dk, dv, 31)
    for i in range(dk):
        xi = dict(x)
        xi["q"] = np.zeros_like(x["q"])
        xi["q"][..., i] = 1.0
        out = _run(xi)
        for j in range(dv):
            lam_d, _ = exact.dense_filter_marginals(
                x["a"][0, 0, :, i], x["pbar"][0, 0, :, i], x["k"][0, 0, :, i], x["lam_v"][0, 0, :, j],
                x["v"][0, 0, :, j], float(x["lam0"][0, 0, i, j]), float(x["eta0"][0, 0, i, j]))
            np.testing.assert_allclose(out["y_var"][0, 0, :, j], 1.0 / lam_d, rtol=1e-9, atol=0)


def test_variance_readout_bounds_and_planted_mistake():
    x = _small(64, 4, 4, 7)
    out = _run(x)
    yv = out["y_var"][0, 0]
    q2 = x["q"][0, 0].astype(np.float64) ** 2
    k2L = x["k"][0, 0, :, :, None].astype(np.float64) ** 2 * x["lam_v"][0, 0, :, None, :]
    assert np.all(yv > 0)
    # λ ≥ k²Λ^v, so y_var ≤ Σ_i q_i² / (k_i² Λ^v_j)
    assert np.all(yv <= np.einsum("ti,tij->tj", q2, 1.0 / k2L) * (1 + 1e-12))
    # reading out the prior variance instead of the posterior one is caught by the closed form
    xr = _small(150, 4, 3, 1)
    xr["a"][:] = 1.0
    xr["pbar"][:] = 0.0
    bad = _run(xr, mutant=10)
    assert np.max(np.abs(bad["y_var"][0, 0] / rls_closed_form(xr) - 1)) > 1e-3
