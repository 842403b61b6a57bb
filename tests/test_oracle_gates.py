"""Pins for the oracle's gate activations (oracle/gates.py): the gated
forward is the plain forward on (softplus, sigmoid, OU-tied) transformed
inputs ("Technische Samenvatting: Kalman Linear Attention (KLA)",
Methodologie §1: a ∈ (0, 1), p̄ > 0, Λ^v > 0; an exactly discretised OU
process has p̄ = s(1 − a²)), and its gradient with respect to the
pre-activations — backward plus the chain rule — must match central finite
differences of that gated forward.
"""
import numpy as np
import pytest

import oracle
from oracle import gates as G

ORDER = ("q", "k", "v", "lam_v", "a", "pbar", "lam0", "eta0")


def problem(seed, B=1, H=2, T=9, dk=3, dv=2):
    rng = np.random.default_rng(seed)
    r = lambda *s: rng.standard_normal(s)
    x = {"q": r(B, H, T, dk) / 2, "k": r(B, H, T, dk) / 2, "v": r(B, H, T, dv), "lam_v": r(B, H, T, dv),
         "a": r(B, H, T, dk) + 2.0, "pbar": r(B, H, T, dk) - 1.0,
         "lam0": 0.5 + np.exp(r(B, H, dk, dv)), "eta0": r(B, H, dk, dv)}
    up = {"dy": r(B, H, T, dv), "dlamT": r(B, H, dk, dv), "detaT": r(B, H, dk, dv)}
    return x, up


def gated_inputs(x, gates):
    L, A, Pb = G.apply(x["lam_v"], x["a"], x["pbar"], gates)
    return dict(x, lam_v=L, a=A, pbar=Pb)


def loss(x, up, gates):
    f = oracle.forward64(*(gated_inputs(x, gates)[n] for n in ORDER))
    return (f["y"] * up["dy"]).sum() + (f["lamT"] * up["dlamT"]).sum() + (f["etaT"] * up["detaT"]).sum()


def gated_grads(x, up, gates, mutant=0):
    xg = gated_inputs(x, gates)
    g = oracle.backward64(*(xg[n] for n in ORDER), up["dy"], up["dlamT"], up["detaT"])
    gL, ga, gp = G.chain(g["dlam_v"], g["da"], g["dpbar"], x["lam_v"], x["a"], x["pbar"], gates, _mutant=mutant)
    return {"lam_v": gL, "a": ga, "pbar": gp}


def fd(x, up, gates, name):
    base = x[name]
    out = np.zeros_like(base)
    for idx in np.ndindex(base.shape):
        h = 1e-6 * max(1.0, abs(base[idx]))
        xp, xm = dict(x), dict(x)
        xp[name] = base.copy()
        xm[name] = base.copy()
        xp[name][idx] += h
        xm[name][idx] -= h
        out[idx] = (loss(xp, up, gates) - loss(xm, up, gates)) / (2 * h)
    return out


@pytest.mark.parametrize("gates", [G.LAMV_SOFTPLUS | G.A_SIGMOID | G.PBAR_SOFTPLUS,
                                   G.LAMV_SOFTPLUS | G.A_SIGMOID | G.PBAR_OU, G.PBAR_OU, G.A_SIGMOID])
def test_gated_gradients_match_finite_differences(gates):
    x, up = problem(3)
    g = gated_grads(x, up, gates)
    for name in ("lam_v", "a", "pbar"):
        want = fd(x, up, gates, name)
        assert np.abs(g[name] - want).max() <= 1e-6 * max(np.abs(want).max(), 1e-12), (gates, name)


def test_planted_chain_rule_mistake_is_caught():
    x, up = problem(4)
    gates = G.A_SIGMOID | G.PBAR_OU
    g = gated_grads(x, up, gates, mutant=1)
    want = fd(x, up, gates, "a")
    assert np.abs(g["a"] - want).max() > 1e-3 * np.abs(want).max()


def test_activation_identities():
    x = np.linspace(-30.0, 30.0, 601)
    assert G.softplus(np.array(0.0)) == pytest.approx(np.log(2.0), rel=1e-15)
    assert np.allclose(G.softplus(x) - G.softplus(-x), x, rtol=1e-13, atol=1e-13)
    assert np.allclose(G.sigmoid(x) + G.sigmoid(-x), 1.0, rtol=0, atol=1e-15)
    L, A, Pb = G.apply(np.array(0.0), np.array(0.0), np.array(0.0), G.LAMV_SOFTPLUS | G.A_SIGMOID | G.PBAR_OU)
    assert (L, A) == (pytest.approx(np.log(2.0)), 0.5)
    assert Pb == pytest.approx(np.log(2.0) * 0.75)
