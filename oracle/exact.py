"""Independent checkers for the oracle — TEST INFRASTRUCTURE ONLY.

Two restatements of the filter that share no arithmetic with ``kla_oracle.cpp``:

* :func:`information_form_exact` — the information-form recursion exactly as
  the summary prints it ("Technische Samenvatting: Kalman Linear Attention
  (KLA)", Methodologie §2 "Parallelisatie via Möbius-transformaties": the
  precision is a Möbius map of the previous precision, the information mean
  follows an affine map), evaluated in exact rational arithmetic
  (``fractions.Fraction``), so its only error is none.
* :func:`dense_filter_marginals` — exact Bayesian filtering by brute force:
  build the joint Gaussian of the whole chain z_0..z_t of one state element
  (Methodologie §1: OU prior with process noise p̄, observation of the token
  through k with value precision Λ^v), condition on the observations up to t
  with a dense linear solve, and read off the marginal of z_t. This pins the
  model itself (which term carries a, a², k, k², p̄) rather than one algebraic
  arrangement of it.

Conventions shared with the oracle: (λ0, η0) is the belief before the first
token; token t first predicts through the OU prior, then absorbs the
observation; the readout y_t = Σ_i q_i · η_t/λ_t uses the posterior that
includes token t.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np


def _fr(x) -> Fraction:
    return x if isinstance(x, Fraction) else Fraction(float(x))


def mobius_coefficients(a, pbar, c):
    """(α, β, γ, δ) of the precision step λ_t = (αλ + β)/(γλ + δ).

    With the OU predict λ_pred = λ/(a² + p̄λ) followed by the update λ_pred + c
    (c = k²Λ^v): α = 1 + c·p̄, β = c·a², γ = p̄, δ = a²."""
    return 1 + c * pbar, c * a * a, pbar, a * a


def information_form_exact(q, k, v, lam_v, a, pbar, lam0=None, eta0=None):
    """Exact-rational information-form scan of one head.

    Arguments are nested sequences (or numpy arrays): q, k, a, pbar ``[T][dk]``;
    v, lam_v ``[T][dv]``; lam0, eta0 ``[dk][dv]`` or None (λ0 = 1, η0 = 0).
    Returns (y ``[T][dv]``, lam ``[T][dk][dv]``, eta ``[T][dk][dv]``) as
    Fractions, lam/eta holding the posterior after every token.
    """
    T = len(q)
    dk = len(q[0]) if T else (len(lam0) if lam0 is not None else 0)
    dv = len(v[0]) if T else (len(lam0[0]) if lam0 is not None else 0)
    lam = [[_fr(lam0[i][j]) if lam0 is not None else Fraction(1) for j in range(dv)] for i in range(dk)]
    eta = [[_fr(eta0[i][j]) if eta0 is not None else Fraction(0) for j in range(dv)] for i in range(dk)]
    ys, lams, etas = [], [], []
    for t in range(T):
        y = [Fraction(0)] * dv
        for i in range(dk):
            ai, pi, ki, qi = _fr(a[t][i]), _fr(pbar[t][i]), _fr(k[t][i]), _fr(q[t][i])
            for j in range(dv):
                Lj, vj = _fr(lam_v[t][j]), _fr(v[t][j])
                c = ki * ki * Lj
                b = ki * Lj * vj
                l_prev = lam[i][j]
                al, be, ga, de = mobius_coefficients(ai, pi, c)
                l_new = (al * l_prev + be) / (ga * l_prev + de)
                l_pred = l_prev / (ai * ai + pi * l_prev)
                e_new = (ai * l_pred / l_prev) * eta[i][j] + b
                lam[i][j], eta[i][j] = l_new, e_new
                y[j] += qi * e_new / l_new
        ys.append(y)
        lams.append([row[:] for row in lam])
        etas.append([row[:] for row in eta])
    return ys, lams, etas


def compose_mobius(mats):
    """Product M_T ⋯ M_1 of 2×2 Möbius matrices [[α, β], [γ, δ]] (exact)."""
    acc = [[Fraction(1), Fraction(0)], [Fraction(0), Fraction(1)]]
    for m in mats:
        acc = [[m[0][0] * acc[0][0] + m[0][1] * acc[1][0], m[0][0] * acc[0][1] + m[0][1] * acc[1][1]],
               [m[1][0] * acc[0][0] + m[1][1] * acc[1][0], m[1][0] * acc[0][1] + m[1][1] * acc[1][1]]]
    return acc


def apply_mobius(m, lam):
    return (m[0][0] * lam + m[0][1]) / (m[1][0] * lam + m[1][1])


def dense_filter_marginals(a, pbar, k, lam_v, v, lam0, eta0):
    """Filtering marginals of ONE scalar state element by dense conditioning.

    Model (one element, tokens t = 1..T, z_0 the state before the first token):
        z_0 ~ N(η0/λ0, 1/λ0)
        z_t = a_t z_{t-1} + w_t,   w_t ~ N(0, p̄_t)          (p̄_t > 0 required)
        v_t = k_t z_t + ε_t,       ε_t ~ N(0, 1/Λ^v_t)
    For every t the joint Gaussian of (z_0..z_t) given v_1..v_t is assembled
    in information form (precision matrix J, information vector h) and solved
    densely: mean = J⁻¹h, variance of z_t = (J⁻¹)_{tt}.
    Returns (lam [T], mu [T]) in float64: λ_t = 1/Var(z_t | v_1..v_t) and
    μ_t = E[z_t | v_1..v_t].
    """
    T = len(a)
    lam_out, mu_out = np.empty(T), np.empty(T)
    for tau in range(1, T + 1):
        n = tau + 1
        J = np.zeros((n, n))
        h = np.zeros(n)
        J[0, 0] += lam0
        h[0] += eta0
        for t in range(1, n):
            at, pt = float(a[t - 1]), float(pbar[t - 1])
            J[t, t] += 1.0 / pt
            J[t - 1, t - 1] += at * at / pt
            J[t, t - 1] -= at / pt
            J[t - 1, t] -= at / pt
            kt, Lt, vt = float(k[t - 1]), float(lam_v[t - 1]), float(v[t - 1])
            J[t, t] += kt * kt * Lt
            h[t] += kt * Lt * vt
        cov = np.linalg.inv(J)
        mean = cov @ h
        lam_out[tau - 1] = 1.0 / cov[tau, tau]
        mu_out[tau - 1] = mean[tau]
    return lam_out, mu_out


def riccati_fixed_point(a, pbar, c):
    """Positive fixed point of λ = (αλ + β)/(γλ + δ) for constant coefficients.

    It solves γλ² + (δ − α)λ − β = 0 (the scalar discrete Riccati equation in
    information form): λ* = [(α − δ) + √((α − δ)² + 4βγ)] / (2γ), γ = p̄ > 0."""
    al, be, ga, de = mobius_coefficients(a, pbar, c)
    return ((al - de) + np.sqrt((al - de) ** 2 + 4 * be * ga)) / (2 * ga)
