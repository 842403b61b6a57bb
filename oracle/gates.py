"""Gate activations of the KLA inputs, in fp64 — TEST INFRASTRUCTURE ONLY
(part of the oracle package; see its header).

Source: "Technische Samenvatting: Kalman Linear Attention (KLA)",
Methodologie §1: the OU prior has decay a ∈ (0, 1) and process noise p̄ > 0,
the observation a precision Λ^v > 0; an exactly discretised OU process with
stationary variance s has p̄ = s·(1 − a²). With a gate bit set an input holds
a pre-activation x:
    bit 1  Λ^v = softplus(x) = log(1 + e^x)
    bit 2  a = sigmoid(x) = 1 / (1 + e^-x)
    bit 4  p̄ = softplus(x)
    bit 8  p̄ = softplus(x) · (1 − a²)
:func:`apply` maps pre-activations to (Λ^v, a, p̄); :func:`chain` maps
gradients with respect to (Λ^v, a, p̄) to gradients with respect to the
pre-activations (the chain rule of those definitions).
"""
from __future__ import annotations

import numpy as np

LAMV_SOFTPLUS, A_SIGMOID, PBAR_SOFTPLUS, PBAR_OU = 1, 2, 4, 8


def softplus(x):
    return np.logaddexp(0.0, x)


def sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def apply(lam_v, a, pbar, gates: int):
    """(Λ^v, a, p̄) from the inputs as given (fp64 arrays)."""
    L = softplus(lam_v) if gates & LAMV_SOFTPLUS else lam_v
    A = sigmoid(a) if gates & A_SIGMOID else a
    if gates & PBAR_OU:
        Pb = softplus(pbar) * (1.0 - A * A)
    elif gates & PBAR_SOFTPLUS:
        Pb = softplus(pbar)
    else:
        Pb = pbar
    return L, A, Pb


def chain(g_lam_v, g_a, g_pbar, lam_v, a, pbar, gates: int, _mutant: int = 0):
    """Gradients with respect to the inputs as given, from the gradients
    with respect to (Λ^v, a, p̄). ``_mutant`` = 1 drops the path from a
    through the OU-tied p̄ (a planted mistake, tests only)."""
    gL = g_lam_v * sigmoid(lam_v) if gates & LAMV_SOFTPLUS else g_lam_v
    A = sigmoid(a) if gates & A_SIGMOID else a
    if gates & PBAR_OU:
        g_p = g_pbar * (1.0 - A * A) * sigmoid(pbar)
        g_A = g_a + (0.0 if _mutant == 1 else g_pbar * softplus(pbar) * (-2.0 * A))
    else:
        g_p = g_pbar * sigmoid(pbar) if gates & PBAR_SOFTPLUS else g_pbar
        g_A = g_a
    g_x = g_A * A * (1.0 - A) if gates & A_SIGMOID else g_A
    return gL, g_x, g_p
