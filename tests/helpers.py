"""Comparison helpers for the GPU parity tests.

Error measure (the north-star tolerance is a "max relative error"; relative
to what is not stated, so the reading here is): every output is compared
against the fp64 oracle on the same rounded inputs, divided by a condition
scale the oracle computes in the same loop —
  y:  Σ_i |q_i| μ̂_ij  (μ̂ = the mean recursion run on absolute values)
  η:  μ̂ / P            λ: λ itself (always > 0)
which bounds the magnitude of everything summed, so the ratio measures
rounding error even where y or η cancel to nearly zero.
Tolerances: 1e-4 for fp32 I/O, 2e-2 for bf16 I/O.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from bayesian_filtering_linear_gb300 import kla

TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}


def to_dev(x: dict, device="cuda") -> dict:
    return {n: t.to(device) for n, t in x.items()}


def run_oracle(x: dict, heads=None, with_state=True) -> dict:
    return oracle.forward(x["q"], x["k"], x["v"], x["lam_v"], x["a"], x["pbar"],
                          x["lam0"] if with_state else None, x["eta0"] if with_state else None, heads=heads)


def errors(y, lamT, etaT, ref: dict, heads=None) -> dict:
    """Max scaled errors of GPU outputs (torch, full batch) against an oracle
    result (numpy, possibly for a subset of flat head indices)."""
    def sel(t):
        a = t.detach().float().cpu().numpy()
        if heads is None:
            return a
        B, H = a.shape[:2]
        return a.reshape((B * H,) + a.shape[2:])[np.asarray(list(heads))][:, None]
    tiny = 1e-30
    out = {"y": float(np.max(np.abs(sel(y) - ref["y"]) / (ref["y_scale"] + tiny)))}
    if lamT is not None:
        out["lam"] = float(np.max(np.abs(sel(lamT) - ref["lamT"]) / ref["lamT"]))
        out["eta"] = float(np.max(np.abs(sel(etaT) - ref["etaT"]) / (ref["eta_scale"] + tiny)))
    return out


def assert_close(errs: dict, tol: float, what: str = ""):
    bad = {k: v for k, v in errs.items() if not (v <= tol)}
    assert not bad, f"{what}: errors {errs} exceed {tol}"


def gpu_forward(xd: dict, with_state=True, **kw):
    return kla.forward(xd["q"], xd["k"], xd["v"], xd["lam_v"], xd["a"], xd["pbar"],
                       xd["lam0"] if with_state else None, xd["eta0"] if with_state else None, **kw)
