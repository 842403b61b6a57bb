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

Beside the scaled error every comparison also reports, for information, the
plain relative error max |gpu − ref| / max(|ref|, 1e-6·max|ref|) (keys
``rel_y``, ``rel_lam``, ``rel_eta``; not asserted: near a cancellation it
measures the cancellation, not the kernel). Every comparison is recorded in
``RECORDS`` and listed at the end of the pytest run.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from bayesian_filtering_linear_gb300 import kla

TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}
RECORDS: list = []  # (what, tolerance, errors) of every assert_close


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
    gy = sel(y)
    out = {"y": float(np.max(np.abs(gy - ref["y"]) / (ref["y_scale"] + tiny))), "rel_y": plain_rel(gy, ref["y"])}
    if lamT is not None:
        gl, ge = sel(lamT), sel(etaT)
        out["lam"] = float(np.max(np.abs(gl - ref["lamT"]) / ref["lamT"]))
        out["eta"] = float(np.max(np.abs(ge - ref["etaT"]) / (ref["eta_scale"] + tiny)))
        out["rel_lam"] = plain_rel(gl, ref["lamT"])
        out["rel_eta"] = plain_rel(ge, ref["etaT"])
    return out


def plain_rel(got, ref) -> float:
    """max |got − ref| / max(|ref|, 1e-6·max|ref|) (informational)."""
    ref = np.asarray(ref, dtype=np.float64)
    if ref.size == 0:
        return 0.0
    floor = 1e-6 * float(np.max(np.abs(ref))) + 1e-300
    return float(np.max(np.abs(np.asarray(got, dtype=np.float64) - ref) / np.maximum(np.abs(ref), floor)))


def assert_close(errs: dict, tol: float, what: str = ""):
    RECORDS.append((what, tol, dict(errs)))
    bad = {k: v for k, v in errs.items() if not k.startswith("rel_") and not (v <= tol)}
    assert not bad, f"{what}: errors {errs} exceed {tol}"


def gpu_forward(xd: dict, with_state=True, **kw):
    return kla.forward(xd["q"], xd["k"], xd["v"], xd["lam_v"], xd["a"], xd["pbar"],
                       xd["lam0"] if with_state else None, xd["eta0"] if with_state else None, **kw)
