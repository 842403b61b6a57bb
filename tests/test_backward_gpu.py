"""GPU parity of the backward pass (kla_backward through the C ABI) against
the fp64 oracle's reverse-mode derivative on the same seeded inputs.

The forward is the scan of "Technische Samenvatting: Kalman Linear Attention
(KLA)", Methodologie §1–§2; the backward is its exact derivative (oracle
pinned by finite differences in test_oracle_backward.py). Error measure: each
gradient entry's |GPU − oracle| divided by the oracle's condition scale for
that entry (the same recursion with every term in absolute value), as for the
forward outputs. Tolerances (written here): 1e-4 for fp32 I/O, 2e-2 for bf16
I/O — the forward's bounds; see BWD_TOL.
"""
import numpy as np
import pytest
import torch

import oracle
from bayesian_filtering_linear_gb300 import kla
from bayesian_filtering_linear_gb300.inputs import make_inputs, make_workload
from helpers import assert_close, plain_rel, to_dev

pytestmark = pytest.mark.gpu

IO = {"f32": torch.float32, "bf16": torch.bfloat16}
# fp32 I/O: the GPU runs the forward recompute and the adjoint recursion in
# fp32 with the hardware reciprocal (≈ 2 ulp per step); the adjoints are
# contractive like the forward, so the error relative to the condition scale
# stays at a few fp32 ulps times the number of terms summed (measured
# ≤ 5e-7), well inside the forward's 1e-4. bf16 I/O: the per-token gradients
# are rounded to bf16 (2^-9 relative) on output, as y is (measured ≤ 3e-3).
BWD_TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}
GRADS = ("gq", "gk", "ga", "gpbar", "gv", "glam_v", "glam0", "geta0")
ORACLE_NAME = {"gq": "dq", "gk": "dk", "ga": "da", "gpbar": "dpbar", "gv": "dv", "glam_v": "dlam_v",
               "glam0": "dlam0", "geta0": "deta0"}


def upstream(B, H, T, dk, dv, io, seed, state=True):
    g = torch.Generator().manual_seed(seed)
    gy = torch.randn(B, H, T, dv, generator=g).to(IO[io])
    if not state:
        return gy, None, None
    return gy, torch.randn(B, H, dk, dv, generator=g), torch.randn(B, H, dk, dv, generator=g)


def bwd_errors(out: dict, ref: dict, heads=None) -> dict:
    errs = {}
    for n in GRADS:
        if n not in out:
            continue
        got = out[n].detach().float().cpu().numpy().astype(np.float64)
        if heads is not None:
            B, H = got.shape[:2]
            got = got.reshape((B * H,) + got.shape[2:])[np.asarray(list(heads))][:, None]
        want, scale = ref[ORACLE_NAME[n]], ref[ORACLE_NAME[n] + "_scale"]
        errs[n] = float(np.max(np.abs(got - want) / (scale + 1e-30))) if want.size else 0.0
        errs["rel_" + n] = plain_rel(got, want)
    return errs


def check(out, ref, io, what, heads=None):
    errs = bwd_errors(out, ref, heads)
    tol = BWD_TOL[IO[io]]
    assert_close(errs, tol, f"backward {what}")


def run_both(x, io, gy, glamT, getaT, with_state=True, state_grads=True, heads=None):
    xd = to_dev(x)
    out = kla.backward(xd["q"], xd["k"], xd["v"], xd["lam_v"], xd["a"], xd["pbar"],
                       xd["lam0"] if with_state else None, xd["eta0"] if with_state else None,
                       gy=gy.cuda() if gy is not None else None,
                       glamT=glamT.cuda() if glamT is not None else None,
                       getaT=getaT.cuda() if getaT is not None else None, state_grads=state_grads)
    torch.cuda.synchronize()
    ref = oracle.backward(x["q"], x["k"], x["v"], x["lam_v"], x["a"], x["pbar"],
                          x["lam0"] if with_state else None, x["eta0"] if with_state else None,
                          gy, glamT, getaT, heads=heads)
    return out, ref


# (B, H, T, dk, dv, io): every head size, ragged chunk tails, one column block
# per head and several (the finish pass), fp32 and bf16.
SHAPES = [
    (1, 1, 40, 16, 16, "f32"),
    (2, 1, 33, 16, 64, "f32"),
    (1, 2, 57, 32, 32, "f32"),
    (2, 2, 64, 64, 64, "f32"),
    (1, 1, 21, 128, 128, "f32"),
    (1, 2, 70, 64, 16, "bf16"),
    (1, 1, 100, 128, 32, "bf16"),
    (3, 1, 17, 32, 128, "bf16"),
    # short and ragged chunks of the 16-token checkpoint interval: one
    # 8-token chunk, one 9-token chunk, a 14-token last chunk
    (1, 1, 8, 16, 16, "f32"),
    (1, 1, 9, 32, 16, "f32"),
    (1, 2, 46, 64, 32, "f32"),
    # head counts for which the planner gives the reverse kernel two or four
    # columns per lane on a 152-SM device, every head size with each (checked
    # on the host in test_abi_host.py): two columns
    (8, 8, 24, 16, 64, "f32"),
    (8, 8, 19, 32, 32, "bf16"),
    (4, 4, 40, 64, 64, "f32"),
    (3, 16, 18, 128, 16, "bf16"),
    # four columns
    (8, 16, 20, 16, 128, "f32"),
    (3, 16, 22, 32, 128, "bf16"),
    (3, 16, 25, 64, 64, "f32"),
    (1, 16, 21, 128, 128, "bf16"),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_backward_matches_oracle(shape):
    B, H, T, dk, dv, io = shape
    x = make_inputs(B, H, T, dk, dv, io=io, seed=500 + T + dk, random_state=True)
    gy, gl, ge = upstream(B, H, T, dk, dv, io, seed=T)
    out, ref = run_both(x, io, gy, gl, ge)
    check(out, ref, io, str(shape))


def test_backward_default_state_and_y_only_upstream():
    x = make_inputs(1, 3, 50, 64, 32, io="f32", seed=9)
    gy, _, _ = upstream(1, 3, 50, 64, 32, "f32", seed=1, state=False)
    out, ref = run_both(x, "f32", gy, None, None, with_state=False)
    check(out, ref, "f32", "default state")


def test_backward_state_upstream_only_and_no_state_grads():
    x = make_inputs(2, 1, 37, 32, 64, io="f32", seed=10, random_state=True)
    _, gl, ge = upstream(2, 1, 37, 32, 64, "f32", seed=2)
    out, ref = run_both(x, "f32", None, gl, ge, state_grads=False)
    assert "glam0" not in out
    check(out, ref, "f32", "no dy")


def test_backward_empty_sequence_gives_state_gradients_only():
    x = make_inputs(1, 2, 0, 16, 16, io="f32", seed=3, random_state=True)
    _, gl, ge = upstream(1, 2, 0, 16, 16, "f32", seed=4)
    out, ref = run_both(x, "f32", None, gl, ge)
    assert out["gq"].numel() == 0
    check(out, ref, "f32", "T=0")


def test_backward_few_heads_split_columns():
    # one head: the planner splits its columns over several blocks (finish pass)
    x = make_inputs(1, 1, 300, 64, 128, io="bf16", seed=12, random_state=True)
    gy, gl, ge = upstream(1, 1, 300, 64, 128, "bf16", seed=5)
    out, ref = run_both(x, "bf16", gy, gl, ge)
    check(out, ref, "bf16", "1 head")


def test_backward_headline_workload_sampled_heads():
    """Full headline size; 32 of the 128 heads against the oracle (its
    per-element reverse pass keeps every forward state, ~0.8 GB of fp64
    gradients and scales for 32 heads)."""
    x = make_workload("headline")
    B, H, T, dk, dv = 8, 16, 4096, 64, 64
    gy, gl, ge = upstream(B, H, T, dk, dv, "bf16", seed=6)
    heads = list(range(0, 128, 4))
    out, ref = run_both(x, "bf16", gy, gl, ge, heads=heads)
    check(out, ref, "bf16", "headline", heads=heads)
    for n in GRADS:
        assert torch.isfinite(out[n].float()).all(), n


def test_backward_long_workload_sampled_head():
    """B1 H16 T65536 d128 bf16 at full size (columns split over blocks, the
    row-sum pass) against the oracle on four heads (one oracle thread per
    head, ~35 s)."""
    x = make_workload("long")
    B, H, T, dk, dv = 1, 16, 65536, 128, 128
    gy, gl, ge = upstream(B, H, T, dk, dv, "bf16", seed=8)
    heads = [0, 5, 10, 15]
    out, ref = run_both(x, "bf16", gy, gl, ge, heads=heads)
    check(out, ref, "bf16", "long", heads=heads)
