"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on
the same seeded inputs, element by element.

Scan definition: "Technische Samenvatting: Kalman Linear Attention (KLA)"
(gist.science/nl/paper/2602.10743), Methodologie §1–§2. Error measure and
tolerances (1e-4 fp32 I/O, 2e-2 bf16 I/O) are described in tests/helpers.py.
"""
import ctypes

import numpy as np
import pytest
import torch

from bayesian_filtering_linear_gb300 import kla
from bayesian_filtering_linear_gb300.inputs import make_inputs, make_workload, WORKLOADS
from helpers import TOL, assert_close, errors, gpu_forward, run_oracle, to_dev

pytestmark = pytest.mark.gpu

IO = {"f32": torch.float32, "bf16": torch.bfloat16}

# (B, H, T, dk, dv, io): several tiles and a ragged tail, every head size.
SHAPES = [
    (1, 1, 256, 16, 16, "f32"),
    (2, 3, 100, 32, 64, "f32"),
    (1, 2, 257, 64, 16, "bf16"),
    (1, 1, 130, 128, 128, "bf16"),
    (2, 2, 77, 128, 32, "f32"),
    (3, 1, 50, 16, 128, "bf16"),
    (2, 1, 1, 64, 64, "f32"),
    (1, 3, 161, 64, 64, "f32"),
]
STRATEGIES = [("auto", 0), ("sequential", 0), ("chunked", 32), ("chunked", 64)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("strategy,chunk_len", STRATEGIES, ids=lambda s: str(s))
def test_small_shapes_match_oracle(shape, strategy, chunk_len):
    B, H, T, dk, dv, io = shape
    x = make_inputs(B, H, T, dk, dv, io=io, seed=100 + T + dk, random_state=True)
    ref = run_oracle(x)
    y, lamT, etaT = gpu_forward(to_dev(x), strategy=strategy, chunk_len=chunk_len)
    torch.cuda.synchronize()
    assert_close(errors(y, lamT, etaT, ref), TOL[IO[io]], f"{shape} {strategy}/{chunk_len}")


# Both scan geometries for the head sizes that have two (rows per lane 4 and
# 8), whichever the planner would pick, on the sequential and chunked paths.
RL_SHAPES = [
    (2, 2, 93, 64, 64, "f32"),
    (1, 2, 130, 64, 32, "bf16"),
    (1, 1, 70, 128, 128, "f32"),
    (2, 1, 161, 128, 16, "bf16"),
]


@pytest.mark.parametrize("shape", RL_SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("rows_per_lane", [4, 8])
@pytest.mark.parametrize("strategy,chunk_len", [("sequential", 0), ("chunked", 32)], ids=lambda s: str(s))
def test_rows_per_lane_choices_match_oracle(shape, rows_per_lane, strategy, chunk_len):
    B, H, T, dk, dv, io = shape
    x = make_inputs(B, H, T, dk, dv, io=io, seed=300 + T + dk, random_state=True)
    ref = run_oracle(x)
    info = kla.plan(B, H, T, dk, dv, io, strategy, chunk_len, rows_per_lane=rows_per_lane)
    assert info["rows_per_lane"] == rows_per_lane
    y, lamT, etaT = gpu_forward(to_dev(x), strategy=strategy, chunk_len=chunk_len, rows_per_lane=rows_per_lane)
    torch.cuda.synchronize()
    assert_close(errors(y, lamT, etaT, ref), TOL[IO[io]], f"{shape} RL{rows_per_lane} {strategy}")


def test_tiny_workload_default_state():
    x = make_workload("tiny")
    ref = run_oracle(x, with_state=False)
    for strategy, cl in STRATEGIES:
        y, lamT, etaT = gpu_forward(to_dev(x), with_state=False, strategy=strategy, chunk_len=cl)
        assert_close(errors(y, lamT, etaT, ref), 1e-4, f"tiny {strategy}")


@pytest.mark.parametrize("strategy,chunk_len", [("auto", 0), ("sequential", 0), ("chunked", 256)])
def test_medium_workload_all_heads(strategy, chunk_len):
    w = WORKLOADS["medium"]
    x = make_workload(w)
    ref = run_oracle(x)
    y, lamT, etaT = gpu_forward(to_dev(x), strategy=strategy, chunk_len=chunk_len)
    assert_close(errors(y, lamT, etaT, ref), 1e-4, f"medium {strategy}")


def test_headline_workload_all_heads():
    """B8 H16 T4096 d64 bf16, every one of the 128 heads against the oracle,
    in the launch configuration the benchmark times."""
    x = make_workload("headline")
    ref = run_oracle(x)
    y, lamT, etaT = gpu_forward(to_dev(x))
    assert_close(errors(y, lamT, etaT, ref), 2e-2, "headline")
    assert torch.isfinite(y.float()).all() and (lamT > 0).all()


def test_long_workload_all_heads():
    """B1 H16 T65536 d128 bf16, all 16 heads, on the planner's path and on the
    chunk-parallel path (one oracle run serves both)."""
    x = make_workload("long")
    ref = run_oracle(x)
    xd = to_dev(x)
    for strategy in ("auto", "chunked"):
        y, lamT, etaT = gpu_forward(xd, strategy=strategy)
        assert_close(errors(y, lamT, etaT, ref), 2e-2, f"long {strategy}")
        assert torch.isfinite(y.float()).all() and (lamT > 0).all()
        del y, lamT, etaT


def test_chunk_length_invariance():
    x = to_dev(make_inputs(2, 2, 1024, 64, 64, io="f32", seed=7, random_state=True))
    y0, l0, e0 = gpu_forward(x, strategy="sequential")
    for cl in (32, 64, 256, 1024 - 32):
        y, l, e = gpu_forward(x, strategy="chunked", chunk_len=cl)
        scale = y0.abs().max()
        assert float((y - y0).abs().max() / scale) < 1e-4, cl
        assert float(((l - l0).abs() / l0).max()) < 1e-4, cl
        assert float((e - e0).abs().max() / e0.abs().max()) < 1e-4, cl


def test_resume_from_state_equals_one_pass():
    x = to_dev(make_inputs(2, 3, 300, 32, 32, io="f32", seed=8, random_state=True))
    y, lamT, etaT = gpu_forward(x)
    T1 = 123
    part = lambda d, s: {n: (t[:, :, s] if t.dim() == 4 and n not in ("lam0", "eta0") else t).contiguous()
                         for n, t in d.items()}
    xa = part(x, slice(0, T1))
    ya, la, ea = gpu_forward(xa)
    xb = part(x, slice(T1, None))
    xb["lam0"], xb["eta0"] = la, ea
    yb, lb, eb = gpu_forward(xb)
    yy = torch.cat([ya, yb], dim=2)
    assert float((yy - y).abs().max() / y.abs().max()) < 1e-5
    assert float(((lb - lamT).abs() / lamT).max()) < 1e-5


@pytest.mark.parametrize("strategy", ["sequential", "chunked"])
def test_in_place_state_update(strategy):
    x = to_dev(make_inputs(1, 2, 200, 64, 32, io="bf16", seed=9, random_state=True))
    y_ref, l_ref, e_ref = gpu_forward(x, strategy=strategy, chunk_len=64 if strategy == "chunked" else 0)
    lam, eta = x["lam0"].clone(), x["eta0"].clone()
    y, l, e = kla.forward(x["q"], x["k"], x["v"], x["lam_v"], x["a"], x["pbar"], lam, eta, lamT=lam, etaT=eta,
                          strategy=strategy, chunk_len=64 if strategy == "chunked" else 0)
    assert torch.equal(y, y_ref) and torch.equal(lam, l_ref) and torch.equal(eta, e_ref)


def test_empty_sequence_copies_initial_state():
    x = to_dev(make_inputs(2, 2, 0, 16, 32, io="f32", seed=10, random_state=True))
    y, l, e = gpu_forward(x)
    assert y.shape == (2, 2, 0, 32)
    assert torch.equal(l, x["lam0"]) and torch.equal(e, x["eta0"])
    y, l, e = gpu_forward(x, with_state=False)
    assert torch.all(l == 1) and torch.all(e == 0)


def test_closed_forms_on_gpu():
    # a = 1, p̄ = 0: recursive least squares; Λ^v = 0: the prior relaxes.
    x = make_inputs(1, 2, 500, 32, 16, io="f32", seed=11, random_state=True)
    x1 = dict(x, a=torch.ones_like(x["a"]), pbar=torch.zeros_like(x["pbar"]))
    ref = run_oracle(x1)
    assert_close(errors(*gpu_forward(to_dev(x1)), ref), 1e-4, "a=1, pbar=0")
    x2 = dict(x, lam_v=torch.zeros_like(x["lam_v"]))
    ref = run_oracle(x2)
    assert_close(errors(*gpu_forward(to_dev(x2)), ref), 1e-4, "lam_v=0")


def test_degenerate_inputs_stay_finite():
    x = make_inputs(1, 1, 96, 64, 64, io="f32", seed=12, random_state=True)
    x["k"][..., :5] = 0.0            # k = 0: no observation
    x["a"][..., 5:9] = 1.0           # no decay
    x["pbar"][..., 9:12] = 0.0       # no process noise
    x["a"][..., 12:14] = 1e-30       # (almost) complete forgetting
    ref = run_oracle(x)
    y, l, e = gpu_forward(to_dev(x))
    assert_close(errors(y, l, e, ref), 1e-4, "degenerate")


def test_decode_steps_match_forward_and_oracle():
    w = WORKLOADS["decode"]
    x = make_workload(w)
    P, S = 1024, w.T - 1024
    xd = to_dev(x)
    y_full, l_full, e_full = gpu_forward(xd)
    pre = {n: (t[:, :, :P] if n not in ("lam0", "eta0") else t).contiguous() for n, t in xd.items()}
    _, lam, eta = gpu_forward(pre)
    ys = []
    for s in range(S):
        t = P + s
        tok = {n: xd[n][:, :, t].contiguous() for n in ("q", "k", "v", "lam_v", "a", "pbar")}
        ys.append(kla.step(tok["q"], tok["k"], tok["v"], tok["lam_v"], tok["a"], tok["pbar"], lam, eta))
    y_steps = torch.stack(ys, dim=2)
    scale = y_full[:, :, P:].abs().amax(dim=(2, 3), keepdim=True) + 1e-30
    assert float(((y_steps - y_full[:, :, P:]).abs() / scale).max()) < 1e-4
    assert float(((lam - l_full).abs() / l_full).max()) < 1e-4
    heads = list(range(0, w.B * w.H, 16))  # 256 of the 4096 heads, spread over the batch
    ref = run_oracle(x, heads=heads)
    e = errors(torch.cat([y_full[:, :, :P], y_steps], dim=2), lam, eta, ref, heads=heads)
    assert_close(e, 1e-4, "decode vs oracle")


@pytest.mark.parametrize("shape", [(2, 3, 20, 64, 32, "bf16"), (1, 2, 12, 128, 16, "bf16"), (3, 1, 9, 16, 128, "f32"),
                                   (1, 1, 15, 32, 64, "f32")], ids=lambda s: "x".join(map(str, s)))
def test_decode_steps_every_head_size_match_oracle(shape):
    """kla_step token by token from the initial state equals the oracle's scan."""
    B, H, T, dk, dv, io = shape
    x = make_inputs(B, H, T, dk, dv, io=io, seed=900 + T, random_state=True)
    ref = run_oracle(x)
    xd = to_dev(x)
    lam, eta = xd["lam0"].clone(), xd["eta0"].clone()
    ys = []
    for t in range(T):
        tok = {n: xd[n][:, :, t].contiguous() for n in ("q", "k", "v", "lam_v", "a", "pbar")}
        ys.append(kla.step(tok["q"], tok["k"], tok["v"], tok["lam_v"], tok["a"], tok["pbar"], lam, eta))
    torch.cuda.synchronize()
    assert_close(errors(torch.stack(ys, dim=2), lam, eta, ref), TOL[IO[io]], f"step {shape}")


def _step_raw(fn, tok, lam, eta, y, io, gates=None):
    """One decode step through the raw C symbol (kla_step, or kla_step_gated)."""
    B, H, dk = tok["q"].shape
    dv = tok["v"].shape[-1]
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    args = [p(tok[n]) for n in ("q", "k", "v", "lam_v", "a", "pbar")] + [p(lam), p(eta), p(y), B, H, dk, dv, io]
    if gates is not None:
        args.append(gates)
    return fn(*args, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("shape", [(2, 3, 40, 64, 32, "f32"), (1, 2, 33, 128, 64, "bf16"), (3, 1, 20, 16, 16, "f32")],
                         ids=lambda s: "x".join(map(str, s)))
def test_ungated_step_symbol_matches_oracle(shape):
    """The C ABI's kla_step (no gate argument), called through ctypes token by
    token from the initial state, against the oracle's scan; and bit-identical
    to kla_step_gated with gates = 0."""
    B, H, T, dk, dv, io = shape
    x = make_inputs(B, H, T, dk, dv, io=io, seed=950 + T, random_state=True)
    ref = run_oracle(x)
    xd = to_dev(x)
    io_code = kla.BF16 if io == "bf16" else kla.F32
    lam, eta = xd["lam0"].clone(), xd["eta0"].clone()
    lam_g, eta_g = xd["lam0"].clone(), xd["eta0"].clone()
    ys = []
    for t in range(T):
        tok = {n: xd[n][:, :, t].contiguous() for n in ("q", "k", "v", "lam_v", "a", "pbar")}
        y = torch.empty((B, H, dv), dtype=xd["q"].dtype, device="cuda")
        y_g = torch.empty_like(y)
        assert _step_raw(kla.LIB.kla_step, tok, lam, eta, y, io_code) == kla.OK
        assert _step_raw(kla.LIB.kla_step_gated, tok, lam_g, eta_g, y_g, io_code, 0) == kla.OK
        torch.cuda.synchronize()
        assert torch.equal(y, y_g)
        ys.append(y)
    assert torch.equal(lam, lam_g) and torch.equal(eta, eta_g)
    assert_close(errors(torch.stack(ys, dim=2), lam, eta, ref), TOL[IO[io]], f"kla_step {shape}")
