"""The coefficient pass of the sequential plan (kla_coef_pass): the per-row
coefficients of each token are computed once per head by their own kernel
and copied by every column block of the head, instead of being built by each
block. Both paths share the per-row arithmetic, so kla_forward must give bit
for bit the same y, λ_T and η_T with and without it — for every head size,
both scan geometries, both I/O types, the gate activations, ragged tiles and
in-place state updates — and match the oracle ("Technische Samenvatting:
Kalman Linear Attention (KLA)", Methodologie §1–§2) where the planner takes it
by itself.
"""
import ctypes

import pytest
import torch

from bayesian_filtering_linear_gb300 import kla
from bayesian_filtering_linear_gb300.inputs import make_inputs
from helpers import TOL, assert_close, errors, gpu_forward, run_oracle, to_dev

pytestmark = pytest.mark.gpu

IO = {"f32": torch.float32, "bf16": torch.bfloat16}
ALL_GATES = kla.GATE_LAMV_SOFTPLUS | kla.GATE_A_SIGMOID | kla.GATE_PBAR_OU

# (B, H, T, dk, dv, io, rows_per_lane): every head size, both geometries where
# there are two, one tile, several tiles with a ragged tail, a single token.
SHAPES = [
    (2, 3, 100, 16, 64, "f32", 4),
    (1, 2, 77, 32, 128, "bf16", 4),
    (2, 2, 161, 64, 64, "f32", 8),
    (1, 3, 33, 64, 32, "bf16", 4),
    (1, 1, 130, 128, 128, "bf16", 8),
    (2, 1, 50, 128, 64, "f32", 4),
    (3, 2, 16, 64, 128, "bf16", 8),
    (2, 2, 1, 32, 32, "f32", 4),
]


def _both(x, **kw):
    off = gpu_forward(x, coef_pass="off", strategy="sequential", **kw)
    on = gpu_forward(x, coef_pass="on", strategy="sequential", **kw)
    torch.cuda.synchronize()
    return off, on


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("gates", [0, ALL_GATES], ids=["plain", "gated"])
def test_bit_identical_with_and_without_the_pass(shape, gates):
    B, H, T, dk, dv, io, rl = shape
    x = to_dev(make_inputs(B, H, T, dk, dv, io=io, seed=500 + T + dk, random_state=True))
    (y0, l0, e0), (y1, l1, e1) = _both(x, rows_per_lane=rl, gates=gates)
    assert torch.equal(y0, y1) and torch.equal(l0, l1) and torch.equal(e0, e1)
    assert torch.isfinite(y1.float()).all()


def test_default_state_and_no_final_state():
    x = to_dev(make_inputs(2, 2, 90, 64, 64, io="f32", seed=511))
    off = gpu_forward(x, with_state=False, coef_pass="off", final_state=False)
    on = gpu_forward(x, with_state=False, coef_pass="on", final_state=False)
    torch.cuda.synchronize()
    assert on[1] is None and torch.equal(off[0], on[0])


def test_in_place_state_update_with_the_pass():
    x = to_dev(make_inputs(2, 2, 70, 64, 64, io="f32", seed=512, random_state=True))
    ref_y, ref_l, ref_e = gpu_forward(x, coef_pass="off")
    lam, eta = x["lam0"].clone(), x["eta0"].clone()
    y, lT, eT = kla.forward(x["q"], x["k"], x["v"], x["lam_v"], x["a"], x["pbar"], lam, eta, lamT=lam, etaT=eta,
                            coef_pass="on", strategy="sequential")
    torch.cuda.synchronize()
    assert lT.data_ptr() == lam.data_ptr()
    assert torch.equal(y, ref_y) and torch.equal(lam, ref_l) and torch.equal(eta, ref_e)


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_planner_takes_the_pass_for_split_heads_and_matches_the_oracle(io):
    # 8 heads of 64 × 64: the planner splits each head's columns over at
    # least four blocks and runs the coefficient pass by itself.
    B, H, T, d = 2, 4, 333, 64
    p = kla.plan(B, H, T, d, d, io)
    assert p["strategy"] == "sequential" and p["coef_pass"], p
    x = make_inputs(B, H, T, d, d, io=io, seed=513, random_state=True)
    ref = run_oracle(x)
    y, lamT, etaT = gpu_forward(to_dev(x))
    torch.cuda.synchronize()
    assert_close(errors(y, lamT, etaT, ref), TOL[IO[io]], f"coef pass {io}")


def test_uncertainty_readout_ignores_the_pass():
    x = to_dev(make_inputs(1, 2, 64, 64, 64, io="f32", seed=514, random_state=True))
    a = gpu_forward(x, coef_pass="off", uncertainty=True)
    b = gpu_forward(x, coef_pass="on", uncertainty=True)
    # through the C ABI directly: asked for, the pass is still not run, so no workspace is needed
    y, yv = torch.empty_like(a[0]), torch.empty_like(a[3])
    lT, eT = torch.empty_like(a[1]), torch.empty_like(a[2])
    opt = kla.options(coef_pass="on")
    st = kla.LIB.kla_forward_uncertainty(*(ctypes.c_void_p(x[n].data_ptr()) for n in
                                           ("q", "k", "v", "lam_v", "a", "pbar", "lam0", "eta0")),
                                         ctypes.c_void_p(y.data_ptr()), ctypes.c_void_p(yv.data_ptr()),
                                         ctypes.c_void_p(lT.data_ptr()), ctypes.c_void_p(eT.data_ptr()),
                                         1, 2, 64, 64, 64, kla.F32, None, 0, ctypes.byref(opt),
                                         ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    assert st == kla.OK
    for u, v in zip(a, b):
        assert torch.equal(u, v)
    for u, v in zip(a, (y, lT, eT, yv)):
        assert torch.equal(u, v)


def test_workspace_too_small_is_refused():
    x = to_dev(make_inputs(1, 2, 64, 64, 64, io="f32", seed=515))
    need = kla.plan(1, 2, 64, 64, 64, "f32", coef_pass="on")["workspace_bytes"]
    assert need == 2 * 64 * 5 * 64 * 4
    small = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(kla.KlaError) as e:
        gpu_forward(x, coef_pass="on", workspace=small)
    assert e.value.status == kla.ERR_WORKSPACE


def test_more_heads_than_one_grid_dimension():
    # the coefficient kernel covers heads in a grid-stride loop over its
    # 65535-wide second grid dimension
    B, H, T, d = 70000, 1, 3, 16
    x = to_dev(make_inputs(B, H, T, d, d, io="f32", seed=516, random_state=True))
    (y0, l0, e0), (y1, l1, e1) = _both(x)
    assert torch.equal(y0, y1) and torch.equal(l0, l1) and torch.equal(e0, e1)
