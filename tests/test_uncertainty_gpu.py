"""GPU parity of kla_forward_uncertainty: the variance readout
y_var[t, j] = Σ_i q_{t,i}² P_{t,i,j} ("Technische Samenvatting: Kalman Linear
Attention (KLA)", Belangrijkste Bijdragen item 3: explicit belief-state
uncertainty) against the fp64 oracle, plus the usual outputs of the same call.
y_var is a sum of positive terms, so its error is plain relative error;
tolerances 1e-4 (fp32 I/O) and 2e-2 (bf16 I/O) as for the other outputs.
"""
import numpy as np
import pytest
import torch

import oracle
from bayesian_filtering_linear_gb300 import kla
from bayesian_filtering_linear_gb300.inputs import make_inputs, make_workload
from helpers import TOL, assert_close, errors, to_dev

pytestmark = pytest.mark.gpu

IO = {"f32": torch.float32, "bf16": torch.bfloat16}


def run(x, heads=None, **kw):
    xd = to_dev(x)
    y, lamT, etaT, yv = kla.forward(xd["q"], xd["k"], xd["v"], xd["lam_v"], xd["a"], xd["pbar"], xd["lam0"],
                                    xd["eta0"], uncertainty=True, **kw)
    torch.cuda.synchronize()
    ref = oracle.forward(x["q"], x["k"], x["v"], x["lam_v"], x["a"], x["pbar"], x["lam0"], x["eta0"],
                         want_var=True, heads=heads)
    got = yv.float().cpu().numpy()
    if heads is not None:
        B, H = got.shape[:2]
        got = got.reshape((B * H,) + got.shape[2:])[np.asarray(heads)][:, None]
    return (y, lamT, etaT), ref, float(np.max(np.abs(got - ref["y_var"]) / ref["y_var"]))


SHAPES = [(1, 1, 100, 16, 16, "f32"), (2, 3, 77, 32, 64, "f32"), (1, 2, 161, 64, 64, "bf16"),
          (1, 1, 70, 128, 128, "f32"), (2, 2, 300, 64, 32, "bf16")]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("strategy,chunk_len", [("sequential", 0), ("chunked", 32)], ids=str)
def test_variance_readout_matches_oracle(shape, strategy, chunk_len):
    B, H, T, dk, dv, io = shape
    x = make_inputs(B, H, T, dk, dv, io=io, seed=700 + T, random_state=True)
    outs, ref, err = run(x, strategy=strategy, chunk_len=chunk_len)
    tol = TOL[IO[io]]
    assert err <= tol, f"y_var error {err}"
    assert_close(errors(*outs, ref), tol, f"{shape} {strategy}")


def test_variance_readout_with_in_place_state_update():
    x = make_inputs(1, 2, 90, 64, 32, io="f32", seed=9, random_state=True)
    xd = to_dev(x)
    lam, eta = xd["lam0"].clone(), xd["eta0"].clone()
    y, _, _, yv = kla.forward(xd["q"], xd["k"], xd["v"], xd["lam_v"], xd["a"], xd["pbar"], lam, eta,
                              lamT=lam, etaT=eta, uncertainty=True)
    torch.cuda.synchronize()
    ref = oracle.forward(x["q"], x["k"], x["v"], x["lam_v"], x["a"], x["pbar"], x["lam0"], x["eta0"], want_var=True)
    assert float(np.max(np.abs(yv.cpu().numpy() - ref["y_var"]) / ref["y_var"])) <= 1e-4
    assert float(np.max(np.abs(lam.cpu().numpy() - ref["lamT"]) / ref["lamT"])) <= 1e-4


def test_variance_readout_headline_all_heads():
    x = make_workload("headline")
    outs, ref, err = run(x)
    assert err <= 2e-2, f"y_var error {err}"
    assert_close(errors(*outs, ref), 2e-2, "headline with the variance readout")
