"""Inputs outside the model's domain give NaN or Inf where the recurrence
carries them and nowhere else — never a trap or a CUDA error (include/kla.h:
"Domain (the caller's contract) … other violations give NaN/Inf and never a
trap"). Every state element (i, j) of a head is its own filter and y_j reads
only column j ("Technische Samenvatting: Kalman Linear Attention (KLA)",
Belangrijkste Bijdragen 1: the diagonal structure), so:

* a NaN value v[t, j] reaches only η and y of column j from token t on;
* a NaN process noise p̄[t, i] reaches row i's λ and η, hence every y_j from
  t on (a NaN decay a does not: the kernels' floor max(a, 2^-40) takes it to
  2^-40, as IEEE max returns its non-NaN operand);
* other heads, and everything before t, are bit for bit the clean run's.
"""
import math

import pytest
import torch

from bayesian_filtering_linear_gb300 import kla
from bayesian_filtering_linear_gb300.inputs import make_conv_inputs, make_inputs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
NAMES = ("q", "k", "v", "lam_v", "a", "pbar", "lam0", "eta0")


def run(x, strategy):
    return kla.forward(*(x[n] for n in NAMES), strategy=strategy, chunk_len=32 if strategy == "chunked" else 0)


@pytest.mark.parametrize("strategy", ["sequential", "chunked"])
def test_nan_value_stays_in_its_column(strategy):
    x = {n: t.to(DEV) for n, t in make_inputs(1, 2, 96, 16, 16, io="f32", seed=31, random_state=True).items()}
    y0, l0, e0 = run(x, strategy)
    bad = dict(x, v=x["v"].clone())
    bad["v"][0, 1, 40, 3] = math.nan
    y, l, e = run(bad, strategy)
    torch.cuda.synchronize()
    assert torch.equal(y[0, 0], y0[0, 0]) and torch.equal(e[0, 0], e0[0, 0])  # the other head
    assert torch.equal(y[0, 1, :40], y0[0, 1, :40])                            # before the token
    assert torch.isnan(y[0, 1, 40:, 3]).all()
    others = [j for j in range(16) if j != 3]
    assert torch.equal(y[0, 1, :, others], y0[0, 1, :, others])                # the other columns
    assert torch.equal(l, l0)                                                  # λ never sees v
    assert torch.isnan(e[0, 1, :, 3]).all() and torch.equal(e[0, 1, :, others], e0[0, 1, :, others])


@pytest.mark.parametrize("strategy", ["sequential", "chunked"])
def test_nan_process_noise_stays_in_its_row(strategy):
    x = {n: t.to(DEV) for n, t in make_inputs(1, 2, 96, 16, 16, io="f32", seed=32, random_state=True).items()}
    y0, l0, e0 = run(x, strategy)
    bad = dict(x, pbar=x["pbar"].clone())
    bad["pbar"][0, 0, 20, 2] = math.nan
    y, l, e = run(bad, strategy)
    torch.cuda.synchronize()
    assert torch.equal(y[0, 1], y0[0, 1]) and torch.equal(l[0, 1], l0[0, 1])
    assert torch.equal(y[0, 0, :20], y0[0, 0, :20])
    assert torch.isnan(y[0, 0, 20:]).all()                                      # every column reads row 2
    rows = [i for i in range(16) if i != 2]
    assert torch.isnan(l[0, 0, 2]).all() and torch.equal(l[0, 0, rows], l0[0, 0, rows])


def test_negative_initial_precision_does_not_trap():
    x = {n: t.to(DEV) for n, t in make_inputs(2, 2, 1, 16, 16, io="f32", seed=33, random_state=True).items()}
    tok = {n: x[n][:, :, 0].contiguous() for n in ("q", "k", "v", "lam_v", "a", "pbar")}
    lam, eta = x["lam0"].clone(), x["eta0"].clone()
    lam_ref, eta_ref = lam.clone(), eta.clone()
    lam[1, 0, 5, 7] = -2.0
    y = kla.step(*(tok[n] for n in ("q", "k", "v", "lam_v", "a", "pbar")), lam, eta)
    y_ref = kla.step(*(tok[n] for n in ("q", "k", "v", "lam_v", "a", "pbar")), lam_ref, eta_ref)
    torch.cuda.synchronize()
    # the other heads and the other elements of the head are untouched
    assert torch.equal(y[0], y_ref[0]) and torch.equal(y[1, 1], y_ref[1, 1])
    mask = torch.ones_like(lam, dtype=torch.bool)
    mask[1, 0, 5, 7] = False
    assert torch.equal(lam[mask], lam_ref[mask]) and torch.equal(eta[mask], eta_ref[mask])
    # and the library keeps working afterwards
    y2 = kla.step(*(tok[n] for n in ("q", "k", "v", "lam_v", "a", "pbar")), lam_ref.clone(), eta_ref.clone())
    torch.cuda.synchronize()
    assert torch.isfinite(y2).all()


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_nan_input_of_the_convolution_reaches_only_its_window(io):
    W = 4
    p = {k: v.to(DEV) for k, v in make_conv_inputs(2, 2, 50, 16, W, io=io, seed=34).items()}
    y0, w0 = kla.conv(p["x"], p["weight"], p["bias"], p["window"])
    bad = p["x"].clone()
    bad[1, 0, 20, 5] = math.nan
    y, w = kla.conv(bad, p["weight"], p["bias"], p["window"])
    torch.cuda.synchronize()
    assert torch.isnan(y[1, 0, 20:20 + W, 5].float()).all()
    mask = torch.ones_like(y, dtype=torch.bool)
    mask[1, 0, 20:20 + W, 5] = False
    assert torch.equal(y[mask], y0[mask])
    assert torch.equal(w, w0)
