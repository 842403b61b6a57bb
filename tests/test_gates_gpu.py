"""GPU parity with fused gate activations (kla_options.gates, kla_step_gated,
kla_backward's gates): the kernels read pre-activations and apply softplus /
sigmoid / the OU tie p̄ = softplus(x)(1 − a²) themselves ("Technische
Samenvatting: Kalman Linear Attention (KLA)", Methodologie §1). The oracle
applies the same definitions in fp64 to the same input values
(oracle/gates.py). Tolerances as for the ungated path.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import gates as G
from bayesian_filtering_linear_gb300 import kla
from helpers import TOL, assert_close

pytestmark = pytest.mark.gpu

IO = {"f32": torch.float32, "bf16": torch.bfloat16}
ALL = G.LAMV_SOFTPLUS | G.A_SIGMOID | G.PBAR_OU


def raw_inputs(B, H, T, dk, dv, io, seed, gates):
    """Pre-activations for the gated inputs; inputs without a gate bit get
    values in their domain (a in (0, 1), p̄ > 0, Λ^v > 0) directly."""
    g = torch.Generator().manual_seed(seed)
    r = lambda *s: torch.randn(*s, generator=g)
    sp = torch.nn.functional.softplus
    x = {"q": r(B, H, T, dk) * dk ** -0.5, "k": r(B, H, T, dk) * dk ** -0.5, "v": r(B, H, T, dv),
         "lam_v": r(B, H, T, dv), "a": r(B, H, T, dk) + 2.0, "pbar": r(B, H, T, dk) - 1.0}
    if not gates & G.LAMV_SOFTPLUS:
        x["lam_v"] = sp(x["lam_v"])
    if not gates & G.A_SIGMOID:
        x["a"] = torch.sigmoid(x["a"])
    if not gates & (G.PBAR_SOFTPLUS | G.PBAR_OU):
        x["pbar"] = sp(x["pbar"])
    x = {n: t.to(IO[io]) for n, t in x.items()}
    x["lam0"] = 0.5 + torch.nn.functional.softplus(r(B, H, dk, dv))
    x["eta0"] = r(B, H, dk, dv)
    return x


def oracle_inputs(x, gates):
    f64 = {n: t.double().numpy() for n, t in x.items()}
    L, A, Pb = G.apply(f64["lam_v"], f64["a"], f64["pbar"], gates)
    return dict(f64, lam_v=L, a=A, pbar=Pb)


def scaled_errors(y, lamT, etaT, ref):
    e = lambda got, want, sc: float(np.max(np.abs(got.float().cpu().numpy() - want) / (sc + 1e-30)))
    return {"y": e(y, ref["y"], ref["y_scale"]), "lam": e(lamT, ref["lamT"], ref["lamT"]),
            "eta": e(etaT, ref["etaT"], ref["eta_scale"])}


@pytest.mark.parametrize("gates", [ALL, G.LAMV_SOFTPLUS | G.A_SIGMOID | G.PBAR_SOFTPLUS, G.PBAR_OU])
@pytest.mark.parametrize("shape", [(2, 2, 77, 64, 32, "f32"), (1, 3, 130, 32, 64, "bf16")], ids=str)
@pytest.mark.parametrize("strategy,chunk_len", [("sequential", 0), ("chunked", 32)], ids=str)
def test_gated_forward_matches_oracle(gates, shape, strategy, chunk_len):
    B, H, T, dk, dv, io = shape
    x = raw_inputs(B, H, T, dk, dv, io, seed=T + gates, gates=gates)
    xd = {n: t.cuda() for n, t in x.items()}
    y, lamT, etaT = kla.forward(*(xd[n] for n in ("q", "k", "v", "lam_v", "a", "pbar", "lam0", "eta0")),
                                strategy=strategy, chunk_len=chunk_len, gates=gates)
    torch.cuda.synchronize()
    xo = oracle_inputs(x, gates)
    ref = oracle.forward64(*(xo[n] for n in ("q", "k", "v", "lam_v", "a", "pbar", "lam0", "eta0")),
                           want_scales=True)
    assert_close(scaled_errors(y, lamT, etaT, ref), TOL[IO[io]], f"gates {gates} {shape} {strategy}")


def test_gated_step_matches_gated_forward():
    x = raw_inputs(2, 2, 40, 64, 64, "f32", seed=5, gates=ALL)
    xd = {n: t.cuda() for n, t in x.items()}
    names = ("q", "k", "v", "lam_v", "a", "pbar")
    y, lamT, etaT = kla.forward(*(xd[n] for n in names), xd["lam0"], xd["eta0"], gates=ALL)
    pre = {n: xd[n][:, :, :39].contiguous() for n in names}
    _, lam, eta = kla.forward(*(pre[n] for n in names), xd["lam0"], xd["eta0"], gates=ALL)
    tok = {n: xd[n][:, :, 39].contiguous() for n in names}
    y_last = kla.step(*(tok[n] for n in names), lam, eta, gates=ALL)
    torch.cuda.synchronize()
    scale = y[:, :, 39].abs().max()
    assert float((y_last - y[:, :, 39]).abs().max() / scale) < 1e-4
    assert float(((lam - lamT).abs() / lamT).max()) < 1e-4


@pytest.mark.parametrize("gates", [ALL, G.LAMV_SOFTPLUS | G.A_SIGMOID | G.PBAR_SOFTPLUS])
@pytest.mark.parametrize("shape", [(2, 2, 50, 64, 64, "f32"), (1, 1, 90, 64, 128, "bf16")], ids=str)
def test_gated_backward_matches_oracle(gates, shape):
    B, H, T, dk, dv, io = shape
    x = raw_inputs(B, H, T, dk, dv, io, seed=gates * 7 + T, gates=gates)
    g = torch.Generator().manual_seed(1)
    gy = torch.randn(B, H, T, dv, generator=g).to(IO[io])
    gl, ge = torch.randn(B, H, dk, dv, generator=g), torch.randn(B, H, dk, dv, generator=g)
    xd = {n: t.cuda() for n, t in x.items()}
    out = kla.backward(*(xd[n] for n in ("q", "k", "v", "lam_v", "a", "pbar", "lam0", "eta0")), gy=gy.cuda(),
                       glamT=gl.cuda(), getaT=ge.cuda(), gates=gates)
    torch.cuda.synchronize()
    xo = oracle_inputs(x, gates)
    ref = oracle.backward64(*(xo[n] for n in ("q", "k", "v", "lam_v", "a", "pbar", "lam0", "eta0")),
                            gy.double().numpy(), gl.double().numpy(), ge.double().numpy(), want_scales=True)
    f64 = {n: t.double().numpy() for n, t in x.items()}
    raw = G.chain(ref["dlam_v"], ref["da"], ref["dpbar"], f64["lam_v"], f64["a"], f64["pbar"], gates)
    # condition scales through the same chain rule with every factor in
    # absolute value (the OU path adds |∂p̄/∂a| = 2a·softplus(x_p))
    A = G.sigmoid(f64["a"]) if gates & G.A_SIGMOID else f64["a"]
    sL = ref["dlam_v_scale"] * (G.sigmoid(f64["lam_v"]) if gates & G.LAMV_SOFTPLUS else 1.0)
    if gates & G.PBAR_OU:
        sp = ref["dpbar_scale"] * (1 - A * A) * G.sigmoid(f64["pbar"])
        sa = ref["da_scale"] + ref["dpbar_scale"] * G.softplus(f64["pbar"]) * 2 * np.abs(A)
    else:
        sp = ref["dpbar_scale"] * (G.sigmoid(f64["pbar"]) if gates & G.PBAR_SOFTPLUS else 1.0)
        sa = ref["da_scale"]
    if gates & G.A_SIGMOID:
        sa = sa * A * (1 - A)
    want = {"gq": (ref["dq"], ref["dq_scale"]), "gk": (ref["dk"], ref["dk_scale"]),
            "gv": (ref["dv"], ref["dv_scale"]), "glam_v": (raw[0], sL), "ga": (raw[1], sa),
            "gpbar": (raw[2], sp), "glam0": (ref["dlam0"], ref["dlam0_scale"]),
            "geta0": (ref["deta0"], ref["deta0_scale"])}
    errs = {n: float(np.max(np.abs(out[n].double().cpu().numpy() - w) / (s + 1e-30))) for n, (w, s) in want.items()}
    tol = 1e-4 if io == "f32" else 2e-2
    assert all(v <= tol for v in errs.values()), errs


def test_gated_uncertainty_chunked_matches_oracle():
    """Gates, the variance readout and the chunk-parallel path together."""
    x = raw_inputs(1, 2, 200, 64, 64, "f32", seed=11, gates=ALL)
    xd = {n: t.cuda() for n, t in x.items()}
    y, lamT, etaT, yv = kla.forward(*(xd[n] for n in ("q", "k", "v", "lam_v", "a", "pbar", "lam0", "eta0")),
                                    strategy="chunked", chunk_len=64, gates=ALL, uncertainty=True)
    torch.cuda.synchronize()
    xo = oracle_inputs(x, ALL)
    ref = oracle.forward64(*(xo[n] for n in ("q", "k", "v", "lam_v", "a", "pbar", "lam0", "eta0")),
                           want_scales=True)
    assert_close(scaled_errors(y, lamT, etaT, ref), 1e-4, "gated chunked")
    # y_var = Σ_i q² / λ_t: the oracle's λ after every token via one-hot q is
    # not needed; compare against the ungated variance readout on the gated values
    xv = {n: torch.from_numpy(v).float() for n, v in xo.items()}
    ref_v = oracle.forward(*(xv[n] for n in ("q", "k", "v", "lam_v", "a", "pbar", "lam0", "eta0")), want_var=True)
    assert float(np.max(np.abs(yv.cpu().numpy() - ref_v["y_var"]) / ref_v["y_var"])) <= 1e-4
