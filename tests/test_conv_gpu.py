"""Parity of the causal depthwise convolution with SiLU (kla_conv,
kla_conv_backward) against the fp64 oracle (oracle/conv.py), element by
element, on seeded inputs from ``inputs.make_conv_inputs``.

Error measure: |gpu − oracle| / (|oracle| + s), with s the same quantity
computed on absolute values (for y: |bias| + Σ_k |w_k x_k|; for gx and the
window gradient: Σ_k |w_k| |gu| + |gwindow_out|; for the tap and bias
gradients: Σ |gu| |x| and Σ |gu|; with |gu| read as |gy|·σ(u)(1 + |u|(1 −
σ(u))), the terms of gy·SiLU'(u) in absolute value), so that cancellation in
a sum is not counted against the kernel. Tolerances: outputs in the I/O dtype 2e-5 (fp32:
a W-term fp32 sum and the hardware exponential and reciprocal in SiLU) or
4e-3 (bf16: round-to-nearest-even of the output, 2^-9 relative); the fp32 tap
and bias gradients 1e-4 (fp32 sums over up to a thousand tokens per thread
and the block and batch partials).

Source of the operation: "Technische Samenvatting: Kalman Linear Attention
(KLA)", Methodologie §4 (Architectuur): 1-D causal convolutions and SiLU
activations in the Mamba-like block around the scan.
"""
import numpy as np
import pytest
import torch

from bayesian_filtering_linear_gb300 import kla
from bayesian_filtering_linear_gb300.inputs import make_conv_inputs
from oracle import conv as C

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
TOL_IO = {"f32": 2e-5, "bf16": 4e-3}
TOL_SUM = 1e-4


def f64(t):
    return None if t is None else t.detach().double().cpu().numpy()


def on_device(d):
    return {k: v.to(DEV) for k, v in d.items()}


def scaled_err(got, want, scale):
    got, want = f64(got) if isinstance(got, torch.Tensor) else got, want
    if want.size == 0:
        return 0.0
    return float(np.max(np.abs(got - want) / (np.abs(want) + scale + 1e-30)))


def oracle_forward(p, act, use_bias, use_window):
    x, w = f64(p["x"]), f64(p["weight"])
    b = f64(p["bias"]) if use_bias else None
    win = f64(p["window"]) if use_window else None
    y, wout = C.conv(x, w, b, win, act)
    scale = C.preactivation(np.abs(x), np.abs(w), None if b is None else np.abs(b),
                            None if win is None else np.abs(win))
    return y, wout, scale


def oracle_backward(p, act, use_bias, use_window, use_gwo=True):
    x, w = f64(p["x"]), f64(p["weight"])
    b = f64(p["bias"]) if use_bias else None
    win = f64(p["window"]) if use_window else None
    gy = f64(p["gy"])
    gwo = f64(p["gwindow_out"]) if use_gwo else None
    g = C.conv_backward(x, w, b, win, gy, gwo, act)
    # scales: the same sums over absolute values. SiLU'(u) = σ(1 + u(1 − σ))
    # cancels to zero near u ≈ −1.28, so its scale is σ(1 + |u|(1 − σ)), the
    # sum of its terms in absolute value, not |SiLU'(u)|
    u = C.preactivation(x, w, b, win)
    sg = C.sigmoid(u)
    gu_abs = np.abs(gy) * sg * (1.0 + np.abs(u) * (1.0 - sg)) if act else np.abs(gy)
    s = C.conv_backward(np.abs(x), np.abs(w), None, None if win is None else np.abs(win), gu_abs,
                        None if gwo is None else np.abs(gwo), activation=False)
    return g, s


def run_forward(p, act, use_bias, use_window, **kw):
    return kla.conv(p["x"], p["weight"], p["bias"] if use_bias else None, p["window"] if use_window else None,
                    activation=kla.ACT_SILU if act else kla.ACT_NONE, **kw)


CASES = [  # B, H, T, D, W
    (2, 3, 37, 16, 4),    # ragged last chunk
    (1, 2, 50, 8, 1),
    (1, 2, 50, 8, 2),
    (1, 2, 50, 8, 3),
    (2, 1, 70, 8, 5),
    (1, 2, 50, 8, 6),
    (1, 2, 50, 8, 7),
    (2, 2, 99, 8, 8),
    (1, 3, 33, 12, 4),    # three channel groups: 85 chunks per block
    (1, 1, 40, 512, 4),   # the widest stream: eight tokens a stage
    (1, 1, 40, 512, 8),   # seven rows of window from the previous stage
    (2, 1, 9, 512, 7),
    (1, 1, 3000, 4, 8),   # one channel group; 8-byte rows in bf16
    (1, 2, 777, 20, 3),   # five channel groups; 8-byte copies in bf16
    (3, 2, 5000, 16, 4),  # several blocks along T: batch and block partials
    (1, 2, 2, 16, 6),     # T < W − 1: the window out keeps part of the window in
    (2, 2, 0, 16, 4),     # T = 0: the window is copied
    (2, 2, 77, 64, 3),    # the compile-time widths of 64 and 128 channels
    (1, 2, 45, 128, 8),
    (1, 1, 2, 64, 6),
    (2, 3, 150, 32, 5),   # the compile-time widths of 16 and 32 channels
    (3, 1, 61, 16, 2),
]


@pytest.mark.parametrize("B,H,T,D,W", CASES)
@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("act,use_bias,use_window", [(True, True, True), (False, False, False),
                                                     (True, False, True), (False, True, False)])
def test_forward_matches_oracle(B, H, T, D, W, io, act, use_bias, use_window):
    p = on_device(make_conv_inputs(B, H, T, D, W, io=io, seed=11 + T + D + W))
    y, wout = run_forward(p, act, use_bias, use_window)
    torch.cuda.synchronize()
    y_ref, wout_ref, scale = oracle_forward(p, act, use_bias, use_window)
    assert scaled_err(y, y_ref, scale) <= TOL_IO[io]
    assert np.array_equal(f64(wout), wout_ref)  # a copy of inputs: exact


@pytest.mark.parametrize("B,H,T,D,W", CASES)
@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("act,use_bias,use_window,use_gwo", [(True, True, True, True), (False, False, False, False),
                                                             (True, False, True, False)])
def test_backward_matches_oracle(B, H, T, D, W, io, act, use_bias, use_window, use_gwo):
    p = on_device(make_conv_inputs(B, H, T, D, W, io=io, seed=23 + T + D + W))
    g = kla.conv_backward(p["x"], p["weight"], p["bias"] if use_bias else None,
                          p["window"] if use_window else None, gy=p["gy"],
                          gwindow_out=p["gwindow_out"] if use_gwo else None,
                          activation=kla.ACT_SILU if act else kla.ACT_NONE)
    torch.cuda.synchronize()
    ref, s = oracle_backward(p, act, use_bias, use_window, use_gwo)
    assert scaled_err(g["gx"], ref["gx"], s["gx"]) <= TOL_IO[io]
    assert scaled_err(g["gwindow"], ref["gwindow"], s["gwindow"]) <= TOL_IO[io]
    assert scaled_err(g["gweight"], ref["gweight"], s["gweight"]) <= TOL_SUM
    assert scaled_err(g["gbias"], ref["gbias"], s["gbias"]) <= TOL_SUM


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_headline_stream_all_heads(io):
    """A q-shaped stream of the headline workload (B8 H16 T4096 d64), every
    element, forward and backward."""
    B, H, T, D, W = 8, 16, 4096, 64, 4
    p = on_device(make_conv_inputs(B, H, T, D, W, io=io, seed=2))
    y, wout = run_forward(p, True, True, True)
    g = kla.conv_backward(p["x"], p["weight"], p["bias"], p["window"], gy=p["gy"], gwindow_out=p["gwindow_out"])
    torch.cuda.synchronize()
    y_ref, wout_ref, scale = oracle_forward(p, True, True, True)
    assert scaled_err(y, y_ref, scale) <= TOL_IO[io]
    assert np.array_equal(f64(wout), wout_ref)
    ref, s = oracle_backward(p, True, True, True)
    for name in ("gx", "gwindow"):
        assert scaled_err(g[name], ref[name], s[name]) <= TOL_IO[io], name
    for name in ("gweight", "gbias"):
        assert scaled_err(g[name], ref[name], s[name]) <= TOL_SUM, name


def test_long_single_head_stream():
    """One head, 65549 tokens, 128 channels: long chunks and many blocks along T."""
    B, H, T, D, W = 1, 1, 65549, 128, 4
    p = on_device(make_conv_inputs(B, H, T, D, W, io="f32", seed=3))
    y, _ = run_forward(p, True, True, True)
    g = kla.conv_backward(p["x"], p["weight"], p["bias"], p["window"], gy=p["gy"], gwindow_out=p["gwindow_out"])
    torch.cuda.synchronize()
    y_ref, _, scale = oracle_forward(p, True, True, True)
    assert scaled_err(y, y_ref, scale) <= TOL_IO["f32"]
    ref, s = oracle_backward(p, True, True, True)
    for name in ("gx", "gwindow"):
        assert scaled_err(g[name], ref[name], s[name]) <= TOL_IO["f32"], name
    for name in ("gweight", "gbias"):
        assert scaled_err(g[name], ref[name], s[name]) <= TOL_SUM, name


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_streaming_and_decoding_equal_one_pass_bit_for_bit(io):
    """Pieces of the sequence with the window carried between calls — and,
    for the last 20 tokens, one token per call with the window updated in
    place — give exactly the outputs of one call."""
    B, H, T, D, W = 2, 4, 300, 64, 4
    p = on_device(make_conv_inputs(B, H, T, D, W, io=io, seed=5))
    y_all, wout_all = run_forward(p, True, True, True)
    win = p["window"].clone()
    ys = []
    for t0, t1 in ((0, 100), (100, 101), (101, 280)):
        y, win = kla.conv(p["x"][:, :, t0:t1].contiguous(), p["weight"], p["bias"], win)
        ys.append(y)
    for t in range(280, T):
        y, win = kla.conv(p["x"][:, :, t:t + 1].contiguous(), p["weight"], p["bias"], win, update_window=True)
        ys.append(y)
    torch.cuda.synchronize()
    assert torch.equal(torch.cat(ys, dim=2), y_all)
    assert torch.equal(win, wout_all)


def test_backward_is_deterministic():
    B, H, T, D, W = 4, 8, 3000, 64, 4
    p = on_device(make_conv_inputs(B, H, T, D, W, io="f32", seed=6))
    runs = [kla.conv_backward(p["x"], p["weight"], p["bias"], p["window"], gy=p["gy"],
                              gwindow_out=p["gwindow_out"]) for _ in range(2)]
    torch.cuda.synchronize()
    for name in ("gx", "gweight", "gbias", "gwindow"):
        assert torch.equal(runs[0][name], runs[1][name]), name


def test_backward_without_gy_or_parameter_gradients():
    """gy = NULL is zero: gx and gwindow are then the window-out gradient
    alone; skipping the tap and bias gradients needs no workspace."""
    B, H, T, D, W = 2, 2, 5, 16, 4
    p = on_device(make_conv_inputs(B, H, T, D, W, io="f32", seed=7))
    g = kla.conv_backward(p["x"], p["weight"], p["bias"], p["window"], gy=None, gwindow_out=p["gwindow_out"],
                          param_grads=False)
    torch.cuda.synchronize()
    gxe = torch.cat([g["gwindow"], g["gx"]], dim=2)  # tokens −3 … 4
    want = torch.zeros_like(gxe)
    want[:, :, -(W - 1):] = p["gwindow_out"]
    assert torch.equal(gxe, want)
    assert "gweight" not in g


def test_many_heads_one_token():
    """4096 heads, one token each (a decode step of the block's convolution)."""
    B, H, T, D, W = 256, 16, 1, 64, 4
    p = on_device(make_conv_inputs(B, H, T, D, W, io="bf16", seed=8))
    y, wout = run_forward(p, True, True, True)
    torch.cuda.synchronize()
    y_ref, wout_ref, scale = oracle_forward(p, True, True, True)
    assert scaled_err(y, y_ref, scale) <= TOL_IO["bf16"]
    assert np.array_equal(f64(wout), wout_ref)


def test_conv_then_scan_layer_prologue():
    """The block's order: q, k, v each through its own convolution and SiLU,
    then the scan, equals the oracle's convolution followed by the oracle's
    scan (the scan oracle on the convolved inputs)."""
    import oracle
    from bayesian_filtering_linear_gb300.inputs import make_inputs
    B, H, T, dk, dv, W = 1, 2, 64, 16, 16, 4
    inp = {k: v.to(DEV) for k, v in make_inputs(B, H, T, dk, dv, io="f32", seed=9).items()}
    conv_in = {n: on_device(make_conv_inputs(B, H, T, dk if n != "v" else dv, W, io="f32", seed=40 + i))
               for i, n in enumerate(("q", "k", "v"))}
    mixed = dict(inp)
    for n in ("q", "k", "v"):
        mixed[n], _ = kla.conv(conv_in[n]["x"], conv_in[n]["weight"], conv_in[n]["bias"])
    y, _, _ = kla.forward(mixed["q"], mixed["k"], mixed["v"], inp["lam_v"], inp["a"], inp["pbar"])
    torch.cuda.synchronize()
    ref_in = {n: C.conv(f64(conv_in[n]["x"]), f64(conv_in[n]["weight"]), f64(conv_in[n]["bias"]))[0]
              for n in ("q", "k", "v")}
    ref = oracle.forward64(ref_in["q"], ref_in["k"], ref_in["v"], f64(inp["lam_v"]), f64(inp["a"]),
                           f64(inp["pbar"]), f64(inp["lam0"]), f64(inp["eta0"]), want_scales=True)
    err = np.max(np.abs(f64(y) - ref["y"]) / (np.abs(ref["y"]) + ref["y_scale"] + 1e-30))
    assert err <= 1e-4


def test_block_backward_chains_scan_and_convolutions():
    """Training a KLA block end to end: q, k, v come from their own causal
    convolutions with SiLU, the scan runs on them, and the gradients flow
    back through kla_backward (dL/dq, dL/dk, dL/dv) into each convolution's
    kla_conv_backward (dL/dx, taps, bias). The same chain in the oracle: the
    fp64 convolutions, the fp64 scan's reverse mode, the fp64 convolution
    backward. Error relative to the largest reference value of each gradient
    (1e-4: fp32 arithmetic through two recursions and two W-term sums)."""
    import oracle
    from bayesian_filtering_linear_gb300.inputs import make_inputs
    B, H, T, dk, dv, W = 1, 2, 96, 16, 16, 4
    inp = {k: v.to(DEV) for k, v in make_inputs(B, H, T, dk, dv, io="f32", seed=12, random_state=True).items()}
    conv_in = {n: on_device(make_conv_inputs(B, H, T, dk if n != "v" else dv, W, io="f32", seed=60 + i))
               for i, n in enumerate(("q", "k", "v"))}
    for n in ("q", "k", "v"):  # keep q, k in the scale of the scan's recipe
        conv_in[n]["weight"] *= 0.5
    mixed = dict(inp)
    for n in ("q", "k", "v"):
        mixed[n], _ = kla.conv(conv_in[n]["x"], conv_in[n]["weight"], conv_in[n]["bias"], conv_in[n]["window"])
    g = torch.Generator().manual_seed(3)
    gy = torch.randn(B, H, T, dv, generator=g).to(DEV)
    gl, ge = torch.randn(B, H, dk, dv, generator=g).to(DEV), torch.randn(B, H, dk, dv, generator=g).to(DEV)
    sg = kla.backward(mixed["q"], mixed["k"], mixed["v"], inp["lam_v"], inp["a"], inp["pbar"], inp["lam0"],
                      inp["eta0"], gy=gy, glamT=gl, getaT=ge)
    cg = {n: kla.conv_backward(conv_in[n]["x"], conv_in[n]["weight"], conv_in[n]["bias"], conv_in[n]["window"],
                               gy=sg["g" + n]) for n in ("q", "k", "v")}
    torch.cuda.synchronize()

    ref_in = {n: C.conv(f64(conv_in[n]["x"]), f64(conv_in[n]["weight"]), f64(conv_in[n]["bias"]),
                        f64(conv_in[n]["window"]))[0] for n in ("q", "k", "v")}
    rs = oracle.backward64(ref_in["q"], ref_in["k"], ref_in["v"], f64(inp["lam_v"]), f64(inp["a"]), f64(inp["pbar"]),
                           f64(inp["lam0"]), f64(inp["eta0"]), f64(gy), f64(gl), f64(ge))
    for n in ("q", "k", "v"):
        rc = C.conv_backward(f64(conv_in[n]["x"]), f64(conv_in[n]["weight"]), f64(conv_in[n]["bias"]),
                             f64(conv_in[n]["window"]), rs["d" + n])
        for name in ("gx", "gweight", "gbias", "gwindow"):
            ref = rc[name]
            err = np.max(np.abs(f64(cg[n][name]) - ref)) / np.max(np.abs(ref))
            assert err <= 1e-4, (n, name, err)
    # the scan's own gradients of the other inputs, for completeness
    for name, key in (("glam_v", "dlam_v"), ("ga", "da"), ("gpbar", "dpbar"), ("glam0", "dlam0")):
        err = np.max(np.abs(f64(sg[name]) - rs[key])) / np.max(np.abs(rs[key]))
        assert err <= 1e-4, (name, err)
