"""Causal depthwise 1-D convolution with an optional SiLU, in fp64 — TEST
INFRASTRUCTURE ONLY (part of the oracle package; see its header).

Source: "Technische Samenvatting: Kalman Linear Attention (KLA)",
Methodologie §4 (Architectuur): the KLA layer is a drop-in sequence mixer
inside a fused, Mamba-like MLP block that adds 1-D causal convolutions and
SiLU activations around the scan. The pages give neither the kernel width
nor the weights; the reading taken here (the depthwise causal convolution of
such blocks) is:

* a stream x is ``[B, H, T, D]``; each channel (h, d) has its own W taps
  ``weight[h, d, 0..W-1]`` and an optional bias ``bias[h, d]``;
* tap k multiplies the input W-1-k tokens back:
      u[t] = bias + sum_k weight[k] * x[t - (W-1) + k]
  (tap W-1 is the current token), so no output depends on a later token;
* inputs before the first token come from a window of the W-1 previous
  inputs (``window[:, :, j]`` is token j - (W-1)), zeros at a sequence start;
  the call also returns the window after its last token, so a sequence cut
  into pieces (or fed one token at a time) gives the same outputs;
* y = SiLU(u) = u * sigmoid(u), or y = u without the activation.

:func:`conv` is that definition; :func:`conv_backward` its reverse-mode
derivative for a loss L with dL/dy = ``gy`` and dL/d(window out) =
``gwindow_out``. ``_mutant`` > 0 plants one mistake (tests only):
1 reverses the taps, 2 returns the window one token early, 3 drops the
u·(1 - sigmoid) term of SiLU', 4 pairs each tap's gradient with the input one
token off.
"""
from __future__ import annotations

import numpy as np


def sigmoid(u):
    return 1.0 / (1.0 + np.exp(-u))


def silu(u):
    return u * sigmoid(u)


def dsilu(u, _mutant: int = 0):
    """d/du of u·sigmoid(u) = sigmoid(u)·(1 + u·(1 − sigmoid(u)))."""
    s = sigmoid(u)
    return s if _mutant == 3 else s * (1.0 + u * (1.0 - s))


def _extended(x, window, W):
    """The window followed by x along T: index W-1+t holds token t."""
    B, H, T, D = x.shape
    if window is None:
        window = np.zeros((B, H, W - 1, D))
    return np.concatenate([np.asarray(window, np.float64), np.asarray(x, np.float64)], axis=2)


def preactivation(x, weight, bias=None, window=None, _mutant: int = 0):
    """u[b, h, t, d] = bias[h, d] + sum_k weight[h, d, k] * x[b, h, t - (W-1) + k, d]."""
    x = np.asarray(x, np.float64)
    weight = np.asarray(weight, np.float64)
    T = x.shape[2]
    W = weight.shape[-1]
    xe = _extended(x, window, W)
    u = np.zeros(x.shape)
    if bias is not None:
        u += np.asarray(bias, np.float64)[None, :, None, :]
    for k in range(W):
        tap = W - 1 - k if _mutant == 1 else k
        u += weight[None, :, None, :, tap] * xe[:, :, k:k + T, :]
    return u


def conv(x, weight, bias=None, window=None, activation: bool = True, _mutant: int = 0):
    """Returns (y [B,H,T,D], window_out [B,H,W-1,D])."""
    W = np.asarray(weight).shape[-1]
    T = np.asarray(x).shape[2]
    u = preactivation(x, weight, bias, window, _mutant)
    y = silu(u) if activation else u
    xe = _extended(x, window, W)
    lo = T - 1 if _mutant == 2 else T
    return y, xe[:, :, lo:lo + W - 1, :].copy()


def conv_backward(x, weight, bias=None, window=None, gy=None, gwindow_out=None, activation: bool = True,
                  _mutant: int = 0):
    """Gradients of L through :func:`conv`: dict with ``gx`` [B,H,T,D],
    ``gweight`` [H,D,W], ``gbias`` [H,D] and ``gwindow`` [B,H,W-1,D]
    (dL/d(window in))."""
    x = np.asarray(x, np.float64)
    weight = np.asarray(weight, np.float64)
    B, H, T, D = x.shape
    W = weight.shape[-1]
    xe = _extended(x, window, W)
    gy = np.zeros(x.shape) if gy is None else np.asarray(gy, np.float64)
    u = preactivation(x, weight, bias, window)
    gu = gy * dsilu(u, _mutant) if activation else gy
    gxe = np.zeros(xe.shape)
    if gwindow_out is not None:  # the window out is a copy of the last W-1 extended inputs
        gxe[:, :, T:T + W - 1, :] += np.asarray(gwindow_out, np.float64)
    gweight = np.zeros((H, D, W))
    for k in range(W):
        gxe[:, :, k:k + T, :] += weight[None, :, None, :, k] * gu
        off = k + 1 if _mutant == 4 and k + 1 + T <= T + W - 1 else k
        gweight[:, :, k] = np.einsum("bhtd,bhtd->hd", gu, xe[:, :, off:off + T, :])
    return {"gx": gxe[:, :, W - 1:, :], "gweight": gweight, "gbias": gu.sum(axis=(0, 2)),
            "gwindow": gxe[:, :, :W - 1, :]}
