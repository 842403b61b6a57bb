"""Seeded synthetic inputs for the KLA scan (shared by the tests, the oracle
checks and the benchmark). This module draws random numbers only; it holds
none of the filter's arithmetic.

Distributions (one workload recipe, parameterised by shape and the mean of
the decay logit):

* q, k ~ N(0, 1/d_k)           per (t, i)       — read as variance 1/d_k
* v ~ N(0, 1)                  per (t, j)
* Λ^v = softplus(N(0, 1))      per (t, j)       — value precision, > 0
* a = sigmoid(N(a_logit_mean, 1))  per (t, i)   — OU decay in (0, 1)
* p̄ = softplus(N(−2, 1))       per (t, i)       — OU process noise, > 0
* λ0 = 1, η0 = 0 unless ``random_state=True`` (then λ0 = 0.5 + softplus(N(0,1)),
  η0 ~ N(0, 1)).

Draw order is fixed — q, k, v, Λ^v, a, p̄, then λ0, η0 — each a full fp32
tensor from one ``torch.Generator`` seeded with ``seed``; the tensors are then
cast to the I/O dtype, and those rounded values are what both the CUDA path
and the oracle read.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    """One synthetic workload: shapes, I/O dtype, seed and decay-logit mean."""
    name: str
    B: int
    H: int
    T: int
    dk: int
    dv: int
    io: str            # "f32" or "bf16"
    seed: int
    a_logit_mean: float = 2.0

    @property
    def tokens(self) -> int:
        return self.B * self.H * self.T


# The five named workloads. ``decode`` holds 1536 tokens: a 1024-token
# forward prefix followed by 512 single-token steps.
WORKLOADS = {
    "tiny": Workload("tiny", 1, 1, 256, 16, 16, "f32", 0),
    "medium": Workload("medium", 4, 8, 2048, 64, 64, "f32", 1),
    "headline": Workload("headline", 8, 16, 4096, 64, 64, "bf16", 2),
    "long": Workload("long", 1, 16, 65536, 128, 128, "bf16", 3, a_logit_mean=4.0),
    "decode": Workload("decode", 256, 16, 1536, 64, 64, "f32", 4),
}
DECODE_PREFIX = 1024

_DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


def io_dtype(io: str) -> torch.dtype:
    return _DTYPES[io]


def make_inputs(B: int, H: int, T: int, dk: int, dv: int, *, io: str = "f32", seed: int = 0,
                a_logit_mean: float = 2.0, random_state: bool = False,
                device: str | torch.device = "cpu") -> dict:
    """Draw one set of inputs. Returns a dict of contiguous tensors on ``device``:
    q, k, a, pbar ``[B,H,T,dk]`` and v, lam_v ``[B,H,T,dv]`` in the I/O dtype,
    lam0, eta0 ``[B,H,dk,dv]`` in fp32.

    With ``device='cpu'`` the values are reproducible across machines (torch's
    CPU generator); a CUDA device uses that device's generator (same recipe,
    different stream of numbers) so that large benchmark inputs need no
    host-to-device copy.
    """
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(int(seed))
    f32 = torch.float32

    def randn(*shape):
        return torch.randn(*shape, generator=g, dtype=f32, device=dev)

    sk, sv = (B, H, T, dk), (B, H, T, dv)
    q = randn(*sk) * dk ** -0.5
    k = randn(*sk) * dk ** -0.5
    v = randn(*sv)
    lam_v = torch.nn.functional.softplus(randn(*sv))
    a = torch.sigmoid(randn(*sk) + a_logit_mean)
    pbar = torch.nn.functional.softplus(randn(*sk) - 2.0)
    if random_state:
        lam0 = 0.5 + torch.nn.functional.softplus(randn(B, H, dk, dv))
        eta0 = randn(B, H, dk, dv)
    else:
        lam0 = torch.ones(B, H, dk, dv, dtype=f32, device=dev)
        eta0 = torch.zeros(B, H, dk, dv, dtype=f32, device=dev)
    dt = _DTYPES[io]
    out = {"q": q, "k": k, "v": v, "lam_v": lam_v, "a": a, "pbar": pbar}
    out = {n: t.to(dt).contiguous() for n, t in out.items()}
    out["lam0"], out["eta0"] = lam0.contiguous(), eta0.contiguous()
    return out


def make_workload(w: Workload | str, *, device: str | torch.device = "cpu", **kw) -> dict:
    if isinstance(w, str):
        w = WORKLOADS[w]
    return make_inputs(w.B, w.H, w.T, w.dk, w.dv, io=w.io, seed=w.seed,
                       a_logit_mean=w.a_logit_mean, device=device, **kw)


def make_conv_inputs(B: int, H: int, T: int, D: int, W: int, *, io: str = "f32", seed: int = 0,
                     device: str | torch.device = "cpu") -> dict:
    """Seeded inputs of the causal convolution that feeds the scan: x
    ``[B,H,T,D]`` ~ N(0, 1) and the carried window ``[B,H,W-1,D]`` ~ N(0, 1)
    in the I/O dtype; fp32 taps ``[H,D,W]`` ~ N(0, 1/W) and bias ``[H,D]`` ~
    N(0, 1/4); and, for the backward, gy ``[B,H,T,D]`` ~ N(0, 1) and
    gwindow_out ``[B,H,W-1,D]`` ~ N(0, 1) in the I/O dtype. Draw order: x,
    window, weight, bias, gy, gwindow_out."""
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(int(seed))

    def randn(*shape):
        return torch.randn(*shape, generator=g, dtype=torch.float32, device=dev)

    dt = _DTYPES[io]
    x = randn(B, H, T, D).to(dt).contiguous()
    window = randn(B, H, W - 1, D).to(dt).contiguous()
    weight = (randn(H, D, W) * W ** -0.5).contiguous()
    bias = (randn(H, D) * 0.5).contiguous()
    gy = randn(B, H, T, D).to(dt).contiguous()
    gwindow_out = randn(B, H, W - 1, D).to(dt).contiguous()
    return {"x": x, "window": window, "weight": weight, "bias": bias, "gy": gy, "gwindow_out": gwindow_out}
