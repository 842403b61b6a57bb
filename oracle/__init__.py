"""Reference oracle for the Kalman Linear Attention scan — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg may import this package. The product path (the CUDA library in
``bayesian_filtering_linear_gb300``) never imports it, and this package never
imports the product path.

Contents
--------
* :func:`forward` — ctypes wrapper of ``kla_oracle.cpp``: the plain per-element
  variance-form Kalman loop in fp64 (or fp32), multithreaded over heads.
* :func:`forward64` — the same loop on fp64 inputs (for finite differences).
* :func:`backward` / :func:`backward64` — its exact reverse-mode derivative in
  fp64 (gradients of a loss with respect to every input, given dL/dy and
  optionally dL/dλ_T, dL/dη_T), with condition scales.
* :mod:`oracle.exact` — exact-rational information-form Möbius recursion and
  dense Gaussian conditioning of the joint chain, used to pin the C++ loop.
* :mod:`oracle.gates` — the gate activations of the inputs and their chain rule.
* :mod:`oracle.conv` — the causal depthwise convolution with SiLU of the block
  around the scan (Methodologie §4), forward and backward, in fp64 numpy.

Source: "Technische Samenvatting: Kalman Linear Attention (KLA)"
(gist.science/nl/paper/2602.10743), Methodologie §1 (model) and §2 (Möbius
precision recursion, affine mean recursion).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kla_oracle.cpp")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "libkla_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False, mutant: int = 0) -> str:
    """Compile ``kla_oracle.cpp`` with g++ -O2 (no fast-math, no FMA
    contraction, so x86-64 and aarch64 round identically) into ``_build/``.
    ``mutant`` > 0 builds a copy with one planted mistake (tests only)."""
    os.makedirs(_BUILD, exist_ok=True)
    lib = _LIB if mutant == 0 else os.path.join(_BUILD, f"libkla_oracle_mutant{mutant}.so")
    if force or not os.path.exists(lib) or os.path.getmtime(lib) < os.path.getmtime(_SRC):
        tmp = lib + f".tmp{os.getpid()}"
        cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-pthread",
               "-fno-fast-math", "-ffp-contract=off", f"-DKLA_ORACLE_MUTANT={int(mutant)}",
               _SRC, "-o", tmp]
        subprocess.run(cmd, check=True)
        os.replace(tmp, lib)
    return lib


def _declare(lib):
    fp = ctypes.c_void_p
    lib.kla_oracle_forward_f64.restype = ctypes.c_longlong
    lib.kla_oracle_forward_f64.argtypes = [fp] * 8 + [ctypes.c_int] * 5 + [fp] * 6 + [ctypes.c_int]
    lib.kla_oracle_forward_f32.restype = ctypes.c_longlong
    lib.kla_oracle_forward_f32.argtypes = [fp] * 8 + [ctypes.c_int] * 5 + [fp] * 3 + [ctypes.c_int]
    lib.kla_oracle_forward_f64in.restype = ctypes.c_longlong
    lib.kla_oracle_forward_f64in.argtypes = [fp] * 8 + [ctypes.c_int] * 5 + [fp] * 5 + [ctypes.c_int]
    for name in ("kla_oracle_backward_f64", "kla_oracle_backward_f64in"):
        f = getattr(lib, name)
        f.restype = ctypes.c_longlong
        f.argtypes = [fp] * 11 + [ctypes.c_int] * 5 + [fp] * 16 + [ctypes.c_int]
    return lib


_mutants = {}


def _load(mutant: int = 0):
    global _lib
    with _lock:
        if mutant:
            if mutant not in _mutants:
                _mutants[mutant] = _declare(ctypes.CDLL(build(mutant=mutant)))
            return _mutants[mutant]
        if _lib is None:
            lib = ctypes.CDLL(build())
            _lib = _declare(lib)
    return _lib


def _f32(x):
    """Widen to a contiguous float32 numpy array (exact for bf16 / fp32 values)."""
    if x is None:
        return None
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().to("cpu", torch.float32).contiguous().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def forward(q, k, v, lam_v, a, pbar, lam0=None, eta0=None, *, precision: str = "f64",
            nthreads: int | None = None, heads=None, want_scales: bool = True, want_var: bool = False,
            _mutant: int = 0) -> dict:
    """Run the oracle over every head (or the flat head indices in ``heads``).

    Shapes: q, k, a, pbar ``[B,H,T,dk]``; v, lam_v ``[B,H,T,dv]``; lam0, eta0
    ``[B,H,dk,dv]`` or None (λ0 = 1, η0 = 0). With ``heads`` given, the
    selected heads are gathered into a ``[n,1,...]`` batch and the returned
    arrays have that leading shape.

    Returns a dict with ``y [B,H,T,dv]``, ``lamT``, ``etaT`` ``[B,H,dk,dv]``,
    (fp64, with ``want_var``) ``y_var [B,H,T,dv]`` = Σ_i q_i² P (all terms ≥ 0,
    so it is its own condition scale),
    (fp64 only) the condition scales ``y_scale`` and ``eta_scale``, and
    ``violations`` — the count of invariant violations (0 expected).
    """
    if heads is not None:
        # gather the selected heads first (before widening), as [n, 1, ...]
        B0, H0 = q.shape[:2]
        idx = list(heads)

        def sel(x):
            if x is None:
                return None
            flat = x.reshape((B0 * H0,) + tuple(x.shape[2:]))
            return flat[idx][:, None] if not isinstance(flat, np.ndarray) else flat[np.asarray(idx)][:, None]
        q, k, v, lam_v, a, pbar, lam0, eta0 = (sel(x) for x in (q, k, v, lam_v, a, pbar, lam0, eta0))
    arrs = [_f32(x) for x in (q, k, v, lam_v, a, pbar)]
    l0, e0 = _f32(lam0), _f32(eta0)
    B, H, T, dk = arrs[0].shape
    dv = arrs[2].shape[-1]
    for x, last in zip(arrs, (dk, dk, dv, dv, dk, dk)):
        if x.shape != (B, H, T, last):
            raise ValueError(f"bad input shape {x.shape}, expected {(B, H, T, last)}")
    for s in (l0, e0):
        if s is not None and s.shape != (B, H, dk, dv):
            raise ValueError(f"bad state shape {s.shape}")
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    lib = _load(_mutant)
    dt = np.float64 if precision == "f64" else np.float32
    y = np.empty((B, H, T, dv), dt)
    lamT = np.empty((B, H, dk, dv), dt)
    etaT = np.empty((B, H, dk, dv), dt)
    out = {"y": y, "lamT": lamT, "etaT": etaT}
    if precision == "f64":
        ys = np.empty((B, H, T, dv), np.float64) if want_scales else None
        es = np.empty((B, H, dk, dv), np.float64) if want_scales else None
        yv = np.empty((B, H, T, dv), np.float64) if want_var else None
        nv = lib.kla_oracle_forward_f64(*[_ptr(x) for x in arrs], _ptr(l0), _ptr(e0),
                                        B, H, T, dk, dv, _ptr(y), _ptr(lamT), _ptr(etaT),
                                        _ptr(ys), _ptr(es), _ptr(yv), int(nthreads))
        if want_scales:
            out["y_scale"], out["eta_scale"] = ys, es
        if want_var:
            out["y_var"] = yv
    elif precision == "f32":
        nv = lib.kla_oracle_forward_f32(*[_ptr(x) for x in arrs], _ptr(l0), _ptr(e0),
                                        B, H, T, dk, dv, _ptr(y), _ptr(lamT), _ptr(etaT),
                                        int(nthreads))
    else:
        raise ValueError("precision must be 'f64' or 'f32'")
    if nv < 0:
        raise ValueError("oracle rejected its arguments")
    out["violations"] = int(nv)
    return out


def _f64(x):
    if x is None:
        return None
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().to("cpu", torch.float64).contiguous().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _shapes(arrs):
    B, H, T, dk = arrs[0].shape
    dv = arrs[2].shape[-1]
    for x, last in zip(arrs, (dk, dk, dv, dv, dk, dk)):
        if x.shape != (B, H, T, last):
            raise ValueError(f"bad input shape {x.shape}, expected {(B, H, T, last)}")
    return B, H, T, dk, dv


def forward64(q, k, v, lam_v, a, pbar, lam0=None, eta0=None, *, nthreads: int | None = None,
              want_scales: bool = False, _mutant: int = 0) -> dict:
    """The fp64 loop of :func:`forward` on fp64 inputs (no rounding of the
    inputs to float32). Returns ``y``, ``lamT``, ``etaT`` (and with
    ``want_scales`` the condition scales ``y_scale``, ``eta_scale``)."""
    arrs = [_f64(x) for x in (q, k, v, lam_v, a, pbar)]
    l0, e0 = _f64(lam0), _f64(eta0)
    B, H, T, dk, dv = _shapes(arrs)
    y = np.empty((B, H, T, dv))
    lamT = np.empty((B, H, dk, dv))
    etaT = np.empty((B, H, dk, dv))
    ys = np.empty((B, H, T, dv)) if want_scales else None
    es = np.empty((B, H, dk, dv)) if want_scales else None
    nv = _load(_mutant).kla_oracle_forward_f64in(*[_ptr(x) for x in arrs], _ptr(l0), _ptr(e0), B, H, T, dk, dv,
                                                 _ptr(y), _ptr(lamT), _ptr(etaT), _ptr(ys), _ptr(es),
                                                 int(nthreads or os.cpu_count() or 1))
    if nv < 0:
        raise ValueError("oracle rejected its arguments")
    out = {"y": y, "lamT": lamT, "etaT": etaT}
    if want_scales:
        out["y_scale"], out["eta_scale"] = ys, es
    return out


GRAD_NAMES = ("dq", "dk", "da", "dpbar", "dv", "dlam_v", "dlam0", "deta0")


def _backward(conv, entry, q, k, v, lam_v, a, pbar, lam0, eta0, dy, dlamT, detaT, nthreads, heads,
              want_scales, _mutant):
    if heads is not None:
        B0, H0 = q.shape[:2]
        idx = np.asarray(list(heads))

        def sel(x):
            if x is None:
                return None
            x = conv(x)
            return x.reshape((B0 * H0,) + x.shape[2:])[idx][:, None]
        q, k, v, lam_v, a, pbar, lam0, eta0, dy, dlamT, detaT = (
            sel(x) for x in (q, k, v, lam_v, a, pbar, lam0, eta0, dy, dlamT, detaT))
    arrs = [conv(x) for x in (q, k, v, lam_v, a, pbar)]
    l0, e0, gy, gl, ge = (conv(x) for x in (lam0, eta0, dy, dlamT, detaT))
    B, H, T, dk, dv = _shapes(arrs)
    shapes = {"dq": (B, H, T, dk), "dk": (B, H, T, dk), "da": (B, H, T, dk), "dpbar": (B, H, T, dk),
              "dv": (B, H, T, dv), "dlam_v": (B, H, T, dv), "dlam0": (B, H, dk, dv), "deta0": (B, H, dk, dv)}
    for name, x in (("dy", gy), ("dlamT", gl), ("detaT", ge)):
        want = (B, H, T, dv) if name == "dy" else (B, H, dk, dv)
        if x is not None and x.shape != want:
            raise ValueError(f"bad {name} shape {x.shape}, expected {want}")
    grads = {n: np.zeros(shapes[n]) for n in GRAD_NAMES}
    scales = {n: np.zeros(shapes[n]) for n in GRAD_NAMES} if want_scales else {n: None for n in GRAD_NAMES}
    lib = _load(_mutant)
    rc = getattr(lib, entry)(*[_ptr(x) for x in arrs], _ptr(l0), _ptr(e0), _ptr(gy), _ptr(gl), _ptr(ge),
                             B, H, T, dk, dv, *[_ptr(grads[n]) for n in GRAD_NAMES],
                             *[_ptr(scales[n]) for n in GRAD_NAMES], int(nthreads or os.cpu_count() or 1))
    if rc < 0:
        raise ValueError("oracle rejected its arguments")
    out = dict(grads)
    if want_scales:
        out.update({n + "_scale": scales[n] for n in GRAD_NAMES})
    return out


def backward(q, k, v, lam_v, a, pbar, lam0=None, eta0=None, dy=None, dlamT=None, detaT=None, *,
             nthreads: int | None = None, heads=None, want_scales: bool = True, _mutant: int = 0) -> dict:
    """Gradients of a scalar loss L with respect to every input, given
    dy = dL/dy ``[B,H,T,dv]`` and optionally dlamT, detaT = dL/dλ_T, dL/dη_T
    ``[B,H,dk,dv]`` (None = 0), in fp64 from the float32 values the GPU reads.
    Returns ``dq, dk, da, dpbar`` ``[B,H,T,dk]``, ``dv, dlam_v`` ``[B,H,T,dv]``,
    ``dlam0, deta0`` ``[B,H,dk,dv]`` and, with ``want_scales``, a ``<name>_scale``
    condition scale for each. ``heads`` selects flat head indices (returned
    as a ``[n,1,...]`` batch), as in :func:`forward`."""
    return _backward(_f32, "kla_oracle_backward_f64", q, k, v, lam_v, a, pbar, lam0, eta0, dy, dlamT, detaT,
                     nthreads, heads, want_scales, _mutant)


def backward64(q, k, v, lam_v, a, pbar, lam0=None, eta0=None, dy=None, dlamT=None, detaT=None, *,
               nthreads: int | None = None, want_scales: bool = False, _mutant: int = 0) -> dict:
    """:func:`backward` on fp64 inputs (for finite-difference checks)."""
    return _backward(_f64, "kla_oracle_backward_f64in", q, k, v, lam_v, a, pbar, lam0, eta0, dy, dlamT, detaT,
                     nthreads, None, want_scales, _mutant)
