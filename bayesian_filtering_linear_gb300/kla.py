"""Thin ctypes binding of ``libkla.so`` (the C ABI in ``include/kla.h``).

Argument marshalling only: tensors are checked for device, dtype and layout,
outputs and workspace are allocated with torch when not given, and the raw
device pointers plus torch's current CUDA stream are passed to the library.
Every step of the scan runs in the library's CUDA kernels; there is no other
implementation here. If the library is missing this module fails to import.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkla.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED_SHAPE, ERR_MISALIGNED, ERR_WORKSPACE, ERR_CUDA, ERR_TIMEOUT = range(7)
F32, BF16 = 0, 1
AUTO, SEQUENTIAL, CHUNKED = 0, 1, 2
_STRATEGIES = {"auto": AUTO, "sequential": SEQUENTIAL, "chunked": CHUNKED}
_IO = {torch.float32: F32, torch.bfloat16: BF16}
# Every function the header declares, for the export check.
EXPORTS = ("kla_plan", "kla_plan_for_sms", "kla_forward_workspace_size", "kla_forward", "kla_step",
           "kla_status_string", "kla_version", "kla_forward_chunked_noalloc", "kla_backward_workspace_size",
           "kla_backward", "kla_forward_uncertainty", "kla_step_gated", "kla_backward_plan_for_sms",
           "kla_shard_map", "kla_shard_start", "kla_conv", "kla_conv_backward_workspace_size",
           "kla_conv_backward")


class Options(ctypes.Structure):
    _fields_ = [("strategy", ctypes.c_int), ("chunk_len", ctypes.c_int), ("rows_per_lane", ctypes.c_int),
                ("gates", ctypes.c_int), ("coef_pass", ctypes.c_int)]


class BackwardPlanInfo(ctypes.Structure):
    _fields_ = [("cols_per_block", ctypes.c_int), ("cols_per_lane", ctypes.c_int), ("threads", ctypes.c_int),
                ("column_blocks", ctypes.c_int), ("workspace_bytes", ctypes.c_size_t)]


class PlanInfo(ctypes.Structure):
    _fields_ = [("strategy", ctypes.c_int), ("chunk_len", ctypes.c_int), ("num_chunks", ctypes.c_int),
                ("cols_per_block", ctypes.c_int), ("workspace_bytes", ctypes.c_size_t),
                ("rows_per_lane", ctypes.c_int), ("coef_pass", ctypes.c_int)]


def load_library(path: str = LIB_PATH):
    """Open a build of the library and declare the C signatures."""
    if not os.path.exists(path):
        raise ImportError(f"{path} is not built; run `python -m bayesian_filtering_linear_gb300.build` "
                          "(needs nvcc) — there is no fallback implementation")
    # RTLD_NOW: an unresolved symbol fails here, not at the first call of the
    # function that needs it.
    lib = ctypes.CDLL(path, mode=os.RTLD_NOW | os.RTLD_LOCAL)
    vp, i, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    lib.kla_status_string.restype = ctypes.c_char_p
    lib.kla_status_string.argtypes = [i]
    lib.kla_version.restype = i
    lib.kla_version.argtypes = []
    lib.kla_plan.restype = i
    lib.kla_plan.argtypes = [i, i, i, i, i, i, ctypes.POINTER(Options), ctypes.POINTER(PlanInfo)]
    lib.kla_backward_plan_for_sms.restype = i
    lib.kla_backward_plan_for_sms.argtypes = [i, i, i, i, i, i, ctypes.POINTER(BackwardPlanInfo)]
    lib.kla_plan_for_sms.restype = i
    lib.kla_plan_for_sms.argtypes = [i, i, i, i, i, i, ctypes.POINTER(Options), i, ctypes.POINTER(PlanInfo)]
    lib.kla_forward_workspace_size.restype = sz
    lib.kla_forward_workspace_size.argtypes = [i, i, i, i, i, ctypes.POINTER(Options)]
    lib.kla_forward.restype = i
    lib.kla_forward.argtypes = [vp] * 11 + [i] * 6 + [vp, sz, ctypes.POINTER(Options), vp]
    lib.kla_step.restype = i
    lib.kla_step.argtypes = [vp] * 9 + [i] * 5 + [vp]
    lib.kla_forward_uncertainty.restype = i
    lib.kla_forward_uncertainty.argtypes = [vp] * 12 + [i] * 6 + [vp, sz, ctypes.POINTER(Options), vp]
    lib.kla_backward_workspace_size.restype = sz
    lib.kla_backward_workspace_size.argtypes = [i] * 5
    lib.kla_backward.restype = i
    lib.kla_backward.argtypes = [vp] * 19 + [i] * 7 + [vp, sz, vp]
    lib.kla_step_gated.restype = i
    lib.kla_step_gated.argtypes = [vp] * 9 + [i] * 6 + [vp]
    lib.kla_shard_map.restype = i
    lib.kla_shard_map.argtypes = [vp] * 7 + [i] * 7 + [vp]
    lib.kla_shard_start.restype = i
    lib.kla_shard_start.argtypes = [vp, i, vp, vp, vp, vp, i, i, i, i, vp]
    lib.kla_conv.restype = i
    lib.kla_conv.argtypes = [vp] * 6 + [i] * 7 + [vp]
    lib.kla_conv_backward_workspace_size.restype = sz
    lib.kla_conv_backward_workspace_size.argtypes = [i] * 5
    lib.kla_conv_backward.restype = i
    lib.kla_conv_backward.argtypes = [vp] * 10 + [i] * 7 + [vp, sz, vp]
    return lib


LIB = load_library()


class KlaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {LIB.kla_status_string(status).decode()} (status {status})")


def _check(status: int, where: str):
    if status != OK:
        raise KlaError(status, where)


def status_string(status: int) -> str:
    return LIB.kla_status_string(status).decode()


# kla_gate bits: the corresponding input holds a pre-activation
GATE_LAMV_SOFTPLUS, GATE_A_SIGMOID, GATE_PBAR_SOFTPLUS, GATE_PBAR_OU = 1, 2, 4, 8


# kla_coef_pass values
_COEF_PASS = {"auto": 0, "off": 1, "on": 2}


def options(strategy: str | int = "auto", chunk_len: int = 0, rows_per_lane: int = 0, gates: int = 0,
            coef_pass: str | int = "auto") -> Options:
    s = _STRATEGIES[strategy] if isinstance(strategy, str) else int(strategy)
    c = _COEF_PASS[coef_pass] if isinstance(coef_pass, str) else int(coef_pass)
    return Options(s, int(chunk_len), int(rows_per_lane), int(gates), c)


def plan(B: int, H: int, T: int, dk: int, dv: int, io: str | int = "bf16", strategy: str | int = "auto",
         chunk_len: int = 0, num_sms: int | None = None, rows_per_lane: int = 0,
         coef_pass: str | int = "auto") -> dict:
    """The launch plan kla_forward uses (for the current device, or for a
    device with ``num_sms`` SMs without touching CUDA)."""
    io_code = {"f32": F32, "bf16": BF16}.get(io, io)
    info = PlanInfo()
    opt = options(strategy, chunk_len, rows_per_lane, coef_pass=coef_pass)
    if num_sms is None:
        st = LIB.kla_plan(B, H, T, dk, dv, io_code, ctypes.byref(opt), ctypes.byref(info))
    else:
        st = LIB.kla_plan_for_sms(B, H, T, dk, dv, io_code, ctypes.byref(opt), int(num_sms), ctypes.byref(info))
    _check(st, "kla_plan")
    return {"strategy": {SEQUENTIAL: "sequential", CHUNKED: "chunked"}[info.strategy],
            "chunk_len": info.chunk_len, "num_chunks": info.num_chunks,
            "cols_per_block": info.cols_per_block, "workspace_bytes": int(info.workspace_bytes),
            "rows_per_lane": info.rows_per_lane, "coef_pass": bool(info.coef_pass)}


def backward_plan(B: int, H: int, T: int, dk: int, dv: int, num_sms: int | None = None) -> dict:
    """The launch geometry kla_backward uses on a device with ``num_sms`` SMs
    (the current device's count when None)."""
    if num_sms is None:
        num_sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    info = BackwardPlanInfo()
    _check(LIB.kla_backward_plan_for_sms(B, H, T, dk, dv, int(num_sms), ctypes.byref(info)), "kla_backward_plan")
    return {"cols_per_block": info.cols_per_block, "cols_per_lane": info.cols_per_lane, "threads": info.threads,
            "column_blocks": info.column_blocks, "workspace_bytes": int(info.workspace_bytes)}


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _need(t, name, dtype, shape, device):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def forward(q, k, v, lam_v, a, pbar, lam0=None, eta0=None, *, y=None, lamT=None, etaT=None,
            strategy: str | int = "auto", chunk_len: int = 0, workspace=None, stream=None,
            final_state: bool = True, rows_per_lane: int = 0, uncertainty: bool = False, y_var=None,
            gates: int = 0, coef_pass: str | int = "auto"):
    """Whole-sequence KLA scan. Returns ``(y, lamT, etaT)`` (the last two are
    None when ``final_state`` is False and none were given); with
    ``uncertainty`` (or a ``y_var`` buffer) also the variance readout
    ``y_var[t, j] = Σ_i q_i² / λ_{t,i,j}`` as a fourth element. ``gates``: kla_gate
    bits (GATE_*), the corresponding inputs being pre-activations.
    ``coef_pass``: "auto", "off" or "on" (kla_coef_pass; results do not depend on it)."""
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("inputs must be CUDA tensors")
    dt = q.dtype
    if dt not in _IO:
        raise TypeError(f"unsupported I/O dtype {dt}")
    for name, t, last in (("q", q, dk), ("k", k, dk), ("a", a, dk), ("pbar", pbar, dk),
                          ("v", v, dv), ("lam_v", lam_v, dv)):
        _need(t, name, dt, (B, H, T, last), dev)
    st_shape = (B, H, dk, dv)
    for name, t in (("lam0", lam0), ("eta0", eta0), ("lamT", lamT), ("etaT", etaT)):
        if t is not None:
            _need(t, name, torch.float32, st_shape, dev)
    if y is None:
        y = torch.empty((B, H, T, dv), dtype=dt, device=dev)
    else:
        _need(y, "y", dt, (B, H, T, dv), dev)
    if final_state and lamT is None:
        lamT = torch.empty(st_shape, dtype=torch.float32, device=dev)
        etaT = torch.empty(st_shape, dtype=torch.float32, device=dev)
    # the uncertainty readout never runs the coefficient pass: size its workspace without it
    want_var = uncertainty or y_var is not None
    opt = options(strategy, chunk_len, rows_per_lane, gates, "off" if want_var else coef_pass)
    with torch.cuda.device(dev):
        if workspace is None:
            info = PlanInfo()
            _check(LIB.kla_plan(B, H, T, dk, dv, _IO[dt], ctypes.byref(opt), ctypes.byref(info)), "kla_plan")
            nbytes = int(info.workspace_bytes)
            workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev) if nbytes else None
        ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
        if want_var:
            if y_var is None:
                y_var = torch.empty((B, H, T, dv), dtype=dt, device=dev)
            else:
                _need(y_var, "y_var", dt, (B, H, T, dv), dev)
            st = LIB.kla_forward_uncertainty(_ptr(q), _ptr(k), _ptr(v), _ptr(lam_v), _ptr(a), _ptr(pbar), _ptr(lam0),
                                             _ptr(eta0), _ptr(y), _ptr(y_var), _ptr(lamT), _ptr(etaT), B, H, T, dk,
                                             dv, _IO[dt], _ptr(workspace), ws_bytes, ctypes.byref(opt),
                                             _stream(stream))
            _check(st, "kla_forward_uncertainty")
            return y, lamT, etaT, y_var
        st = LIB.kla_forward(_ptr(q), _ptr(k), _ptr(v), _ptr(lam_v), _ptr(a), _ptr(pbar), _ptr(lam0), _ptr(eta0),
                             _ptr(y), _ptr(lamT), _ptr(etaT), B, H, T, dk, dv, _IO[dt],
                             _ptr(workspace), ws_bytes, ctypes.byref(opt), _stream(stream))
    _check(st, "kla_forward")
    return y, lamT, etaT


def step(q, k, v, lam_v, a, pbar, lam, eta, *, y=None, stream=None, gates: int = 0):
    """One decode step: q, k, a, pbar ``[B,H,dk]``, v, lam_v ``[B,H,dv]``;
    updates the fp32 state (lam, eta) ``[B,H,dk,dv]`` in place; returns y."""
    B, H, dk = q.shape
    dv = v.shape[-1]
    dev, dt = q.device, q.dtype
    if dt not in _IO:
        raise TypeError(f"unsupported I/O dtype {dt}")
    for name, t, last in (("q", q, dk), ("k", k, dk), ("a", a, dk), ("pbar", pbar, dk),
                          ("v", v, dv), ("lam_v", lam_v, dv)):
        _need(t, name, dt, (B, H, last), dev)
    _need(lam, "lam", torch.float32, (B, H, dk, dv), dev)
    _need(eta, "eta", torch.float32, (B, H, dk, dv), dev)
    if y is None:
        y = torch.empty((B, H, dv), dtype=dt, device=dev)
    else:
        _need(y, "y", dt, (B, H, dv), dev)
    with torch.cuda.device(dev):
        if gates:
            st = LIB.kla_step_gated(_ptr(q), _ptr(k), _ptr(v), _ptr(lam_v), _ptr(a), _ptr(pbar), _ptr(lam),
                                    _ptr(eta), _ptr(y), B, H, dk, dv, _IO[dt], int(gates), _stream(stream))
        else:
            st = LIB.kla_step(_ptr(q), _ptr(k), _ptr(v), _ptr(lam_v), _ptr(a), _ptr(pbar), _ptr(lam), _ptr(eta),
                              _ptr(y), B, H, dk, dv, _IO[dt], _stream(stream))
    _check(st, "kla_step")
    return y


def backward(q, k, v, lam_v, a, pbar, lam0=None, eta0=None, *, gy=None, glamT=None, getaT=None,
             state_grads: bool = True, workspace=None, stream=None, gates: int = 0):
    """Gradients of a scalar loss through :func:`forward`, given ``gy`` = dL/dy
    ``[B,H,T,dv]`` (I/O dtype) and optionally ``glamT``, ``getaT`` = dL/dλ_T,
    dL/dη_T (fp32 ``[B,H,dk,dv]``). Returns a dict with ``gq, gk, ga, gpbar``
    ``[B,H,T,dk]`` and ``gv, glam_v`` ``[B,H,T,dv]`` in the I/O dtype and, with
    ``state_grads``, ``glam0, geta0`` (fp32)."""
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    dev, dt = q.device, q.dtype
    if dev.type != "cuda":
        raise ValueError("inputs must be CUDA tensors")
    if dt not in _IO:
        raise TypeError(f"unsupported I/O dtype {dt}")
    for name, t, last in (("q", q, dk), ("k", k, dk), ("a", a, dk), ("pbar", pbar, dk),
                          ("v", v, dv), ("lam_v", lam_v, dv)):
        _need(t, name, dt, (B, H, T, last), dev)
    st_shape = (B, H, dk, dv)
    for name, t in (("lam0", lam0), ("eta0", eta0), ("glamT", glamT), ("getaT", getaT)):
        if t is not None:
            _need(t, name, torch.float32, st_shape, dev)
    if gy is not None:
        _need(gy, "gy", dt, (B, H, T, dv), dev)
    out = {n: torch.empty((B, H, T, dk), dtype=dt, device=dev) for n in ("gq", "gk", "ga", "gpbar")}
    out.update({n: torch.empty((B, H, T, dv), dtype=dt, device=dev) for n in ("gv", "glam_v")})
    if state_grads:
        out["glam0"] = torch.empty(st_shape, dtype=torch.float32, device=dev)
        out["geta0"] = torch.empty(st_shape, dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):
        if workspace is None:
            nbytes = LIB.kla_backward_workspace_size(B, H, T, dk, dv)
            if nbytes == ctypes.c_size_t(-1).value:
                raise KlaError(ERR_CUDA, "kla_backward_workspace_size")
            workspace = torch.empty(max(int(nbytes), 16), dtype=torch.uint8, device=dev)
        ws_bytes = workspace.numel() * workspace.element_size()
        st = LIB.kla_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(lam_v), _ptr(a), _ptr(pbar), _ptr(lam0), _ptr(eta0),
                              _ptr(gy), _ptr(glamT), _ptr(getaT), _ptr(out["gq"]), _ptr(out["gk"]), _ptr(out["gv"]),
                              _ptr(out["glam_v"]), _ptr(out["ga"]), _ptr(out["gpbar"]), _ptr(out.get("glam0")),
                              _ptr(out.get("geta0")), B, H, T, dk, dv, _IO[dt], int(gates), _ptr(workspace),
                              ws_bytes, _stream(stream))
    _check(st, "kla_backward")
    return out


# ---- context-parallel sharding over T -----------------------------------------

def shard_map(q, k, v, lam_v, a, pbar, *, gates: int = 0, out=None, stream=None):
    """The composed map of a shard (all of its tokens), ``[7, B, H, dk, dv]``
    fp32 (kla_shard_map): (A, B, C, D, E, F, G) take the state (P, μ) before
    the shard to P' = (A P + B)/(C P + D), μ' = (E P + F + G μ)/(C P + D)."""
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    dev, dt = q.device, q.dtype
    if dt not in _IO:
        raise TypeError(f"unsupported I/O dtype {dt}")
    for name, t, last in (("q", q, dk), ("k", k, dk), ("a", a, dk), ("pbar", pbar, dk),
                          ("v", v, dv), ("lam_v", lam_v, dv)):
        _need(t, name, dt, (B, H, T, last), dev)
    if out is None:
        out = torch.empty((7, B, H, dk, dv), dtype=torch.float32, device=dev)
    else:
        _need(out, "out", torch.float32, (7, B, H, dk, dv), dev)
    with torch.cuda.device(dev):
        st = LIB.kla_shard_map(_ptr(q), _ptr(k), _ptr(v), _ptr(lam_v), _ptr(a), _ptr(pbar), _ptr(out),
                               B, H, T, dk, dv, _IO[dt], int(gates), _stream(stream))
    _check(st, "kla_shard_map")
    return out


def shard_start(maps, lam0=None, eta0=None, *, lam_out=None, eta_out=None, stream=None):
    """Start state (λ, η) of the shard after those whose maps are stacked in
    ``maps`` ``[n, 7, B, H, dk, dv]`` (in sequence order), from (λ0, η0) (None:
    λ0 = 1, η0 = 0). Returns ``(lam, eta)`` fp32 ``[B, H, dk, dv]``."""
    n, seven, B, H, dk, dv = maps.shape
    if seven != 7:
        raise ValueError("maps must be [n, 7, B, H, dk, dv]")
    dev = maps.device
    _need(maps, "maps", torch.float32, tuple(maps.shape), dev)
    st_shape = (B, H, dk, dv)
    for name, t in (("lam0", lam0), ("eta0", eta0), ("lam_out", lam_out), ("eta_out", eta_out)):
        if t is not None:
            _need(t, name, torch.float32, st_shape, dev)
    lam_out = torch.empty(st_shape, dtype=torch.float32, device=dev) if lam_out is None else lam_out
    eta_out = torch.empty(st_shape, dtype=torch.float32, device=dev) if eta_out is None else eta_out
    with torch.cuda.device(dev):
        st = LIB.kla_shard_start(_ptr(maps) if n else None, n, _ptr(lam0), _ptr(eta0), _ptr(lam_out),
                                 _ptr(eta_out), B, H, dk, dv, _stream(stream))
    _check(st, "kla_shard_start")
    return lam_out, eta_out


def exchange_maps(local_map, group=None):
    """All-gather every rank's shard map, ``[world, 7, B, H, dk, dv]`` in rank
    order. With the NCCL backend the device tensors are gathered in place;
    with another backend (gloo) through host copies."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    nccl = dist.get_backend(group) == "nccl"
    src = local_map if nccl else local_map.cpu()
    parts = [torch.empty_like(src) for _ in range(world)]
    dist.all_gather(parts, src.contiguous(), group=group)
    out = torch.stack(parts)
    return out if out.device == local_map.device else out.to(local_map.device)


def forward_context_parallel(q, k, v, lam_v, a, pbar, lam0=None, eta0=None, *, group=None, gates: int = 0,
                             stream=None, **forward_kw):
    """KLA forward over a sequence cut along T across the ranks of ``group``
    (rank r holds the r-th contiguous token range of the same heads). Each
    rank composes its shard's map (kla_shard_map), the maps are all-gathered
    (the one exchange step), each rank applies the maps of the shards before
    its own to (λ0, η0) (kla_shard_start) and scans its shard from that state
    (kla_forward). Returns this rank's ``(y, lamT, etaT)``: y of its tokens and
    the state after its shard (the last rank's is the sequence's final state).
    λ0, η0 must be the same on every rank."""
    import torch.distributed as dist
    rank = dist.get_rank(group)
    local = shard_map(q, k, v, lam_v, a, pbar, gates=gates, stream=stream)
    maps = exchange_maps(local, group)
    lam_s, eta_s = shard_start(maps[:rank].contiguous(), lam0, eta0, stream=stream)
    return forward(q, k, v, lam_v, a, pbar, lam_s, eta_s, gates=gates, stream=stream, **forward_kw)


# ---- causal depthwise convolution with SiLU (the block around the scan) -------

ACT_NONE, ACT_SILU = 0, 1


def _conv_shapes(x, weight, window, W):
    B, H, T, D = x.shape
    if tuple(weight.shape) != (H, D, W):
        raise ValueError(f"weight has shape {tuple(weight.shape)}, expected {(H, D, W)}")
    return B, H, T, D


def conv(x, weight, bias=None, window=None, *, activation: int = ACT_SILU, y=None, window_out=None,
         update_window: bool = False, stream=None):
    """Causal depthwise convolution of ``x`` ``[B,H,T,D]`` with taps ``weight``
    ``[H,D,W]`` (fp32; tap W-1 multiplies the current token), optional
    ``bias`` ``[H,D]`` and SiLU (kla_conv). ``window`` ``[B,H,W-1,D]`` holds
    the W-1 inputs before the first token (None: zeros). Returns ``(y,
    window_out)``; with ``update_window`` the window is updated in place and
    returned as window_out."""
    W = weight.shape[-1]
    B, H, T, D = _conv_shapes(x, weight, window, W)
    dev, dt = x.device, x.dtype
    if dt not in _IO:
        raise TypeError(f"unsupported I/O dtype {dt}")
    _need(weight, "weight", torch.float32, (H, D, W), dev)
    if bias is not None:
        _need(bias, "bias", torch.float32, (H, D), dev)
    wshape = (B, H, W - 1, D)
    if window is not None:
        _need(window, "window", dt, wshape, dev)
    if y is None:
        y = torch.empty((B, H, T, D), dtype=dt, device=dev)
    else:
        _need(y, "y", dt, (B, H, T, D), dev)
    if update_window:
        if window is None:
            raise ValueError("update_window needs a window")
        window_out = window
    elif window_out is None:
        window_out = torch.empty(wshape, dtype=dt, device=dev)
    else:
        _need(window_out, "window_out", dt, wshape, dev)
    with torch.cuda.device(dev):
        st = LIB.kla_conv(_ptr(x), _ptr(weight), _ptr(bias), _ptr(window), _ptr(y), _ptr(window_out),
                          B, H, T, D, W, _IO[dt], int(activation), _stream(stream))
    _check(st, "kla_conv")
    return y, window_out


def conv_backward(x, weight, bias=None, window=None, *, gy=None, gwindow_out=None, activation: int = ACT_SILU,
                  param_grads: bool = True, window_grad: bool = True, workspace=None, stream=None):
    """Gradients through :func:`conv` (kla_conv_backward) given ``gy`` = dL/dy
    and optionally ``gwindow_out`` = dL/d(window out). Returns a dict with
    ``gx`` and, with ``window_grad``, ``gwindow`` (I/O dtype), and with
    ``param_grads`` ``gweight`` ``[H,D,W]`` and ``gbias`` ``[H,D]`` (fp32)."""
    W = weight.shape[-1]
    B, H, T, D = _conv_shapes(x, weight, window, W)
    dev, dt = x.device, x.dtype
    if dt not in _IO:
        raise TypeError(f"unsupported I/O dtype {dt}")
    _need(weight, "weight", torch.float32, (H, D, W), dev)
    if bias is not None:
        _need(bias, "bias", torch.float32, (H, D), dev)
    wshape = (B, H, W - 1, D)
    for name, t in (("window", window), ("gwindow_out", gwindow_out)):
        if t is not None:
            _need(t, name, dt, wshape, dev)
    if gy is not None:
        _need(gy, "gy", dt, (B, H, T, D), dev)
    out = {"gx": torch.empty((B, H, T, D), dtype=dt, device=dev)}
    if window_grad:
        out["gwindow"] = torch.empty(wshape, dtype=dt, device=dev)
    if param_grads:
        out["gweight"] = torch.empty((H, D, W), dtype=torch.float32, device=dev)
        out["gbias"] = torch.empty((H, D), dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):
        if workspace is None and param_grads:
            nbytes = LIB.kla_conv_backward_workspace_size(B, H, T, D, W)
            if nbytes == ctypes.c_size_t(-1).value:
                raise KlaError(ERR_CUDA, "kla_conv_backward_workspace_size")
            workspace = torch.empty(max(int(nbytes), 16), dtype=torch.uint8, device=dev)
        ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
        st = LIB.kla_conv_backward(_ptr(x), _ptr(weight), _ptr(bias), _ptr(window), _ptr(gy), _ptr(gwindow_out),
                                   _ptr(out["gx"]), _ptr(out.get("gweight")), _ptr(out.get("gbias")),
                                   _ptr(out.get("gwindow")), B, H, T, D, W, _IO[dt], int(activation),
                                   _ptr(workspace), ws_bytes, _stream(stream))
    _check(st, "kla_conv_backward")
    return out


# ---- autograd: the entry points as differentiable torch operations ------------

class _ScanFunction(torch.autograd.Function):
    """kla_forward with kla_backward as its derivative."""

    @staticmethod
    def forward(ctx, q, k, v, lam_v, a, pbar, lam0, eta0, gates):
        y, lamT, etaT = forward(q, k, v, lam_v, a, pbar, lam0, eta0, gates=gates)
        ctx.save_for_backward(q, k, v, lam_v, a, pbar, lam0, eta0)
        ctx.gates = gates
        return y, lamT, etaT

    @staticmethod
    def backward(ctx, gy, glamT, getaT):
        q, k, v, lam_v, a, pbar, lam0, eta0 = ctx.saved_tensors
        g = backward(q, k, v, lam_v, a, pbar, lam0, eta0,
                     gy=None if gy is None else gy.to(q.dtype).contiguous(),
                     glamT=None if glamT is None else glamT.contiguous(),
                     getaT=None if getaT is None else getaT.contiguous(),
                     state_grads=lam0 is not None, gates=ctx.gates)
        return (g["gq"], g["gk"], g["gv"], g["glam_v"], g["ga"], g["gpbar"], g.get("glam0"), g.get("geta0"), None)


def scan(q, k, v, lam_v, a, pbar, lam0=None, eta0=None, *, gates: int = 0):
    """Differentiable KLA scan (autograd): returns ``(y, lamT, etaT)`` like
    :func:`forward`; gradients come from kla_backward."""
    return _ScanFunction.apply(q, k, v, lam_v, a, pbar, lam0, eta0, int(gates))


class _ConvFunction(torch.autograd.Function):
    """kla_conv with kla_conv_backward as its derivative."""

    @staticmethod
    def forward(ctx, x, weight, bias, window, activation):
        y, wout = conv(x, weight, bias, window, activation=activation)
        ctx.save_for_backward(x, weight, bias, window)
        ctx.activation = activation
        return y, wout

    @staticmethod
    def backward(ctx, gy, gwindow_out):
        x, weight, bias, window = ctx.saved_tensors
        g = conv_backward(x, weight, bias, window,
                          gy=None if gy is None else gy.to(x.dtype).contiguous(),
                          gwindow_out=None if gwindow_out is None else gwindow_out.to(x.dtype).contiguous(),
                          activation=ctx.activation, window_grad=window is not None)
        return (g["gx"], g["gweight"], None if bias is None else g["gbias"], g.get("gwindow"), None)


def causal_conv(x, weight, bias=None, window=None, *, activation: int = ACT_SILU):
    """Differentiable causal convolution with SiLU (autograd): returns
    ``(y, window_out)`` like :func:`conv`; gradients come from
    kla_conv_backward."""
    return _ConvFunction.apply(x, weight, bias, window, int(activation))
