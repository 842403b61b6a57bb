"""GPU test of kla_forward_chunked_noalloc, the entry point for callers that
cannot allocate device memory (allocator callbacks, allocation-free real-time
loops, frameworks that own every device allocation). It runs the
chunk-parallel scan with the library's own fixed 32 MiB device scratch
instead of a caller-provided workspace.

Checked through the C ABI against kla_forward on the same inputs with the
same chunk length, on two calls in a row with different shapes (the second
must not see stale scratch from the first), with an explicit, the automatic
and a one-chunk chunk length, and that a call needing more than 32 MiB of
scratch is refused before anything is launched. Kept in its own file, collected
last, so that a stop-at-first-failure run has already run every other test.
"""
import ctypes

import pytest
import torch

from bayesian_filtering_linear_gb300 import kla
from bayesian_filtering_linear_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 2e-2}
NAMES = ("q", "k", "v", "lam_v", "a", "pbar")


def _entry():
    fn = kla.LIB.kla_forward_chunked_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p] * 11 + [ctypes.c_int] * 7 + [ctypes.c_void_p]
    return fn


def _noalloc(x, io, chunk_len):
    B, H, T, dk = x["q"].shape
    dv = x["v"].shape[-1]
    y = torch.empty((B, H, T, dv), dtype=x["q"].dtype, device="cuda")
    lamT = torch.empty_like(x["lam0"])
    etaT = torch.empty_like(x["eta0"])
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    st = _entry()(*[p(x[n]) for n in NAMES], p(x["lam0"]), p(x["eta0"]), p(y), p(lamT), p(etaT),
                  B, H, T, dk, dv, kla.BF16 if io == "bf16" else kla.F32, chunk_len,
                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st, y, lamT, etaT


def _compare(x, io, chunk_len):
    B, H, T, dk = x["q"].shape
    dv = x["v"].shape[-1]
    y_ref, l_ref, e_ref = kla.forward(*[x[n] for n in NAMES], x["lam0"], x["eta0"], strategy="chunked",
                                      chunk_len=chunk_len)
    st, y, l, e = _noalloc(x, io, chunk_len)
    torch.cuda.synchronize()
    assert st == kla.OK, kla.status_string(st)
    scale = y_ref.float().abs().max()
    assert float((y.float() - y_ref.float()).abs().max() / scale) <= TOL[io]
    assert float(((l - l_ref).abs() / l_ref).max()) <= TOL[io]
    assert float((e - e_ref).abs().max() / e_ref.abs().max()) <= TOL[io]


# Two calls in a row with different shapes (the second call's scratch layout
# differs from the first's, so stale contents would show): an explicit chunk
# length, the automatic one (0), and a sequence no longer than one chunk
# (the plan then runs one chunk and uses no scratch).
@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("chunk_len,shapes", [
    (128, [(2, 3, 700, 64, 32), (1, 5, 1000, 32, 64)]),
    (0, [(1, 2, 900, 64, 64), (3, 1, 513, 128, 32)]),
    (256, [(2, 2, 200, 64, 32), (1, 3, 256, 16, 16)]),
], ids=["chunk128", "auto", "one-chunk"])
def test_noalloc_matches_kla_forward_on_two_calls(io, chunk_len, shapes):
    for seed, (B, H, T, dk, dv) in enumerate(shapes, start=21):
        x = {n: t.cuda() for n, t in make_inputs(B, H, T, dk, dv, io=io, seed=seed, random_state=True).items()}
        need = kla.plan(B, H, T, dk, dv, io, strategy="chunked", chunk_len=chunk_len)
        assert need["workspace_bytes"] <= 32 << 20
        if T > max(chunk_len, 32):
            assert need["strategy"] == "chunked" and need["workspace_bytes"] > 0
        _compare(x, io, chunk_len)


def test_noalloc_refuses_more_than_its_scratch():
    B, H, T, d = 64, 16, 64, 128
    need = kla.plan(B, H, T, d, d, "bf16", strategy="chunked", chunk_len=32)
    assert need["workspace_bytes"] > 32 << 20
    x = {n: t.cuda() for n, t in make_inputs(B, H, T, d, d, io="bf16", seed=3).items()}
    st, *_ = _noalloc(x, "bf16", 32)
    torch.cuda.synchronize()
    assert st == kla.ERR_WORKSPACE
