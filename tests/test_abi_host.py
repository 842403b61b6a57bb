"""C-ABI checks that need no GPU: the library loads, exports every function
``include/kla.h`` declares, rejects bad arguments with the documented status
before making any CUDA call, and plans launches deterministically.

Only argument combinations that fail validation are passed with placeholder
pointers, so nothing here can reach a kernel even on a machine with a GPU.
"""
import ctypes
import os
import re
import subprocess

import pytest
import torch

from bayesian_filtering_linear_gb300 import kla

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kla.h")
L = kla.LIB
P = ctypes.c_void_p(0x10000)      # 16-byte aligned placeholder (never dereferenced)
MIS = ctypes.c_void_p(0x10004)    # misaligned placeholder


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kla_[a-z_]+)\s*\(", text)))


def test_library_exports_every_declared_function():
    declared = header_functions()
    assert set(declared) == set(kla.EXPORTS)
    out = subprocess.run(["nm", "-D", "--defined-only", kla.LIB_PATH], capture_output=True, text=True, check=True)
    exported = set(re.findall(r"\bT (kla_[a-z_]+)", out.stdout))
    missing = [f for f in declared if f not in exported]
    assert not missing, missing
    for f in declared:
        assert hasattr(L, f)


def test_version_and_status_strings():
    assert L.kla_version() == 100
    for s in range(7):
        assert kla.status_string(s)
    assert "unknown" in kla.status_string(99)


def fwd(B=1, H=1, T=8, dk=16, dv=16, io=kla.F32, ptrs=None, lam0=None, eta0=None, lamT=None, etaT=None,
        ws=None, ws_bytes=0, opt=None):
    ptrs = ptrs or {}
    g = lambda n: ptrs.get(n, P)
    return L.kla_forward(g("q"), g("k"), g("v"), g("lam_v"), g("a"), g("pbar"), lam0, eta0, g("y"), lamT, etaT,
                         B, H, T, dk, dv, io, ws, ws_bytes, opt, None)


@pytest.mark.parametrize("dk,dv", [(8, 16), (16, 24), (256, 16), (48, 64), (0, 16)])
def test_unsupported_head_dims(dk, dv):
    assert fwd(dk=dk, dv=dv) == kla.ERR_UNSUPPORTED_SHAPE


@pytest.mark.parametrize("B,H,T", [(-1, 1, 8), (1, -2, 8), (1, 1, -5)])
def test_negative_sizes(B, H, T):
    assert fwd(B=B, H=H, T=T) == kla.ERR_INVALID_ARG


@pytest.mark.parametrize("name", ["q", "k", "v", "lam_v", "a", "pbar", "y"])
def test_null_required_pointer(name):
    assert fwd(ptrs={name: None}) == kla.ERR_INVALID_ARG


@pytest.mark.parametrize("name", ["q", "k", "v", "lam_v", "a", "pbar", "y"])
def test_misaligned_pointer(name):
    assert fwd(ptrs={name: MIS}) == kla.ERR_MISALIGNED


def test_state_pointers_must_come_in_pairs_and_not_overlap():
    assert fwd(lam0=P) == kla.ERR_INVALID_ARG
    assert fwd(lamT=P) == kla.ERR_INVALID_ARG
    assert fwd(lam0=P, eta0=MIS) == kla.ERR_MISALIGNED
    a, b = ctypes.c_void_p(0x20000), ctypes.c_void_p(0x20000 + 16)
    # 16x16 fp32 state = 1 KiB: lamT starting 16 bytes into lam0 is a partial overlap
    assert fwd(lam0=a, eta0=ctypes.c_void_p(0x40000), lamT=b, etaT=ctypes.c_void_p(0x60000)) == kla.ERR_INVALID_ARG
    assert fwd(lamT=a, etaT=a) == kla.ERR_INVALID_ARG


def test_bad_io_and_options():
    assert fwd(io=7) == kla.ERR_INVALID_ARG
    for c in (-1, 3):
        assert fwd(opt=ctypes.byref(kla.Options(kla.AUTO, 0, 0, 0, c))) == kla.ERR_INVALID_ARG
    assert fwd(opt=ctypes.byref(kla.Options(9, 0))) == kla.ERR_INVALID_ARG
    assert fwd(opt=ctypes.byref(kla.Options(kla.CHUNKED, 48))) == kla.ERR_INVALID_ARG
    assert fwd(opt=ctypes.byref(kla.Options(kla.CHUNKED, -32))) == kla.ERR_INVALID_ARG
    for rl in (-4, 2, 6, 16):
        assert fwd(opt=ctypes.byref(kla.Options(kla.AUTO, 0, rl))) == kla.ERR_INVALID_ARG
    # eight rows per lane needs a head of at least 64 rows
    assert fwd(dk=32, opt=ctypes.byref(kla.Options(kla.AUTO, 0, 8))) == kla.ERR_INVALID_ARG


def test_empty_batch_is_ok_without_any_cuda_call():
    assert fwd(B=0, ptrs={n: None for n in ("q", "k", "v", "lam_v", "a", "pbar", "y")}) == kla.OK
    assert L.kla_step(None, None, None, None, None, None, None, None, None, 0, 4, 16, 16, kla.F32, None) == kla.OK


def test_step_validation():
    s = lambda **kw: L.kla_step(*(kw.get(n, P) for n in ("q", "k", "v", "lam_v", "a", "pbar", "lam", "eta", "y")),
                                kw.get("B", 1), 1, kw.get("dk", 16), 16, kw.get("io", kla.F32), None)
    assert s(dk=20) == kla.ERR_UNSUPPORTED_SHAPE
    assert s(lam=None) == kla.ERR_INVALID_ARG
    assert s(y=MIS) == kla.ERR_MISALIGNED
    assert s(io=3) == kla.ERR_INVALID_ARG
    assert s(B=-1) == kla.ERR_INVALID_ARG
    assert s(lam=P, eta=P) == kla.ERR_INVALID_ARG


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_valid_arguments_without_a_device_report_cuda_error():
    # Validation passes, so the first CUDA call (device query) fails cleanly.
    assert fwd() == kla.ERR_CUDA
    info = kla.PlanInfo()
    assert L.kla_plan(1, 1, 8, 16, 16, kla.F32, None, ctypes.byref(info)) == kla.ERR_CUDA
    assert L.kla_forward_workspace_size(1, 1, 8, 16, 16, None) == ctypes.c_size_t(-1).value


def test_planner_headline_shape_is_sequential_on_152_sms():
    p = kla.plan(8, 16, 4096, 64, 64, "bf16", num_sms=152)
    assert p["strategy"] == "sequential" and p["num_chunks"] == 1 and p["workspace_bytes"] == 0
    assert 64 % p["cols_per_block"] == 0


def test_planner_coefficient_pass():
    """kla_coef_pass: automatic when a head's columns span four or more
    blocks of at most 16 columns (the medium and long workloads on 152 SMs),
    never for one block per head (the headline) or on the chunked plan; its
    buffer is B·H·T·5·d_k fp32 and is the plan's whole workspace."""
    coef_bytes = lambda B, H, T, dk: B * H * T * 5 * dk * 4
    med = kla.plan(4, 8, 2048, 64, 64, "f32", num_sms=152)
    assert med["strategy"] == "sequential" and 64 // med["cols_per_block"] >= 4
    assert med["coef_pass"] and med["workspace_bytes"] == coef_bytes(4, 8, 2048, 64)
    long_ = kla.plan(1, 16, 65536, 128, 128, "bf16", num_sms=152)
    assert long_["strategy"] == "sequential" and long_["coef_pass"]
    assert long_["workspace_bytes"] == coef_bytes(1, 16, 65536, 128)
    head = kla.plan(8, 16, 4096, 64, 64, "bf16", num_sms=152)
    assert head["cols_per_block"] == 64 and not head["coef_pass"] and head["workspace_bytes"] == 0
    # four blocks of 32 columns, or two of 32: the per-row work weighs too little there
    for shape in ((8, 8, 2048, 128, 128, "f32"), (4, 16, 4096, 64, 64, "bf16")):
        p = kla.plan(*shape, num_sms=152)
        assert p["cols_per_block"] == 32 and not p["coef_pass"] and p["workspace_bytes"] == 0, (shape, p)
    # forced on / off; the geometry does not depend on it
    on = kla.plan(8, 16, 4096, 64, 64, "bf16", coef_pass="on", num_sms=152)
    assert on["coef_pass"] and on["workspace_bytes"] == coef_bytes(8, 16, 4096, 64)
    assert {k: v for k, v in on.items() if k not in ("coef_pass", "workspace_bytes")} == \
        {k: v for k, v in head.items() if k not in ("coef_pass", "workspace_bytes")}
    off = kla.plan(4, 8, 2048, 64, 64, "f32", coef_pass="off", num_sms=152)
    assert not off["coef_pass"] and off["workspace_bytes"] == 0 and off["cols_per_block"] == med["cols_per_block"]
    # the chunked plan never takes it, even when asked to
    ch = kla.plan(1, 2, 16384, 64, 64, "bf16", strategy="chunked", coef_pass="on", num_sms=152)
    assert ch["strategy"] == "chunked" and not ch["coef_pass"]
    # empty sequences and batches need nothing
    assert kla.plan(4, 8, 0, 64, 64, "f32", coef_pass="on", num_sms=152)["workspace_bytes"] == 0
    assert kla.plan(0, 8, 64, 64, 64, "f32", coef_pass="on", num_sms=152)["workspace_bytes"] == 0
    # above 16 GiB the automatic choice leaves it out
    big = kla.plan(1, 16, 1 << 21, 128, 128, "bf16", strategy="sequential", num_sms=152)
    assert coef_bytes(1, 16, 1 << 21, 128) > 16 << 30 and not big["coef_pass"] and big["workspace_bytes"] == 0


def test_planner_low_parallelism_goes_chunked_and_sizes_workspace():
    p = kla.plan(1, 2, 16384, 64, 64, "bf16", num_sms=152)
    assert p["strategy"] == "chunked"
    S, elems = p["num_chunks"], 2 * 64 * 64
    assert p["chunk_len"] % 32 == 0 and S == -(-16384 // p["chunk_len"]) and S >= 2
    assert p["workspace_bytes"] == (7 * (S - 1) + 2 * S) * elems * 4


def test_planner_forced_strategies_and_chunk_len():
    seq = kla.plan(1, 2, 16384, 64, 64, "f32", strategy="sequential", coef_pass="off", num_sms=152)
    assert seq["strategy"] == "sequential" and seq["workspace_bytes"] == 0 and not seq["coef_pass"]
    ch = kla.plan(8, 16, 4096, 64, 64, "bf16", strategy="chunked", chunk_len=1024, num_sms=152)
    assert ch["strategy"] == "chunked" and ch["chunk_len"] == 1024 and ch["num_chunks"] == 4
    # a chunk as long as the sequence leaves nothing to parallelise: sequential
    one = kla.plan(1, 1, 64, 16, 16, "f32", strategy="chunked", chunk_len=64, num_sms=152)
    assert one["strategy"] == "sequential"
    with pytest.raises(kla.KlaError):
        kla.plan(1, 1, 64, 16, 16, "f32", strategy="chunked", chunk_len=40, num_sms=152)


@pytest.mark.parametrize("dk,dv,io", [(16, 16, "f32"), (32, 128, "bf16"), (128, 16, "f32"), (128, 128, "bf16"),
                                      (64, 32, "f32")])
def test_planner_blocks_fit_the_hardware(dk, dv, io):
    for B, H, T in [(1, 1, 33), (4, 8, 2048), (1, 16, 65536), (256, 16, 1)]:
        p = kla.plan(B, H, T, dk, dv, io, num_sms=152)
        cc = p["cols_per_block"]
        assert dv % cc == 0 and cc * (2 if io == "bf16" else 4) % 16 == 0


def test_planner_rows_per_lane_choice():
    # Many heads: eight rows per lane (fewer coefficient loads per element).
    assert kla.plan(8, 16, 4096, 64, 64, "bf16", num_sms=152)["rows_per_lane"] == 8
    # Few heads: four rows per lane gives twice as many column blocks.
    assert kla.plan(4, 8, 2048, 64, 64, "f32", num_sms=152)["rows_per_lane"] == 4
    # Small heads only have four.
    assert kla.plan(8, 16, 4096, 32, 64, "bf16", num_sms=152)["rows_per_lane"] == 4
    for dk in (64, 128):
        for rl in (4, 8):
            for strategy, cl in (("sequential", 0), ("chunked", 64)):
                p = kla.plan(2, 3, 1000, dk, 64, "f32", strategy, cl, num_sms=152, rows_per_lane=rl)
                assert p["rows_per_lane"] == rl and p["strategy"] == strategy
                # the column block is a whole number of warps of that geometry
                wc = 32 // (dk // rl) * 2
                assert p["cols_per_block"] % wc == 0
    with pytest.raises(kla.KlaError):
        kla.plan(1, 1, 64, 16, 16, "f32", rows_per_lane=8, num_sms=152)


def bwd(B=1, H=1, T=8, dk=16, dv=16, io=kla.F32, ptrs=None, lam0=None, eta0=None, glam0=None, geta0=None,
        ws=None, ws_bytes=0, gates=0):
    ptrs = ptrs or {}
    g = lambda n: ptrs.get(n, P)
    return L.kla_backward(g("q"), g("k"), g("v"), g("lam_v"), g("a"), g("pbar"), lam0, eta0, ptrs.get("gy"),
                          ptrs.get("glamT"), ptrs.get("getaT"), g("gq"), g("gk"), g("gv"), g("glam_v"), g("ga"),
                          g("gpbar"), glam0, geta0, B, H, T, dk, dv, io, gates, ws, ws_bytes, None)


def test_backward_validation_before_any_cuda_call():
    assert bwd(dk=24) == kla.ERR_UNSUPPORTED_SHAPE
    assert bwd(T=-1) == kla.ERR_INVALID_ARG
    assert bwd(io=5) == kla.ERR_INVALID_ARG
    assert bwd(lam0=P) == kla.ERR_INVALID_ARG                 # eta0 missing
    assert bwd(glam0=P) == kla.ERR_INVALID_ARG                # geta0 missing
    for out in ("gq", "gk", "gv", "glam_v", "ga", "gpbar", "q", "lam_v"):
        assert bwd(ptrs={out: None}) == kla.ERR_INVALID_ARG, out
    for name in ("gq", "gy", "glamT", "v"):
        assert bwd(ptrs={name: MIS}) == kla.ERR_MISALIGNED, name
    assert bwd(glam0=P, geta0=P) == kla.ERR_INVALID_ARG       # the two outputs alias
    assert bwd(gates=16) == kla.ERR_INVALID_ARG               # unknown gate bit
    assert bwd(gates=kla.GATE_PBAR_SOFTPLUS | kla.GATE_PBAR_OU) == kla.ERR_INVALID_ARG
    # nothing to do: OK without touching CUDA
    assert bwd(B=0, ptrs={n: None for n in ("q", "k", "v", "lam_v", "a", "pbar", "gq", "gk", "gv", "glam_v",
                                              "ga", "gpbar")}) == kla.OK


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_backward_without_a_device_reports_cuda_error():
    assert bwd() == kla.ERR_CUDA
    assert L.kla_backward_workspace_size(1, 1, 8, 16, 16) == ctypes.c_size_t(-1).value
    assert L.kla_backward_workspace_size(0, 4, 8, 16, 16) == 0
    assert L.kla_backward_workspace_size(1, 1, 8, 20, 16) == ctypes.c_size_t(-1).value


def test_backward_plan_geometry_on_a_152_sm_device():
    """Eight columns per lane when the blocks fill the SMs with warps (many
    heads), four or two when eight would leave few warps per SM (few heads);
    the workspace is the 16-token checkpoints plus, with split columns, the
    fp32 per-row partial sums."""
    bp = lambda *shape, sms=152: kla.backward_plan(*shape, num_sms=sms)
    head = bp(8, 16, 4096, 64, 64)
    assert (head["cols_per_lane"], head["cols_per_block"], head["threads"], head["column_blocks"]) == (8, 64, 512, 1)
    assert head["workspace_bytes"] == (4096 // 16 + 1) * 2 * 128 * 64 * 64 * 4
    med = bp(4, 8, 2048, 64, 64)
    assert (med["cols_per_lane"], med["cols_per_block"], med["threads"], med["column_blocks"]) == (2, 16, 512, 4)
    assert med["workspace_bytes"] == (2048 // 16 + 1) * 2 * 32 * 64 * 64 * 4 + 4 * 32 * 2048 * 64 * 4
    assert bp(1, 16, 65536, 128, 128)["cols_per_lane"] == 4
    # the GPU parity shapes of tests/test_backward_gpu.py: each head size with two and four columns per lane
    for shape, cpl in (((8, 8, 24, 16, 64), 2), ((8, 8, 19, 32, 32), 2), ((4, 4, 40, 64, 64), 2),
                       ((3, 16, 18, 128, 16), 2), ((8, 16, 20, 16, 128), 4), ((3, 16, 22, 32, 128), 4),
                       ((3, 16, 25, 64, 64), 4), ((1, 16, 21, 128, 128), 4)):
        assert bp(*shape)["cols_per_lane"] == cpl, shape
    # no block narrower than 8 columns (a staged bf16 column row is then at least 16 bytes)
    for sms in (152, 132, 16):
        for dk in (16, 32, 64, 128):
            for dv in (16, 32, 64, 128):
                for bh in (1, 2, 3, 5, 8, 13, 32, 64, 128, 1024):
                    assert bp(1, bh, 40, dk, dv, sms=sms)["cols_per_block"] >= 8
    assert bp(1, 1, 40, 16, 16)["cols_per_lane"] == 8
    for shape in ((8, 16, 4096, 64, 64), (4, 8, 2048, 64, 64), (3, 5, 77, 32, 128)):
        p = bp(*shape)
        assert p["cols_per_block"] * p["column_blocks"] == shape[4]
        assert p["threads"] % 32 == 0 and 32 <= p["threads"] <= 512
    assert bp(0, 4, 8, 16, 16) == {"cols_per_block": 0, "cols_per_lane": 0, "threads": 0, "column_blocks": 0,
                                   "workspace_bytes": 0}
    info = kla.BackwardPlanInfo()
    assert L.kla_backward_plan_for_sms(1, 1, 8, 20, 16, 152, ctypes.byref(info)) == kla.ERR_UNSUPPORTED_SHAPE
    assert L.kla_backward_plan_for_sms(1, 1, 8, 16, 16, 0, ctypes.byref(info)) == kla.ERR_INVALID_ARG
    assert L.kla_backward_plan_for_sms(1, 1, 8, 16, 16, 152, None) == kla.ERR_INVALID_ARG


def test_forward_uncertainty_validation_before_any_cuda_call():
    def fu(y_var=P, y=ctypes.c_void_p(0x30000), **kw):
        g = lambda n: kw.get(n, P)
        return L.kla_forward_uncertainty(g("q"), g("k"), g("v"), g("lam_v"), g("a"), g("pbar"), None, None, y,
                                         y_var, None, None, 1, 1, 8, 16, 16, kla.F32, None, 0, None, None)
    assert fu(y_var=None) == kla.ERR_INVALID_ARG
    assert fu(y_var=ctypes.c_void_p(0x30000)) == kla.ERR_INVALID_ARG        # same buffer as y
    assert fu(y_var=ctypes.c_void_p(0x30000 + 64)) == kla.ERR_INVALID_ARG   # overlaps y (8x16 fp32 = 512 B)
    assert fu(y_var=MIS) == kla.ERR_MISALIGNED


def test_gate_bits_are_validated_before_any_cuda_call():
    for g in (16, 32, kla.GATE_PBAR_SOFTPLUS | kla.GATE_PBAR_OU):
        assert fwd(opt=ctypes.byref(kla.Options(kla.AUTO, 0, 0, g))) == kla.ERR_INVALID_ARG
        assert L.kla_step_gated(P, P, P, P, P, P, P, ctypes.c_void_p(0x50000), P, 1, 1, 16, 16, kla.F32, g,
                                None) == kla.ERR_INVALID_ARG


def test_shard_entry_points_validate_before_any_cuda_call():
    # kla_shard_map(q, k, v, lam_v, a, pbar, map, B, H, T, dk, dv, io, gates, stream)
    m = L.kla_shard_map
    assert m(P, P, P, P, P, P, P, 1, 1, 8, 24, 64, kla.F32, 0, None) == kla.ERR_UNSUPPORTED_SHAPE
    assert m(P, P, P, P, P, P, P, -1, 1, 8, 64, 64, kla.F32, 0, None) == kla.ERR_INVALID_ARG
    assert m(P, P, P, P, P, P, None, 1, 1, 8, 64, 64, kla.F32, 0, None) == kla.ERR_INVALID_ARG
    assert m(P, None, P, P, P, P, P, 1, 1, 8, 64, 64, kla.F32, 0, None) == kla.ERR_INVALID_ARG
    assert m(P, P, P, P, P, P, MIS, 1, 1, 8, 64, 64, kla.F32, 0, None) == kla.ERR_MISALIGNED
    assert m(P, P, P, P, P, P, P, 1, 1, 8, 64, 64, 7, 0, None) == kla.ERR_INVALID_ARG
    assert m(P, P, P, P, P, P, P, 1, 1, 8, 64, 64, kla.F32, 12, None) == kla.ERR_INVALID_ARG  # both p̄ gates
    assert m(None, None, None, None, None, None, None, 0, 4, 8, 64, 64, kla.F32, 0, None) == kla.OK
    # kla_shard_start(maps, n_maps, lam0, eta0, lam_start, eta_start, B, H, dk, dv, stream)
    s = L.kla_shard_start
    assert s(P, -1, None, None, P, ctypes.c_void_p(0x20000), 1, 1, 64, 64, None) == kla.ERR_INVALID_ARG
    assert s(None, 2, None, None, P, ctypes.c_void_p(0x20000), 1, 1, 64, 64, None) == kla.ERR_INVALID_ARG
    assert s(P, 1, P, None, ctypes.c_void_p(0x30000), ctypes.c_void_p(0x40000), 1, 1, 64, 64,
             None) == kla.ERR_INVALID_ARG                                    # lam0 without eta0
    assert s(P, 1, None, None, MIS, ctypes.c_void_p(0x40000), 1, 1, 64, 64, None) == kla.ERR_MISALIGNED
    # outputs overlapping the maps (one map is 7·64·64·4 bytes from 0x10000)
    assert s(P, 1, None, None, ctypes.c_void_p(0x10000 + 4096), ctypes.c_void_p(0x900000), 1, 1, 64, 64,
             None) == kla.ERR_INVALID_ARG
    assert s(P, 1, None, None, ctypes.c_void_p(0x900000), ctypes.c_void_p(0x900000), 1, 1, 64, 64,
             None) == kla.ERR_INVALID_ARG                                    # lam_start == eta_start
    assert s(P, 1, None, None, P, P, 1, 1, 24, 64, None) == kla.ERR_UNSUPPORTED_SHAPE
    assert s(None, 0, None, None, None, None, 0, 3, 64, 64, None) == kla.OK  # empty batch


def test_shard_entry_points_without_a_device_report_cuda_error():
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    a, b = ctypes.c_void_p(0x100000), ctypes.c_void_p(0x200000)
    assert L.kla_shard_start(None, 0, None, None, a, b, 1, 1, 16, 16, None) == kla.ERR_CUDA


def conv_call(B=1, H=1, T=8, D=16, W=4, io=kla.F32, act=kla.ACT_SILU, x=None, weight=None, bias=None,
              win=None, y=None, wout=None):
    """kla_conv with distinct, non-overlapping placeholder regions by default."""
    x = ctypes.c_void_p(0x100000) if x is None else x
    weight = ctypes.c_void_p(0x200000) if weight is None else weight
    y = ctypes.c_void_p(0x300000) if y is None else y
    return L.kla_conv(x, weight, bias, win, y, wout, B, H, T, D, W, io, act, None)


def test_conv_validates_before_any_cuda_call():
    assert conv_call(D=6) == kla.ERR_UNSUPPORTED_SHAPE       # not a multiple of 4
    assert conv_call(D=1024) == kla.ERR_UNSUPPORTED_SHAPE
    assert conv_call(W=0) == kla.ERR_UNSUPPORTED_SHAPE
    assert conv_call(W=9) == kla.ERR_UNSUPPORTED_SHAPE
    assert conv_call(T=-1) == kla.ERR_INVALID_ARG
    assert conv_call(io=5) == kla.ERR_INVALID_ARG
    assert conv_call(act=2) == kla.ERR_INVALID_ARG
    assert conv_call(weight=ctypes.c_void_p(0)) == kla.ERR_INVALID_ARG
    assert conv_call(x=ctypes.c_void_p(0)) == kla.ERR_INVALID_ARG
    assert conv_call(y=ctypes.c_void_p(0)) == kla.ERR_INVALID_ARG
    assert conv_call(bias=MIS) == kla.ERR_MISALIGNED
    assert conv_call(win=MIS) == kla.ERR_MISALIGNED
    # y over x (8 tokens × 16 channels × 4 bytes from 0x100000)
    assert conv_call(y=ctypes.c_void_p(0x100000 + 256)) == kla.ERR_INVALID_ARG
    # window out over x, partially over the window in, over y
    assert conv_call(win=ctypes.c_void_p(0x400000), wout=ctypes.c_void_p(0x100000)) == kla.ERR_INVALID_ARG
    assert conv_call(win=ctypes.c_void_p(0x400000), wout=ctypes.c_void_p(0x400000 + 64)) == kla.ERR_INVALID_ARG
    assert conv_call(wout=ctypes.c_void_p(0x300000)) == kla.ERR_INVALID_ARG
    # empty batch: nothing to do, no CUDA call
    assert conv_call(B=0, x=ctypes.c_void_p(0), y=ctypes.c_void_p(0), weight=ctypes.c_void_p(0)) == kla.OK


def test_conv_with_one_tap_ignores_the_window_pointers():
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    # misaligned / overlapping window pointers are ignored for W = 1, so validation passes and the
    # missing device is reported
    assert conv_call(W=1, win=MIS, wout=ctypes.c_void_p(0x100000)) == kla.ERR_CUDA
    assert conv_call(W=4, win=MIS) == kla.ERR_MISALIGNED


def test_conv_backward_validates_before_any_cuda_call():
    b = L.kla_conv_backward
    x, wt, gy, gx = (ctypes.c_void_p(a) for a in (0x100000, 0x200000, 0x300000, 0x400000))
    gw, gb, gwin = (ctypes.c_void_p(a) for a in (0x500000, 0x600000, 0x700000))

    def call(**kw):
        args = dict(x=x, weight=wt, bias=None, win=None, gy=gy, gwo=None, gx=gx, gw=gw, gb=gb, gwin=gwin,
                    B=1, H=1, T=8, D=16, W=4, io=kla.F32, act=kla.ACT_SILU, ws=ctypes.c_void_p(0x800000),
                    ws_bytes=1 << 20)
        args.update(kw)
        a = args
        return b(a["x"], a["weight"], a["bias"], a["win"], a["gy"], a["gwo"], a["gx"], a["gw"], a["gb"],
                 a["gwin"], a["B"], a["H"], a["T"], a["D"], a["W"], a["io"], a["act"], a["ws"], a["ws_bytes"],
                 None)

    assert call(D=12 + 2) == kla.ERR_UNSUPPORTED_SHAPE
    assert call(W=10) == kla.ERR_UNSUPPORTED_SHAPE
    assert call(act=-1) == kla.ERR_INVALID_ARG
    assert call(gx=None) == kla.ERR_INVALID_ARG
    assert call(weight=None) == kla.ERR_INVALID_ARG
    assert call(gw=MIS) == kla.ERR_MISALIGNED
    assert call(ws=MIS) == kla.ERR_MISALIGNED
    assert call(gx=ctypes.c_void_p(0x100000 + 64)) == kla.ERR_INVALID_ARG       # gx over x
    assert call(gwin=ctypes.c_void_p(0x400000 + 128)) == kla.ERR_INVALID_ARG    # gwindow over gx
    assert call(gb=ctypes.c_void_p(0x200000)) == kla.ERR_INVALID_ARG            # gbias over the taps
    # no batch, no weight gradient wanted: nothing to do
    assert call(B=0, x=None, gx=None, gy=None, gw=None, gb=None, ws=None, ws_bytes=0) == kla.OK
    if not torch.cuda.is_available():
        assert L.kla_conv_backward_workspace_size(1, 1, 8, 16, 4) == ctypes.c_size_t(-1).value
        assert call() == kla.ERR_CUDA
    assert L.kla_conv_backward_workspace_size(1, 1, 8, 18, 4) == ctypes.c_size_t(-1).value
    assert L.kla_conv_backward_workspace_size(0, 3, 8, 16, 4) == 0
