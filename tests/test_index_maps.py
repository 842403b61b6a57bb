"""CPU models of the index arithmetic of two kernels, checked before they
run on a GPU: every element is covered exactly once and every access stays
inside its buffer, for the launch shapes the host code produces.

* kla_coef_kernel (csrc/kla_scan_kernel.cuh, launched by
  csrc/kla_scan_inst_y_pre.cu): a block covers 64 tokens of one head
  (grid.x) for heads blockIdx.y, blockIdx.y + gridDim.y, ...; a thread
  handles four consecutive rows of a token and writes five float4
  coefficients; it reads k of the token before when t > 0. The scan's MODE 4
  producers then copy tl·5·d_k floats of a tile from the same buffer.
* kla_bwd_kernel's lane geometry (BwdGeo / BwdLane in csrc/kla_backward.cu):
  a warp covers RW = min(32, d_k) rows and 32/RW column groups of CPL
  columns; a block has d_k/RW row warps × cc/(32/RW·CPL) column warps; lane
  (warp, lane) owns row wr·RW + lane % RW and columns
  wc·WCOLS + (lane / RW)·CPL + [0, CPL). Checked for every geometry the
  backward planner chooses (kla_backward_plan_for_sms), two columns per lane
  included.
"""
import itertools

import pytest

from bayesian_filtering_linear_gb300 import kla

COEF_TOKENS, COEF_THREADS = 64, 256


def coef_kernel_accesses(bh_count, T, DK):
    """Yield ('r'|'w', flat index, length) of every global access of the
    coefficient kernel, in units of the buffer's element."""
    R4 = DK // 4
    grid_x = (T + COEF_TOKENS - 1) // COEF_TOKENS
    grid_y = min(bh_count, 65535)
    for bx, by in itertools.product(range(grid_x), range(grid_y)):
        t0 = bx * COEF_TOKENS
        tl = min(COEF_TOKENS, T - t0)
        for bh in range(by, bh_count, grid_y):
            row0 = bh * T
            for tid in range(COEF_THREADS):
                for g in range(tid, tl * R4, COEF_THREADS):
                    tt, i = g // R4, 4 * (g % R4)
                    t = t0 + tt
                    o = (row0 + t) * DK + i
                    yield ("r", "in", o, 4)
                    if t > 0:
                        yield ("r", "in", o - DK, 4)
                    for c in range(5):
                        yield ("w", "coef", (row0 + t) * 5 * DK + i + c * DK, 4)


@pytest.mark.parametrize("bh,T,DK", [(1, 1, 16), (3, 63, 32), (2, 64, 64), (2, 65, 128), (5, 130, 16),
                                     (65537, 1, 16), (65536 + 3, 2, 16)])
def test_coefficient_kernel_writes_every_coefficient_once_in_bounds(bh, T, DK):
    n_in, n_coef = bh * T * DK, bh * T * 5 * DK
    written = bytearray(n_coef)
    for kind, buf, o, ln in coef_kernel_accesses(bh, T, DK):
        assert 0 <= o and o + ln <= (n_in if buf == "in" else n_coef), (kind, buf, o)
        assert o % 4 == 0  # 16-byte (fp32) or 8-byte (bf16) aligned vector accesses
        if kind == "w":
            for x in range(o, o + ln):
                assert not written[x], f"coefficient {x} written twice"
                written[x] = 1
    assert all(written)


@pytest.mark.parametrize("T", [1, 15, 16, 17, 33, 100])
@pytest.mark.parametrize("DK", [16, 64, 128])
def test_scan_copy_mode_reads_stay_in_the_head_and_fit_the_tile(T, DK):
    """MODE 4: tile m of a head reads tl·5·d_k floats from
    coefs + (bh·T + m·16)·5·d_k in 16-byte pieces into a 16·5·d_k-float
    buffer."""
    TC, bh_count = 16, 3
    for bh in range(bh_count):
        head_lo, head_hi = bh * T * 5 * DK, (bh + 1) * T * 5 * DK
        for m in range((T + TC - 1) // TC):
            tl = min(TC, T - m * TC)
            src = (bh * T + m * TC) * 5 * DK
            chunks = tl * (5 * DK // 4)
            assert src % 4 == 0 and head_lo <= src and src + 4 * chunks <= head_hi
            assert 4 * chunks <= TC * 5 * DK


def lane_owners(DK, CPL, cc):
    RW = min(32, DK)
    CG = 32 // RW
    WCOLS = CG * CPL
    NWR = DK // RW
    warps = NWR * (cc // WCOLS)
    owned = {}
    for warp, lane in itertools.product(range(warps), range(32)):
        wr, wc = warp % NWR, warp // NWR
        i = wr * RW + lane % RW
        jl = wc * WCOLS + (lane // RW) * CPL
        for j in range(jl, jl + CPL):
            owned.setdefault((i, j), []).append((warp, lane))
    return owned, warps


def test_reverse_kernel_lanes_own_every_element_once_for_every_planned_geometry():
    seen = set()
    for sms in (152, 132, 16):
        for dk, dv in itertools.product((16, 32, 64, 128), repeat=2):
            for bh in (1, 2, 3, 8, 32, 64, 128, 1024):
                p = kla.backward_plan(1, bh, 40, dk, dv, num_sms=sms)
                key = (dk, p["cols_per_lane"], p["cols_per_block"])
                if key in seen:
                    continue
                seen.add(key)
                cpl, cc = p["cols_per_lane"], p["cols_per_block"]
                owned, warps = lane_owners(dk, cpl, cc)
                assert 32 * warps == p["threads"], key
                assert set(owned) == {(i, j) for i in range(dk) for j in range(cc)}, key
                assert all(len(v) == 1 for v in owned.values()), key
                assert cc * p["column_blocks"] == dv
    assert any(k[1] == 2 for k in seen) and any(k[1] == 4 for k in seen) and any(k[1] == 8 for k in seen)
