"""Context-parallel sharding over T, host side (no GPU; gloo, world size 2).

The sequence is cut into contiguous token ranges, one per rank. The maps of
the filter compose associatively ("Technische Samenvatting: Kalman Linear
Attention (KLA)", Methodologie §2), so each rank needs only the composed maps
of the shards before its own to know where its shard starts; the exchange
step is one all-gather of the per-shard maps (kla.exchange_maps).

Here every rank composes its shard's map in numpy (fp64 products of the
per-token homogeneous matrices, as the pages' Möbius form gives them), the
maps go through kla.exchange_maps over gloo, each rank applies the maps of
the ranks before it to the initial state, runs the oracle over its own
shard from there, and the result must equal the oracle's single pass over
the whole sequence: y on the rank's tokens and, on the last rank, the final
state. The GPU kernels that compose and apply maps on the device are
checked in test_context_parallel_gpu.py.
"""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

B, H, T, DK, DV = 1, 2, 60, 4, 3


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs():
    from bayesian_filtering_linear_gb300.inputs import make_inputs
    return {n: t.numpy() for n, t in make_inputs(B, H, T, DK, DV, io="f32", seed=5, random_state=True).items()}


def shard_map_fp64(x, t0, t1):
    """[7, B, H, dk, dv] map (A, B, C, D, E, F, G) of tokens [t0, t1): the
    product of the per-token matrices M_t = [[a², p̄, 0], [c a², 1 + c p̄, 0],
    [b a², b p̄, a]] acting on (n, m, e) with P = n/m, μ = e/m."""
    a, pb, k = (x[n][:, :, t0:t1].astype(np.float64) for n in ("a", "pbar", "k"))
    L, v = (x[n][:, :, t0:t1].astype(np.float64) for n in ("lam_v", "v"))
    M = np.zeros((B, H, DK, DV, 3, 3))
    M[..., 0, 0] = M[..., 1, 1] = M[..., 2, 2] = 1.0
    for t in range(t1 - t0):
        a2 = (a[:, :, t] ** 2)[..., None]
        p = pb[:, :, t][..., None] + np.zeros((1, 1, 1, DV))
        c = (k[:, :, t] ** 2)[..., None] * L[:, :, t][:, :, None, :]
        b = k[:, :, t][..., None] * (L[:, :, t] * v[:, :, t])[:, :, None, :]
        at = a[:, :, t][..., None] + np.zeros((1, 1, 1, DV))
        Mt = np.zeros_like(M)
        Mt[..., 0, 0], Mt[..., 0, 1] = a2, p
        Mt[..., 1, 0], Mt[..., 1, 1] = c * a2, 1 + c * p
        Mt[..., 2, 0], Mt[..., 2, 1], Mt[..., 2, 2] = b * a2, b * p, at
        M = Mt @ M
    return np.stack([M[..., 0, 0], M[..., 0, 1], M[..., 1, 0], M[..., 1, 1], M[..., 2, 0], M[..., 2, 1],
                     M[..., 2, 2]])


def apply_maps_fp64(maps, lam0, eta0):
    P, mu = 1.0 / lam0.astype(np.float64), eta0.astype(np.float64) / lam0
    for m in maps:
        A, Bm, C, D, E, F, G = m
        den = C * P + D
        P, mu = (A * P + Bm) / den, (E * P + F + G * mu) / den
    return 1.0 / P, mu / P


def _worker(rank, world, port, cuts, q):
    import torch
    import torch.distributed as dist
    import oracle
    from bayesian_filtering_linear_gb300 import kla
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        x = _inputs()
        t0, t1 = cuts[rank], cuts[rank + 1]
        local = torch.from_numpy(shard_map_fp64(x, t0, t1))
        maps = kla.exchange_maps(local).numpy()
        assert maps.shape == (world, 7, B, H, DK, DV)
        assert np.array_equal(maps[rank], local.numpy())  # rank order
        lam_s, eta_s = apply_maps_fp64(maps[:rank], x["lam0"], x["eta0"])
        sl = {n: x[n][:, :, t0:t1] for n in ("q", "k", "v", "lam_v", "a", "pbar")}
        out = oracle.forward64(*(sl[n] for n in ("q", "k", "v", "lam_v", "a", "pbar")), lam_s, eta_s)
        q.put((rank, out["y"], out["lamT"], out["etaT"]))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("cuts", [[0, 25, 60], [0, 0, 60], [0, 60, 60]], ids=["ragged", "empty-first", "empty-last"])
def test_sharded_scan_over_gloo_matches_one_pass(cuts):
    import oracle
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, cuts, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
        assert p.exitcode == 0
    res = {r: (y, l, e) for r, y, l, e in (q.get(timeout=10) for _ in range(2))}
    x = _inputs()
    ref = oracle.forward64(*(x[n] for n in ("q", "k", "v", "lam_v", "a", "pbar", "lam0", "eta0")), want_scales=True)
    y = np.concatenate([res[0][0], res[1][0]], axis=2)
    assert np.max(np.abs(y - ref["y"]) / ref["y_scale"]) < 1e-10
    assert np.max(np.abs(res[1][1] - ref["lamT"]) / ref["lamT"]) < 1e-10
    assert np.max(np.abs(res[1][2] - ref["etaT"]) / ref["eta_scale"]) < 1e-10
