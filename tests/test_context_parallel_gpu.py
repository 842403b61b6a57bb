"""GPU parity of context-parallel sharding over T: kla_shard_map and
kla_shard_start (through the C ABI), and kla.forward_context_parallel.

The maps of the filter compose associatively ("Technische Samenvatting:
Kalman Linear Attention (KLA)", Methodologie §2): a rank that holds a
contiguous token range starts from the initial state pushed through the
composed maps of the ranges before it. Checked against the fp64 oracle's
single pass over the whole sequence (scaled errors, 1e-4 fp32 I/O, 2e-2 bf16
I/O) and against one kla_forward call:

* ranks emulated in one process, one after another (no collective): every
  shard's map, the start states from the maps before each shard, and each
  shard's forward from its start; ragged shards and an empty one;
* two processes on the one GPU joined by a gloo process group, each running
  kla.forward_context_parallel on its half (the maps go through host
  copies; the processes' kernels never wait on one another).
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from bayesian_filtering_linear_gb300 import kla
from bayesian_filtering_linear_gb300.inputs import make_inputs
from helpers import TOL, assert_close, errors, run_oracle, to_dev

pytestmark = pytest.mark.gpu
IO = {"f32": torch.float32, "bf16": torch.bfloat16}
NAMES = ("q", "k", "v", "lam_v", "a", "pbar")


def _slice(xd, t0, t1):
    return {n: xd[n][:, :, t0:t1].contiguous() for n in NAMES}


@pytest.mark.parametrize("shape,cuts", [
    ((2, 3, 700, 64, 32, "f32"), [0, 123, 123, 500, 700]),
    ((1, 2, 1000, 128, 64, "bf16"), [0, 256, 512, 768, 1000]),
    ((3, 1, 333, 16, 128, "f32"), [0, 1, 332, 333]),
], ids=["f32-ragged-empty", "bf16-d128", "f32-one-token-shards"])
def test_emulated_ranks_match_one_pass_and_oracle(shape, cuts):
    B, H, T, dk, dv, io = shape
    x = make_inputs(B, H, T, dk, dv, io=io, seed=40 + T, random_state=True)
    xd = to_dev(x)
    maps = torch.stack([kla.shard_map(*(_slice(xd, t0, t1)[n] for n in NAMES)) for t0, t1 in zip(cuts, cuts[1:])])
    ys = []
    for r, (t0, t1) in enumerate(zip(cuts, cuts[1:])):
        lam_s, eta_s = kla.shard_start(maps[:r].contiguous(), xd["lam0"], xd["eta0"])
        y, lamT, etaT = kla.forward(*(_slice(xd, t0, t1)[n] for n in NAMES), lam_s, eta_s)
        ys.append(y)
    torch.cuda.synchronize()
    y = torch.cat(ys, dim=2)
    ref = run_oracle(x)
    assert_close(errors(y, lamT, etaT, ref), TOL[IO[io]], f"sharded {shape}")
    # the last shard's start from all maps but its own equals the state one
    # forward over those tokens reaches
    y1, l1, e1 = kla.forward(*(_slice(xd, 0, cuts[-2])[n] for n in NAMES), xd["lam0"], xd["eta0"])
    lam_s, eta_s = kla.shard_start(maps[:-1].contiguous(), xd["lam0"], xd["eta0"])
    torch.cuda.synchronize()
    assert float(((lam_s - l1).abs() / l1).max()) < TOL[IO[io]]
    assert float((eta_s - e1).abs().max() / e1.abs().max()) < TOL[IO[io]]


def test_empty_shard_map_is_the_identity_and_no_maps_keep_the_state():
    x = to_dev(make_inputs(2, 2, 0, 32, 16, io="f32", seed=3, random_state=True))
    m = kla.shard_map(*(x[n] for n in NAMES))
    eye = torch.zeros_like(m)
    eye[0] = eye[3] = eye[6] = 1.0
    assert torch.equal(m, eye)
    lam, eta = kla.shard_start(torch.empty((0,) + tuple(m.shape), device="cuda"), x["lam0"], x["eta0"])
    torch.cuda.synchronize()
    assert float(((lam - x["lam0"]).abs() / x["lam0"]).max()) < 1e-6
    assert float((eta - x["eta0"]).abs().max()) < 1e-5


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


SHAPE = (2, 2, 600, 64, 64, "bf16")


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        torch.cuda.set_device(0)
        B, H, T, dk, dv, io = SHAPE
        x = to_dev(make_inputs(B, H, T, dk, dv, io=io, seed=77, random_state=True))
        cut = [0, 250, T]
        sl = _slice(x, cut[rank], cut[rank + 1])
        y, lamT, etaT = kla.forward_context_parallel(*(sl[n] for n in NAMES), x["lam0"], x["eta0"])
        torch.cuda.synchronize()
        q.put((rank, y.float().cpu().numpy(), lamT.cpu().numpy(), etaT.cpu().numpy()))
    finally:
        dist.destroy_process_group()


def test_forward_context_parallel_two_processes_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(2):
        r, y, l, e = q.get(timeout=300)
        res[r] = (y, l, e)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    B, H, T, dk, dv, io = SHAPE
    x = make_inputs(B, H, T, dk, dv, io=io, seed=77, random_state=True)
    ref = run_oracle(x)
    y = torch.from_numpy(np.concatenate([res[0][0], res[1][0]], axis=2))
    assert_close(errors(y, torch.from_numpy(res[1][1]), torch.from_numpy(res[1][2]), ref), TOL[IO[io]],
                 "context-parallel, 2 ranks")
