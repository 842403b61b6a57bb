"""GPU parity at the size extremes, against the fp64 oracle: a very long
sequence on one small head (2^20 tokens: the planner cuts it into chunks; the
sequential path runs it in one block) and very many heads of a single token
(65,536 heads). The filter: "Technische Samenvatting: Kalman Linear Attention
(KLA)", Methodologie §1–§2; error measure and tolerances as in
tests/helpers.py."""
import pytest
import torch

from bayesian_filtering_linear_gb300 import kla
from bayesian_filtering_linear_gb300.inputs import make_inputs
from helpers import assert_close, errors, gpu_forward, run_oracle, to_dev

pytestmark = pytest.mark.gpu


def test_million_token_sequence_on_one_head():
    x = make_inputs(1, 1, 1 << 20, 16, 16, io="f32", seed=31, random_state=True)
    ref = run_oracle(x)
    xd = to_dev(x)
    assert kla.plan(1, 1, 1 << 20, 16, 16, "f32")["strategy"] == "chunked"
    for strategy in ("auto", "sequential"):
        y, lamT, etaT = gpu_forward(xd, strategy=strategy)
        torch.cuda.synchronize()
        assert_close(errors(y, lamT, etaT, ref), 1e-4, f"2^20 tokens, {strategy}")
        del y, lamT, etaT


def test_sixty_five_thousand_single_token_heads():
    x = make_inputs(256, 256, 1, 16, 32, io="bf16", seed=32, random_state=True)
    ref = run_oracle(x)
    y, lamT, etaT = gpu_forward(to_dev(x))
    torch.cuda.synchronize()
    assert_close(errors(y, lamT, etaT, ref), 2e-2, "65536 heads, T = 1")
