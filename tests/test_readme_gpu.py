"""The Python example in README.md runs as written (forward, a decode step,
the convolution and a backward pass through autograd) and produces finite
results and a gradient."""
import os
import re

import pytest
import torch

pytestmark = pytest.mark.gpu

README = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "README.md")


def test_readme_example_runs():
    text = open(README).read()
    blocks = re.findall(r"```python\n(.*?)```", text, flags=re.S)
    assert blocks, "no python example"
    scope = {}
    exec(compile(blocks[0], "README.md", "exec"), scope)
    torch.cuda.synchronize()
    assert torch.isfinite(scope["y"].float()).all()
    assert torch.isfinite(scope["y_t"].float()).all()
    assert scope["w"].grad is not None and torch.isfinite(scope["w"].grad).all()
