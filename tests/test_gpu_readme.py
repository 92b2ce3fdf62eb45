"""The README's Python example runs as written (GPU): its code block is
executed with a small synthetic batch bound to the names it uses."""
import os
import re

import pytest
import torch

from asr_tiled_tanh_gb300 import synthetic
from tests.helpers import to_device

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_readme_example_runs():
    text = open(os.path.join(ROOT, "README.md")).read()
    blocks = re.findall(r"```python\n(.*?)```", text, flags=re.S)
    assert blocks, "no python example in README.md"
    inp = synthetic.custom(B=3, T=40, U=6, HA=64, HL=64, H=64, V=128, dtype="bf16", seed=5)
    dev = to_device(inp)
    ns = dict(B=3, T=40, U=6, HA=64, HL=64, H=64, V=128, **dev)
    exec(compile(blocks[0], "README.md", "exec"), ns)
    torch.cuda.synchronize()
    assert ns["loss"].shape == (3,) and bool(torch.isfinite(ns["loss"]).all())
    assert set(ns["grads"]) == {"dhA", "dhL", "dWA", "dWL", "dbZ", "dWO", "dbO"}
    assert ns["r"].status() == (0, 0)
