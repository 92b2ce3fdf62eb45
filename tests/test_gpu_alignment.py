"""On the bf16 (tensor-core) path, gradient outputs that are not 16-byte
aligned are refused before anything is launched (GPU).  The kernels write
them by 16-byte stores and vector reductions, so the refusal happens on the
host; the test checks the status and that the buffer around the view is
untouched."""
import pytest
import torch

import asr_tiled_tanh_gb300 as rn
from asr_tiled_tanh_gb300 import synthetic
from tests.helpers import to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    rn.load(build_if_missing=True)


def test_unaligned_gradient_outputs_are_refused_and_untouched():
    inp = synthetic.custom(B=2, T=20, U=5, HA=64, HL=64, H=64, V=128, dtype="bf16", seed=71)
    dev = to_device(inp)
    r = rn.Rnnt.for_inputs(inp)
    params = rn.make_params(dev["WA"], dev["WL"], dev["bZ"], dev["WO"], dev["bO"])
    args = (dev["hA"], dev["hL"], params, dev["labels"], dev["T_len"], dev["U_len"])
    r.fwd(*args)
    torch.cuda.synchronize()
    g = r.alloc_grads()
    for name in ("dhA", "dhL", "dWA", "dWL", "dWO"):
        n = g[name].numel()
        big = torch.full((n + 4,), 7.0, dtype=torch.float32, device="cuda")
        gg = dict(g)
        gg[name] = big[1:1 + n].view_as(g[name])  # 4 bytes past a 16-byte boundary
        code = rn.rnnt_bwd(r.dims, *args, None, r.saved, gg["dhA"], gg["dhL"], gg["dWA"],
                           gg["dWL"], gg["dbZ"], gg["dWO"], gg["dbO"], r.ws, check=False)
        torch.cuda.synchronize()
        assert code == 1, name  # RNNT_ERR_INVALID_ARG
        assert bool((big == 7.0).all()), name
    # aligned buffers still work after the refusals
    out = r.bwd(*args)
    torch.cuda.synchronize()
    assert r.status() == (0, 0)
    assert torch.isfinite(out["dWO"]).all()
