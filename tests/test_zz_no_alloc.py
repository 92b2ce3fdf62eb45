"""rnnt_fwd_noalloc, the forward pass for callers that cannot allocate (GPU).

Some callers cannot allocate device memory: hosts that reserve all memory up
front, plugin interfaces that provide no allocator, latency-critical loops.
rnnt_fwd_noalloc takes its scratch from a fixed device array inside the
library instead of a caller buffer.  This test calls it through the C ABI
twice in a row and checks that both calls give what rnnt_fwd gives with a
caller-provided workspace; it runs last (file name) so that a failure here
never hides the rest of the suite, and it needs no earlier test's state.
"""
import ctypes

import numpy as np
import pytest
import torch

import asr_tiled_tanh_gb300 as rn
from asr_tiled_tanh_gb300 import binding, synthetic
from tests.helpers import TOL, to_device

pytestmark = pytest.mark.gpu


def _noalloc_fn():
    lib = rn.load(build_if_missing=True)
    f = lib.rnnt_fwd_noalloc
    P = ctypes.c_void_p
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.POINTER(binding.RnntDims), P, P, ctypes.POINTER(binding.RnntParams),
                  P, P, P, P, P, P]
    return f


def _saved_state(r):
    sa = r.saved_arrays()
    return {k: getattr(sa, k).clone() for k in ("lnP", "lpb", "lpl", "lnPD", "alpha", "beta")}


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_noalloc_forward_matches_rnnt_fwd_twice(dtype):
    H, V = (128, 256) if dtype == "bf16" else (64, 96)
    inp = synthetic.custom(B=4, T=60, U=20, HA=H, HL=H, H=H, V=V, dtype=dtype, seed=23,
                           bias_std=0.1)
    dev = to_device(inp)
    params = rn.make_params(dev["WA"], dev["WL"], dev["bZ"], dev["WO"], dev["bO"])
    ref = rn.Rnnt.for_inputs(inp)
    ref_loss = ref.fwd(dev["hA"], dev["hL"], params, dev["labels"], dev["T_len"], dev["U_len"])
    torch.cuda.synchronize()
    ref_state = _saved_state(ref)
    assert rn.rnnt_workspace_bytes(ref.dims) <= 32 << 20

    f = _noalloc_fn()
    stream = torch.cuda.current_stream().cuda_stream
    tl = TOL[dtype][0]
    for call in range(2):
        r = rn.Rnnt.for_inputs(inp)   # fresh `saved`; scratch comes from the library
        loss = torch.full((inp.wl.B,), float("nan"), device="cuda")
        code = f(ctypes.byref(r.dims), dev["hA"].data_ptr(), dev["hL"].data_ptr(),
                 ctypes.byref(params), dev["labels"].data_ptr(), dev["T_len"].data_ptr(),
                 dev["U_len"].data_ptr(), loss.data_ptr(), r.saved.data_ptr(), stream)
        assert code == 0, rn.rnnt_status_string(code)
        torch.cuda.synchronize()
        assert r.status() == (0, 0)
        got, want = loss.double().cpu().numpy(), ref_loss.double().cpu().numpy()
        assert np.all(np.abs(got - want) <= tl * np.abs(want)), (call, got, want)
        state = _saved_state(r)
        for k, v in ref_state.items():
            a, b = state[k].cpu().numpy(), v.cpu().numpy()
            assert np.array_equal(np.isneginf(a), np.isneginf(b)), (call, k)
            fin = np.isfinite(b)
            assert np.allclose(a[fin], b[fin], rtol=tl, atol=tl), (call, k)


def test_noalloc_rejects_problems_beyond_its_scratch():
    f = _noalloc_fn()
    # the large-batch 40 s workload needs far more than the fixed scratch
    dims = rn.make_dims(1024, 1000, 101, 512, 512, 512, 4096, 0, rn.RNNT_BF16, rn.RNNT_TILED, 0)
    assert rn.rnnt_workspace_bytes(dims) > 32 << 20
    params = rn.make_params(None, None, None, None, None)
    code = f(ctypes.byref(dims), None, None, ctypes.byref(params), None, None, None, None, None,
             None)
    assert code == 3  # RNNT_ERR_WORKSPACE_TOO_SMALL
