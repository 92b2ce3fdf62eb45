"""rnnt_fwd_noalloc, the forward pass for callers that cannot allocate (GPU).

Some callers cannot allocate device memory: hosts that reserve all memory up
front, plugin interfaces that provide no allocator, latency-critical loops.
rnnt_fwd_noalloc takes its scratch from a fixed device array inside the
library instead of a caller buffer.  This test calls it through the C ABI
several times in a row (different values, lengths and chunk counts) and checks
that every call gives what rnnt_fwd gives with a fresh caller-provided
workspace; it runs last (file name) so that a failure here never hides the
rest of the suite, and it needs no earlier test's state.
"""
import numpy as np
import pytest
import torch

import asr_tiled_tanh_gb300 as rn
from asr_tiled_tanh_gb300 import synthetic
from tests.helpers import TOL, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    rn.load(build_if_missing=True)


def _saved_state(r):
    sa = r.saved_arrays()
    return {k: getattr(sa, k).clone() for k in ("lnP", "lpb", "lpl", "lnPD", "alpha", "beta")}


def _call_noalloc(r, dev, params, B):
    loss = torch.full((B,), float("nan"), device="cuda")
    code = rn.rnnt_fwd_noalloc(r.dims, dev["hA"], dev["hL"], params, dev["labels"], dev["T_len"],
                               dev["U_len"], loss, r.saved, check=False)
    assert code == 0, rn.rnnt_status_string(code)
    torch.cuda.synchronize()
    return loss


def _check_against_rnnt_fwd(inp, tile_cells, tag, e4m3=False):
    """One rnnt_fwd_noalloc call against rnnt_fwd with a fresh caller workspace."""
    dtype = inp.wl.dtype
    dev = to_device(inp)
    params = rn.make_params(dev["WA"], dev["WL"], dev["bZ"], dev["WO"], dev["bO"])
    ref = rn.Rnnt.for_inputs(inp, tile_cells=tile_cells, e4m3_scores=e4m3)
    assert rn.rnnt_workspace_bytes(ref.dims) <= 32 << 20
    ref_loss = ref.fwd(dev["hA"], dev["hL"], params, dev["labels"], dev["T_len"], dev["U_len"])
    torch.cuda.synchronize()
    assert ref.status() == (0, 0)
    ref_state = _saved_state(ref)
    # fresh `saved`; scratch from the library
    r = rn.Rnnt.for_inputs(inp, tile_cells=tile_cells, e4m3_scores=e4m3)
    loss = _call_noalloc(r, dev, params, inp.wl.B)
    assert r.status() == (0, 0)
    tl = TOL[dtype][0]
    got, want = loss.double().cpu().numpy(), ref_loss.double().cpu().numpy()
    assert np.all(np.abs(got - want) <= tl * np.abs(want)), (tag, got, want)
    state = _saved_state(r)
    for k, v in ref_state.items():
        a, b = state[k].cpu().numpy(), v.cpu().numpy()
        assert np.array_equal(np.isneginf(a), np.isneginf(b)), (tag, k)
        fin = np.isfinite(b)
        assert np.allclose(a[fin], b[fin], rtol=tl, atol=tl), (tag, k)


@pytest.mark.parametrize("mode", ["bf16", "bf16-e4m3", "f32"])
def test_noalloc_forward_matches_rnnt_fwd_on_calls_in_a_row(mode):
    # Three calls in a row share the library's scratch array, each left with
    # the previous call's contents: full-ish lengths; then other values with
    # much shorter lattices (more positions of the same tiles outside every
    # lattice); then a plan of several chunks (small tile buffers), so that
    # every chunk reuses tile buffers the previous one wrote.
    dtype = "f32" if mode == "f32" else "bf16"
    e4m3 = mode == "bf16-e4m3"  # (the quantized output layer lives in the scratch too)
    H, V = (128, 256) if dtype == "bf16" else (64, 96)
    cases = [
        (synthetic.custom(B=4, T=60, U=20, HA=H, HL=H, H=H, V=V, dtype=dtype, seed=23,
                          bias_std=0.1), 0, "first"),
        (synthetic.custom(B=4, T=60, U=20, HA=H, HL=H, H=H, V=V, dtype=dtype, seed=24,
                          t_frac=0.1, u_frac=0.1, full_first=False, bias_std=0.2), 0,
         "shorter lengths"),
        (synthetic.custom(B=4, T=60, U=20, HA=H, HL=H, H=H, V=V, dtype=dtype, seed=25,
                          bias_std=0.1), 3 * 128, "three tiles per chunk"),
    ]
    for inp, tile_cells, tag in cases:
        _check_against_rnnt_fwd(inp, tile_cells, tag, e4m3)


def test_noalloc_rejects_problems_beyond_its_scratch():
    # the large-batch 40 s workload needs far more than the fixed scratch
    dims = rn.make_dims(1024, 1000, 101, 512, 512, 512, 4096, 0, rn.RNNT_BF16, rn.RNNT_TILED, 0)
    assert rn.rnnt_workspace_bytes(dims) > 32 << 20
    params = rn.make_params(None, None, None, None, None)
    code = rn.rnnt_fwd_noalloc(dims, None, None, params, None, None, None, None, None,
                               check=False)
    assert code == 3  # RNNT_ERR_WORKSPACE_TOO_SMALL
