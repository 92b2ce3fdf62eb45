"""rnnt_bwd_ex: the encoder-side gradients handed over in bf16, and the joint
projections' gradients dA, dL for an encoder that folds dh^A = dA W^A and
dh^L = dL W^L into its own backward (GPU).

dA and dL are checked through what defines them: dA W^A = dh^A and
dL W^L = dh^L (against the plain backward's fp32 outputs, which the parity
tests hold to the oracle) and sum over frames of dA = db^Z.
"""
import numpy as np
import pytest
import torch

import asr_tiled_tanh_gb300 as rn
from asr_tiled_tanh_gb300 import synthetic
from tests.helpers import TOL, rel_l2, run_oracle, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    rn.load(build_if_missing=True)


def _setup(dtype, e4m3=False):
    H = 128 if dtype == "bf16" else 48
    inp = synthetic.custom(B=3, T=30, U=8, HA=H + 32, HL=H - 16, H=H, V=256, dtype=dtype,
                           seed=61, bias_std=0.2)
    dev = to_device(inp)
    r = rn.Rnnt.for_inputs(inp, e4m3_scores=e4m3)
    params = rn.make_params(dev["WA"], dev["WL"], dev["bZ"], dev["WO"], dev["bO"])
    args = (dev["hA"], dev["hL"], params, dev["labels"], dev["T_len"], dev["U_len"])
    return inp, dev, r, args


def _np(t):
    return t.double().cpu().numpy()


@pytest.mark.parametrize("e4m3", [False, True])
def test_bf16_handoff(e4m3):
    inp, dev, r, args = _setup("bf16", e4m3)
    g = np.array([1.0, 0.5, -1.5])
    r.fwd(*args)
    ref = r.bwd(*args, grad_loss=torch.tensor(g, dtype=torch.float32, device="cuda"))
    out = r.bwd_ex(*args, grad_loss=g, enc_dtype="bf16", handoff=True)
    torch.cuda.synchronize()
    assert r.status() == (0, 0)
    assert out["dhA"].dtype == torch.bfloat16 and out["dA"].dtype == torch.bfloat16
    # dh^A, dh^L in bf16: the fp32 result rounded (fp32 atomic order aside)
    for k in ("dhA", "dhL"):
        a, b = _np(out[k]), _np(ref[k])
        assert np.all(np.abs(a - b) <= 2.0 ** -8 * np.abs(b) + 1e-5 * np.abs(b).max()), k
    # the projections' gradients: dA W^A = dh^A, dL W^L = dh^L, sum of dA = db^Z
    WA, WL = _np(dev["WA"]), _np(dev["WL"])
    assert rel_l2(_np(out["dA"]) @ WA, _np(ref["dhA"])) < 1e-2
    assert rel_l2(_np(out["dL"]) @ WL, _np(ref["dhL"])) < 1e-2
    assert rel_l2(_np(out["dA"]).sum(axis=(0, 1)), _np(ref["dbZ"])) < 1e-2
    # zero outside each sample's lengths
    T_len, U_len = inp.T_len.numpy(), inp.U_len.numpy()
    for b in range(inp.wl.B):
        assert not _np(out["dA"])[b, T_len[b]:].any()
        assert not _np(out["dL"])[b, U_len[b] + 1:].any()
    # parameter gradients are those of the plain backward
    for k in ("dWA", "dWL", "dbZ", "dWO", "dbO"):
        assert rel_l2(_np(out[k]), _np(ref[k])) < 1e-4, k


def test_handoff_without_encoder_products():
    # dh^A, dh^L left to the caller (NULL): the rest is unchanged
    inp, dev, r, args = _setup("bf16")
    r.fwd(*args)
    full = r.bwd_ex(*args, enc_dtype="bf16", handoff=True)
    r.fwd(*args)
    part = r.bwd_ex(*args, enc_dtype="bf16", handoff=True, skip_enc=True)
    torch.cuda.synchronize()
    assert part["dhA"] is None and part["dhL"] is None
    for k in ("dA", "dL", "dWA", "dWL", "dbZ", "dWO", "dbO"):
        assert rel_l2(_np(part[k]), _np(full[k])) < 1e-4, k


def test_fp32_handoff_against_the_oracle():
    inp, dev, r, args = _setup("f32")
    r.fwd(*args)
    out = r.bwd_ex(*args, enc_dtype="f32", handoff=True)
    torch.cuda.synchronize()
    orc = run_oracle(inp)
    tg = TOL["f32"][1]
    assert rel_l2(_np(out["dhA"]), orc.grads["dhA"]) < tg
    assert rel_l2(_np(out["dA"]) @ _np(dev["WA"]), orc.grads["dhA"]) < tg
    assert rel_l2(_np(out["dL"]) @ _np(dev["WL"]), orc.grads["dhL"]) < tg
    assert rel_l2(_np(out["dA"]).sum(axis=(0, 1)), orc.grads["dbZ"]) < tg


def test_handoff_option_errors():
    inp, dev, r, args = _setup("f32")
    r.fwd(*args)
    g = r.alloc_grads()
    for opts in (rn.RnntBwdOpts(rn.RNNT_BF16, None, None),   # bf16 hand-off of an fp32 problem
                 rn.RnntBwdOpts(7, None, None)):               # unknown element type
        code = rn.rnnt_bwd_ex(r.dims, *args, None, r.saved, g["dhA"], g["dhL"], g["dWA"],
                              g["dWL"], g["dbZ"], g["dWO"], g["dbO"], r.ws, opts, check=False)
        assert code == 1
