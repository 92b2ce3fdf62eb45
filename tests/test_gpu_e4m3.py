"""The e4m3 output-layer scores (dtype RNNT_BF16_E4M3) against the oracle (GPU).

The library quantizes W^O per block of 256 rows (power-of-two scales) and
runs the two score products on e4m3 tensor cores; the layer it computes, in
the forward and the backward alike, is W^O_q.  The oracle is fed W^O_q from
the host reference (tests/e4m3ref.py, PyTorch's float8 conversion) and
nothing else changes, so the only rounding the GPU adds beyond the bf16 path
is z entering the score products as e4m3(2^8 z).
"""
import numpy as np
import pytest
import torch

import asr_tiled_tanh_gb300 as rn
from asr_tiled_tanh_gb300 import binding, synthetic
from tests import e4m3ref
from tests.helpers import GRAD_KEYS, rel_l2, run_oracle, to_device

pytestmark = pytest.mark.gpu

# Tolerances of the e4m3 scores against the oracle fed W^O_q: the bf16 ones
# (loss relative error 2e-3, gradient relative L2 1e-2).  Why they hold: the
# only rounding beyond the bf16 path is z -> e4m3(2^8 z), a relative error of
# at most 2^-4 per element (3 mantissa bits, nearest even), uniform, so a score
# h_v = sum_k W_vk z_k picks up an error of about 2^-4 / sqrt(3) times
# sqrt(sum_k W_vk^2 z_k^2) ~ 0.036 rms(z) |W_v| ~ 0.02-0.03 here, independent
# from position to position; ln P is a posterior-weighted sum of T+U such
# per-position errors against |ln P| ~ (T+U) ln V, so the loss moves by
# ~0.03 / (ln V sqrt(T+U)) ~ 5e-4 at T+U ~ 50; the gradients see the score
# error through the softmax factor of dh, ~3% of its softmax part, which the
# sums over positions average down to a few 1e-3.  Measured on these tests:
# loss 4.5e-4 - 5.9e-4, gradients at most 6.8e-3 at H <= 512 and 9.2e-3 at the
# large-vocabulary shapes (H = 1024, V = 16384), the thinnest margin.
E4M3_TOL = {"loss": 2e-3, "grad": 1e-2}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    rn.load(build_if_missing=True)


@pytest.mark.parametrize("case", ["spread", "zero block"])
def test_quantizer_matches_the_host_reference_bit_for_bit(case):
    g = torch.Generator().manual_seed(7)
    V, H = 1000, 512   # four blocks, the last one ragged
    WO = (torch.randn(V, H, generator=g) / H ** 0.5)
    WO[256:512] *= 30.0
    WO[512:768] *= 1e-3
    WO[768:] = 0.0
    WO[999, 3] = 5e-3   # a lone value in an otherwise empty block
    if case == "zero block":
        WO[512:768] = 0.0   # an all-zero block: scale 1, every byte 0
    WO = WO.to(torch.bfloat16)
    q_ref, Wq_ref, s_ref = e4m3ref.quantize_wo(WO)
    dev = WO.cuda()
    q = torch.empty(V, H, dtype=torch.uint8, device="cuda")
    Wdq = torch.empty(V, H, dtype=torch.bfloat16, device="cuda")
    ns = torch.empty((V + 255) // 256, dtype=torch.float32, device="cuda")
    binding.rnnt_testing_quantize_wo(dev, q, Wdq, ns)
    torch.cuda.synchronize()
    assert torch.equal(q.cpu(), q_ref)
    assert torch.equal(Wdq.cpu().double(), Wq_ref)
    assert torch.equal(ns.cpu().double(), s_ref / e4m3ref.Z_SCALE)


def _run(inp, mode="tiled", tile_cells=0, grad_loss=None):
    dev = to_device(inp)
    r = rn.Rnnt.for_inputs(inp, mode=mode, tile_cells=tile_cells, e4m3_scores=True)
    params = rn.make_params(dev["WA"], dev["WL"], dev["bZ"], dev["WO"], dev["bO"])
    args = (dev["hA"], dev["hL"], params, dev["labels"], dev["T_len"], dev["U_len"])
    loss = r.fwd(*args)
    g = None if grad_loss is None else torch.as_tensor(grad_loss, dtype=torch.float32,
                                                       device="cuda")
    grads = r.bwd(*args, grad_loss=g)
    torch.cuda.synchronize()
    assert r.status() == (0, 0)
    out = {k: v.cpu().numpy() for k, v in grads.items()}
    out["loss"] = loss.double().cpu().numpy()
    return out


def _errors(gpu, orc):
    lrel = float(np.max(np.abs(gpu["loss"] - orc.loss) / np.abs(orc.loss)))
    return lrel, {k: rel_l2(gpu[k], orc.grads[k]) for k in GRAD_KEYS}


@pytest.mark.parametrize("mode,tile_cells", [("tiled", 0), ("tiled", 128 * 3), ("untiled", 0)])
def test_e4m3_scores_against_the_oracle(mode, tile_cells):
    inp = synthetic.custom(B=4, T=40, U=12, HA=256, HL=256, H=256, V=1024, dtype="bf16",
                           seed=51, bias_std=0.1)
    gpu = _run(inp, mode, tile_cells)
    orc = run_oracle(e4m3ref.with_quantized_wo(inp))
    lrel, gerr = _errors(gpu, orc)
    print(mode, tile_cells, "loss", lrel, "grads", gerr)
    assert lrel <= E4M3_TOL["loss"], lrel
    assert max(gerr.values()) <= E4M3_TOL["grad"], gerr


def test_e4m3_scores_bigger_vocabulary_several_blocks():
    # V = 4096: 16 W^O blocks with their own scales (the 40 s workload's V and H)
    inp = synthetic.custom(B=2, T=30, U=10, HA=512, HL=512, H=512, V=4096, dtype="bf16",
                           seed=52, bias_std=0.1)
    g = np.array([1.0, -0.5])
    gpu = _run(inp, grad_loss=g)
    orc = run_oracle(e4m3ref.with_quantized_wo(inp), grad_loss=g)
    lrel, gerr = _errors(gpu, orc)
    print("V4096 loss", lrel, "grads", gerr)
    assert lrel <= E4M3_TOL["loss"], lrel
    assert max(gerr.values()) <= E4M3_TOL["grad"], gerr


def test_e4m3_tiled_and_untiled_agree():
    inp = synthetic.custom(B=3, T=33, U=9, HA=128, HL=128, H=128, V=512, dtype="bf16", seed=53,
                           bias_std=0.2)
    runs = [_run(inp, "tiled", 128), _run(inp, "tiled", 0), _run(inp, "untiled", 0)]
    np.testing.assert_array_equal(runs[0]["loss"], runs[1]["loss"])
    np.testing.assert_allclose(runs[2]["loss"], runs[0]["loss"], rtol=1e-6)
    for r in runs[1:]:
        for k in GRAD_KEYS:
            assert rel_l2(r[k], runs[0][k]) < 1e-2, k


def test_e4m3_needs_h_multiple_of_16():
    dims = rn.make_dims(2, 8, 4, 64, 64, 72, 64, 0, rn.RNNT_BF16_E4M3, rn.RNNT_TILED, 0)
    assert rn.rnnt_workspace_bytes(dims) > 0
    inp = synthetic.custom(B=2, T=8, U=3, HA=64, HL=64, H=72, V=64, dtype="bf16", seed=1)
    dev = to_device(inp)
    r = rn.Rnnt(2, 8, 4, 64, 64, 72, 64, 0, "bf16-e4m3")
    params = rn.make_params(dev["WA"], dev["WL"], dev["bZ"], dev["WO"], dev["bO"])
    loss = torch.empty(2, device="cuda")
    code = rn.rnnt_fwd(r.dims, dev["hA"], dev["hL"], params, dev["labels"], dev["T_len"],
                       dev["U_len"], loss, r.saved, r.ws, check=False)
    assert code == 2  # RNNT_ERR_UNSUPPORTED_SHAPE


def test_e4m3_training_step_call_and_graph_capture():
    # rnnt_fwd_bwd with e4m3 scores (the backward rebuilds both the e4m3 and
    # the bf16 z rows) equals the separate calls, eagerly and replayed from a
    # CUDA graph of the step
    inp = synthetic.custom(B=3, T=40, U=10, HA=128, HL=128, H=128, V=512, dtype="bf16",
                           seed=54, bias_std=0.2)
    dev = to_device(inp)
    params = rn.make_params(dev["WA"], dev["WL"], dev["bZ"], dev["WO"], dev["bO"])
    args = (dev["hA"], dev["hL"], params, dev["labels"], dev["T_len"], dev["U_len"])
    sep = _run(inp)
    r = rn.Rnnt.for_inputs(inp, e4m3_scores=True)
    assert rn.rnnt_graph_capturable(r.dims) == 1
    loss, grads = r.fwd_bwd(*args)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(loss.double().cpu().numpy(), sep["loss"])
    for k in GRAD_KEYS:
        assert rel_l2(grads[k].cpu().numpy(), sep[k]) < 1e-3, k
    # the same step captured into a CUDA graph and replayed
    loss2 = torch.empty_like(loss)
    g2 = r.alloc_grads()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        r.fwd_bwd(*args, loss=loss2, grads=g2, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        r.fwd_bwd(*args, loss=loss2, grads=g2, stream=s)
    loss2.fill_(float("nan"))
    graph.replay()
    torch.cuda.synchronize()
    assert r.status() == (0, 0)
    np.testing.assert_array_equal(loss2.double().cpu().numpy(), sep["loss"])
    for k in GRAD_KEYS:
        assert rel_l2(g2[k].cpu().numpy(), sep[k]) < 1e-3, k


def test_e4m3_scores_large_vocabulary_shapes():
    # the large-vocabulary configuration's shapes (H = 1024, V = 16384: 64 W^O
    # blocks, Zipf labels) on short lattices, tiled over several chunks
    inp = synthetic.custom(B=2, T=20, U=6, HA=1024, HL=1024, H=1024, V=16384, dtype="bf16",
                           seed=55, labels="zipf1.1", bias_std=0.1)
    gpu = _run(inp, "tiled", 128)
    orc = run_oracle(e4m3ref.with_quantized_wo(inp))
    lrel, gerr = _errors(gpu, orc)
    print("bigvocab e4m3 loss", lrel, "grads", gerr)
    assert lrel <= E4M3_TOL["loss"], lrel
    assert max(gerr.values()) <= E4M3_TOL["grad"], gerr


def test_e4m3_ragged_vocabulary_and_partial_k_block():
    # V = 1000: the last W^O block holds 232 rows and the last N tile is
    # ragged; H = HA = HL = 48: one e4m3 K block of 128 bytes of which 48 hold
    # data (the MMA issues two of its four 32-wide steps)
    inp = synthetic.custom(B=3, T=29, U=7, HA=48, HL=48, H=48, V=1000, dtype="bf16", seed=56,
                           t_frac=0.3, u_frac=0.0, bias_std=0.3)
    g = np.array([0.7, 1.3, -0.4])
    for mode, tc in (("tiled", 128), ("untiled", 0)):
        gpu = _run(inp, mode, tc, grad_loss=g)
        orc = run_oracle(e4m3ref.with_quantized_wo(inp), grad_loss=g)
        lrel, gerr = _errors(gpu, orc)
        print("ragged", mode, "loss", lrel, "grads", gerr)
        assert lrel <= E4M3_TOL["loss"], (mode, lrel)
        assert max(gerr.values()) <= E4M3_TOL["grad"], (mode, gerr)
