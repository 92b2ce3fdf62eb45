"""Parity at the full workload sizes (GPU).

The oracle cannot run whole batches of these sizes in seconds, so each test
runs the full batch on the GPU in the configuration the benchmark uses and
checks (a) the losses of sampled samples against the oracle run on just those
samples, (b) the gradients of a sub-batch of those samples against the
oracle, and (c) properties that hold at any size: every loss finite and
positive, the output-bias gradient summing to zero over the vocabulary
(sum_v dh = 0 at every position), batched = sum of sample-wise, and the tile
buffer, not the lattice, setting the memory.  The large-vocabulary shapes get
full gradient parity on short lattices, and the 40 s batch's longest lattice
(full T and U) its loss parity.
"""
import numpy as np
import pytest
import torch

import functools

import asr_tiled_tanh_gb300 as rn
from asr_tiled_tanh_gb300 import synthetic
from tests.helpers import TOL, assert_parity, rel_l2, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


@functools.lru_cache(maxsize=1)
def _workload(name):
    return synthetic.make(name)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    rn.load(build_if_missing=True)


def _shortest(inp, k):
    cells = (inp.T_len.long() * (inp.U_len.long() + 1)).numpy()
    return [int(i) for i in np.argsort(cells, kind="stable")[:k]]


def _check_full_batch(inp, full, n_loss, n_grad, tile_cells=0, want_grad_parity=True):
    tl, tg = TOL[inp.wl.dtype]
    assert full["status"] == (0, 0)
    assert np.all(np.isfinite(full["loss"])) and np.all(full["loss"] > 0)
    # sum_v dh = 0 at every position, so sum_v db^O = 0 (relative to its size)
    dbO = full["dbO"]
    assert abs(dbO.sum()) <= 1e-3 * np.abs(dbO).sum() + 1e-6
    for k in ("dhA", "dhL", "dWA", "dWL", "dbZ", "dWO", "dbO"):
        assert np.all(np.isfinite(full[k])), k
    # sampled losses against the oracle, from the full-batch run
    idx = _shortest(inp, n_loss)
    sub = inp.subset(idx)
    orc = run_oracle(sub, want_grad=False)
    lrel = np.abs(full["loss"][idx] - orc.loss) / np.abs(orc.loss)
    assert lrel.max() <= tl, lrel
    # gradients of a sub-batch (identical tensors) against the oracle
    if want_grad_parity:
        gsub = inp.subset(idx[:n_grad])
        g = run_gpu(gsub, tile_cells=tile_cells)
        o = run_oracle(gsub)
        assert_parity(g, o, gsub)


def test_audio20_workload():
    inp = _workload("audio20")
    full = run_gpu(inp, keep_saved=False)
    _check_full_batch(inp, full, n_loss=3, n_grad=2)


def test_bigvocab_workload():
    inp = _workload("bigvocab")
    full = run_gpu(inp, keep_saved=False)
    # the oracle costs ~2e7 multiply-adds per position here: losses of the two
    # shortest samples, gradients through the properties and the smaller configs
    _check_full_batch(inp, full, n_loss=2, n_grad=0, want_grad_parity=False)
    # batched = sum of sample-wise (sample-wise paper §4), on two samples
    idx = _shortest(inp, 2)
    pair = run_gpu(inp.subset(idx), keep_saved=False)
    ones = [run_gpu(inp.subset([i]), keep_saved=False) for i in idx]
    for j, o in enumerate(ones):
        assert o["loss"][0] == pair["loss"][j]
    for k in ("dWO", "dbO", "dWA", "dbZ"):
        assert rel_l2(ones[0][k] + ones[1][k], pair[k]) < 1e-4, k


@pytest.mark.parametrize("mode,tile_cells", [("tiled", 0), ("tiled", 128), ("untiled", 0)])
def test_bigvocab_shapes_gradients_against_oracle(mode, tile_cells):
    # The large-vocabulary configuration's shapes (H = HA = HL = 1024,
    # V = 16384, Zipf(1.1) labels) on lattices short enough for the oracle's
    # gradients: every gradient compared with the oracle, in one chunk, in one
    # tile per chunk (several chunks) and untiled.
    inp = synthetic.custom(B=3, T=20, U=6, HA=1024, HL=1024, H=1024, V=16384, dtype="bf16",
                           seed=41, t_frac=0.5, u_frac=0.5, labels="zipf1.1", bias_std=0.1)
    gpu = run_gpu(inp, mode=mode, tile_cells=tile_cells)
    assert gpu["status"] == (0, 0)
    orc = _oracle_cached(inp.wl)
    errs = assert_parity(gpu, orc, inp)
    print(mode, tile_cells, "gradient rel L2:", errs)


@functools.lru_cache(maxsize=1)
def _oracle_cached(wl):
    inp = synthetic.make(wl, bias_std=0.1)
    return run_oracle(inp)


def test_audio40_large_batch_workload():
    inp = _workload("audio40")
    torch.cuda.reset_peak_memory_stats()
    full = run_gpu(inp, keep_saved=False)
    peak = torch.cuda.max_memory_allocated()
    _check_full_batch(inp, full, n_loss=2, n_grad=2)
    # the longest lattice: sample 0 has the full T = 1000 frames and U = 100
    # labels (101,000 positions, |ln P| ~ 9e3); its loss from the full-batch
    # run against the oracle's forward on that sample alone
    assert int(inp.T_len[0]) == inp.wl.T and int(inp.U_len[0]) == inp.wl.U
    o0 = run_oracle(inp.subset([0]), want_grad=False)
    lrel = abs(full["loss"][0] - o0.loss[0]) / abs(o0.loss[0])
    assert lrel <= TOL["bf16"][0], (full["loss"][0], o0.loss[0], lrel)
    # memory is set by the tile buffer, not by B*T*(U+1)*V (847 GB of bf16 scores)
    nominal_scores = inp.wl.B * inp.wl.T * inp.wl.U1 * inp.wl.V * 2
    assert peak < nominal_scores / 40, peak


def test_audio40_memory_tracks_tile_size():
    inp = _workload("audio40")
    dev = {k: getattr(inp, k).cuda() for k in ("hA", "hL", "WA", "WL", "bZ", "WO", "bO",
                                                "labels", "T_len", "U_len")}
    params = rn.make_params(dev["WA"], dev["WL"], dev["bZ"], dev["WO"], dev["bO"])
    peaks, ws = [], []
    losses = []
    for tc in (128 * 152, 128 * 608):
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        base = torch.cuda.memory_allocated()
        torch.cuda.reset_peak_memory_stats()
        r = rn.Rnnt.for_inputs(inp, tile_cells=tc)
        loss = r.fwd(dev["hA"], dev["hL"], params, dev["labels"], dev["T_len"], dev["U_len"])
        g = r.bwd(dev["hA"], dev["hL"], params, dev["labels"], dev["T_len"], dev["U_len"])
        torch.cuda.synchronize()
        peaks.append(torch.cuda.max_memory_allocated() - base)
        ws.append(r.ws.numel())
        losses.append(loss.cpu())
        del r, g, loss
    # the difference in peak memory is the difference in tile buffers (allocator slack 64 MiB)
    assert abs((peaks[1] - peaks[0]) - (ws[1] - ws[0])) < 64 << 20
    assert torch.equal(losses[0], losses[1])


def test_untiled_mode_refuses_the_40s_batch():
    # Untiled mode keeps z and the scores of every lattice position: at the
    # 40 s, batch-1024 shapes that is ~0.9 TB of bf16 scores, more than the
    # device holds, so rnnt_fwd refuses the plan before it looks at any buffer
    # (the pointers are all NULL: no launch can happen whatever the outcome;
    # a missing check would show as RNNT_ERR_INVALID_ARG instead)
    dims = rn.make_dims(1024, 1000, 101, 512, 512, 512, 4096, 0, rn.RNNT_BF16, rn.RNNT_UNTILED, 0)
    assert rn.rnnt_saved_bytes(dims) > torch.cuda.get_device_properties(0).total_memory
    params = rn.make_params(None, None, None, None, None)
    code = rn.rnnt_fwd(dims, None, None, params, None, None, None, None, None, None,
                       check=False)
    assert code == 3  # RNNT_ERR_WORKSPACE_TOO_SMALL
    # the same shapes tiled are a valid plan (they fail here only on the NULL buffers)
    tiled = rn.make_dims(1024, 1000, 101, 512, 512, 512, 4096, 0, rn.RNNT_BF16, rn.RNNT_TILED, 0)
    code = rn.rnnt_fwd(tiled, None, None, params, None, None, None, None, None, None,
                       check=False)
    assert code == 1  # RNNT_ERR_INVALID_ARG


def test_audio40_under_a_memory_budget():
    # the tile size chosen for a 13 GB budget: the library's whole footprint
    # (saved + workspace) fits it, the chunks are whole waves of SMs, and the
    # losses are those of the default plan (the forward is the same per tile)
    inp = _workload("audio40")
    budget = 13 * 10 ** 9
    dims = rn.make_dims(inp.wl.B, inp.wl.T, inp.wl.U1, inp.wl.HA, inp.wl.HL, inp.wl.H, inp.wl.V,
                        0, rn.RNNT_BF16, rn.RNNT_TILED, 0)
    tc = rn.rnnt_tile_cells_for_budget(dims, budget)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert tc > 0 and (tc // 128) % sms == 0
    dev = {k: getattr(inp, k).cuda() for k in ("hA", "hL", "WA", "WL", "bZ", "WO", "bO",
                                                "labels", "T_len", "U_len")}
    params = rn.make_params(dev["WA"], dev["WL"], dev["bZ"], dev["WO"], dev["bO"])
    args = (dev["hA"], dev["hL"], params, dev["labels"], dev["T_len"], dev["U_len"])
    losses = []
    for tile_cells in (tc, 0):
        r = rn.Rnnt.for_inputs(inp, tile_cells=tile_cells)
        if tile_cells == tc:
            assert r.saved.numel() + r.ws.numel() <= budget
        losses.append(r.fwd(*args).cpu())
        torch.cuda.synchronize()
        assert r.status() == (0, 0)
        del r
    assert torch.equal(losses[0], losses[1])
