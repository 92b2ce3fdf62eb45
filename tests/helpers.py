"""Shared test plumbing: run the library and the oracle on the same inputs."""
from __future__ import annotations

import numpy as np
import torch

import asr_tiled_tanh_gb300 as rn
from asr_tiled_tanh_gb300 import synthetic

GRAD_KEYS = ("dhA", "dhL", "dWA", "dWL", "dbZ", "dWO", "dbO")

# Tolerances (loss relative error, gradient relative L2 error) by dtype.
TOL = {"f32": (1e-5, 1e-4), "bf16": (2e-3, 1e-2)}

# fp32 unit roundoff.
U32 = 2.0 ** -24


def fp32_grad_tol(T: int, U: int, V: int) -> float:
    """Gradient tolerance of the fp32 path on a lattice of T frames and U
    labels over V symbols.

    alpha and beta are stored in fp32 (the saved state of the boundary) and
    reach |ln P| ~ (T + U) ln V; each of the three terms of a posterior's
    exponent, alpha + beta - ln P, then carries an absolute error of a few
    units of roundoff times that magnitude, and exp turns an absolute error
    in log space into the same relative error of the posterior and of every
    gradient built from it.  The bound is 8 u (T + U) ln V (u = 2^-24; the
    factor 8 covers the three terms and the accumulation along the
    recursion), and never below the 1e-4 the pages' fp32 target states.  It
    is a limit of this implementation's fp32 saved alpha/beta, not of the
    method.  Among the stated configurations only the tiny one is fp32:
    (32 + 8) ln 32 gives 6.6e-5, so 1e-4 holds there; the bound passes 1e-4
    once (T + U) ln V exceeds about 210 (e.g. T + U = 324, V = 48: 6.0e-4).
    """
    return max(TOL["f32"][1], 8.0 * U32 * (T + U) * np.log(V))


def to_device(inp: synthetic.Inputs, device="cuda"):
    d = {k: getattr(inp, k).to(device) for k in ("hA", "hL", "WA", "WL", "bZ", "WO", "bO",
                                                  "labels", "T_len", "U_len")}
    return d


def run_gpu(inp: synthetic.Inputs, mode="tiled", tile_cells=0, grad_loss=None, dev=None,
            want_grad=True, keep_saved=True):
    """Forward (+ backward) through the C ABI; returns host numpy arrays."""
    dev = dev if dev is not None else to_device(inp)
    r = rn.Rnnt.for_inputs(inp, mode=mode, tile_cells=tile_cells)
    params = rn.make_params(dev["WA"], dev["WL"], dev["bZ"], dev["WO"], dev["bO"])
    loss = r.fwd(dev["hA"], dev["hL"], params, dev["labels"], dev["T_len"], dev["U_len"])
    out = dict(loss=loss.double().cpu().numpy())
    if keep_saved:
        sa = r.saved_arrays()
        out.update({k: getattr(sa, k).double().cpu().numpy()
                    for k in ("lnP", "lpb", "lpl", "lnPD", "alpha", "beta")})
    if want_grad:
        g = None if grad_loss is None else torch.as_tensor(grad_loss, dtype=torch.float32,
                                                           device="cuda")
        grads = r.bwd(dev["hA"], dev["hL"], params, dev["labels"], dev["T_len"], dev["U_len"],
                      grad_loss=g)
        out.update({k: v.cpu().numpy() for k, v in grads.items()})
    code, word = r.status()
    out["status"] = (code, word)
    torch.cuda.synchronize()
    return out


def run_oracle(inp: synthetic.Inputs, grad_loss=None, want_grad=True, nthreads=0):
    import oracle
    f = lambda t: t.double().numpy()
    return oracle.rnnt(f(inp.hA), f(inp.hL), f(inp.WA), f(inp.WL), f(inp.bZ), f(inp.WO),
                       f(inp.bO), inp.labels.numpy(), inp.T_len.numpy(), inp.U_len.numpy(),
                       blank=0, grad_loss=grad_loss, want_grad=want_grad, nthreads=nthreads)


def rel_l2(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    nb = np.linalg.norm(b)
    if nb == 0:
        return float(np.linalg.norm(a))
    return float(np.linalg.norm(a - b) / nb)


def valid_mask(inp):
    B, T, U1 = inp.wl.B, inp.wl.T, inp.wl.U1
    t = np.arange(T)[None, :, None]
    u = np.arange(U1)[None, None, :]
    return (t < inp.T_len.numpy()[:, None, None]) & (u <= inp.U_len.numpy()[:, None, None])


def assert_parity(gpu, orc, inp, dtype=None, grads=True, check_saved=True):
    """Compare a GPU run with the oracle at the tolerance of the dtype."""
    dtype = dtype or inp.wl.dtype
    tl, tg = TOL[dtype]
    lrel = np.abs(gpu["loss"] - orc.loss) / np.abs(orc.loss)
    assert lrel.max() <= tl, f"loss rel err {lrel.max():.3e} > {tl}"
    if check_saved:
        # indexing is exact: the -inf pattern of every saved array matches;
        # the finite values match to the loss tolerance relative to their
        # magnitude (alpha(0,0) = 0 and values below 1 in magnitude get that
        # tolerance as an absolute one)
        for k in ("lpb", "lpl", "lnPD", "alpha", "beta"):
            g, o = gpu[k], getattr(orc, k)
            assert np.array_equal(np.isneginf(g), np.isneginf(o)), f"{k}: -inf mask differs"
            fin = np.isfinite(o)
            assert np.all(np.isfinite(g[fin])), f"{k}: non-finite where the oracle is finite"
            err = np.abs(g[fin] - o[fin]) / np.maximum(1.0, np.abs(o[fin]))
            assert err.size == 0 or err.max() <= tl, \
                f"{k}: value error {err.max():.3e} > {tl} (at {np.argmax(err)} of {err.size})"
    if grads:
        errs = {k: rel_l2(gpu[k], orc.grads[k]) for k in GRAD_KEYS}
        bad = {k: v for k, v in errs.items() if v > tg}
        assert not bad, f"gradient rel L2 errors above {tg}: {bad} (all: {errs})"
        return errs
    return {}
