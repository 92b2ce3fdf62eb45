"""Pins of the fp64 oracle against things other than itself (CPU only).

Each test names what fixes the expected value: path enumeration, a closed
form, a hand-worked lattice, central finite differences, or an identity that
holds for every transducer lattice.  Together they fail on a dropped term
(biases are non-zero), a wrong sign, a wrong label or length index (distinct
labels, mixed lengths), or a transposed weight (HA, HL, H and V all differ).
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from tests import bruteforce

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_case(seed, B=3, T=6, U=4, HA=5, HL=4, H=7, V=6, bias=0.3, full_first=True):
    rng = np.random.default_rng(seed)
    U1 = U + 1
    T_len = rng.integers(1, T + 1, B)
    U_len = rng.integers(0, U + 1, B)
    if full_first:
        T_len[0], U_len[0] = T, U
    labels = rng.integers(1, V, (B, U1))
    labels[:, 0] = 0
    return dict(
        hA=rng.normal(size=(B, T, HA)), hL=rng.normal(size=(B, U1, HL)),
        WA=rng.normal(size=(H, HA)) / math.sqrt(HA), WL=rng.normal(size=(H, HL)) / math.sqrt(HL),
        bZ=rng.normal(size=H) * bias, WO=rng.normal(size=(V, H)) * 1.5 / math.sqrt(H),
        bO=rng.normal(size=V) * bias, labels=labels.astype(np.int32),
        T_len=T_len.astype(np.int32), U_len=U_len.astype(np.int32))


def _valid_mask(T_len, U_len, T, U1):
    t = np.arange(T)[None, :, None]
    u = np.arange(U1)[None, None, :]
    return (t < np.asarray(T_len)[:, None, None]) & (u <= np.asarray(U_len)[:, None, None])


# --- path enumeration -------------------------------------------------------

@pytest.mark.parametrize("seed", range(6))
def test_loss_matches_path_enumeration(seed):
    c = _rand_case(seed)
    r = oracle.rnnt(**c, want_grad=False)
    bf = bruteforce.losses(**c)
    np.testing.assert_allclose(r.loss, bf, rtol=1e-12, atol=0)


def test_path_count_formula():
    # the enumerator itself: C(T+U-1, U) distinct paths, each ending with a blank
    for Tb, Ub in [(1, 0), (1, 3), (4, 0), (3, 2), (5, 4)]:
        ps = list(bruteforce.paths(Tb, Ub))
        assert len(ps) == len(set(ps)) == bruteforce.n_paths(Tb, Ub)
        assert all(p[-1] == "b" and p.count("b") == Tb and p.count("l") == Ub for p in ps)


def test_log_probs_at_every_cell_match_numpy_softmax():
    c = _rand_case(11, B=2, T=5, U=3)
    r = oracle.rnnt(**c, want_grad=False)
    lp = bruteforce.log_probs(c["hA"], c["hL"], c["WA"], c["WL"], c["bZ"], c["WO"], c["bO"])
    for b in range(2):
        for t in range(c["T_len"][b]):
            for u in range(c["U_len"][b] + 1):
                assert abs(r.lpb[b, t, u] - lp[b, t, u, 0]) < 1e-12
                if u < c["U_len"][b]:
                    assert abs(r.lpl[b, t, u] - lp[b, t, u, c["labels"][b, u + 1]]) < 1e-12
                else:
                    assert r.lpl[b, t, u] == -np.inf


# --- hand-worked lattices and closed forms ---------------------------------

def test_golden_constant_softmax_lattices():
    g = json.load(open(os.path.join(GOLDEN, "constant_softmax_lattices.json")))
    V, H, HA, HL = g["V"], g["H"], g["HA"], g["HL"]
    rng = np.random.default_rng(0)
    for case in g["cases"]:
        T, lab = case["T"], np.array(case["labels"], np.int32)[None, :]
        U1 = lab.shape[1]
        r = oracle.rnnt(hA=rng.normal(size=(1, T, HA)), hL=rng.normal(size=(1, U1, HL)),
                        WA=rng.normal(size=(H, HA)), WL=rng.normal(size=(H, HL)),
                        bZ=rng.normal(size=H), WO=np.zeros((V, H)), bO=np.array(g["bO"]),
                        labels=lab, T_len=[T], U_len=[U1 - 1], blank=g["blank"])
        assert abs(r.loss[0] - case["loss"]) < 1e-12, case["name"]
        np.testing.assert_allclose(r.grads["dbO"], case["dbO"], atol=1e-12, rtol=0)
        for k in ("dhA", "dhL", "dWA", "dWL", "dbZ"):
            assert np.all(r.grads[k] == 0.0), (case["name"], k)


def test_uniform_output_closed_form():
    # W^O = 0, b^O = 0: every emission has probability 1/V, so
    # -ln P = (T_b + U_b) ln V - ln C(T_b + U_b - 1, U_b) and no gradient reaches z.
    c = _rand_case(5, B=5, T=30, U=10, V=13, full_first=True)
    c["WO"][:] = 0.0
    c["bO"][:] = 0.0
    r = oracle.rnnt(**c)
    for b in range(5):
        Tb, Ub = int(c["T_len"][b]), int(c["U_len"][b])
        expect = (Tb + Ub) * math.log(13) - math.log(math.comb(Tb + Ub - 1, Ub))
        assert abs(r.loss[b] - expect) <= 1e-12 * expect
    for k in ("dhA", "dhL", "dWA", "dWL", "dbZ"):
        assert np.all(r.grads[k] == 0.0), k


def test_single_frame_and_blank_only_reductions():
    c = _rand_case(7, B=4, T=9, U=5)
    c["T_len"][:] = [1, 9, 1, 4]
    c["U_len"][:] = [5, 0, 0, 3]
    r = oracle.rnnt(**c, want_grad=False)
    # T_b = 1: one path, all labels then the final blank, all at t = 0
    for b in (0, 2):
        Ub = c["U_len"][b]
        expect = r.lpl[b, 0, :Ub].sum() + r.lpb[b, 0, Ub]
        assert abs(-r.loss[b] - expect) < 1e-12
    # U_b = 0: one path, a blank at every frame
    expect = r.lpb[1, :9, 0].sum()
    assert abs(-r.loss[1] - expect) < 1e-12


# --- lattice identities ------------------------------------------------------

def _posteriors(r, c):
    B, T, U1 = r.alpha.shape
    pb = np.zeros((B, T, U1))
    pl = np.zeros((B, T, U1))
    for b in range(B):
        Tb, Ub = int(c["T_len"][b]), int(c["U_len"][b])
        lnP = -r.loss[b]
        for t in range(Tb):
            for u in range(Ub + 1):
                bn = r.beta[b, t + 1, u] if t + 1 < Tb else (0.0 if u == Ub else -np.inf)
                pb[b, t, u] = math.exp(r.alpha[b, t, u] + r.lpb[b, t, u] + bn - lnP)
                if u < Ub:
                    pl[b, t, u] = math.exp(r.alpha[b, t, u] + r.lpl[b, t, u]
                                           + r.beta[b, t, u + 1] - lnP)
    return pb, pl


def test_alpha_beta_likelihoods_agree():
    c = _rand_case(3, B=4, T=40, U=12, V=20, H=16, HA=9, HL=11)
    r = oracle.rnnt(**c, want_grad=False)
    np.testing.assert_allclose(-r.loss, r.lnP_beta, rtol=1e-9, atol=0)


def test_occupancy_one_blank_per_frame_and_each_label_once():
    c = _rand_case(4, B=3, T=12, U=6, V=9)
    r = oracle.rnnt(**c, want_grad=False)
    pb, pl = _posteriors(r, c)
    for b in range(3):
        Tb, Ub = int(c["T_len"][b]), int(c["U_len"][b])
        np.testing.assert_allclose(pb[b, :Tb].sum(axis=1), 1.0, atol=1e-12)
        if Ub:
            np.testing.assert_allclose(pl[b, :Tb, :Ub].sum(axis=0), 1.0, atol=1e-12)


def test_dh_sums_to_zero_and_matches_posteriors():
    c = _rand_case(8, B=3, T=7, U=4, V=8)
    g = np.array([1.0, -0.5, 2.0])
    r = oracle.rnnt(**c, grad_loss=g, want_dh=True)
    mask = _valid_mask(c["T_len"], c["U_len"], 7, 5)
    s = r.dh.sum(axis=-1)
    assert np.all(np.abs(s[mask]) < 1e-12)
    assert np.all(r.dh[~mask] == 0.0)
    # the blank column: g * ((pb+pl) softmax_blank - pb)
    np.testing.assert_allclose(r.grads["dbO"].sum(), 0.0, atol=1e-12)
    pb, pl = _posteriors(r, c)
    sm_blank = np.exp(r.lpb)
    b_idx, t_idx, u_idx = np.nonzero(mask)
    expect = g[b_idx] * ((pb + pl)[mask] * sm_blank[mask] - pb[mask])
    got = r.dh[b_idx, t_idx, u_idx, 0]
    np.testing.assert_allclose(got, expect, atol=1e-12)


def test_saved_state_is_minus_inf_outside_the_lattice():
    c = _rand_case(9, B=4, T=8, U=5)
    r = oracle.rnnt(**c, want_grad=False)
    mask = _valid_mask(c["T_len"], c["U_len"], 8, 6)
    for a in (r.lpb, r.lpl, r.lnPD, r.alpha, r.beta):
        assert np.all(a[~mask] == -np.inf)
    for a in (r.lpb, r.lnPD, r.alpha, r.beta):
        assert np.all(np.isfinite(a[mask]))
    # lpl is -inf exactly on the last label row
    for b in range(4):
        Tb, Ub = c["T_len"][b], c["U_len"][b]
        assert np.all(r.lpl[b, :Tb, Ub] == -np.inf)
        assert np.all(np.isfinite(r.lpl[b, :Tb, :Ub]))


# --- gradients ---------------------------------------------------------------

def test_gradients_match_central_finite_differences():
    c = _rand_case(21, B=2, T=4, U=3, HA=3, HL=2, H=5, V=6, bias=0.1)
    c["T_len"][1], c["U_len"][1] = 3, 1
    g = np.array([0.7, 1.3])
    r = oracle.rnnt(**c, grad_loss=g)

    def total(cc):
        return float(np.dot(g, oracle.rnnt(**cc, want_grad=False, nthreads=1).loss))

    name_of = dict(hA="dhA", hL="dhL", WA="dWA", WL="dWL", bZ="dbZ", WO="dWO", bO="dbO")
    for key, gk in name_of.items():
        an = r.grads[gk]
        fd = np.zeros_like(an)
        base = c[key]
        for idx in np.ndindex(base.shape):
            x0 = base[idx]
            eps = 1e-6 * max(1.0, abs(x0))
            base[idx] = x0 + eps
            fp = total(c)
            base[idx] = x0 - eps
            fm = total(c)
            base[idx] = x0
            fd[idx] = (fp - fm) / (2 * eps)
        scale = max(np.abs(an).max(), 1e-30)
        err = np.abs(fd - an) / np.maximum(np.abs(an), 0.01 * scale)
        assert err.max() <= 1e-6, (key, err.max())


# --- properties the pages state ---------------------------------------------

def test_batched_equals_sum_of_single_samples():
    # Sample-wise paper §4: accumulating per-sample gradients "is identical to
    # batched computation".
    c = _rand_case(13, B=4, T=7, U=4)
    full = oracle.rnnt(**c)
    acc = {k: np.zeros_like(v) for k, v in full.grads.items() if k not in ("dhA", "dhL")}
    for b in range(4):
        cb = {k: (v[b:b + 1] if k in ("hA", "hL", "labels", "T_len", "U_len") else v)
              for k, v in c.items()}
        rb = oracle.rnnt(**cb)
        assert rb.loss[0] == full.loss[b]
        np.testing.assert_allclose(rb.grads["dhA"][0], full.grads["dhA"][b], rtol=0, atol=1e-14)
        np.testing.assert_allclose(rb.grads["dhL"][0], full.grads["dhL"][b], rtol=0, atol=1e-14)
        for k in acc:
            acc[k] += rb.grads[k]
    for k in acc:
        np.testing.assert_allclose(acc[k], full.grads[k], rtol=1e-12, atol=1e-14)


def test_padding_is_never_read():
    c = _rand_case(17, B=4, T=8, U=5)
    clean = oracle.rnnt(**c)
    d = {k: v.copy() for k, v in c.items()}
    for b in range(4):
        Tb, Ub = d["T_len"][b], d["U_len"][b]
        d["hA"][b, Tb:] = np.nan
        d["hL"][b, Ub + 1:] = np.nan
        d["labels"][b, Ub + 1:] = -7
        d["labels"][b, 0] = 12345   # the prepended blank slot is never read either
    dirty = oracle.rnnt(**d)
    np.testing.assert_array_equal(clean.loss, dirty.loss)
    for k in clean.grads:
        np.testing.assert_array_equal(clean.grads[k], dirty.grads[k])
    for b in range(4):
        assert np.all(dirty.grads["dhA"][b, d["T_len"][b]:] == 0.0)
        assert np.all(dirty.grads["dhL"][b, d["U_len"][b] + 1:] == 0.0)


@pytest.mark.parametrize("field,value", [("T_len", 0), ("T_len", 9), ("U_len", 6),
                                         ("U_len", -1)])
def test_rejects_bad_lengths(field, value):
    c = _rand_case(1, B=2, T=8, U=5)
    c[field][1] = value
    with pytest.raises(ValueError, match="length"):
        oracle.rnnt(**c, want_grad=False)


@pytest.mark.parametrize("value", [-1, 6])
def test_rejects_bad_labels(value):
    c = _rand_case(1, B=2, T=8, U=5, V=6)
    c["U_len"][1] = 3
    c["labels"][1, 2] = value
    with pytest.raises(ValueError, match="label"):
        oracle.rnnt(**c, want_grad=False)


def test_thread_count_does_not_change_forward_values():
    c = _rand_case(23, B=5, T=9, U=4)
    r1 = oracle.rnnt(**c, nthreads=1)
    r4 = oracle.rnnt(**c, nthreads=4)
    np.testing.assert_array_equal(r1.loss, r4.loss)
    for k in r1.grads:
        np.testing.assert_allclose(r1.grads[k], r4.grads[k], rtol=1e-12, atol=1e-15)
