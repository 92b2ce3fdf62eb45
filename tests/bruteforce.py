"""Brute-force transducer likelihood by enumerating every alignment.

Used only to pin the oracle.  It shares nothing with ``oracle/``: the joint
network and output layer are evaluated with numpy matrix products over whole
sequences, the log-softmax with ``scipy.special.log_softmax``, and ln P is the
log-sum over an explicit list of alignment paths instead of a recursion.

An alignment of sample b is a sequence of T_b blank moves and U_b label moves
ending with a blank (the final blank leaves the lattice from (T_b-1, U_b)).
The label move out of label position u emits labels[b, u+1] (the labels carry
a prepended blank at index 0, "Neural transducer training: reduced memory
consumption with sample-wise computation", §2).  There are
C(T_b + U_b - 1, U_b) such paths.
"""
from __future__ import annotations

import itertools
import math

import numpy as np
from scipy.special import log_softmax, logsumexp


def log_probs(hA, hL, WA, WL, bZ, WO, bO):
    """Full [B,T,U1,V] log-softmax of the output scores, by whole-tensor numpy."""
    hA, hL, WA, WL, WO = (np.asarray(x, np.float64) for x in (hA, hL, WA, WL, WO))
    bZ = np.zeros(WA.shape[0]) if bZ is None else np.asarray(bZ, np.float64)
    bO = np.zeros(WO.shape[0]) if bO is None else np.asarray(bO, np.float64)
    pa = np.einsum("bti,hi->bth", hA, WA)
    pl = np.einsum("bui,hi->buh", hL, WL)
    z = np.tanh(pa[:, :, None, :] + pl[:, None, :, :] + bZ)
    h = np.einsum("btuh,vh->btuv", z, WO) + bO
    return log_softmax(h, axis=-1)


def paths(Tb: int, Ub: int):
    """Every alignment as a tuple of moves, 'b' (blank) or 'l' (label)."""
    n = Tb - 1 + Ub  # moves before the final blank
    for pos in itertools.combinations(range(n), Ub):
        mv = ["b"] * n
        for p in pos:
            mv[p] = "l"
        yield tuple(mv) + ("b",)


def n_paths(Tb: int, Ub: int) -> int:
    return math.comb(Tb - 1 + Ub, Ub)


def log_likelihood(lp, labels, Tb, Ub, blank=0):
    """ln P(y|x) of one sample from its [T,U1,V] log-probs, by path enumeration."""
    terms = []
    for mv in paths(Tb, Ub):
        t = u = 0
        s = 0.0
        for m in mv:
            if m == "b":
                s += lp[t, u, blank]
                t += 1
            else:
                s += lp[t, u, labels[u + 1]]
                u += 1
        assert t == Tb and u == Ub
        terms.append(s)
    return float(logsumexp(terms))


def losses(hA, hL, WA, WL, bZ, WO, bO, labels, T_len, U_len, blank=0):
    lp = log_probs(hA, hL, WA, WL, bZ, WO, bO)
    return np.array([-log_likelihood(lp[b], np.asarray(labels[b]), int(T_len[b]), int(U_len[b]),
                                     blank) for b in range(lp.shape[0])])
