"""fp64 CPU oracle for the RNN-T joint network, output layer and transducer loss.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
benchmark's CPU-baseline leg may import this package.  The product library
(``asr_tiled_tanh_gb300``) never imports, links or runs anything here, and
this package imports nothing from it.

The arithmetic lives in ``rnnt_oracle.c`` (plain definition, fp64, one cell at
a time; see its header for the equations and the readings of the pages).  This
module compiles it with gcc and marshals numpy arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle_rnnt.so")
_SRC = os.path.join(_HERE, "rnnt_oracle.c")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liboracle_rnnt.so``."""
    os.makedirs(_BUILD, exist_ok=True)
    stale = (not os.path.exists(_SO)) or os.path.getmtime(_SO) < max(
        os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "rnnt_oracle.h")))
    if force or stale:
        tmp = _SO + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O3", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _SO)
    return _SO


class _Dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("B", "T", "U1", "HA", "HL", "H", "V", "blank")]


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        lib.oracle_rnnt.restype = ctypes.c_int
        lib.oracle_rnnt.argtypes = [ctypes.POINTER(_Dims)] + [P] * 26 + [ctypes.c_int]
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_num_threads.argtypes = [ctypes.c_int]
        _lib = lib
    return _lib


def num_threads(nthreads: int = 0) -> int:
    return _load().oracle_num_threads(nthreads)


ERRORS = {1: "dims", 2: "length", 3: "label", 4: "alloc"}


@dataclass
class OracleResult:
    loss: np.ndarray           # [B]   -ln P(y_b|x_b)
    lnP_beta: np.ndarray       # [B]   beta(0,0)
    lpb: np.ndarray            # [B,T,U1]
    lpl: np.ndarray
    lnPD: np.ndarray
    alpha: np.ndarray
    beta: np.ndarray
    dh: np.ndarray | None      # [B,T,U1,V] when asked for
    grads: dict | None         # dhA, dhL, dWA, dWL, dbZ, dWO, dbO


def _f64(x):
    return None if x is None else np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _i32(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def rnnt(hA, hL, WA, WL, bZ, WO, bO, labels, T_len, U_len, blank=0, grad_loss=None,
         want_grad=True, want_dh=False, nthreads=0) -> OracleResult:
    """Run the oracle on host arrays (any float dtype; widened to fp64)."""
    hA, hL, WA, WL, WO = map(_f64, (hA, hL, WA, WL, WO))
    bZ, bO, grad_loss = _f64(bZ), _f64(bO), _f64(grad_loss)
    labels, T_len, U_len = _i32(labels), _i32(T_len), _i32(U_len)
    B, T, HA = hA.shape
    U1, HL = hL.shape[1], hL.shape[2]
    H, V = WA.shape[0], WO.shape[0]
    assert hL.shape[0] == B and labels.shape == (B, U1)
    assert WA.shape == (H, HA) and WL.shape == (H, HL) and WO.shape == (V, H)
    d = _Dims(B, T, U1, HA, HL, H, V, blank)
    cells = (B, T, U1)
    loss = np.zeros(B)
    lnPb = np.zeros(B)
    lpb, lpl, lnPD, al, be = (np.zeros(cells) for _ in range(5))
    dh = np.zeros(cells + (V,)) if want_dh else None
    g = None
    if want_grad:
        g = dict(dhA=np.zeros((B, T, HA)), dhL=np.zeros((B, U1, HL)), dWA=np.zeros((H, HA)),
                 dWL=np.zeros((H, HL)), dbZ=np.zeros(H), dWO=np.zeros((V, H)), dbO=np.zeros(V))
    gp = [None] * 7 if g is None else [_ptr(g[k]) for k in ("dhA", "dhL", "dWA", "dWL", "dbZ",
                                                             "dWO", "dbO")]
    st = _load().oracle_rnnt(
        ctypes.byref(d), _ptr(hA), _ptr(hL), _ptr(WA), _ptr(WL), _ptr(bZ), _ptr(WO), _ptr(bO),
        _ptr(labels), _ptr(T_len), _ptr(U_len), _ptr(grad_loss), _ptr(loss), _ptr(lpb),
        _ptr(lpl), _ptr(lnPD), _ptr(al), _ptr(be), _ptr(lnPb), _ptr(dh), *gp, nthreads)
    if st != 0:
        raise ValueError(f"oracle rejected the inputs: {ERRORS.get(st, st)}")
    return OracleResult(loss, lnPb, lpb, lpl, lnPD, al, be, dh, g)
