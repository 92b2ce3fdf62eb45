"""Thin ctypes binding of librnnt_gb300 (include/rnnt.h).

Argument marshalling only: torch tensors are used for device memory and
streams, and their data pointers are handed to the C functions of the same
names.  Every step of the computation runs in the library's CUDA kernels; if
the library is not built this module raises instead of computing anything
another way.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

from . import build as _build

RNNT_OK = 0
STATUS_NAMES = {0: "RNNT_OK", 1: "RNNT_ERR_INVALID_ARG", 2: "RNNT_ERR_UNSUPPORTED_SHAPE",
                3: "RNNT_ERR_WORKSPACE_TOO_SMALL", 4: "RNNT_ERR_LENGTH_RANGE",
                5: "RNNT_ERR_LABEL_RANGE", 6: "RNNT_ERR_TIMEOUT", 7: "RNNT_ERR_CUDA"}
RNNT_F32, RNNT_BF16, RNNT_BF16_E4M3 = 0, 1, 2
# Rnnt(dtype=...) names
DTYPES = {"f32": RNNT_F32, "bf16": RNNT_BF16, "bf16-e4m3": RNNT_BF16_E4M3}
RNNT_TILED, RNNT_UNTILED = 0, 1

# Every function include/rnnt.h and include/rnnt_profile.h declare (the test
# hooks of include/rnnt_testing.h are called by their own tests).
EXPORTS = ("rnnt_saved_bytes", "rnnt_saved_layout", "rnnt_workspace_bytes",
           "rnnt_graph_capturable", "rnnt_tile_cells_for_budget", "rnnt_fwd", "rnnt_bwd",
           "rnnt_bwd_ex", "rnnt_fwd_bwd", "rnnt_fwd_noalloc",
           "rnnt_device_status",
           "rnnt_status_string", "rnnt_profile_start", "rnnt_profile_stop", "rnnt_profile_entry")


class RnntError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS_NAMES.get(code, code)} ({rnnt_status_string(code)})")


class RnntDims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("T", ctypes.c_int), ("U1", ctypes.c_int),
                ("HA", ctypes.c_int), ("HL", ctypes.c_int), ("H", ctypes.c_int),
                ("V", ctypes.c_int), ("blank", ctypes.c_int), ("dtype", ctypes.c_int),
                ("mode", ctypes.c_int), ("tile_cells", ctypes.c_longlong)]


class RnntParams(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("WA", "WL", "bZ", "WO", "bO")]


class RnntBwdOpts(ctypes.Structure):
    _fields_ = [("enc_grad_dtype", ctypes.c_int), ("dA", ctypes.c_void_p),
                ("dL", ctypes.c_void_p)]


class RnntSavedOffsets(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in ("status", "lnP", "lpb", "lpl", "lnPD", "alpha",
                                               "beta", "z", "h", "total")]


_lib = None


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False):
    """Load the shared library (fails loudly if it is not built)."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        if build_if_missing:
            _build.build_library()
        else:
            raise RuntimeError(f"{path} is not built; run asr_tiled_tanh_gb300.build.build_library()")
    lib = ctypes.CDLL(path)
    P, S = ctypes.c_void_p, ctypes.c_size_t
    D = ctypes.POINTER(RnntDims)
    lib.rnnt_saved_bytes.restype = S
    lib.rnnt_saved_bytes.argtypes = [D]
    lib.rnnt_workspace_bytes.restype = S
    lib.rnnt_workspace_bytes.argtypes = [D]
    lib.rnnt_tile_cells_for_budget.restype = ctypes.c_longlong
    lib.rnnt_tile_cells_for_budget.argtypes = [D, S]
    lib.rnnt_graph_capturable.restype = ctypes.c_int
    lib.rnnt_graph_capturable.argtypes = [D]
    lib.rnnt_saved_layout.restype = ctypes.c_int
    lib.rnnt_saved_layout.argtypes = [D, ctypes.POINTER(RnntSavedOffsets)]
    lib.rnnt_fwd.restype = ctypes.c_int
    lib.rnnt_fwd.argtypes = [D, P, P, ctypes.POINTER(RnntParams), P, P, P, P, P, P, S, P]
    lib.rnnt_bwd.restype = ctypes.c_int
    lib.rnnt_bwd.argtypes = [D, P, P, ctypes.POINTER(RnntParams), P, P, P, P, P,
                             P, P, P, P, P, P, P, P, S, P]
    lib.rnnt_bwd_ex.restype = ctypes.c_int
    lib.rnnt_bwd_ex.argtypes = [D, P, P, ctypes.POINTER(RnntParams), P, P, P, P, P,
                                P, P, P, P, P, P, P, P, S, ctypes.POINTER(RnntBwdOpts), P]
    lib.rnnt_fwd_bwd.restype = ctypes.c_int
    lib.rnnt_fwd_bwd.argtypes = [D, P, P, ctypes.POINTER(RnntParams), P, P, P, P, P, P,
                                 P, P, P, P, P, P, P, P, S, P]
    lib.rnnt_fwd_noalloc.restype = ctypes.c_int
    lib.rnnt_fwd_noalloc.argtypes = [D, P, P, ctypes.POINTER(RnntParams), P, P, P, P, P, P]
    lib.rnnt_device_status.restype = ctypes.c_int
    lib.rnnt_device_status.argtypes = [D, P, P, ctypes.POINTER(ctypes.c_int32)]
    lib.rnnt_status_string.restype = ctypes.c_char_p
    lib.rnnt_status_string.argtypes = [ctypes.c_int]
    lib.rnnt_profile_start.restype = ctypes.c_int
    lib.rnnt_profile_start.argtypes = [ctypes.c_int]
    lib.rnnt_profile_stop.restype = ctypes.c_int
    lib.rnnt_profile_stop.argtypes = []
    lib.rnnt_profile_entry.restype = ctypes.c_int
    lib.rnnt_profile_entry.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_char_p),
                                       ctypes.POINTER(ctypes.c_double),
                                       ctypes.POINTER(ctypes.c_int)]
    lib.rnnt_testing_gemm_bf16.restype = ctypes.c_int
    lib.rnnt_testing_gemm_bf16.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, P,
                                           ctypes.c_int, P, ctypes.c_int, P, ctypes.c_int,
                                           ctypes.c_int, ctypes.c_int, P]
    lib.rnnt_testing_quantize_wo.restype = ctypes.c_int
    lib.rnnt_testing_quantize_wo.argtypes = [ctypes.c_int, ctypes.c_int, P, P, P, P, P]
    lib.rnnt_testing_gemm_timeout.restype = ctypes.c_int
    lib.rnnt_testing_gemm_timeout.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P, P,
                                              P, ctypes.c_ulonglong, P]
    _lib = lib
    return lib


def _p(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(code: int, where: str):
    if code != RNNT_OK:
        raise RnntError(code, where)


def make_dims(B, T, U1, HA, HL, H, V, blank=0, dtype=RNNT_BF16, mode=RNNT_TILED,
              tile_cells=0) -> RnntDims:
    return RnntDims(B, T, U1, HA, HL, H, V, blank, dtype, mode, tile_cells)


def make_params(WA, WL, bZ, WO, bO) -> RnntParams:
    return RnntParams(_p(WA), _p(WL), _p(bZ), _p(WO), _p(bO))


# --- the C functions, same names --------------------------------------------

def rnnt_saved_bytes(dims: RnntDims) -> int:
    return int(load().rnnt_saved_bytes(ctypes.byref(dims)))


def rnnt_workspace_bytes(dims: RnntDims) -> int:
    return int(load().rnnt_workspace_bytes(ctypes.byref(dims)))


def rnnt_tile_cells_for_budget(dims, budget_bytes: int) -> int:
    """tile_cells whose saved + workspace footprint fits budget_bytes (0: none)."""
    return int(load().rnnt_tile_cells_for_budget(ctypes.byref(dims), int(budget_bytes)))


def rnnt_graph_capturable(dims: RnntDims) -> int:
    """1 if rnnt_fwd / rnnt_bwd for dims make no host synchronization (they
    can be captured into a CUDA graph), 0 if not, -1 for invalid dims."""
    return int(load().rnnt_graph_capturable(ctypes.byref(dims)))


def rnnt_saved_layout(dims: RnntDims) -> RnntSavedOffsets:
    out = RnntSavedOffsets()
    _check(load().rnnt_saved_layout(ctypes.byref(dims), ctypes.byref(out)), "rnnt_saved_layout")
    return out


def rnnt_status_string(code: int) -> str:
    return load().rnnt_status_string(int(code)).decode()


def rnnt_fwd(dims, hA, hL, params: RnntParams, labels, T_len, U_len, loss, saved, ws,
             stream=None, check=True) -> int:
    code = load().rnnt_fwd(ctypes.byref(dims), _p(hA), _p(hL), ctypes.byref(params), _p(labels),
                           _p(T_len), _p(U_len), _p(loss), _p(saved), _p(ws),
                           ws.numel() * ws.element_size() if ws is not None else 0,
                           _stream(stream))
    if check:
        _check(code, "rnnt_fwd")
    return code


def rnnt_bwd(dims, hA, hL, params: RnntParams, labels, T_len, U_len, grad_loss, saved, dhA, dhL,
             dWA, dWL, dbZ, dWO, dbO, ws, stream=None, check=True) -> int:
    code = load().rnnt_bwd(ctypes.byref(dims), _p(hA), _p(hL), ctypes.byref(params), _p(labels),
                           _p(T_len), _p(U_len), _p(grad_loss), _p(saved), _p(dhA), _p(dhL),
                           _p(dWA), _p(dWL), _p(dbZ), _p(dWO), _p(dbO), _p(ws),
                           ws.numel() * ws.element_size() if ws is not None else 0,
                           _stream(stream))
    if check:
        _check(code, "rnnt_bwd")
    return code


def rnnt_bwd_ex(dims, hA, hL, params: RnntParams, labels, T_len, U_len, grad_loss, saved, dhA,
                dhL, dWA, dWL, dbZ, dWO, dbO, ws, opts: RnntBwdOpts, stream=None,
                check=True) -> int:
    code = load().rnnt_bwd_ex(ctypes.byref(dims), _p(hA), _p(hL), ctypes.byref(params),
                              _p(labels), _p(T_len), _p(U_len), _p(grad_loss), _p(saved),
                              _p(dhA), _p(dhL), _p(dWA), _p(dWL), _p(dbZ), _p(dWO), _p(dbO),
                              _p(ws), ws.numel() * ws.element_size() if ws is not None else 0,
                              ctypes.byref(opts) if opts is not None else None,
                              _stream(stream))
    if check:
        _check(code, "rnnt_bwd_ex")
    return code


def rnnt_fwd_bwd(dims, hA, hL, params: RnntParams, labels, T_len, U_len, loss, grad_loss, saved,
                 dhA, dhL, dWA, dWL, dbZ, dWO, dbO, ws, stream=None, check=True) -> int:
    code = load().rnnt_fwd_bwd(ctypes.byref(dims), _p(hA), _p(hL), ctypes.byref(params),
                               _p(labels), _p(T_len), _p(U_len), _p(loss), _p(grad_loss),
                               _p(saved), _p(dhA), _p(dhL), _p(dWA), _p(dWL), _p(dbZ), _p(dWO),
                               _p(dbO), _p(ws),
                               ws.numel() * ws.element_size() if ws is not None else 0,
                               _stream(stream))
    if check:
        _check(code, "rnnt_fwd_bwd")
    return code


def rnnt_fwd_noalloc(dims, hA, hL, params: RnntParams, labels, T_len, U_len, loss, saved,
                     stream=None, check=True) -> int:
    code = load().rnnt_fwd_noalloc(ctypes.byref(dims), _p(hA), _p(hL), ctypes.byref(params),
                                   _p(labels), _p(T_len), _p(U_len), _p(loss), _p(saved),
                                   _stream(stream))
    if check:
        _check(code, "rnnt_fwd_noalloc")
    return code


def rnnt_device_status(dims, saved, stream=None):
    """(status code, raw status word)."""
    w = ctypes.c_int32(0)
    code = load().rnnt_device_status(ctypes.byref(dims), _p(saved), _stream(stream),
                                     ctypes.byref(w))
    return code, int(w.value)


def rnnt_profile_start(capacity: int = 65536):
    _check(load().rnnt_profile_start(int(capacity)), "rnnt_profile_start")


def rnnt_profile_stop() -> dict:
    """{kernel name: (total ms, timed launches)} of the session just closed."""
    lib = load()
    n = lib.rnnt_profile_stop()
    if n < 0:
        raise RnntError(7, "rnnt_profile_stop")
    out = {}
    for i in range(n):
        name, ms, cnt = ctypes.c_char_p(), ctypes.c_double(), ctypes.c_int()
        _check(lib.rnnt_profile_entry(i, ctypes.byref(name), ctypes.byref(ms), ctypes.byref(cnt)),
               "rnnt_profile_entry")
        out[name.value.decode()] = (ms.value, cnt.value)
    return out


def rnnt_testing_gemm_bf16(A, a_mn, B, b_mn, C, M, N, K, accumulate=0, k_splits=1, bn=256,
                           stream=None):
    """The library's tcgen05 GEMM alone (include/rnnt_testing.h)."""
    _check(load().rnnt_testing_gemm_bf16(M, N, K, _p(A), a_mn, _p(B), b_mn, _p(C), accumulate,
                                         k_splits, bn, _stream(stream)),
           "rnnt_testing_gemm_bf16")


def rnnt_testing_quantize_wo(WO, Q, Wdq, nscale, stream=None):
    """The e4m3 W^O quantization alone (include/rnnt_testing.h)."""
    V, H = WO.shape
    _check(load().rnnt_testing_quantize_wo(V, H, _p(WO), _p(Q), _p(Wdq), _p(nscale),
                                           _stream(stream)),
           "rnnt_testing_quantize_wo")


def rnnt_testing_gemm_timeout(A, B, C, status, M, N, K, wait_ns, stream=None):
    """The GEMM with a stage that is never filled (include/rnnt_testing.h)."""
    _check(load().rnnt_testing_gemm_timeout(M, N, K, _p(A), _p(B), _p(C), _p(status),
                                            int(wait_ns), _stream(stream)),
           "rnnt_testing_gemm_timeout")


# --- convenience: buffers owned by torch -------------------------------------

@dataclass
class SavedArrays:
    lnP: torch.Tensor
    lpb: torch.Tensor
    lpl: torch.Tensor
    lnPD: torch.Tensor
    alpha: torch.Tensor
    beta: torch.Tensor


class Rnnt:
    """Owns the `saved` and `ws` buffers of one problem size (torch allocations)."""

    def __init__(self, B, T, U1, HA, HL, H, V, blank=0, dtype="bf16", mode="tiled",
                 tile_cells=0, device="cuda"):
        self.dims = make_dims(B, T, U1, HA, HL, H, V, blank, DTYPES[dtype],
                              RNNT_UNTILED if mode == "untiled" else RNNT_TILED, tile_cells)
        sb, wb = rnnt_saved_bytes(self.dims), rnnt_workspace_bytes(self.dims)
        if sb == 0 or wb == 0:
            raise RnntError(1, "Rnnt(dims)")
        self.saved = torch.empty(sb, dtype=torch.uint8, device=device)
        self.ws = torch.empty(wb, dtype=torch.uint8, device=device)
        self.layout = rnnt_saved_layout(self.dims)
        self.device = device

    @classmethod
    def for_inputs(cls, inp, mode="tiled", tile_cells=0, device="cuda", e4m3_scores=False):
        """Buffers for a batch of `inp`'s shapes; e4m3_scores: bf16 inputs with
        the score products on e4m3 tensor cores (RNNT_BF16_E4M3)."""
        wl = inp.wl
        dtype = "bf16-e4m3" if e4m3_scores else wl.dtype
        if e4m3_scores and wl.dtype != "bf16":
            raise ValueError("e4m3 scores take bf16 inputs")
        return cls(wl.B, wl.T, wl.U1, wl.HA, wl.HL, wl.H, wl.V, 0, dtype, mode, tile_cells,
                   device)

    def fwd(self, hA, hL, params, labels, T_len, U_len, loss=None, stream=None):
        if loss is None:
            loss = torch.empty(self.dims.B, dtype=torch.float32, device=self.device)
        rnnt_fwd(self.dims, hA, hL, params, labels, T_len, U_len, loss, self.saved, self.ws,
                 stream)
        return loss

    def alloc_grads(self):
        d, f = self.dims, dict(dtype=torch.float32, device=self.device)
        return dict(dhA=torch.empty(d.B, d.T, d.HA, **f), dhL=torch.empty(d.B, d.U1, d.HL, **f),
                    dWA=torch.empty(d.H, d.HA, **f), dWL=torch.empty(d.H, d.HL, **f),
                    dbZ=torch.empty(d.H, **f), dWO=torch.empty(d.V, d.H, **f),
                    dbO=torch.empty(d.V, **f))

    def bwd(self, hA, hL, params, labels, T_len, U_len, grad_loss=None, grads=None, stream=None):
        g = grads if grads is not None else self.alloc_grads()
        rnnt_bwd(self.dims, hA, hL, params, labels, T_len, U_len, grad_loss, self.saved,
                 g["dhA"], g["dhL"], g["dWA"], g["dWL"], g["dbZ"], g["dWO"], g["dbO"], self.ws,
                 stream)
        return g

    def bwd_ex(self, hA, hL, params, labels, T_len, U_len, grad_loss=None, enc_dtype="f32",
               handoff=False, skip_enc=False, stream=None):
        """rnnt_bwd_ex: dhA/dhL (and, with handoff, the projections' gradients
        dA [B,T,H], dL [B,U1,H]) in enc_dtype ("f32" or "bf16"); skip_enc
        leaves dhA/dhL out (NULL)."""
        d = self.dims
        et = torch.bfloat16 if enc_dtype == "bf16" else torch.float32
        g = self.alloc_grads()
        g["dhA"] = None if skip_enc else torch.empty(d.B, d.T, d.HA, dtype=et, device=self.device)
        g["dhL"] = None if skip_enc else torch.empty(d.B, d.U1, d.HL, dtype=et, device=self.device)
        opts = RnntBwdOpts(RNNT_BF16 if enc_dtype == "bf16" else RNNT_F32, None, None)
        if handoff:
            g["dA"] = torch.empty(d.B, d.T, d.H, dtype=et, device=self.device)
            g["dL"] = torch.empty(d.B, d.U1, d.H, dtype=et, device=self.device)
            opts.dA, opts.dL = g["dA"].data_ptr(), g["dL"].data_ptr()
        gl = None if grad_loss is None else torch.as_tensor(grad_loss, dtype=torch.float32,
                                                             device=self.device)
        rnnt_bwd_ex(d, hA, hL, params, labels, T_len, U_len, gl, self.saved, g["dhA"], g["dhL"],
                    g["dWA"], g["dWL"], g["dbZ"], g["dWO"], g["dbO"], self.ws, opts, stream)
        return g

    def fwd_bwd(self, hA, hL, params, labels, T_len, U_len, loss=None, grad_loss=None,
                grads=None, stream=None):
        """One training step (rnnt_fwd_bwd): returns (loss, grads)."""
        if loss is None:
            loss = torch.empty(self.dims.B, dtype=torch.float32, device=self.device)
        g = grads if grads is not None else self.alloc_grads()
        rnnt_fwd_bwd(self.dims, hA, hL, params, labels, T_len, U_len, loss, grad_loss,
                     self.saved, g["dhA"], g["dhL"], g["dWA"], g["dWL"], g["dbZ"], g["dWO"],
                     g["dbO"], self.ws, stream)
        return loss, g

    def saved_arrays(self) -> SavedArrays:
        d, L = self.dims, self.layout
        n = d.B * d.T * d.U1

        def view(off, count, shape):
            return self.saved[off:off + 4 * count].view(torch.float32).view(*shape)

        cells = (d.B, d.T, d.U1)
        return SavedArrays(view(L.lnP, d.B, (d.B,)), view(L.lpb, n, cells), view(L.lpl, n, cells),
                           view(L.lnPD, n, cells), view(L.alpha, n, cells),
                           view(L.beta, n, cells))

    def status(self, stream=None):
        return rnnt_device_status(self.dims, self.saved, stream)
