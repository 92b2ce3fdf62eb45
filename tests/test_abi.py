"""The C-ABI library loads and exports what include/*.h declares (CPU only)."""
import ctypes
import glob
import os
import re

import pytest

import asr_tiled_tanh_gb300 as rn
from asr_tiled_tanh_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build_library()
    return rn.load()


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        for m in re.finditer(r"\b(rnnt_[a-z0-9_]+)\s*\(", src):
            names.add(m.group(1))
    return names


def test_every_declared_symbol_is_exported(lib):
    declared = _declared_functions()
    assert declared, "no declarations found"
    assert set(rn.EXPORTS) <= declared
    for name in declared:
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_strings(lib):
    for code in range(8):
        assert rn.rnnt_status_string(code)
    assert rn.rnnt_status_string(99) == "unknown status"


@pytest.mark.parametrize("bad", [dict(B=-1), dict(T=0), dict(U1=0), dict(H=0), dict(V=0),
                                 dict(blank=32), dict(blank=-1), dict(dtype=7), dict(mode=3),
                                 dict(tile_cells=-5)])
def test_invalid_dims_give_zero_sizes(lib, bad):
    kw = dict(B=2, T=32, U1=9, HA=64, HL=64, H=64, V=32, blank=0, dtype=rn.RNNT_F32,
              mode=rn.RNNT_TILED, tile_cells=0)
    kw.update(bad)
    d = rn.make_dims(**kw)
    assert rn.rnnt_saved_bytes(d) == 0
    assert rn.rnnt_workspace_bytes(d) == 0
    with pytest.raises(rn.RnntError):
        rn.rnnt_saved_layout(d)


def test_saved_layout_is_aligned_and_sized(lib):
    for mode in (rn.RNNT_TILED, rn.RNNT_UNTILED):
        d = rn.make_dims(3, 37, 12, 24, 40, 48, 37, 0, rn.RNNT_F32, mode)
        L = rn.rnnt_saved_layout(d)
        n = 3 * 37 * 12
        offs = [L.status, L.lnP, L.lpb, L.lpl, L.lnPD, L.alpha, L.beta]
        assert all(o % 256 == 0 for o in offs)
        assert sorted(offs) == offs
        assert L.beta + 4 * n <= L.total == rn.rnnt_saved_bytes(d)
        if mode == rn.RNNT_UNTILED:
            assert L.z > L.beta and L.h > L.z
        else:
            assert L.z == 0 and L.h == 0


def test_tile_buffer_tracks_tile_cells(lib):
    # the tile workspace grows with tile_cells and not with the lattice size
    big = dict(B=1024, T=1000, U1=101, HA=512, HL=512, H=512, V=4096, blank=0,
               dtype=rn.RNNT_BF16, mode=rn.RNNT_TILED)
    w1 = rn.rnnt_workspace_bytes(rn.make_dims(**big, tile_cells=128 * 152))
    w2 = rn.rnnt_workspace_bytes(rn.make_dims(**big, tile_cells=128 * 304))
    assert w2 > w1
    per_cell_elems = 512 + 4096
    assert w2 - w1 <= 128 * 152 * per_cell_elems * 8 + 4096
    nominal_scores = 1024 * 1000 * 101 * 4096 * 2
    assert w2 < nominal_scores / 50


def test_untiled_saved_grows_with_lattice(lib):
    small = rn.make_dims(8, 200, 51, 512, 512, 512, 1024, 0, rn.RNNT_BF16, rn.RNNT_UNTILED)
    tiled = rn.make_dims(8, 200, 51, 512, 512, 512, 1024, 0, rn.RNNT_BF16, rn.RNNT_TILED)
    assert rn.rnnt_saved_bytes(small) > 8 * 200 * 51 * 1024 * 2
    # tiled: 20 B per position + the fp32 joint projections, nothing per vocabulary entry
    assert rn.rnnt_saved_bytes(tiled) < 8 * 200 * 51 * 24 + 4 * (8 * 200 + 8 * 51) * 512 + 65536


def test_graph_capturable_follows_the_chunking(lib):
    kw = dict(B=8, T=200, U1=51, HA=512, HL=512, H=512, V=1024, blank=0, dtype=rn.RNNT_BF16)
    assert rn.rnnt_graph_capturable(rn.make_dims(**kw, mode=rn.RNNT_TILED)) == 1
    assert rn.rnnt_graph_capturable(rn.make_dims(**kw, mode=rn.RNNT_UNTILED)) == 1
    # one tile per chunk: the calls read the tile count back, no capture
    assert rn.rnnt_graph_capturable(rn.make_dims(**kw, mode=rn.RNNT_TILED, tile_cells=128)) == 0
    assert rn.rnnt_graph_capturable(rn.make_dims(**dict(kw, T=0), mode=rn.RNNT_TILED)) == -1


def _declared_arity():
    """Parameter count of every rnnt_* prototype in include/*.h."""
    out = {}
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        for m in re.finditer(r"\b(rnnt_[a-z0-9_]+)\s*\(([^()]*)\)\s*;", src):
            params = m.group(2).strip()
            out[m.group(1)] = 0 if params in ("", "void") else params.count(",") + 1
    return out


def test_binding_argument_counts_match_the_headers(lib):
    # a ctypes prototype with the wrong number of arguments would pass garbage
    # to the library (or fail only on a GPU machine): every function the binding
    # declares must take exactly the header's parameters
    arity = _declared_arity()
    assert "rnnt_fwd" in arity and arity["rnnt_fwd"] == 12
    checked = 0
    for name, n in arity.items():
        fn = getattr(lib, name)
        if fn.argtypes is None:
            continue
        assert len(fn.argtypes) == n, (name, len(fn.argtypes), n)
        checked += 1
    assert checked >= len(rn.EXPORTS) - 3


def test_bf16_operands_must_be_16_byte_aligned(lib):
    # The tensor-core path reads hA, hL and the parameters by TMA and 16-byte
    # vector loads: a pointer that is bf16- but not 16-byte aligned is refused
    # on the host, before the driver is touched.  The addresses are fake and
    # never dereferenced.
    d = rn.make_dims(2, 32, 9, 64, 64, 64, 64, 0, rn.RNNT_BF16, rn.RNNT_TILED, 0)
    nws = rn.rnnt_workspace_bytes(d)
    assert nws > 0
    base = {"hA": 0x10000, "hL": 0x20000, "WA": 0x30000, "WL": 0x40000, "bZ": 0x50000,
            "WO": 0x60000, "bO": 0x70000}
    for name in base:
        a = dict(base)
        a[name] += 2
        params = rn.RnntParams(a["WA"], a["WL"], a["bZ"], a["WO"], a["bO"])
        code = lib.rnnt_fwd(ctypes.byref(d), a["hA"], a["hL"], ctypes.byref(params), 0x80000,
                            0x90000, 0xA0000, 0xB0000, 0x100000, 0x200000, nws, None)
        assert code == 1, name  # RNNT_ERR_INVALID_ARG
