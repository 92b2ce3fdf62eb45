"""Memory-bounded scheduling (rnnt_tile_cells_for_budget) on the host (CPU).

The library allocates nothing: its device footprint is rnnt_saved_bytes +
rnnt_workspace_bytes.  The budget function must return the largest tile size
whose footprint fits, and one tile more must not fit.
"""
import pytest

import asr_tiled_tanh_gb300 as rn

AUDIO40 = dict(B=1024, T=1000, U1=101, HA=512, HL=512, H=512, V=4096, blank=0)


def _dims(tile_cells=0, dtype=rn.RNNT_BF16, mode=rn.RNNT_TILED, **kw):
    d = dict(AUDIO40)
    d.update(kw)
    return rn.make_dims(**d, dtype=dtype, mode=mode, tile_cells=tile_cells)


def _footprint(tc, **kw):
    d = _dims(tc, **kw)
    return rn.rnnt_saved_bytes(d) + rn.rnnt_workspace_bytes(d)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    rn.load(build_if_missing=True)


@pytest.mark.parametrize("budget_gb", [12.8, 13.0, 14.0, 20.0])
@pytest.mark.parametrize("dtype", [rn.RNNT_BF16, rn.RNNT_BF16_E4M3])
def test_budget_gives_the_largest_fitting_tile(budget_gb, dtype):
    budget = int(budget_gb * 1e9)
    tc = rn.rnnt_tile_cells_for_budget(_dims(dtype=dtype), budget)
    assert tc > 0 and tc % 128 == 0
    assert _footprint(tc, dtype=dtype) <= budget
    # (no device here, so no rounding to whole waves: one tile more does not fit)
    assert _footprint(tc + 128, dtype=dtype) > budget


def test_budget_edges():
    # below the fixed part (saved state and per-frame vectors): nothing fits
    assert rn.rnnt_tile_cells_for_budget(_dims(), 10 ** 9) == 0
    # enough for the whole lattice: one chunk, capped at every possible tile
    small = _dims(B=4, T=50, U1=11, HA=64, HL=64, H=64, V=128)
    tc = rn.rnnt_tile_cells_for_budget(small, 1 << 40)
    assert tc == 4 * 2 * 3 * 128        # B * ceil(T/32) * ceil(U1/4) tiles of 32 x 4 tiles
    assert rn.rnnt_graph_capturable(rn.make_dims(4, 50, 11, 64, 64, 64, 128, 0, rn.RNNT_BF16,
                                                 rn.RNNT_TILED, tc)) == 1
    # untiled plans and invalid dims have no tile size
    assert rn.rnnt_tile_cells_for_budget(_dims(mode=rn.RNNT_UNTILED), 1 << 50) == 0
    assert rn.rnnt_tile_cells_for_budget(_dims(V=0), 1 << 40) == 0
