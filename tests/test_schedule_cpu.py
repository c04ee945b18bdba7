"""The fused attention kernel's work schedule, computed on the host by
bsp_diag_attention_schedule (the same routine the launcher uploads): every
(tile, batch entry) item assigned exactly once, each CTA's items in
longest-first order with the tile's own step range, and the per-CTA work
within the greedy bound of the optimum."""

import numpy as np
import pytest

from sparse_attention_layout_gb300 import bsp
from sparse_attention_layout_gb300 import workloads as W


def _check(L, Z, grid):
    tab = L.tiles()
    nt = tab["n_tiles"]
    ptr, items = bsp.bsp_diag_attention_schedule(L, Z, grid)
    assert ptr[0] == 0 and ptr[-1] == Z * nt
    assert np.all(np.diff(ptr) >= 0)
    # every (tile, batch entry) exactly once, with the tile's own steps
    seen = np.zeros((nt, Z), np.int32)
    sp = tab["tile_step_ptr"]
    for t, s0, ns, z in items:
        seen[t, z] += 1
        assert s0 == sp[t] and ns == sp[t + 1] - sp[t]
    assert np.all(seen == 1)
    # each CTA's items longest-first; the work per CTA (steps + 1 per item)
    # within the longest-processing-time-first bound: no CTA exceeds the mean
    # by more than one item's weight
    weights = items[:, 2].astype(np.int64) + 1
    loads = np.array([weights[ptr[c]:ptr[c + 1]].sum() for c in range(grid)])
    for c in range(grid):
        w = weights[ptr[c]:ptr[c + 1]]
        assert np.all(np.diff(w) <= 0)
    if Z * nt:
        assert loads.max() <= weights.sum() / grid + weights.max()
        # no CTA idle while there are at least as many items as CTAs
        if Z * nt >= grid:
            assert np.all(np.diff(ptr) > 0)
    return loads


@pytest.mark.parametrize("name", ["bigbird", "band", "strided", "tiny"])
def test_schedule_of_the_workloads(name):
    w = W.ATTENTION_WORKLOADS[name]
    L = bsp.bsp_layout_plan(w.layout(), w.B)
    nt = L.tiles()["n_tiles"]
    grid = min(w.Z * nt, 152)
    loads = _check(L, w.Z, grid)
    if name == "bigbird":
        # the global-row tiles are ~10x the others: greedy placement keeps the
        # busiest CTA close to the mean (round-robin over the longest-first
        # order gave one CTA a long tile plus a full share of short ones)
        assert loads.max() <= 1.1 * loads.mean() + 1


@pytest.mark.parametrize("seed", range(8))
def test_schedule_random_layouts(seed):
    rng = np.random.default_rng(900 + seed)
    B = int(rng.choice([16, 32, 64, 128]))
    nb = int(rng.integers(1, 40))
    H = int(rng.integers(1, 4))
    lay = (rng.random((H, nb, nb)) < rng.uniform(0.0, 0.6)).astype(np.uint8)
    L = bsp.bsp_layout_plan(lay, B)
    nt = L.tiles()["n_tiles"]
    for Z in (1, 3):
        for grid in sorted({1, 5, max(1, Z * nt), 152}):
            _check(L, Z, grid)


def test_schedule_rejects_bad_arguments():
    L = bsp.bsp_layout_plan(np.ones((1, 2, 2), np.uint8), 64)
    for Z, grid in ((0, 4), (2, 0), (-1, 1)):
        with pytest.raises(bsp.BspError) as e:
            bsp.bsp_diag_attention_schedule(L, Z, grid)
        assert e.value.code == -1
