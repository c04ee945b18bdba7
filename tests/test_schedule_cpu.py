"""The fused attention kernel's work schedule, computed on the host by
bsp_diag_attention_schedule (the routine the launcher uploads): every
(tile, batch entry) covered exactly once -- whole, or cut into pieces whose
step ranges partition the tile's -- each CTA's items longest-first, the
per-CTA work within the greedy bound, and long tiles cut only when that
shortens the makespan."""

import ctypes

import numpy as np
import pytest
import torch

from sparse_attention_layout_gb300 import bsp
from sparse_attention_layout_gb300 import workloads as W

N_SM = 152
F32_MAX_STEPS = 32
DT = {"f32": torch.float32, "bf16": torch.bfloat16}


def _check(L, Z, n_sm, dtype=torch.bfloat16):
    tab = L.tiles()
    nt = tab["n_tiles"]
    sc = bsp.bsp_diag_attention_schedule(L, Z, n_sm, dtype)
    grid, ptr, items, part, comb = sc["grid"], sc["ptr"], sc["items"], sc["part"], sc["combine"]
    n = len(items)
    assert grid == min(n, n_sm)
    assert ptr[0] == 0 and ptr[-1] == n and np.all(np.diff(ptr) >= 0)
    sp = tab["tile_step_ptr"]
    # the cut tiles: consecutive slots, pieces partitioning the tile's steps in slot order
    cut = {}
    slots = []
    for t, z, s0, npc in comb:
        assert npc >= 2 and (t, z) not in cut
        cut[(t, z)] = (s0, npc)
        slots.extend(range(s0, s0 + npc))
    assert sorted(slots) == list(range(len(slots)))
    by_slot = {}
    seen = np.zeros((nt, Z), np.int32)
    for (t, s0, ns, z), p in zip(items, part):
        if p < 0:
            assert (t, z) not in cut
            assert s0 == sp[t] and ns == sp[t + 1] - sp[t]
            seen[t, z] += 1
        else:
            assert p not in by_slot
            by_slot[p] = (t, z, s0, ns)
    for (t, z), (first, npc) in cut.items():
        s = sp[t]
        for k in range(npc):
            tt, zz, s0, ns = by_slot[first + k]
            assert (tt, zz) == (t, z) and s0 == s and ns >= 1
            s += ns
        assert s == sp[t + 1]
        seen[t, z] += 1
    assert len(by_slot) == len(slots)
    assert np.all(seen == 1)
    if dtype == torch.float32:  # fp32 accumulations span at most 32 steps
        assert np.all(items[:, 2] <= F32_MAX_STEPS)
    # each CTA's items longest-first; no CTA idle; greedy bound
    weights = items[:, 2].astype(np.int64) + 1
    loads = np.array([weights[ptr[c]:ptr[c + 1]].sum() for c in range(grid)])
    for c in range(grid):
        assert np.all(np.diff(weights[ptr[c]:ptr[c + 1]]) <= 0)
    if n:
        assert np.all(np.diff(ptr) > 0)
        assert loads.max() <= weights.sum() / grid + weights.max()
    return sc, loads


@pytest.mark.parametrize("name", ["bigbird", "band", "strided", "tiny"])
def test_schedule_of_the_workloads(name):
    w = W.ATTENTION_WORKLOADS[name]
    L = bsp.bsp_layout_plan(w.layout(), w.B)
    sc, loads = _check(L, w.Z, N_SM, DT[w.dtype])
    # whole tiles already balance these (cutting would not gain enough), and
    # BigBird's fp32 global-row tiles (32 steps) stay within the fp32 limit
    assert len(sc["combine"]) == 0
    if name == "bigbird":
        # the global-row tiles are ~10x the others: greedy placement keeps the
        # busiest CTA close to the mean (round-robin over the longest-first
        # order gave one CTA a long tile plus a full share of short ones)
        assert loads.max() <= 1.1 * loads.mean() + 1


def test_short_cuts_are_not_taken():
    # BigBird over S = 4096 with one batch entry: cutting the 32-step
    # global-row tiles would shorten the greedy makespan from 33 to 22 steps,
    # less than the 24 steps the combine pass must save (measured: 10 % slower)
    lay = W.layout_bigbird(64, 12, window=3, n_global=2, n_random=3, seed=2)
    L = bsp.bsp_layout_plan(lay, 64)
    sc, _ = _check(L, 1, N_SM)
    assert len(sc["combine"]) == 0


def test_long_global_rows_are_cut():
    # BigBird over S = 16384: a global-row tile has 128 steps against a fair
    # share of ~80, so whole tiles cannot balance; the automatic setting cuts
    lay = W.layout_bigbird(256, 12, window=3, n_global=2, n_random=3, seed=2)
    L = bsp.bsp_layout_plan(lay, 64)
    bsp.bsp_diag_attention_split(L, -1)
    _, whole = _check(L, 1, N_SM)
    bsp.bsp_diag_attention_split(L, 0)
    sc, loads = _check(L, 1, N_SM)
    assert len(sc["combine"]) == 12  # one global-row tile per head
    # fp32 cuts them into pieces of at most 32 steps with any setting
    for split in (0, -1, 40):
        bsp.bsp_diag_attention_split(L, split)
        sc32, _ = _check(L, 1, N_SM, torch.float32)
        assert len(sc32["combine"]) == 12 and np.all(sc32["combine"][:, 3] >= 4)
    bsp.bsp_diag_attention_split(L, 0)
    assert loads.max() * 10 < whole.max() * 9
    assert loads.max() <= 1.1 * loads.mean() + 4


@pytest.mark.parametrize("seed", range(8))
@pytest.mark.parametrize("split", [0, -1, 1, 3])
def test_schedule_random_layouts(seed, split):
    rng = np.random.default_rng(900 + seed)
    B = int(rng.choice([16, 32, 64, 128]))
    nb = int(rng.integers(1, 40))
    H = int(rng.integers(1, 4))
    lay = (rng.random((H, nb, nb)) < rng.uniform(0.0, 0.6)).astype(np.uint8)
    if seed % 2:
        lay[0, 0, :] = 1  # one long block-row
    L = bsp.bsp_layout_plan(lay, B)
    bsp.bsp_diag_attention_split(L, split)
    nt = L.tiles()["n_tiles"]
    for Z in (1, 3):
        for n_sm in sorted({1, 5, max(1, Z * nt), N_SM}):
            _check(L, Z, n_sm, torch.float32)
            sc, _ = _check(L, Z, n_sm)
            if split > 0:
                assert np.all(sc["items"][sc["part"] >= 0, 2] <= split)
                longest = max((L.tiles()["tile_step_ptr"][1:] - L.tiles()["tile_step_ptr"][:-1]).max(), 0)
                assert (len(sc["combine"]) > 0) == (longest > split)
            if split < 0:
                assert len(sc["combine"]) == 0


def test_schedule_rejects_bad_arguments():
    L = bsp.bsp_layout_plan(np.ones((1, 2, 2), np.uint8), 64)
    for Z, n_sm in ((0, 4), (2, 0), (-1, 1)):
        with pytest.raises(bsp.BspError) as e:
            bsp.bsp_diag_attention_schedule(L, Z, n_sm)
        assert e.value.code == -1
    n = ctypes.c_int()
    assert bsp.lib().bsp_diag_attention_schedule(L.handle, 7, 1, 4, ctypes.byref(n), ctypes.byref(n),
                                                  ctypes.byref(n), None, None, None, None) == -1
    assert bsp.lib().bsp_diag_attention_split(None, 0) == -1
