"""Host-side checks of the C ABI (no GPU needed): the library loads and
exports every symbol of include/bsp.h, the layout compiler's tables are
bit-exact with the oracle's, the tensor-core work lists cover every block
exactly once, and argument errors return the documented codes without
touching a device."""

import ctypes
import os
import re

import numpy as np
import pytest

from sparse_attention_layout_gb300 import bsp, build, workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return bsp.lib()


def header_symbols():
    text = open(os.path.join(ROOT, "include", "bsp.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bsp_[a-z_]+)\s*\(", text)))


def test_header_symbols_exported(lib):
    syms = header_symbols()
    assert "bsp_attention" in syms and "bsp_layout_compile" in syms and len(syms) >= 14
    for s in syms:
        assert hasattr(lib, s), f"libbsp.so does not export {s}"


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5, -6, -7):
        assert lib.bsp_status_string(code)
    assert b"sm_103a" in lib.bsp_version()


def _layouts():
    out = {}
    for name, w in W.ATTENTION_WORKLOADS.items():
        out[name] = (w.layout(), w.B)
    for d in W.SPMM_DENSITIES:
        out[f"spmm{int(d * 100)}"] = (W.SPMM.layout(d), W.SPMM.B)
    rng = np.random.default_rng(7)
    out["all_zero"] = (np.zeros((2, 8, 8), np.uint8), 16)
    out["single"] = (np.pad(np.ones((1, 1, 1), np.uint8), ((0, 0), (3, 4), (2, 5))), 32)
    out["all_ones"] = (np.ones((3, 5, 5), np.uint8), 64)
    lay = (rng.random((2, 9, 9)) < 0.3).astype(np.uint8)
    lay[0, 4, :] = 0
    lay[1, :, 6] = 0
    out["empty_rows_cols"] = (lay, 128)
    return out


LAYOUTS = _layouts()


@pytest.mark.parametrize("name", sorted(LAYOUTS))
def test_luts_bit_exact_with_oracle(lib, oracle, name):
    lay, B = LAYOUTS[name]
    L = bsp.bsp_layout_plan(lay, B)
    got = L.luts()
    want = oracle.luts(lay)
    assert L.nnz == oracle.nnz(lay)
    for k in want:
        assert got[k].dtype == np.int32
        assert np.array_equal(got[k], want[k]), k


@pytest.mark.parametrize("name", sorted(LAYOUTS))
def test_tiles_cover_every_block_once(lib, name):
    lay, B = LAYOUTS[name]
    L = bsp.bsp_layout_plan(lay, B)
    T = L.tiles()
    H, nb = lay.shape[0], lay.shape[1]
    G = T["G"]
    assert G == 128 // B
    ngroups = -(-nb // G)
    assert T["n_tiles"] == H * ngroups
    ids = -np.ones(lay.shape, np.int64)
    hs, is_, js = np.nonzero(lay)
    ids[hs, is_, js] = np.arange(hs.size)
    seen = np.zeros(hs.size, np.int64)
    ptr = T["tile_step_ptr"]
    for t in range(T["n_tiles"]):
        h, g = divmod(t, ngroups)
        rows = [g * G + a for a in range(G)]
        union = sorted({j for i in rows if i < nb for j in np.flatnonzero(lay[h, i])})
        steps = range(ptr[t], ptr[t + 1])
        assert len(steps) == -(-len(union) // G)
        cols = [c for s in steps for c in T["step_col"][s]]
        assert cols[:len(union)] == union and all(c == -1 for c in cols[len(union):])
        for s in steps:
            for a in range(G):
                for b in range(G):
                    c, i = T["step_col"][s][b], g * G + a
                    want = ids[h, i, c] if (c >= 0 and i < nb) else -1
                    assert T["step_blk"][s][a][b] == want
                    if want >= 0:
                        seen[want] += 1
    assert np.all(seen == 1)
    steps_per_tile = np.diff(ptr)
    order = T["tile_order"]
    assert sorted(order.tolist()) == list(range(T["n_tiles"]))
    assert np.all(np.diff(steps_per_tile[order]) <= 0)


@pytest.mark.parametrize("orient", [0, 1])
@pytest.mark.parametrize("name", sorted(LAYOUTS))
def test_groups_cover_every_block_once(lib, name, orient):
    """The DSD / DDS line groups: per group the ascending union of its lines'
    block indices, the id of every present (line, index) block, each block
    exactly once, groups ordered by size."""
    lay, B = LAYOUTS[name]
    L = bsp.bsp_layout_plan(lay, B)
    T = L.groups(orient)
    H, nb = lay.shape[0], lay.shape[1]
    G = T["G"]
    ngroups = -(-nb // G)
    assert T["n_groups"] == H * ngroups
    ids = -np.ones(lay.shape, np.int64)
    hs, is_, js = np.nonzero(lay)
    ids[hs, is_, js] = np.arange(hs.size)
    lines = lay if orient == 0 else lay.transpose(0, 2, 1)   # [h, line, index]
    lids = ids if orient == 0 else ids.transpose(0, 2, 1)
    seen = np.zeros(hs.size, np.int64)
    ptr = T["grp_ptr"]
    for t in range(T["n_groups"]):
        h, g = divmod(t, ngroups)
        members = [g * G + a for a in range(G) if g * G + a < nb]
        union = sorted({u for m in members for u in np.flatnonzero(lines[h, m])})
        slots = range(ptr[t], ptr[t + 1])
        assert [T["slot_idx"][s] for s in slots] == union
        for s in slots:
            u = T["slot_idx"][s]
            for a in range(G):
                m = g * G + a
                want = lids[h, m, u] if m < nb else -1
                assert T["slot_blk"][s][a] == want
                if want >= 0:
                    seen[want] += 1
    assert np.all(seen == 1)
    order = T["grp_order"]
    assert sorted(order.tolist()) == list(range(T["n_groups"]))
    assert np.all(np.diff(np.diff(ptr)[order]) <= 0)


def test_groups_reject_bad_orient(lib):
    L = bsp.bsp_layout_plan(np.ones((1, 2, 2), np.uint8), 64)
    assert lib.bsp_layout_groups(L.handle, 2, None, None, None, None, None, None, None) == -1


def test_plan_rejects_bad_arguments(lib):
    h = ctypes.c_void_p()
    lay = np.ones((1, 4, 4), np.uint8)
    p = ctypes.c_void_p(lay.ctypes.data)
    assert lib.bsp_layout_plan(p, 1, 4, 48, ctypes.byref(h)) == -1       # block size
    assert lib.bsp_layout_plan(p, 0, 4, 16, ctypes.byref(h)) == -1       # H
    assert lib.bsp_layout_plan(p, 1, 0, 16, ctypes.byref(h)) == -1       # nb
    assert lib.bsp_layout_plan(None, 1, 4, 16, ctypes.byref(h)) == -1    # NULL layout
    bad = lay.copy()
    bad[0, 1, 2] = 2
    assert lib.bsp_layout_plan(ctypes.c_void_p(bad.ctypes.data), 1, 4, 16, ctypes.byref(h)) == -1
    assert h.value is None


def test_compute_calls_reject_host_only_handle(lib):
    L = bsp.bsp_layout_plan(np.ones((1, 2, 2), np.uint8), 16)
    buf = (ctypes.c_char * 4096)()
    a = ctypes.c_void_p(ctypes.addressof(buf) + (-ctypes.addressof(buf)) % 16)
    assert lib.bsp_sdd(L.handle, 1, a, a, a, 1, 16, 0, 1, None) == -1
    assert lib.bsp_dsd(L.handle, 1, a, a, a, 1, 16, 0, 0, None) == -1
    assert lib.bsp_dds(L.handle, 1, a, a, a, 1, 16, 0, 0, None) == -1
    assert lib.bsp_softmax(L.handle, 1, a, a, 1, ctypes.c_float(1.0), 0, None, None) == -1
    assert lib.bsp_attention(L.handle, 1, a, a, a, a, 1, 64, ctypes.c_float(1.0), 0, None, None) == -1
    assert lib.bsp_status_check(L.handle, None) == -1
    assert lib.bsp_sdd(None, 1, a, a, a, 1, 16, 0, 1, None) == -1
    assert lib.bsp_layout_destroy(None) == 0


def test_info_reports_sizes(lib):
    lay = W.layout_band(10, 2, H=3)
    L = bsp.bsp_layout_plan(lay, 32)
    assert (L.H, L.nb, L.B, L.nnz, L.S) == (3, 10, 32, int(lay.sum()), 320)
