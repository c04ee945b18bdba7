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


def _chunk_layouts():
    out = dict(LAYOUTS)
    lay = np.eye(1100, dtype=np.uint8)[None].copy()
    lay[0, 550, :] = 1  # one row of 1100 blocks of 16: 35 KB in bf16, 70 KB in fp32
    out["one_long_row"] = (lay, 16)
    return out


CHUNK_LAYOUTS = _chunk_layouts()


@pytest.mark.parametrize("elt", [2, 4])
@pytest.mark.parametrize("name", sorted(CHUNK_LAYOUTS))
def test_softmax_chunks_cover_every_row_once(lib, name, elt):
    """The softmax chunk list: every row of every non-empty block-row exactly
    once, block-rows in memory order; R a power of two, the largest within the
    documented budget (twice the longest row's bytes, 24 KB to 64 KB); the first
    block id is the block-row's first row-major position; the list is marked
    unusable exactly when a row alone exceeds the budget."""
    lay, B = CHUNK_LAYOUTS[name]
    L = bsp.bsp_layout_plan(lay, B)
    C = L.softmax_chunks(elt)
    H, nb = lay.shape[0], lay.shape[1]
    row_len = (lay.reshape(H * nb, nb) != 0).sum(axis=1)
    first = np.concatenate([[0], np.cumsum(row_len)[:-1]])
    budget = min(64 * 1024, max(24 * 1024, 2 * int(row_len.max()) * B * elt))
    items = C["items"]
    keys = items[:, 0]
    assert np.all(np.diff(keys) >= 0)
    covered = {}
    for key, p0, n, w in items.tolist():
        r0, R = w & 0xFFFF, w >> 16
        assert p0 == first[key] and n == row_len[key] and n > 0
        assert R >= 1 and R & (R - 1) == 0 and r0 % R == 0 and r0 + R <= B
        if C["fits"]:
            assert R * n * B * elt <= budget
            assert R == B or 2 * R * n * B * elt > budget  # the largest such power of two
        covered.setdefault(key, []).extend(range(r0, r0 + R))
    assert sorted(covered) == [k for k in range(H * nb) if row_len[k] > 0]
    for key, rows in covered.items():
        assert sorted(rows) == list(range(B)), f"block-row {key}: rows {rows}"
    assert C["fits"] == bool(int(row_len.max()) * B * elt <= budget)
    if len(items):
        assert C["max_bytes"] == max((w >> 16) * n * B * elt for _, _, n, w in items.tolist())


@pytest.mark.parametrize("n_long,budget,fits", [(96, 24 * 1024, True), (97, 2 * 97 * 128, True),
                                                (256, 64 * 1024, True), (257, 64 * 1024, True),
                                                (513, 64 * 1024, False)])
def test_softmax_chunk_budget_boundaries(lib, n_long, budget, fits):
    """Budget = twice the longest row (blocks of 64, bf16: 128 bytes a block),
    24 KB at least and 64 KB at most; a 96-block row (12 KB) sits on the lower
    bound, a 513-block row (65.7 KB) no longer fits a chunk."""
    nb = max(n_long, 4)
    lay = np.eye(nb, dtype=np.uint8)[None].copy()
    lay[0, 1, :n_long] = 1
    L = bsp.bsp_layout_plan(lay, 64)
    C = L.softmax_chunks(2)
    assert C["fits"] == fits
    items = C["items"]
    long_rows = items[items[:, 0] == 1]
    R = int(long_rows[0, 3]) >> 16
    row_bytes = n_long * 64 * 2
    if fits:
        assert R * row_bytes <= budget and (R == 64 or 2 * R * row_bytes > budget)
    short = items[items[:, 0] == 0]
    assert int(short[0, 3]) >> 16 == 64  # one-block rows: the whole block-row in one chunk


def test_softmax_chunks_reject_bad_element_size(lib):
    L = bsp.bsp_layout_plan(np.ones((1, 2, 2), np.uint8), 64)
    assert lib.bsp_layout_softmax_chunks(L.handle, 8, None, None, None, None) == -1


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
    assert lib.bsp_attention_host(L.handle, 1, a, a, a, a, 1, 64, ctypes.c_float(1.0), 0, None, a,
                                  ctypes.c_size_t(1 << 20), 0, None) == -1
    # workspace for slices of one batch entry: 2 slots x (Q, K, V, O) x H S D x 2 bytes
    assert lib.bsp_attention_host_workspace(L.handle, 1, 64, 1) == 2 * 4 * 1 * 32 * 64 * 2
    assert lib.bsp_sdd(None, 1, a, a, a, 1, 16, 0, 1, None) == -1
    assert lib.bsp_layout_destroy(None) == 0


def test_info_reports_sizes(lib):
    lay = W.layout_band(10, 2, H=3)
    L = bsp.bsp_layout_plan(lay, 32)
    assert (L.H, L.nb, L.B, L.nnz, L.S) == (3, 10, 32, int(lay.sum()), 320)


# ------------------------------------------------------ affine geometry ----

def _affine_cases():
    """Small heads: every band / column-term family member the rules allow on
    nb = 6, random affine pairs, and random layouts (mostly not affine)."""
    rng = np.random.default_rng(11)
    heads = []
    nb = 6
    for bb in range(-(nb - 1), nb):
        for bk in range(1, nb - bb + 1):
            heads.append(("band", nb, [(1, bb, 1, bk, 0)]))
    for _ in range(60):
        nb = int(rng.integers(2, 10))
        bb = int(rng.integers(-(nb - 1), nb))
        bk = int(rng.integers(1, nb - bb + 1))
        cb = int(rng.integers(0, nb))
        cs = int(rng.integers(1, nb))
        ck = int(rng.integers(1, (nb - 1 - cb) // cs + 2))
        cs = 1 if ck == 1 else cs
        terms = [(0, cb, cs, ck, int(rng.integers(0, 2)))]
        if rng.random() < 0.7:
            terms.insert(0, (1, bb, 1, bk, 0))
        heads.append(("pair", nb, terms))
    for k in range(60):
        nb = int(rng.integers(1, 9))
        heads.append(("random", nb, (rng.random((nb, nb)) < rng.choice([0.2, 0.5, 0.8])).astype(np.uint8)))
    return heads


AFFINE_CASES = _affine_cases()


def _check_terms(nb, n, t):
    """The rules of bsp_affine_term_t for the first n rows of t [2, 5]."""
    kinds = [int(x[0]) for x in t[:n]]
    assert kinds in ([], [1], [0], [1, 0])
    for a, b, s, k, c in t[:n]:
        assert k >= 1
        if a == 1:
            assert s == 1 and c == 0 and -(nb - 1) <= b and b + k - 1 <= nb - 1
        else:
            assert s >= 1 and c in (0, 1) and b >= 0 and b + s * (k - 1) <= nb - 1 and (k > 1 or s == 1)
    assert not t[n:].any()


@pytest.mark.parametrize("idx", range(len(AFFINE_CASES)))
def test_geometry_exact_and_complete(lib, oracle, idx):
    # exact: the terms the library reports expand (oracle) to the head; complete:
    # it reports none only when the oracle's exhaustive search finds none
    kind, nb, spec = AFFINE_CASES[idx]
    if kind == "random":
        head = spec
    else:
        n0 = np.array([len(spec)], np.int32)
        t0 = np.zeros((1, 2, 5), np.int32)
        t0[0, :len(spec)] = spec
        head = oracle.affine_expand(n0, t0, nb)[0]
    L = bsp.bsp_layout_plan(head[None], 16)
    n, t = L.geometry()
    if n[0] < 0:
        assert not oracle.affine_describable(head), f"{kind}: a description exists but none was found"
    else:
        _check_terms(nb, n[0], t[0])
        assert np.array_equal(oracle.affine_expand(n, t, nb)[0], head)
        if kind != "random":
            assert oracle.affine_describable(head)


def test_geometry_of_the_workloads(lib):
    want = {"band": (1, [(1, -4, 1, 9, 0)]), "strided": (2, [(1, -3, 1, 4, 0), (0, 0, 16, 16, 1)]),
            "tiny": (-1, []), "bigbird": (-1, [])}
    for name, (n_want, terms) in want.items():
        w = W.ATTENTION_WORKLOADS[name]
        n, t = bsp.bsp_layout_plan(w.layout(), w.B).geometry()
        assert (n == n_want).all(), name
        for h in range(len(n)):
            for k, term in enumerate(terms):
                assert tuple(t[h, k]) == term, (name, h, k)
    n, _ = bsp.bsp_layout_plan(W.SPMM.layout(0.1), W.SPMM.B).geometry()
    assert (n == -1).all()


def test_geometry_mixed_heads(lib):
    lay = np.stack([W.layout_band(8, 1)[0], np.eye(8, dtype=np.uint8)[::-1].copy(), np.zeros((8, 8), np.uint8)])
    n, t = bsp.bsp_layout_plan(lay, 32).geometry()
    assert list(n) == [1, -1, 0]
    assert tuple(t[0, 0]) == (1, -1, 1, 3, 0) and not t[1:].any()


@pytest.mark.parametrize("terms", [
    [(2, 0, 1, 1, 0)],                         # alpha not 0 / 1
    [(1, 0, 2, 2, 0)],                         # band with stride
    [(1, 0, 1, 2, 1)],                         # causal band
    [(1, -8, 1, 1, 0)],                        # band offset below -(nb - 1)
    [(1, 6, 1, 3, 0)],                         # band past the last column
    [(0, -1, 1, 1, 0)],                        # column before 0
    [(0, 4, 2, 3, 0)],                         # column past nb
    [(0, 1, 2, 1, 0)],                         # one column with a stride
    [(0, 1, 1, 0, 0)],                         # kappa 0
    [(0, 1, 1, 2, 2)],                         # causal not 0 / 1
    [(1, 0, 1, 1, 0), (1, 1, 1, 1, 0)],        # two bands
    [(0, 0, 1, 1, 0), (1, 0, 1, 1, 0)],        # band not first
])
def test_compile_affine_rejects_bad_terms(lib, terms):
    # checked on the host before any device work
    nb = 8
    n = np.array([len(terms)], np.int32)
    t = np.zeros((1, 2, 5), np.int32)
    t[0, :len(terms)] = terms
    with pytest.raises(bsp.BspError) as e:
        bsp.bsp_layout_compile_affine(n, t, nb, 32, stream=0)
    assert e.value.code == -1
    with pytest.raises(bsp.BspError) as e:
        bsp.bsp_layout_compile_affine(np.array([3], np.int32), np.zeros((1, 2, 5), np.int32), nb, 32, stream=0)
    assert e.value.code == -1


@pytest.mark.parametrize("B", [16, 32, 64, 128])
@pytest.mark.parametrize("seed", range(6))
def test_geometry_steps_equal_step_tables(lib, oracle, B, seed):
    # the attention kernel's column / presence arithmetic (evaluated on the
    # host by bsp_diag_geometry_steps) against the compiler's step tables
    rng = np.random.default_rng(500 + seed)
    nb = int(rng.integers(3, 70))
    H = 3
    n = np.zeros(H, np.int32)
    t = np.zeros((H, 2, 5), np.int32)
    for h in range(H):
        bb = int(rng.integers(-(nb - 1), nb))
        bk = int(rng.integers(1, nb - bb + 1))
        cb = int(rng.integers(0, nb))
        cs = int(rng.integers(1, nb))
        ck = int(rng.integers(1, (nb - 1 - cb) // cs + 2))
        cs = 1 if ck == 1 else cs
        terms = [[(1, bb, 1, bk, 0)], [(0, cb, cs, ck, int(rng.integers(0, 2)))],
                 [(1, bb, 1, bk, 0), (0, cb, cs, ck, int(rng.integers(0, 2)))], []][int(rng.integers(0, 4))]
        n[h] = len(terms)
        if terms:
            t[h, :len(terms)] = terms
    lay = oracle.affine_expand(n, t, nb)
    L = bsp.bsp_layout_plan(lay, B)
    assert (L.geometry()[0] >= 0).all()
    tab = L.tiles()
    G, ns = tab["G"], tab["n_steps"]
    col = np.zeros(max(ns * G, 1), np.int32)
    blk = np.zeros(max(ns * G * G, 1), np.int32)
    assert lib.bsp_diag_geometry_steps(L.handle, ctypes.c_void_p(col.ctypes.data), ctypes.c_void_p(blk.ctypes.data)) == 0
    assert np.array_equal(col[:ns * G].reshape(ns, G), tab["step_col"])
    assert np.array_equal(blk[:ns * G * G].reshape(ns, G, G), (tab["step_blk"] >= 0).astype(np.int32))


def test_geometry_steps_of_the_workloads(lib):
    for name in ("band", "strided"):
        w = W.ATTENTION_WORKLOADS[name]
        L = bsp.bsp_layout_plan(w.layout(), w.B)
        tab = L.tiles()
        G, ns = tab["G"], tab["n_steps"]
        col = np.zeros(ns * G, np.int32)
        blk = np.zeros(ns * G * G, np.int32)
        assert lib.bsp_diag_geometry_steps(L.handle, ctypes.c_void_p(col.ctypes.data),
                                           ctypes.c_void_p(blk.ctypes.data)) == 0
        assert np.array_equal(col.reshape(ns, G), tab["step_col"]), name
        assert np.array_equal(blk.reshape(ns, G, G), (tab["step_blk"] >= 0).astype(np.int32)), name
    L = bsp.bsp_layout_plan(W.ATTENTION_WORKLOADS["bigbird"].layout(), 64)
    z = np.zeros(4, np.int32)
    assert lib.bsp_diag_geometry_steps(L.handle, ctypes.c_void_p(z.ctypes.data), ctypes.c_void_p(z.ctypes.data)) == -2


def test_blocksparse_module_rejects_unknown_mode(lib):
    from sparse_attention_layout_gb300 import blocksparse
    assert blocksparse.MODES == ("sdd", "dsd", "dds")
    with pytest.raises(ValueError):
        blocksparse.matmul(np.ones((1, 2, 2), np.uint8), 32, "sds")


def test_new_entry_points_validate_arguments(lib):
    # checked on the host before any device work: NULL handle / host-only
    # handle, bad scale, bad mask kind, missing dense mask
    L = bsp.bsp_layout_plan(np.ones((1, 2, 2), np.uint8), 16)
    buf = (ctypes.c_char * 4096)()
    a = ctypes.c_void_p(ctypes.addressof(buf) + (-ctypes.addressof(buf)) % 16)
    one = ctypes.c_float(1.0)
    f = lib.bsp_sdd_softmax
    assert f(None, 1, a, a, a, 1, 16, 0, 1, one, 0, None, None) == -1
    assert f(L.handle, 1, a, a, a, 1, 16, 0, 1, one, 0, None, None) == -1       # host-only handle
    assert lib.bsp_layout_geometry(None, None, None) == -1
    n = np.zeros(1, np.int32)
    assert lib.bsp_layout_geometry(L.handle, ctypes.c_void_p(n.ctypes.data), None) == 0 and n[0] == 1  # a full 2 x 2 head is one band
    assert lib.bsp_attention_host(None, 1, a, a, a, a, 1, 64, one, 0, None, a, ctypes.c_size_t(1 << 20), 0, None) == -1
    assert lib.bsp_attention_host_workspace(None, 1, 64, 1) == 0
    assert lib.bsp_attention_host_workspace(L.handle, 1, 64, 0) == 0
    assert lib.bsp_diag_geometry_steps(None, a, a) == -1
    assert lib.bsp_attention_lse(None, 1, a, a, a, a, a, 1, 64, one, 0, None, None) == -1
    assert lib.bsp_attention_lse(L.handle, 1, a, a, a, a, a, 1, 64, one, 0, None, None) == -1  # host-only handle
    assert lib.bsp_attention_backward_lse(None, 1, a, a, a, a, a, a, a, a, a, 1, 64, one, 0, None, a, a, None) == -1


def test_diag_wait_limit_needs_a_compiled_handle(lib):
    # a host-only plan has no device status word or kernels: rejected without a GPU
    L = bsp.bsp_layout_plan(np.ones((1, 2, 2), np.uint8), 32)
    assert lib.bsp_diag_wait_limit(L.handle, ctypes.c_uint64(1000), 0) == -1
    assert lib.bsp_diag_wait_limit(None, ctypes.c_uint64(0), 0) == -1
