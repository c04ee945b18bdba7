"""On-device layout compilation (bsp_layout_compile_device) against the host
compiler: every table (softmax chunk lists included) bit-exact on the workload
layouts and edge layouts, the
compute calls give identical results with either handle, invalid values and
oversize layouts are rejected."""

import numpy as np
import pytest
import torch

from sparse_attention_layout_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bsp():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from sparse_attention_layout_gb300 import build
    build.build()
    from sparse_attention_layout_gb300 import bsp as m
    return m


def layouts():
    out = {}
    for name, w in W.ATTENTION_WORKLOADS.items():
        out[name] = (w.layout(), w.B)
    for d in W.SPMM_DENSITIES:
        out[f"spmm{int(d * 100)}"] = (W.SPMM.layout(d), W.SPMM.B)
    out["spmm_b16"] = (W.SPMM_BLOCKS[16].layout(0.1), 16)
    rng = np.random.default_rng(9)
    out["all_zero"] = (np.zeros((2, 8, 8), np.uint8), 16)
    out["all_ones"] = (np.ones((3, 5, 5), np.uint8), 64)
    out["ragged_groups"] = ((rng.random((3, 13, 13)) < 0.3).astype(np.uint8), 16)  # 13 rows, G = 8
    lay = (rng.random((2, 9, 9)) < 0.3).astype(np.uint8)
    lay[0, 4, :] = 0
    lay[1, :, 6] = 0
    out["empty_rows_cols"] = (lay, 128)
    return out


LAYOUTS = layouts()


@pytest.mark.parametrize("name", sorted(LAYOUTS))
def test_device_tables_equal_host_tables(bsp, name):
    lay, B = LAYOUTS[name]
    host = bsp.bsp_layout_compile(lay, B)
    dev = bsp.bsp_layout_compile_device(torch.from_numpy(lay).cuda(), B)
    assert dev.nnz == host.nnz
    hl, dl = host.luts(), dev.luts()
    for k in hl:
        assert np.array_equal(hl[k], dl[k]), k
    ht, dt = host.tiles(), dev.tiles()
    for k in ("G", "n_tiles", "n_steps"):
        assert ht[k] == dt[k], k
    for k in ("tile_step_ptr", "tile_order", "step_col", "step_blk"):
        assert np.array_equal(ht[k], dt[k]), k
    for o in (0, 1):
        hg, dg = host.groups(o), dev.groups(o)
        assert hg["n_slots"] == dg["n_slots"]
        for k in ("grp_ptr", "grp_order", "slot_idx", "slot_blk"):
            assert np.array_equal(hg[k], dg[k]), (o, k)
    for elt in (2, 4):
        hc, dc = host.softmax_chunks(elt), dev.softmax_chunks(elt)
        assert hc["fits"] == dc["fits"] and hc["max_bytes"] == dc["max_bytes"], elt
        assert np.array_equal(hc["items"], dc["items"]), elt


@pytest.mark.parametrize("name", ["tiny", "strided", "bigbird"])
def test_ops_identical_with_either_handle(bsp, name):
    w = W.ATTENTION_WORKLOADS[name]
    lay = w.layout()
    Lh = bsp.bsp_layout_compile(lay, w.B)
    Ld = bsp.bsp_layout_compile_device(torch.from_numpy(lay).cuda(), w.B)
    q, k, v = (t.cuda() for t in w.qkv())
    if name == "strided":  # a smaller batch of heads keeps the test short
        q, k, v = q[:, :4], k[:, :4], v[:, :4]
        lay4 = lay[:4]
        Lh = bsp.bsp_layout_compile(lay4, w.B)
        Ld = bsp.bsp_layout_compile_device(torch.from_numpy(lay4).cuda(), w.B)
    o1 = bsp.bsp_attention(Lh, q, k, v, None, w.scale, w.mask_kind)
    o2 = bsp.bsp_attention(Ld, q, k, v, None, w.scale, w.mask_kind)
    p1 = bsp.bsp_softmax(Lh, bsp.bsp_sdd(Lh, q, k), None, w.scale, w.mask_kind)
    p2 = bsp.bsp_softmax(Ld, bsp.bsp_sdd(Ld, q, k), None, w.scale, w.mask_kind)
    d1, d2 = bsp.bsp_dsd(Lh, p1, v), bsp.bsp_dsd(Ld, p2, v)
    # the softmax backward (BigBird's global rows take its chunk kernel, the
    # other layouts its row kernel)
    g = W.randn(tuple(p1.shape), w.dtype, 9).cuda()
    b1, b2 = bsp.bsp_softmax_backward(Lh, p1, g, None, w.scale), bsp.bsp_softmax_backward(Ld, p2, g, None, w.scale)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(p1, p2) and torch.equal(d1, d2) and torch.equal(b1, b2)


def test_device_compile_rejects_bad_values_and_sizes(bsp):
    lay = torch.ones(1, 4, 4, dtype=torch.uint8, device="cuda")
    lay[0, 1, 2] = 2
    with pytest.raises(bsp.BspError) as e:
        bsp.bsp_layout_compile_device(lay, 32)
    assert e.value.code == -1
    with pytest.raises(bsp.BspError) as e:
        bsp.bsp_layout_compile_device(torch.zeros(1, 4100, 4100, dtype=torch.uint8, device="cuda"), 16)
    assert e.value.code == -2
