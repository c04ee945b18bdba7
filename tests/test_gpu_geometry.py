"""Affine geometry on the GPU: handles compiled from per-head terms
(bsp_layout_compile_affine) against the host compiler on the expanded layout
(every table bit-exact), and the fused attention kernel's geometry variant
(BSP_GEOMETRY=1: key blocks computed from the terms) against the variant
that reads the step tables (identical bytes) and against the fp64 oracle
(normwise 2e-2 for bf16 / fp16), over block sizes, head sizes, mask kinds,
ragged last tiles and the full-size banded and strided workloads."""

import numpy as np
import pytest
import torch

from gpu_util import TOL, dev, normwise_err, to_np
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


def random_terms(H, nb, seed):
    """Per-head band and / or column terms within the rules (head 0 a band
    only, head 1 a causal column term only when H > 2)."""
    rng = np.random.default_rng(seed)
    n = np.zeros(H, np.int32)
    t = np.zeros((H, 2, 5), np.int32)
    for h in range(H):
        bb = int(rng.integers(-min(nb - 1, 6), min(nb, 4)))
        bk = int(rng.integers(1, min(nb - bb, 9) + 1))
        cb = int(rng.integers(0, nb))
        cs = int(rng.integers(1, max(2, nb // 3)))
        ck = int(rng.integers(1, (nb - 1 - cb) // cs + 2))
        cs = 1 if ck == 1 else cs
        band, col = (1, bb, 1, bk, 0), (0, cb, cs, ck, int(rng.integers(0, 2)))
        terms = [band] if h == 0 else [(0, cb, cs, ck, 1)] if (h == 1 and H > 2) else [band, col]
        n[h] = len(terms)
        t[h, :len(terms)] = terms
    return n, t


def tables_equal(a, b):
    la, lb = a.luts(), b.luts()
    for k in la:
        assert np.array_equal(la[k], lb[k]), k
    ta, tb = a.tiles(), b.tiles()
    for k in ("G", "n_tiles", "n_steps"):
        assert ta[k] == tb[k], k
    for k in ("tile_step_ptr", "tile_order", "step_col", "step_blk"):
        assert np.array_equal(ta[k], tb[k]), k
    for o in (0, 1):
        ga, gb = a.groups(o), b.groups(o)
        for k in ("grp_ptr", "grp_order", "slot_idx", "slot_blk"):
            assert np.array_equal(ga[k], gb[k]), (o, k)


@pytest.mark.parametrize("B,nb,seed", [(16, 37, 1), (32, 30, 2), (64, 20, 3), (128, 9, 4), (64, 256, 5)])
def test_compile_affine_tables_equal_host_compile(bsp, oracle, B, nb, seed):
    n, t = random_terms(4, nb, seed)
    lay = oracle.affine_expand(n, t, nb)
    La = bsp.bsp_layout_compile_affine(n, t, nb, B)
    Lh = bsp.bsp_layout_compile(lay, B)
    assert La.nnz == Lh.nnz
    tables_equal(La, Lh)
    na, ta = La.geometry()
    assert np.array_equal(na, n) and np.array_equal(ta, t)


def _attn(bsp, L, q, k, v, scale, kind, mask, geo):
    """Attention with the geometry variant switched on (BSP_GEOMETRY=1) or off."""
    import os
    old = os.environ.get("BSP_GEOMETRY")
    os.environ["BSP_GEOMETRY"] = "1" if geo else "0"
    try:
        o = bsp.bsp_attention(L, q, k, v, None, scale, kind, mask)
        torch.cuda.synchronize()
    finally:
        if old is None:
            del os.environ["BSP_GEOMETRY"]
        else:
            os.environ["BSP_GEOMETRY"] = old
    return o


@pytest.mark.parametrize("B,nb", [(16, 37), (32, 23), (64, 13), (128, 6)])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("kind", [0, 1, 2])
@pytest.mark.parametrize("dt", ["bf16", "f16"])
def test_attention_geometry_equals_tables_and_oracle(bsp, oracle, B, nb, D, kind, dt):
    dtype = {"bf16": torch.bfloat16, "f16": torch.float16}[dt]
    Z, H = 2, 3
    S = nb * B
    n, t = random_terms(H, nb, 100 + B + D + kind)
    lay = oracle.affine_expand(n, t, nb)
    L = bsp.bsp_layout_compile(lay, B)
    assert (L.geometry()[0] >= 0).all()
    Q, K, V = (W.randn((Z, H, S, D), dt, 200 + s) for s in range(3))
    mask = W.random_mask(S, 0.8, 210) if kind == W.MASK_DENSE else None
    dmask = None if mask is None else torch.from_numpy(mask).cuda()
    scale = 1.0 / np.sqrt(D)
    o_geo = _attn(bsp, L, dev(Q), dev(K), dev(V), scale, kind, dmask, True)
    o_tab = _attn(bsp, L, dev(Q), dev(K), dev(V), scale, kind, dmask, False)
    assert torch.equal(o_geo, o_tab)
    want = oracle.attention(lay, B, Q, K, V, scale, kind, mask)
    err = normwise_err(to_np(o_geo), want)
    assert err <= TOL[dtype], f"normwise error {err:.3e}"


def test_attention_compile_affine_handle(bsp, oracle):
    # a handle built from terms gives the same output as one built from the layout
    B, nb, D, Z, H = 64, 40, 128, 1, 4
    n, t = random_terms(H, nb, 7)
    lay = oracle.affine_expand(n, t, nb)
    La = bsp.bsp_layout_compile_affine(n, t, nb, B)
    Lh = bsp.bsp_layout_compile(lay, B)
    q, k, v = (dev(W.randn((Z, H, nb * B, D), "bf16", 300 + s)) for s in range(3))
    o1 = _attn(bsp, La, q, k, v, 0.1, W.MASK_DIAG_CAUSAL, None, True)
    o2 = _attn(bsp, Lh, q, k, v, 0.1, W.MASK_DIAG_CAUSAL, None, False)
    assert torch.equal(o1, o2)


@pytest.mark.parametrize("name", ["band", "strided"])
def test_full_size_geometry_equals_tables(bsp, name):
    # the bench's launch configuration on the full workloads
    w = W.ATTENTION_WORKLOADS[name]
    L = bsp.bsp_layout_compile(w.layout(), w.B)
    assert (L.geometry()[0] >= 0).all()
    q, k, v = (dev(x) for x in w.qkv())
    o_geo = _attn(bsp, L, q, k, v, w.scale, w.mask_kind, None, True)
    o_tab = _attn(bsp, L, q, k, v, w.scale, w.mask_kind, None, False)
    assert torch.equal(o_geo, o_tab)
    assert torch.isfinite(o_geo).all()
