"""GPU parity at the workloads' full sizes, in the launch configuration the
bench times, on sampled outputs the oracle computes one by one (plus whole-
tensor properties that hold at any size: finiteness, softmax rows summing to 1,
exact zeros of empty rows).

Workloads: tiny (Z1 H1 S256 D64 B16 fp32), bigbird (Z2 H12 S4096 D64 B64
fp32, diagonal-causal), band (Z4 H16 S8192 D128 B128 bf16), strided (Z1 H32
S16384 D128 B64 bf16, diagonal-causal) and the spMM workload (8192^2 sparse,
block 32, bf16, 10/25/50 % density).  Tolerance: normwise max |g - r| / max |r|
<= 1e-5 (fp32) or 2e-2 (bf16), and every sampled entry within its own bound
(tests/gpu_util.py): softmax rows elementwise, products by their forward error
bound against the product of the operands' absolute values.  Row sums of the
whole softmax output: |sum - 1| <= u + 1e-4 for 16-bit outputs (u the unit
roundoff: each probability is rounded once, so the rounding moves a sum of 1
by at most u) and <= 1e-5 for fp32; entries that the diagonal-causal mask
removes are exactly 0 in the whole output."""

import numpy as np
import pytest
import torch

from gpu_util import PROB_TOL, U, assert_close, attention_acc, check_softmax_backward_elementwise, gamma, to_np
from sparse_attention_layout_gb300 import workloads as W

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


@pytest.fixture(scope="module")
def bsp():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from sparse_attention_layout_gb300 import build
    build.build()
    from sparse_attention_layout_gb300 import bsp as m
    return m


def rowsum_tol(dtype):
    """|sum of a softmax row - 1|: one rounding of each probability to the
    output type moves the sum by at most u; the fp32 exponentials and the
    normalisation by far less than 1e-4."""
    return 1e-5 if dtype == torch.float32 else U[dtype] + 1e-4


def check_rowsums_and_masked_zeros(w, lay, P):
    """Every present row of the block-format softmax output P sums to 1, and
    the entries above the diagonal of every diagonal block are exactly 0 when
    the workload masks them (diagonal-causal)."""
    hs, is_, js = np.nonzero(lay)
    key = torch.from_numpy(hs * w.nb + is_).cuda()
    rowsum = torch.zeros(w.Z, w.H * w.nb, w.B, device="cuda", dtype=torch.float64)
    rowsum.index_add_(1, key, P.double().sum(dim=3))
    present = torch.from_numpy(lay.sum(axis=2).reshape(-1) > 0).cuda()
    dev = (rowsum[:, present] - 1.0).abs().max().item()
    assert dev <= rowsum_tol(DT[w.dtype]), f"{w.name}: a row sums to 1 +- {dev:.3e}"
    if w.mask_kind == W.MASK_DIAG_CAUSAL:
        diag = torch.from_numpy(np.flatnonzero(is_ == js)).cuda()
        upper = torch.triu(torch.ones(w.B, w.B, dtype=torch.bool, device="cuda"), 1)
        leaked = (P[:, diag] != 0) & upper
        assert not leaked.any(), f"{w.name}: {int(leaked.sum())} masked entries are not exactly 0"


def sample_rows(w, lay, n, seed):
    """Random rows plus edge rows: first/last row of every sampled (z, h), rows
    of the last block-row and of the longest block-row."""
    rng = np.random.default_rng(seed)
    total = w.Z * w.H * w.S
    rows = set(rng.choice(total, size=n, replace=False).tolist())
    counts = lay.sum(axis=2)  # [H, nb]
    h_long, i_long = np.unravel_index(np.argmax(counts), counts.shape)
    for z in range(w.Z):
        for h in (0, w.H - 1, int(h_long)):
            base = (z * w.H + h) * w.S
            rows.update([base, base + w.S - 1, base + w.S - w.B, base + int(i_long) * w.B + w.B // 2])
    return np.array(sorted(rows), dtype=np.int64)


@pytest.mark.parametrize("name", ["tiny", "bigbird", "band", "strided"])
def test_attention_workload(bsp, oracle, name):
    w = W.ATTENTION_WORKLOADS[name]
    lay = w.layout()
    L = bsp.bsp_layout_compile(lay, w.B)
    Q, K, V = w.qkv()
    q, k, v = (t.cuda() for t in (Q, K, V))
    o = torch.empty_like(q)
    bsp.bsp_attention(L, q, k, v, o, w.scale, w.mask_kind)  # the bench's call
    torch.cuda.synchronize()
    assert bsp.bsp_status_check(L) == 0
    assert torch.isfinite(o).all()
    sel = sample_rows(w, lay, 48, 7)
    got = to_np(o.reshape(-1, w.D)[torch.from_numpy(sel).cuda()])
    want = oracle.attention(lay, w.B, Q, K, V, w.scale, w.mask_kind, sel=sel)
    mag = oracle.attention(lay, w.B, Q, K, V.abs(), w.scale, w.mask_kind, sel=sel)
    acc = attention_acc(q, k, w.scale, DT[w.dtype], w.S).reshape(-1, 1)[sel]
    assert_close(got, want, DT[w.dtype], f"{name} fused attention, {sel.size} sampled rows", mag=mag, acc=acc)


@pytest.mark.parametrize("name", ["tiny", "bigbird", "band", "strided"])
def test_unfused_chain_workload(bsp, oracle, name):
    """SDD -> softmax -> DSD at full size: sampled SDD blocks and sampled rows
    of the chain's output against the oracle."""
    w = W.ATTENTION_WORKLOADS[name]
    lay = w.layout()
    L = bsp.bsp_layout_compile(lay, w.B)
    Q, K, V = w.qkv()
    q, k, v = (t.cuda() for t in (Q, K, V))
    P = bsp.bsp_sdd(L, q, k)
    torch.cuda.synchronize()
    rng = np.random.default_rng(3)
    blocks = np.unique(np.concatenate([rng.choice(w.Z * L.nnz, size=24, replace=False),
                                       [0, w.Z * L.nnz - 1]])).astype(np.int64)
    got_s = to_np(P.reshape(-1, w.B, w.B)[torch.from_numpy(blocks).cuda()])
    want_s = oracle.sdd(lay, w.B, Q, K, sel=blocks)
    mag_s = oracle.sdd(lay, w.B, Q.abs(), K.abs(), sel=blocks)
    assert_close(got_s, want_s, DT[w.dtype], f"{name} SDD, {blocks.size} sampled blocks", mag=mag_s,
                 acc=gamma(w.D))
    bsp.bsp_softmax(L, P, P, w.scale, w.mask_kind)
    O = bsp.bsp_dsd(L, P, v)
    torch.cuda.synchronize()
    assert torch.isfinite(O).all()
    sel = sample_rows(w, lay, 48, 11)
    got = to_np(O.reshape(-1, w.D)[torch.from_numpy(sel).cuda()])
    want = oracle.attention(lay, w.B, Q, K, V, w.scale, w.mask_kind, sel=sel)
    mag = oracle.attention(lay, w.B, Q, K, V.abs(), w.scale, w.mask_kind, sel=sel)
    # the chain rounds the scores and the probabilities to the data type between its steps
    acc = attention_acc(q, k, w.scale, DT[w.dtype], w.S, scores_rounded=True).reshape(-1, 1)[sel]
    assert_close(got, want, DT[w.dtype], f"{name} unfused chain, {sel.size} sampled rows", mag=mag, acc=acc)


@pytest.mark.parametrize("name", ["tiny", "bigbird", "band", "strided"])
def test_sdd_softmax_chain_workload(bsp, oracle, name):
    """Fused SDD + softmax, then DSD, at full size: every present row of P sums
    to 1, sampled rows of the output against the oracle's attention."""
    w = W.ATTENTION_WORKLOADS[name]
    lay = w.layout()
    L = bsp.bsp_layout_compile(lay, w.B)
    Q, K, V = w.qkv()
    q, k, v = (t.cuda() for t in (Q, K, V))
    P = bsp.bsp_sdd_softmax(L, q, k, None, w.scale, w.mask_kind)
    O = bsp.bsp_dsd(L, P, v)
    torch.cuda.synchronize()
    assert torch.isfinite(P).all() and torch.isfinite(O).all()
    check_rowsums_and_masked_zeros(w, lay, P)
    sel = sample_rows(w, lay, 48, 13)
    got = to_np(O.reshape(-1, w.D)[torch.from_numpy(sel).cuda()])
    want = oracle.attention(lay, w.B, Q, K, V, w.scale, w.mask_kind, sel=sel)
    mag = oracle.attention(lay, w.B, Q, K, V.abs(), w.scale, w.mask_kind, sel=sel)
    # scores stay fp32 inside the fused kernel; P is rounded once before DSD
    acc = attention_acc(q, k, w.scale, DT[w.dtype], w.S).reshape(-1, 1)[sel]
    assert_close(got, want, DT[w.dtype], f"{name} fused SDD+softmax chain, {sel.size} sampled rows", mag=mag,
                 acc=acc)


@pytest.mark.parametrize("name", ["tiny", "bigbird", "band", "strided"])
def test_softmax_backward_workload(bsp, oracle, name):
    """The softmax backward at full size on a softmax output: sampled
    block-rows (the longest, the first and last, random ones), each against
    the oracle run on a layout holding that block-row alone, every entry
    within the fp32 evaluation's error bound; over the whole output, dX is
    exactly 0 wherever Y is 0."""
    w = W.ATTENTION_WORKLOADS[name]
    lay = w.layout()
    L = bsp.bsp_layout_compile(lay, w.B)
    Y = bsp.bsp_softmax(L, W.randn((w.Z, L.nnz, w.B, w.B), w.dtype, 81).cuda(), None, w.scale, w.mask_kind)
    dY = W.randn((w.Z, L.nnz, w.B, w.B), w.dtype, 82).cuda()
    dX = bsp.bsp_softmax_backward(L, Y, dY, None, w.scale)
    torch.cuda.synchronize()
    assert bsp.bsp_status_check(L) == 0
    assert not dX.masked_select(Y == 0).any()
    H, nb = lay.shape[0], lay.shape[1]
    cnt = lay.reshape(-1, nb).sum(axis=1).astype(np.int64)
    ptr = np.concatenate([[0], np.cumsum(cnt)])
    keys = set(np.random.default_rng(83).choice(H * nb, 6, replace=False).tolist())
    keys |= {int(np.argmax(cnt)), 0, H * nb - 1}
    for k in sorted(keys):
        a, b = int(ptr[k]), int(ptr[k + 1])
        if a == b:
            continue
        h, i = divmod(k, nb)
        sub = np.zeros((1, nb, nb), np.uint8)
        sub[0, i] = lay[h, i]
        ys, gs, xs = Y[:, a:b].cpu(), dY[:, a:b].cpu(), dX[:, a:b].cpu()
        want = oracle.softmax_backward(sub, w.B, ys, gs, w.scale)
        check_softmax_backward_elementwise(sub, w.B, ys, gs, xs, want, w.scale, DT[w.dtype],
                                           f"{name} softmax backward, head {h} block-row {i}")


@pytest.mark.parametrize("name", ["tiny", "bigbird", "band", "strided"])
def test_softmax_workload(bsp, oracle, name):
    """The softmax alone on random SDD-shaped input at full size: sampled rows
    against the oracle, every row of the whole output sums to 1."""
    w = W.ATTENTION_WORKLOADS[name]
    lay = w.layout()
    L = bsp.bsp_layout_compile(lay, w.B)
    X = W.randn((w.Z, L.nnz, w.B, w.B), w.dtype, 77)
    Y = bsp.bsp_softmax(L, X.cuda(), None, w.scale, w.mask_kind)
    torch.cuda.synchronize()
    assert torch.isfinite(Y).all()
    check_rowsums_and_masked_zeros(w, lay, Y)
    hs, is_, js = np.nonzero(lay)
    sel = sample_rows(w, lay, 48, 5)
    want = oracle.softmax_rows(lay, w.B, X, w.scale, w.mask_kind, sel=sel)  # dense rows [n, S]
    Yh = to_np(Y)
    ids = -np.ones(lay.shape, np.int64)
    ids[hs, is_, js] = np.arange(hs.size)
    got = np.zeros_like(want)
    keep = np.zeros(want.shape, dtype=bool)
    cols = np.arange(w.S)
    for t, u in enumerate(sel):
        zh, r = divmod(int(u), w.S)
        z, h = divmod(zh, w.H)
        i, a = divmod(r, w.B)
        for j in np.flatnonzero(lay[h, i]):
            got[t, j * w.B:(j + 1) * w.B] = Yh[z, ids[h, i, j], a]
        keep[t] = np.repeat(lay[h, i].astype(bool), w.B)
        if w.mask_kind == W.MASK_DIAG_CAUSAL:
            keep[t] &= (cols // w.B != i) | (cols <= r)
    assert_close(got, want, DT[w.dtype], f"{name} softmax, {sel.size} sampled rows", rel=PROB_TOL[DT[w.dtype]],
                 zeros=~keep)


@pytest.mark.parametrize("B,density", [(32, d) for d in W.SPMM_DENSITIES] +
                         [(b, d) for b in (16, 64, 128) for d in W.SPMM_BLOCK_DENSITIES])
def test_spmm_workload(bsp, oracle, B, density):
    sp = W.SPMM_BLOCKS[B]
    lay = sp.layout(density)
    L = bsp.bsp_layout_compile(lay, sp.B)
    A = sp.sparse_values(L.nnz, density)
    Bd = sp.dense_dsd(density)
    Ad = sp.dense_dds(density)
    C1 = bsp.bsp_dsd(L, A.cuda(), Bd.cuda())
    C2 = bsp.bsp_dds(L, Ad.cuda(), A.cuda())
    torch.cuda.synchronize()
    assert torch.isfinite(C1).all() and torch.isfinite(C2).all()
    rng = np.random.default_rng(int(density * 100))
    empty_rows = np.flatnonzero(lay[0].sum(axis=1) == 0)
    rows = np.unique(np.concatenate([rng.choice(sp.S, 10, replace=False), [0, sp.S - 1],
                                     empty_rows[:2] * sp.B])).astype(np.int64)
    got = to_np(C1[0, 0][torch.from_numpy(rows).cuda()])
    assert_close(got, oracle.dsd(lay, sp.B, A, Bd, sel=rows), torch.bfloat16, f"DSD spMM B={B} {density}",
                 mag=oracle.dsd(lay, sp.B, A.abs(), Bd.abs(), sel=rows), acc=gamma(sp.S))
    mrows = np.unique(np.concatenate([rng.choice(sp.N, 6, replace=False), [0, sp.N - 1]])).astype(np.int64)
    got = to_np(C2[0, 0][torch.from_numpy(mrows).cuda()])
    assert_close(got, oracle.dds(lay, sp.B, Ad, A, sel=mrows), torch.bfloat16, f"DDS spMM B={B} {density}",
                 mag=oracle.dds(lay, sp.B, Ad.abs(), A.abs(), sel=mrows), acc=gamma(sp.S))
    # block-rows without any block are exactly zero in the DSD output
    for i in empty_rows[:4]:
        assert (C1[0, 0, i * sp.B:(i + 1) * sp.B] == 0).all()


def test_long_sequence_band(bsp, oracle):
    """A maximum-size case: S = 262144 tokens (4096 blocks of 64, the largest
    block count the on-device compiler takes), band of +-2 blocks, causal
    inside the diagonal blocks, bf16.  Fused attention and the fused
    SDD + softmax -> DSD chain on sampled rows (first, last, random) against
    the oracle; the layout compiled on the device equals the host compile's
    tiles."""
    from types import SimpleNamespace
    B, nb, H, Z, D = 64, 4096, 1, 1, 128
    S = nb * B
    lay = W.layout_band(nb, 2, H)
    L = bsp.bsp_layout_compile(lay, B)
    Ld = bsp.bsp_layout_compile_device(torch.from_numpy(lay).cuda(), B)
    assert np.array_equal(L.tiles()["step_col"], Ld.tiles()["step_col"])
    Q, K, V = (W.randn((Z, H, S, D), "bf16", 500 + s) for s in range(3))
    q, k, v = (t.cuda() for t in (Q, K, V))
    scale = 1.0 / np.sqrt(D)
    o = bsp.bsp_attention(Ld, q, k, v, None, scale, W.MASK_DIAG_CAUSAL)
    o2 = bsp.bsp_dsd(Ld, bsp.bsp_sdd_softmax(Ld, q, k, None, scale, W.MASK_DIAG_CAUSAL), v)
    torch.cuda.synchronize()
    assert torch.isfinite(o).all() and torch.isfinite(o2).all()
    w = SimpleNamespace(Z=Z, H=H, S=S, B=B)
    sel = sample_rows(w, lay, 40, 17)
    want = oracle.attention(lay, B, Q, K, V, scale, W.MASK_DIAG_CAUSAL, sel=sel)
    mag = oracle.attention(lay, B, Q, K, V.abs(), scale, W.MASK_DIAG_CAUSAL, sel=sel)
    acc = attention_acc(q, k, scale, torch.bfloat16, 5 * B).reshape(-1, 1)[sel]
    for got, what in ((o, "fused attention"), (o2, "fused SDD + softmax -> DSD")):
        g = to_np(got.reshape(-1, D)[torch.from_numpy(sel).cuda()])
        assert_close(g, want, torch.bfloat16, f"S={S} {what}, {sel.size} sampled rows", mag=mag, acc=acc)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_long_global_rows_cut(bsp, oracle, dt):
    """BigBird over S = 16384 (Z1 H12 D64 B64, window 3, 2 global, 3 random,
    diagonal-causal): each head's global-row tile has 128 steps against a fair
    share of ~80, so the automatic schedule cuts those tiles and merges their
    pieces.  Sampled rows (the global rows included) against the oracle; the
    result without cuts for balance within the same bound."""
    from types import SimpleNamespace
    B, nb, H, Z, D = 64, 256, 12, 1, 64
    S = nb * B
    lay = W.layout_bigbird(nb, H, window=3, n_global=2, n_random=3, seed=2)
    L = bsp.bsp_layout_compile(lay, B)
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    assert len(bsp.bsp_diag_attention_schedule(L, Z, n_sm, DT[dt])["combine"]) == H
    Q, K, V = (W.randn((Z, H, S, D), dt, 520 + s) for s in range(3))
    q, k, v = (t.cuda() for t in (Q, K, V))
    o = bsp.bsp_attention(L, q, k, v, None, 0.125, W.MASK_DIAG_CAUSAL)
    # no cuts for balance (fp32 still cuts at 32 steps: one accumulation of
    # all 16384 keys in tensor memory missed 1e-5, normwise 1.5e-5)
    bsp.bsp_diag_attention_split(L, -1)
    assert len(bsp.bsp_diag_attention_schedule(L, Z, n_sm, DT[dt])["combine"]) == (H if dt == "f32" else 0)
    o_whole = bsp.bsp_attention(L, q, k, v, None, 0.125, W.MASK_DIAG_CAUSAL)
    torch.cuda.synchronize()
    assert bsp.bsp_status_check(L) == 0
    w = SimpleNamespace(Z=Z, H=H, S=S, B=B)
    sel = np.unique(np.concatenate([sample_rows(w, lay, 40, 19),
                                    [h * S + r for h in (0, 5, 11) for r in (0, 63, 64, 127)]])).astype(np.int64)
    want = oracle.attention(lay, B, Q, K, V, 0.125, W.MASK_DIAG_CAUSAL, sel=sel)
    mag = oracle.attention(lay, B, Q, K, V.abs(), 0.125, W.MASK_DIAG_CAUSAL, sel=sel)
    acc = attention_acc(q, k, 0.125, DT[dt], S).reshape(-1, 1)[sel]
    for got, what in ((o, "cut"), (o_whole, "whole tiles")):
        g = to_np(got.reshape(-1, D)[torch.from_numpy(sel).cuda()])
        assert_close(g, want, DT[dt], f"BigBird S={S} {dt} {what}, {sel.size} sampled rows", mag=mag, acc=acc)


@pytest.mark.parametrize("name", ["band", "strided"])
def test_backward_paths_agree_at_full_size(bsp, name):
    """The two attention backwards at full size (the fp64 oracle's backward
    is dense S x S per head, too slow here): the recomputing chain (P from a
    two-pass fused softmax, dX with rowsum(P .* dP) accumulated in a first
    pass) and the one from the forward's O and log-sum-exp (P and dX in one
    pass each, rowsum from dO . O) reach P and dX through different kernels
    and formulas; their gradients agree within the 16-bit chain's tolerance
    (normwise 3e-2: each rounds P and dX to bf16), and are finite."""
    from gpu_util import normwise_err
    w = W.ATTENTION_WORKLOADS[name]
    lay = w.layout()
    L = bsp.bsp_layout_compile(lay, w.B)
    q, k, v = (t.cuda() for t in w.qkv())
    g = W.randn(q.shape, w.dtype, 909).cuda()
    r1 = bsp.attention_backward(L, q, k, v, g, w.scale, w.mask_kind)
    O, lse = bsp.bsp_attention_lse(L, q, k, v, None, None, w.scale, w.mask_kind)
    r2 = bsp.attention_backward_lse(L, q, k, v, O, g, lse, w.scale, w.mask_kind)
    torch.cuda.synchronize()
    assert bsp.bsp_status_check(L) == 0
    for a, b_, what in zip(r1, r2, ("dQ", "dK", "dV")):
        assert torch.isfinite(b_).all(), f"{name} {what} not finite"
        err = normwise_err(to_np(b_), to_np(a))
        assert err <= 3e-2, f"{name} {what}: the two backwards differ by {err:.3e} (normwise)"
