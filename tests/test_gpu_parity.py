"""GPU parity: every op through the C ABI against the fp64 oracle on the same
seeded inputs, at sizes spanning several tiles with ragged tails, each block
size, each dtype, each mask kind and both kernel paths (tensor-core where it
applies, CUDA-core forced with BSP_FORCE_SIMT=1).

Tolerance (normwise max |g - r| / max |r|): 1e-5 for fp32 outputs, 2e-2 for
bf16 / fp16 outputs; on top of it every entry is bounded (tests/gpu_util.py):
softmax outputs by an elementwise relative bound from the output's unit
roundoff, with the entries the oracle defines as 0 (masked, empty rows) exactly
0; products by their forward error bound against the same product of the
operands' absolute values."""

import os

import numpy as np
import pytest
import torch

from gpu_util import (PROB_TOL, assert_close, attention_acc, dev, gamma, softmax_rel_bound,
                      softmax_zero_positions, to_np)
from sparse_attention_layout_gb300 import workloads as W

pytestmark = pytest.mark.gpu

DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


@pytest.fixture(scope="module")
def bsp():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from sparse_attention_layout_gb300 import build
    build.build()
    from sparse_attention_layout_gb300 import bsp as m
    return m


@pytest.fixture(params=["tc", "simt"])
def path(request, monkeypatch):
    if request.param == "simt":
        monkeypatch.setenv("BSP_FORCE_SIMT", "1")
    else:
        monkeypatch.delenv("BSP_FORCE_SIMT", raising=False)
    return request.param


def rlayout(H, nb, p, seed, diag=False):
    lay = (np.random.default_rng(seed).random((H, nb, nb)) < p).astype(np.uint8)
    if diag:
        lay[:, np.arange(nb), np.arange(nb)] = 1
    if nb > 3:
        lay[0, 2, :] = 0   # an empty block-row
        lay[0, :, 1] = 0   # an empty block-column
    return lay


def randn(shape, dtype, seed):
    return W.randn(shape, {torch.float32: "f32", torch.bfloat16: "bf16", torch.float16: "f16"}[dtype], seed)


# ----------------------------------------------------------- softmax ----

@pytest.mark.parametrize("B", [16, 32, 64, 128])
@pytest.mark.parametrize("dt", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("kind", [0, 1, 2])
def test_softmax(bsp, oracle, B, dt, kind):
    dtype = DTYPES[dt]
    H, Z = 2, 2
    nb = max(3, 512 // B) + 1
    S = nb * B
    lay = rlayout(H, nb, 0.4, B + kind, diag=True)
    L = bsp.bsp_layout_compile(lay, B)
    mask = W.random_mask(S, 0.8, 3) if kind == 1 else None
    X = randn((Z, L.nnz, B, B), dtype, 10 + B)
    Y = bsp.bsp_softmax(L, dev(X), scale=0.3, mask_kind=kind,
                        mask=None if mask is None else dev(torch.from_numpy(mask)))
    torch.cuda.synchronize()
    want = oracle.softmax(lay, B, X, 0.3, kind, mask)
    assert_close(to_np(Y), want, dtype, f"softmax B={B} {dt} kind={kind}", rel=PROB_TOL[dtype],
                 zeros=softmax_zero_positions(lay, B, Z, kind, mask))
    assert bsp.bsp_status_check(L) == 0


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("nb", [80, 100])
def test_softmax_long_rows_and_in_place(bsp, oracle, dt, nb):
    # rows at and past the register-resident limit (two-pass online path)
    dtype = DTYPES[dt]
    B, H = 16, 1
    lay = np.ones((H, nb, nb), np.uint8)
    lay[0, 5, 7:] = 0
    L = bsp.bsp_layout_compile(lay, B)
    X = randn((1, L.nnz, B, B), dtype, 21)
    Xd = dev(X)
    bsp.bsp_softmax(L, Xd, Xd, scale=1.7, mask_kind=2)
    torch.cuda.synchronize()
    want = oracle.softmax(lay, B, X, 1.7, 2)
    assert_close(to_np(Xd), want, dtype, f"softmax long/in-place nb={nb}", rel=PROB_TOL[dtype],
                 zeros=softmax_zero_positions(lay, B, 1, 2))


@pytest.mark.parametrize("B,dt,nb,kind", [(128, "bf16", 260, 0), (128, "bf16", 260, 2),
                                           (16, "f32", 1040, 0), (16, "f32", 1040, 1), (16, "f32", 1040, 2)])
def test_softmax_rows_longer_than_a_chunk(bsp, oracle, B, dt, nb, kind):
    # one block-row holds every block, so its rows exceed the largest softmax
    # chunk (64 KB) and the whole layout takes the one-warp-per-row kernel
    # (online pass and normalising pass for the long rows, registers for the
    # others); sampled rows against the oracle
    dtype = DTYPES[dt]
    S = nb * B
    assert S * torch.tensor([], dtype=dtype).element_size() > 64 * 1024
    lay = np.eye(nb, dtype=np.uint8)[None].copy()
    lay[0, nb // 2, :] = 1
    lay[0, 3, :5] = 1
    L = bsp.bsp_layout_compile(lay, B)
    X = randn((1, L.nnz, B, B), dtype, 31)
    mask = None
    if kind == 1:
        mask = (np.random.default_rng(4).integers(0, 5, size=(S, S), dtype=np.uint8) != 0).astype(np.uint8)
    Y = bsp.bsp_softmax(L, dev(X), scale=0.6, mask_kind=kind,
                        mask=None if mask is None else dev(torch.from_numpy(mask)))
    torch.cuda.synchronize()
    assert bsp.bsp_status_check(L) == 0
    i_long = nb // 2
    sel = sorted({0, B - 1, 3 * B, 3 * B + B - 1, S - 1, i_long * B, i_long * B + 1,
                  i_long * B + B // 2, i_long * B + B - 1} |
                 set(np.random.default_rng(5).choice(S, size=8, replace=False).tolist()))
    sel = np.array(sel, dtype=np.int64)
    want = oracle.softmax_rows(lay, B, X, 0.6, kind, mask, sel=sel)
    ids = -np.ones(lay.shape, np.int64)
    hs, is_, js = np.nonzero(lay)
    ids[hs, is_, js] = np.arange(hs.size)
    Yh = to_np(Y)
    got = np.zeros_like(want)
    for t, r in enumerate(sel):
        i, a = divmod(int(r), B)
        for j in np.flatnonzero(lay[0, i]):
            got[t, j * B:(j + 1) * B] = Yh[0, ids[0, i, j], a]
    # zeros of the dense rows: outside the row's blocks, masked, or the row keeps nothing
    keep = np.ones((sel.size, S), dtype=bool)
    for t, r in enumerate(sel):
        keep[t] = np.repeat(lay[0, int(r) // B].astype(bool), B)
        if kind == 1:
            keep[t] &= mask[int(r)].astype(bool)
        elif kind == 2:
            keep[t] &= (np.arange(S) // B != int(r) // B) | (np.arange(S) <= int(r))
    keep &= keep.any(axis=1, keepdims=True)
    assert_close(got, want, dtype, f"softmax rows > 64 KB B={B} {dt} kind={kind}", rel=PROB_TOL[dtype],
                 zeros=~keep)


# --------------------------------------------------------------- SDD ----

@pytest.mark.parametrize("B", [16, 32, 64, 128])
@pytest.mark.parametrize("dt", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("trans", [(0, 1), (0, 0), (1, 0), (1, 1)])
def test_sdd(bsp, oracle, path, B, dt, trans):
    dtype = DTYPES[dt]
    ta, tb = trans
    Z, H, K = 2, 3, 64 if B < 128 else 128
    nb = max(3, 384 // B) + 1
    S = nb * B
    lay = rlayout(H, nb, 0.35, B, diag=True)
    L = bsp.bsp_layout_compile(lay, B)
    A = randn((Z, H, K, S) if ta else (Z, H, S, K), dtype, 31)
    Bm = randn((Z, H, S, K) if tb else (Z, H, K, S), dtype, 32)
    C = bsp.bsp_sdd(L, dev(A), dev(Bm), trans_a=ta, trans_b=tb)
    torch.cuda.synchronize()
    want = oracle.sdd(lay, B, A, Bm, ta, tb)
    mag = oracle.sdd(lay, B, A.abs(), Bm.abs(), ta, tb)
    assert_close(to_np(C), want, dtype, f"sdd B={B} {dt} trans={trans} {path}", mag=mag, acc=gamma(K))


@pytest.mark.parametrize("B", [32, 128])
@pytest.mark.parametrize("K", [16, 40, 48, 96, 128])
@pytest.mark.parametrize("trans", [(0, 1), (0, 0), (1, 0), (1, 1)])
def test_sdd_contraction_lengths(bsp, oracle, path, B, K, trans):
    # the tensor-core kernel takes an operand stored [K][S] for K a multiple
    # of 16 (K = 40 runs on the CUDA cores); ragged last row tile (S = 5 * 64
    # or 3 * 128 + ... rows)
    dtype = torch.bfloat16
    ta, tb = trans
    Z, H = 1, 2
    nb = 10 if B == 32 else 5
    S = nb * B
    lay = rlayout(H, nb, 0.4, B + K, diag=True)
    L = bsp.bsp_layout_compile(lay, B)
    A = randn((Z, H, K, S) if ta else (Z, H, S, K), dtype, 33)
    Bm = randn((Z, H, S, K) if tb else (Z, H, K, S), dtype, 34)
    C = bsp.bsp_sdd(L, dev(A), dev(Bm), trans_a=ta, trans_b=tb)
    torch.cuda.synchronize()
    assert_close(to_np(C), oracle.sdd(lay, B, A, Bm, ta, tb), dtype, f"sdd B={B} K={K} trans={trans} {path}",
                 mag=oracle.sdd(lay, B, A.abs(), Bm.abs(), ta, tb), acc=gamma(K))


@pytest.mark.parametrize("B", [16, 32, 64, 128])
@pytest.mark.parametrize("dt", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("kind", [0, 1, 2])
def test_sdd_softmax(bsp, oracle, path, B, dt, kind):
    # fused SDD + softmax against the oracle's softmax of its SDD (fp64); the
    # tensor-core path keeps the scores in fp32, the fallback rounds them to
    # the dtype between the two steps
    dtype = DTYPES[dt]
    Z, H, K = 2, 3, 64 if B < 128 else 128
    nb = max(3, 384 // B) + 1
    S = nb * B
    lay = rlayout(H, nb, 0.35, 3 * B + kind, diag=True)
    L = bsp.bsp_layout_compile(lay, B)
    A, Bm = randn((Z, H, S, K), dtype, 35), randn((Z, H, S, K), dtype, 36)
    mask = W.random_mask(S, 0.7, 37) if kind == 1 else None
    P = bsp.bsp_sdd_softmax(L, dev(A), dev(Bm), scale=0.2, mask_kind=kind,
                            mask=None if mask is None else dev(torch.from_numpy(mask)))
    torch.cuda.synchronize()
    s_ref = oracle.sdd(lay, B, A, Bm)
    want = oracle.softmax(lay, B, s_ref, 0.2, kind, mask)
    rel = softmax_rel_bound(lay, B, s_ref, oracle.sdd(lay, B, A.abs(), Bm.abs()), 0.2, K, dtype,
                            scores_rounded=(path == "simt"))
    assert_close(to_np(P), want, dtype, f"sdd_softmax B={B} {dt} kind={kind} {path}", rel=rel,
                 zeros=softmax_zero_positions(lay, B, Z, kind, mask))
    assert bsp.bsp_status_check(L) == 0


@pytest.mark.parametrize("trans", [(0, 0), (1, 0), (1, 1)])
def test_sdd_softmax_orientations(bsp, oracle, path, trans):
    ta, tb = trans
    B, Z, H, K, nb = 64, 1, 2, 64, 7
    S = nb * B
    lay = rlayout(H, nb, 0.4, 90, diag=True)
    L = bsp.bsp_layout_compile(lay, B)
    A = randn((Z, H, K, S) if ta else (Z, H, S, K), torch.bfloat16, 38)
    Bm = randn((Z, H, S, K) if tb else (Z, H, K, S), torch.bfloat16, 39)
    P = bsp.bsp_sdd_softmax(L, dev(A), dev(Bm), scale=0.15, mask_kind=2, trans_a=ta, trans_b=tb)
    torch.cuda.synchronize()
    s_ref = oracle.sdd(lay, B, A, Bm, ta, tb)
    want = oracle.softmax(lay, B, s_ref, 0.15, 2)
    rel = softmax_rel_bound(lay, B, s_ref, oracle.sdd(lay, B, A.abs(), Bm.abs(), ta, tb), 0.15, K,
                            torch.bfloat16, scores_rounded=(path == "simt"))
    assert_close(to_np(P), want, torch.bfloat16, f"sdd_softmax trans={trans} {path}", rel=rel,
                 zeros=softmax_zero_positions(lay, B, Z, 2))


def test_sdd_leaves_absent_blocks_untouched(bsp, path):
    # the output has exactly nnz blocks; guard regions around it keep a canary
    B, H, nb, Z, K = 64, 2, 6, 2, 64
    lay = rlayout(H, nb, 0.3, 5, diag=True)
    L = bsp.bsp_layout_compile(lay, B)
    n = Z * L.nnz * B * B
    guard = 4096
    buf = torch.full((n + 2 * guard,), float("nan"), dtype=torch.bfloat16, device="cuda")
    C = buf[guard:guard + n].view(Z, L.nnz, B, B)
    A = dev(randn((Z, H, nb * B, K), torch.bfloat16, 6))
    bsp.bsp_sdd(L, A, A, C)
    torch.cuda.synchronize()
    assert torch.isnan(buf[:guard]).all() and torch.isnan(buf[guard + n:]).all()
    assert torch.isfinite(C).all()


# --------------------------------------------------------------- DSD ----

@pytest.mark.parametrize("B", [16, 32, 64, 128])
@pytest.mark.parametrize("dt", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("trans", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("N", [200, 72])
def test_dsd(bsp, oracle, path, B, dt, trans, N):
    dtype = DTYPES[dt]
    ta, tb = trans
    Z, H = 2, 2  # N not a multiple of the column tile; 72 takes the 128-wide tile
    nb = max(3, 384 // B) + 1
    S = nb * B
    lay = rlayout(H, nb, 0.35, 40 + B)
    L = bsp.bsp_layout_compile(lay, B)
    Asp = randn((Z, L.nnz, B, B), dtype, 41)
    Bd = randn((Z, H, N, S) if tb else (Z, H, S, N), dtype, 42)
    C = bsp.bsp_dsd(L, dev(Asp), dev(Bd), trans_a=ta, trans_b=tb)
    torch.cuda.synchronize()
    want = oracle.dsd(lay, B, Asp, Bd, ta, tb)
    mag = oracle.dsd(lay, B, Asp.abs(), Bd.abs(), ta, tb)
    assert_close(to_np(C), want, dtype, f"dsd B={B} {dt} trans={trans} {path}", mag=mag, acc=gamma(S))


# --------------------------------------------------------------- DDS ----

@pytest.mark.parametrize("B", [16, 32, 64, 128])
@pytest.mark.parametrize("dt", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("trans", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("M", [200, 72])
def test_dds(bsp, oracle, path, B, dt, trans, M):
    dtype = DTYPES[dt]
    ta, tb = trans
    Z, H = 2, 2
    nb = max(3, 384 // B) + 1
    S = nb * B
    lay = rlayout(H, nb, 0.35, 50 + B)
    L = bsp.bsp_layout_compile(lay, B)
    Bsp = randn((Z, L.nnz, B, B), dtype, 51)
    Ad = randn((Z, H, S, M) if ta else (Z, H, M, S), dtype, 52)
    C = bsp.bsp_dds(L, dev(Ad), dev(Bsp), trans_a=ta, trans_b=tb)
    torch.cuda.synchronize()
    want = oracle.dds(lay, B, Ad, Bsp, ta, tb)
    mag = oracle.dds(lay, B, Ad.abs(), Bsp.abs(), ta, tb)
    assert_close(to_np(C), want, dtype, f"dds B={B} {dt} trans={trans} {path}", mag=mag, acc=gamma(S))


# --------------------------------------------------------- attention ----

@pytest.mark.parametrize("B", [16, 32, 64, 128])
@pytest.mark.parametrize("dt", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("kind", [0, 1, 2])
def test_attention(bsp, oracle, path, B, dt, D, kind):
    dtype = DTYPES[dt]
    Z, H = 2, 2
    nb = max(3, 512 // B) + 1
    S = nb * B
    lay = rlayout(H, nb, 0.3, 60 + B + kind, diag=(kind == 2))
    L = bsp.bsp_layout_compile(lay, B)
    mask = W.random_mask(S, 0.8, 61) if kind == 1 else None
    Q, K, V = (randn((Z, H, S, D), dtype, 62 + k) for k in range(3))
    scale = 1.0 / np.sqrt(D)
    O = bsp.bsp_attention(L, dev(Q), dev(K), dev(V), scale=scale, mask_kind=kind,
                          mask=None if mask is None else dev(torch.from_numpy(mask)))
    torch.cuda.synchronize()
    want = oracle.attention(lay, B, Q, K, V, scale, kind, mask)
    mag = oracle.attention(lay, B, Q, K, V.abs(), scale, kind, mask)
    assert_close(to_np(O), want, dtype, f"attention B={B} {dt} D={D} kind={kind} {path}", mag=mag,
                 acc=attention_acc(Q, K, scale, dtype, S))
    assert bsp.bsp_status_check(L) == 0


@pytest.mark.parametrize("B", [16, 64])
@pytest.mark.parametrize("dt", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("D", [16, 32, 96])
@pytest.mark.parametrize("kind", [0, 2])
def test_attention_other_head_sizes(bsp, oracle, B, dt, D, kind):
    # head sizes outside the tensor-core kernels' (64, 128) take the CUDA-core
    # kernel; its O and log-sum-exp against the oracle's
    dtype = DTYPES[dt]
    Z, H = 2, 2
    nb = max(3, 384 // B) + 1
    S = nb * B
    lay = rlayout(H, nb, 0.3, 90 + B + kind, diag=(kind == 2))
    L = bsp.bsp_layout_compile(lay, B)
    Q, K, V = (randn((Z, H, S, D), dtype, 92 + k) for k in range(3))
    scale = 1.0 / np.sqrt(D)
    O, lse = bsp.bsp_attention_lse(L, dev(Q), dev(K), dev(V), None, None, scale, kind)
    O0 = bsp.bsp_attention(L, dev(Q), dev(K), dev(V), scale=scale, mask_kind=kind)
    torch.cuda.synchronize()
    assert bsp.bsp_status_check(L) == 0
    assert torch.equal(O, O0), "bsp_attention_lse's O differs from bsp_attention's"
    want = oracle.attention(lay, B, Q, K, V, scale, kind, None)
    mag = oracle.attention(lay, B, Q, K, V.abs(), scale, kind, None)
    assert_close(to_np(O), want, dtype, f"attention B={B} {dt} D={D} kind={kind}", mag=mag,
                 acc=attention_acc(Q, K, scale, dtype, S))
    wl = oracle.attention_lse(lay, B, Q, K, scale, kind, None)
    got = lse.cpu().double().numpy()
    empty = np.isneginf(wl)
    assert np.all(np.isneginf(got[empty]))
    qn = Q.double().norm(dim=-1)
    kmax = K.double().norm(dim=-1).amax(dim=-1, keepdim=True)
    bound = (scale * gamma(D) * qn * kmax + (S + 4) * 2.0 ** -22).numpy() + 2.0 ** -22 * np.abs(wl)
    err = np.abs(got[~empty] - wl[~empty])
    assert np.all(err <= bound[~empty]), f"lse B={B} {dt} D={D} kind={kind}: {err.max():.3e}"


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_unfused_chain_matches_oracle(bsp, oracle, dt):
    dtype = DTYPES[dt]
    B, H, Z, D = 64, 2, 2, 64
    nb = 7
    lay = rlayout(H, nb, 0.4, 70, diag=True)
    L = bsp.bsp_layout_compile(lay, B)
    Q, K, V = (randn((Z, H, nb * B, D), dtype, 71 + k) for k in range(3))
    O = bsp.attention_unfused(L, dev(Q), dev(K), dev(V), 0.125, 2)
    torch.cuda.synchronize()
    want = oracle.attention(lay, B, Q, K, V, 0.125, 2)
    mag = oracle.attention(lay, B, Q, K, V.abs(), 0.125, 2)
    # the chain rounds the scores and P to the data type between its steps
    assert_close(to_np(O), want, dtype, "unfused chain", mag=mag,
                 acc=attention_acc(Q, K, 0.125, dtype, nb * B, scores_rounded=True))


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("where", ["host", "device"])
def test_attention_batch_sizes_on_one_handle(bsp, oracle, dt, where):
    # the tensor-core kernels keep one work schedule per batch size: calls of
    # changing Z on one handle (a handle compiled on the host, or on the
    # device, whose schedule is built from tables read back) each match the
    # oracle, and a repeated Z gives the same bytes
    dtype = DTYPES[dt]
    B, H, D = 64, 3, 64
    nb = 9
    lay = rlayout(H, nb, 0.35, 90, diag=True)
    lay[1, 0, :] = 1  # one long block-row
    L = (bsp.bsp_layout_compile(lay, B) if where == "host"
         else bsp.bsp_layout_compile_device(torch.from_numpy(lay).cuda(), B))
    first = {}
    for Z in (3, 1, 2, 3, 1):
        Q, K, V = (randn((Z, H, nb * B, D), dtype, 91 + k) for k in range(3))
        O = bsp.bsp_attention(L, dev(Q), dev(K), dev(V), scale=0.125, mask_kind=2)
        torch.cuda.synchronize()
        assert bsp.bsp_status_check(L) == 0
        if Z in first:
            assert torch.equal(O.cpu(), first[Z]), f"Z={Z} repeated"
            continue
        first[Z] = O.cpu()
        want = oracle.attention(lay, B, Q, K, V, 0.125, 2)
        mag = oracle.attention(lay, B, Q, K, V.abs(), 0.125, 2)
        assert_close(to_np(O), want, dtype, f"attention Z={Z} {dt} {where}", mag=mag,
                     acc=attention_acc(Q, K, 0.125, dtype, nb * B))


@pytest.mark.parametrize("B", [16, 64, 128])
@pytest.mark.parametrize("dt", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("kind", [0, 1, 2])
@pytest.mark.parametrize("cut", [1, 3])
def test_attention_cut_tiles(bsp, oracle, B, dt, kind, cut):
    # long block-rows cut into pieces of at most `cut` steps, merged by the
    # combine pass: the oracle's result, the same bytes on a second call
    # (the merge order is fixed), and the result without cuts for balance
    # within the tolerance
    dtype = DTYPES[dt]
    Z, H, D = 2, 3, 64
    nb = max(4, 1024 // B) + 1
    S = nb * B
    lay = rlayout(H, nb, 0.25, 95 + B + kind, diag=(kind == 2))
    lay[0, 0, :] = 1           # a long first block-row
    lay[2, nb - 1, :] = 1      # and a long last one (ragged tile)
    if kind == 2:
        lay[:, np.arange(nb), np.arange(nb)] = 1
    L = bsp.bsp_layout_compile(lay, B)
    mask = W.random_mask(S, 0.8, 96) if kind == 1 else None
    dmask = None if mask is None else dev(torch.from_numpy(mask))
    Q, K, V = (randn((Z, H, S, D), dtype, 97 + k) for k in range(3))
    q, k, v = dev(Q), dev(K), dev(V)
    bsp.bsp_diag_attention_split(L, cut)
    sc = bsp.bsp_diag_attention_schedule(L, Z, torch.cuda.get_device_properties(0).multi_processor_count, dtype)
    assert len(sc["combine"]) > 0
    O1 = bsp.bsp_attention(L, q, k, v, scale=0.125, mask_kind=kind, mask=dmask)
    O2 = bsp.bsp_attention(L, q, k, v, scale=0.125, mask_kind=kind, mask=dmask)
    bsp.bsp_diag_attention_split(L, -1)
    O0 = bsp.bsp_attention(L, q, k, v, scale=0.125, mask_kind=kind, mask=dmask)
    # the combine pass also writes the cut rows' log-sum-exp
    bsp.bsp_diag_attention_split(L, cut)
    _, lse = bsp.bsp_attention_lse(L, q, k, v, None, None, 0.125, kind, dmask)
    torch.cuda.synchronize()
    assert bsp.bsp_status_check(L) == 0
    assert torch.equal(O1, O2)
    want_lse = oracle.attention_lse(lay, B, Q, K, 0.125, kind, mask)
    kept = ~np.isneginf(want_lse)
    got_lse = lse.cpu().double().numpy()
    assert np.all(np.isneginf(got_lse[~kept]))
    assert np.abs(got_lse[kept] - want_lse[kept]).max() < 1e-3, "lse of cut tiles"
    want = oracle.attention(lay, B, Q, K, V, 0.125, kind, mask)
    mag = oracle.attention(lay, B, Q, K, V.abs(), 0.125, kind, mask)
    acc = attention_acc(Q, K, 0.125, dtype, S)
    assert_close(to_np(O1), want, dtype, f"cut tiles B={B} {dt} kind={kind} cut={cut}", mag=mag, acc=acc)
    assert_close(to_np(O0), want, dtype, f"uncut B={B} {dt} kind={kind}", mag=mag, acc=acc)


def test_attention_cut_tiles_two_streams(bsp, oracle):
    # two streams sharing one handle whose schedule cuts tiles: the workspace
    # is taken in turn, both results equal the single-stream one
    B, Z, H, D = 64, 2, 2, 64
    nb = 17
    lay = rlayout(H, nb, 0.3, 98, diag=True)
    lay[:, 0, :] = 1
    L = bsp.bsp_layout_compile(lay, B)
    bsp.bsp_diag_attention_split(L, 2)
    Q, K, V = (randn((Z, H, nb * B, D), torch.bfloat16, 99 + k) for k in range(3))
    Q2 = randn((Z, H, nb * B, D), torch.bfloat16, 102)
    q, k, v, q2 = dev(Q), dev(K), dev(V), dev(Q2)
    ref1 = bsp.bsp_attention(L, q, k, v, scale=0.125, mask_kind=2)
    ref2 = bsp.bsp_attention(L, q2, k, v, scale=0.125, mask_kind=2)
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    outs = []
    for _ in range(8):
        o1, o2 = torch.empty_like(q), torch.empty_like(q)
        bsp.bsp_attention(L, q, k, v, o1, 0.125, 2, stream=s1)
        bsp.bsp_attention(L, q2, k, v, o2, 0.125, 2, stream=s2)
        outs.append((o1, o2))
    torch.cuda.synchronize()
    assert bsp.bsp_status_check(L) == 0
    for o1, o2 in outs:
        assert torch.equal(o1, ref1) and torch.equal(o2, ref2)
    want = oracle.attention(lay, B, Q, K, V, 0.125, 2)
    assert_close(to_np(ref1), want, torch.bfloat16, "cut tiles, two streams")


def test_edge_empty_layout_and_zero_batch(bsp, oracle):
    B, H, nb, D = 64, 2, 4, 64
    lay = np.zeros((H, nb, nb), np.uint8)
    L = bsp.bsp_layout_compile(lay, B)
    Q = torch.randn(1, H, nb * B, D, device="cuda", dtype=torch.bfloat16)
    O = torch.full_like(Q, 7.0)
    bsp.bsp_attention(L, Q, Q, Q, O, scale=0.1)
    torch.cuda.synchronize()
    assert (O == 0).all()  # no kept entries: rows are 0
    C = torch.full((1, H, nb * B, 32), 5.0, device="cuda", dtype=torch.bfloat16)
    bsp.bsp_dsd(L, torch.zeros(1, 1, B, B, device="cuda", dtype=torch.bfloat16),
                torch.randn(1, H, nb * B, 32, device="cuda", dtype=torch.bfloat16), C)
    torch.cuda.synchronize()
    assert (C == 0).all()
    # Z = 0 is a no-op
    empty = torch.empty(0, H, nb * B, D, device="cuda", dtype=torch.bfloat16)
    bsp.bsp_attention(L, empty, empty, empty, empty, scale=0.1)


def test_error_codes_on_device(bsp):
    B, H, nb = 32, 1, 4
    L = bsp.bsp_layout_compile(np.ones((H, nb, nb), np.uint8), B)
    Q = torch.randn(1, H, nb * B, 64, device="cuda", dtype=torch.bfloat16)
    with pytest.raises(bsp.BspError) as e:   # D not a multiple of 16
        bsp.bsp_attention(L, Q[..., :40].contiguous(), Q[..., :40].contiguous(),
                          Q[..., :40].contiguous(), scale=0.1)
    assert e.value.code == -1
    raw = torch.empty(Q.numel() * 2 + 8, dtype=torch.bfloat16, device="cuda")
    mis = raw[1:1 + Q.numel()].view_as(Q)    # 2-byte offset: not 16-byte aligned
    with pytest.raises(bsp.BspError) as e:
        bsp.bsp_attention(L, mis, Q, Q, scale=0.1)
    assert e.value.code == -3
    with pytest.raises(bsp.BspError) as e:   # dense mask kind without a mask
        bsp.bsp_softmax(L, torch.empty(1, L.nnz, B, B, device="cuda"), scale=1.0, mask_kind=1)
    assert e.value.code == -1


def test_device_luts_bit_exact(bsp, oracle):
    for w in W.ATTENTION_WORKLOADS.values():
        lay = w.layout()
        L = bsp.bsp_layout_compile(lay, w.B)
        got, want = L.luts(), oracle.luts(lay)
        for k in want:
            assert np.array_equal(got[k], want[k]), (w.name, k)
