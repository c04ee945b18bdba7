"""Pins for the fp64 oracle: library routines on special cases, closed forms
and invariants.  None of these re-types the oracle's own loops.

Passages the pins follow:
 - "question on blocksparse" (openai/triton issue 117): SDD / DSD / DDS
   definitions, 0/1 block layout, block softmax equal to the dense softmax of
   the present entries, dense masks for diagonal blocks;
 - Triton-Puzzles blog, Puzzle 8 (stable softmax) and Puzzle 9 (attention as a
   softmax-weighted sum of value rows).
"""

import numpy as np
import pytest
from scipy.special import softmax as sp_softmax

import libref
from sparse_attention_layout_gb300 import workloads as W

RNG = np.random.default_rng(1234)


def rand(*shape, seed=0):
    return np.random.default_rng(seed).standard_normal(shape).astype(np.float32)


def random_layout(H, nb, p, seed):
    """Random layout that is guaranteed to contain an empty block-row and an
    empty block-column in head 0 (when nb > 2)."""
    lay = (np.random.default_rng(seed).random((H, nb, nb)) < p).astype(np.uint8)
    if nb > 2:
        lay[0, 1, :] = 0
        lay[0, :, 2] = 0
    return lay


# ---------------------------------------------------------------- LUTs ----

@pytest.mark.parametrize("H,nb,p,seed", [(1, 1, 1.0, 0), (2, 5, 0.4, 1), (3, 8, 0.25, 2),
                                         (1, 16, 0.0, 3), (2, 7, 1.0, 4)])
def test_luts_match_numpy_enumeration(oracle, H, nb, p, seed):
    lay = random_layout(H, nb, p, seed)
    L = oracle.luts(lay)
    nnz = int(lay.sum())
    assert oracle.nnz(lay) == nnz
    # CSR: np.nonzero enumerates (h, i, j) in row-major order = block-id order
    hs, is_, js = np.nonzero(lay)
    assert np.array_equal(L["col_idx"], js.astype(np.int32))
    assert np.array_equal(L["blk_id"], np.arange(nnz, dtype=np.int32))
    counts = lay.sum(axis=2)  # [H, nb]
    for h in range(H):
        start = counts[:h].sum()
        want = start + np.concatenate([[0], np.cumsum(counts[h])])
        assert np.array_equal(L["row_ptr"][h * (nb + 1):(h + 1) * (nb + 1)], want)
    # CSC: nonzero of the per-head transpose enumerates (h, j, i)
    ids = -np.ones(lay.shape, dtype=np.int64)
    ids[hs, is_, js] = np.arange(nnz)
    ht, jt, it = np.nonzero(np.transpose(lay, (0, 2, 1)))
    assert np.array_equal(L["row_idx"], it.astype(np.int32))
    assert np.array_equal(L["blk_id_csc"], ids[ht, it, jt].astype(np.int32))
    ccounts = lay.sum(axis=1)
    for h in range(H):
        start = ccounts[:h].sum()
        want = start + np.concatenate([[0], np.cumsum(ccounts[h])])
        assert np.array_equal(L["col_ptr"][h * (nb + 1):(h + 1) * (nb + 1)], want)
    # CSR and CSC describe the same set; blk_id_csc is a permutation
    assert np.array_equal(np.sort(L["blk_id_csc"]), np.arange(nnz))


# ----------------------------------------------------------------- SDD ----

@pytest.mark.parametrize("trans_a,trans_b", [(0, 1), (0, 0), (1, 0), (1, 1)])
def test_sdd_matches_numpy_matmul(oracle, trans_a, trans_b):
    Z, H, nb, B, K = 2, 2, 4, 8, 12
    S = nb * B
    lay = random_layout(H, nb, 0.4, 11)
    A = rand(Z, H, K, S, seed=1) if trans_a else rand(Z, H, S, K, seed=1)
    Bm = rand(Z, H, S, K, seed=2) if trans_b else rand(Z, H, K, S, seed=2)
    opA = np.swapaxes(A, -1, -2) if trans_a else A
    opB = np.swapaxes(Bm, -1, -2) if trans_b else Bm
    full = np.matmul(opA.astype(np.float64), opB.astype(np.float64))
    want = libref.dense_to_blocks(lay, B, full)
    got = oracle.sdd(lay, B, A, Bm, trans_a, trans_b)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_sdd_single_block_is_dense_gemm(oracle):
    # B = S: one 1x1 all-ones layout, SDD is the plain GEMM A B^T
    A, Bm = rand(1, 1, 32, 16, seed=3), rand(1, 1, 32, 16, seed=4)
    got = oracle.sdd(np.ones((1, 1, 1), np.uint8), 32, A, Bm)
    np.testing.assert_allclose(got[0, 0], A[0, 0].astype(np.float64) @ Bm[0, 0].T.astype(np.float64),
                               rtol=1e-12, atol=1e-12)


def test_sdd_selection_matches_full(oracle):
    lay = random_layout(2, 4, 0.5, 5)
    A, Bm = rand(2, 2, 32, 8, seed=5), rand(2, 2, 32, 8, seed=6)
    full = oracle.sdd(lay, 8, A, Bm)
    nnz = full.shape[1]
    sel = np.array([0, nnz + 1, 2 * nnz - 1])
    got = oracle.sdd(lay, 8, A, Bm, sel=sel)
    np.testing.assert_array_equal(got, full.reshape(-1, 8, 8)[sel])


# ------------------------------------------------------------- softmax ----

def test_softmax_all_ones_is_dense_softmax(oracle):
    Z, H, nb, B = 2, 3, 4, 8
    S = nb * B
    lay = np.ones((H, nb, nb), np.uint8)
    Xd = rand(Z, H, S, S, seed=7)
    X = libref.dense_to_blocks(lay, B, Xd).astype(np.float32)
    got = libref.blocks_to_dense(lay, B, oracle.softmax(lay, B, X, 0.37))
    np.testing.assert_allclose(got, sp_softmax(0.37 * Xd.astype(np.float64), axis=-1), rtol=1e-12, atol=1e-15)


def test_softmax_block_causal_with_diag_mask_is_dense_causal(oracle):
    Z, H, nb, B = 1, 2, 5, 4
    S = nb * B
    lay = W.layout_causal_blocks(nb, H)
    Xd = rand(Z, H, S, S, seed=8)
    X = libref.dense_to_blocks(lay, B, Xd).astype(np.float32)
    got = libref.blocks_to_dense(lay, B, oracle.softmax(lay, B, X, 1.3, W.MASK_DIAG_CAUSAL))
    tril = np.tril(np.ones((S, S), bool))
    np.testing.assert_allclose(got, libref.masked_softmax(1.3 * Xd.astype(np.float64), tril),
                               rtol=1e-12, atol=1e-15)


@pytest.mark.parametrize("kind", [W.MASK_NONE, W.MASK_DENSE, W.MASK_DIAG_CAUSAL])
def test_softmax_random_layout_matches_masked_dense(oracle, kind):
    Z, H, nb, B = 2, 2, 6, 8
    S = nb * B
    lay = random_layout(H, nb, 0.35, 9)
    mask = W.random_mask(S, 0.7, 10) if kind == W.MASK_DENSE else None
    Xd = rand(Z, H, S, S, seed=11)
    X = libref.dense_to_blocks(lay, B, Xd).astype(np.float32)
    got = libref.blocks_to_dense(lay, B, oracle.softmax(lay, B, X, 0.5, kind, mask))
    M = libref.expand_mask(lay, B).astype(bool) & libref.keep_mask(S, B, kind, mask)[None]
    want = libref.masked_softmax(0.5 * Xd.astype(np.float64), M[None])
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-15)
    # rows sum to one (or zero when nothing is kept), entries are >= 0
    sums = got.sum(-1)
    kept = M.any(-1)
    np.testing.assert_allclose(sums[:, kept], 1.0, rtol=1e-12)
    assert np.all(sums[:, ~kept] == 0.0) and np.all(got >= 0)


def test_softmax_constant_input_closed_form(oracle):
    H, nb, B = 2, 6, 4
    lay = random_layout(H, nb, 0.5, 12)
    nnz = int(lay.sum())
    X = np.full((1, nnz, B, B), 3.25, np.float32)
    got = libref.blocks_to_dense(lay, B, oracle.softmax(lay, B, X, 0.9))
    M = libref.expand_mask(lay, B).astype(bool)
    count = M.sum(-1, keepdims=True)
    want = np.where(M, 1.0 / np.maximum(count, 1), 0.0)
    np.testing.assert_allclose(got[0], want, rtol=1e-14)


def test_softmax_is_stable_for_large_inputs(oracle):
    # the max is subtracted first (Puzzle 8): huge logits stay finite and equal
    # to the softmax of the shifted logits
    H, nb, B = 1, 4, 8
    lay = random_layout(H, nb, 0.6, 13)
    nnz = int(lay.sum())
    # values on a 2^-12 grid so that X + 2000 is exact in float32
    X = (np.round(rand(1, nnz, B, B, seed=14) * 4096) / 4096).astype(np.float32)
    got_big = oracle.softmax(lay, B, X + np.float32(2000.0), 1.0)
    got = oracle.softmax(lay, B, X, 1.0)
    assert np.all(np.isfinite(got_big))
    np.testing.assert_allclose(got_big, got, rtol=1e-9, atol=1e-12)


@pytest.mark.parametrize("kind", [W.MASK_NONE, W.MASK_DENSE, W.MASK_DIAG_CAUSAL])
def test_softmax_rows_matches_full(oracle, kind):
    Z, H, nb, B = 2, 2, 5, 4
    S = nb * B
    lay = random_layout(H, nb, 0.5, 15)
    nnz = int(lay.sum())
    X = rand(Z, nnz, B, B, seed=16)
    mask = W.random_mask(S, 0.7, 17) if kind == W.MASK_DENSE else None
    full = libref.blocks_to_dense(lay, B, oracle.softmax(lay, B, X, 0.8, kind, mask))
    sel = np.array([0, 7, S + 3, 2 * H * S - 1])
    got = oracle.softmax_rows(lay, B, X, 0.8, kind, mask, sel=sel)
    np.testing.assert_allclose(got, full.reshape(-1, S)[sel], rtol=1e-15, atol=0)


# ----------------------------------------------------------------- DSD ----

@pytest.mark.parametrize("trans_a,trans_b", [(0, 0), (0, 1), (1, 0), (1, 1)])
def test_dsd_matches_numpy_matmul(oracle, trans_a, trans_b):
    Z, H, nb, B, N = 2, 2, 5, 4, 6
    S = nb * B
    lay = random_layout(H, nb, 0.4, 17)
    nnz = int(lay.sum())
    Asp = rand(Z, nnz, B, B, seed=18)
    Bd = rand(Z, H, N, S, seed=19) if trans_b else rand(Z, H, S, N, seed=19)
    Ad = libref.blocks_to_dense(lay, B, Asp)
    opA = np.swapaxes(Ad, -1, -2) if trans_a else Ad
    opB = np.swapaxes(Bd, -1, -2) if trans_b else Bd
    want = np.matmul(opA, opB.astype(np.float64))
    got = oracle.dsd(lay, B, Asp, Bd, trans_a, trans_b)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_dsd_identity_blocks_give_dense_operand(oracle):
    H, nb, B, N = 2, 4, 8, 5
    lay = np.broadcast_to(np.eye(nb, dtype=np.uint8), (H, nb, nb)).copy()
    Asp = np.broadcast_to(np.eye(B, dtype=np.float32), (1, H * nb, B, B)).copy()
    Bd = rand(1, H, nb * B, N, seed=20)
    np.testing.assert_array_equal(oracle.dsd(lay, B, Asp, Bd), Bd.astype(np.float64))


def test_dsd_empty_rows_are_zero(oracle):
    lay = random_layout(1, 6, 0.5, 21)  # block-row 1 is empty
    nnz = int(lay.sum())
    got = oracle.dsd(lay, 4, rand(1, nnz, 4, 4, seed=22), rand(1, 1, 24, 3, seed=23))
    assert np.all(got[0, 0, 4:8] == 0.0)


# ----------------------------------------------------------------- DDS ----

@pytest.mark.parametrize("trans_a,trans_b", [(0, 0), (0, 1), (1, 0), (1, 1)])
def test_dds_matches_numpy_matmul(oracle, trans_a, trans_b):
    Z, H, nb, B, M = 2, 2, 5, 4, 7
    S = nb * B
    lay = random_layout(H, nb, 0.4, 24)
    nnz = int(lay.sum())
    Bsp = rand(Z, nnz, B, B, seed=25)
    Ad = rand(Z, H, S, M, seed=26) if trans_a else rand(Z, H, M, S, seed=26)
    Bdn = libref.blocks_to_dense(lay, B, Bsp)
    opA = np.swapaxes(Ad, -1, -2) if trans_a else Ad
    opB = np.swapaxes(Bdn, -1, -2) if trans_b else Bdn
    want = np.matmul(opA.astype(np.float64), opB)
    got = oracle.dds(lay, B, Ad, Bsp, trans_a, trans_b)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_dds_empty_cols_are_zero(oracle):
    lay = random_layout(1, 6, 0.5, 27)  # block-column 2 is empty
    nnz = int(lay.sum())
    got = oracle.dds(lay, 4, rand(1, 1, 5, 24, seed=28), rand(1, nnz, 4, 4, seed=29))
    assert np.all(got[0, 0, :, 8:12] == 0.0)


@pytest.mark.parametrize("trans_a,trans_b", [(0, 0), (1, 1)])
def test_dsd_dds_selection_matches_full(oracle, trans_a, trans_b):
    # the sampled-row forms used by the full-size GPU tests
    Z, H, nb, B, N = 2, 2, 5, 4, 6
    S = nb * B
    lay = random_layout(H, nb, 0.4, 30)
    nnz = int(lay.sum())
    Sp = rand(Z, nnz, B, B, seed=31)
    Bd = rand(Z, H, N, S, seed=32) if trans_b else rand(Z, H, S, N, seed=32)
    full = oracle.dsd(lay, B, Sp, Bd, trans_a, trans_b)
    sel = np.array([0, 9, S + 4, Z * H * S - 1])
    np.testing.assert_array_equal(oracle.dsd(lay, B, Sp, Bd, trans_a, trans_b, sel=sel), full.reshape(-1, N)[sel])
    Ad = rand(Z, H, S, N, seed=33) if trans_a else rand(Z, H, N, S, seed=33)
    full = oracle.dds(lay, B, Ad, Sp, trans_a, trans_b)
    sel = np.array([0, 5, N + 1, Z * H * N - 1])
    np.testing.assert_array_equal(oracle.dds(lay, B, Ad, Sp, trans_a, trans_b, sel=sel), full.reshape(-1, S)[sel])


# ----------------------------------------------------------- attention ----

def test_attention_all_ones_is_dense_attention(oracle):
    Z, H, S, D, B = 2, 2, 32, 16, 8
    lay = np.ones((H, S // B, S // B), np.uint8)
    Q, K, V = rand(Z, H, S, D, seed=30), rand(Z, H, S, D, seed=31), rand(Z, H, S, D, seed=32)
    got = oracle.attention(lay, B, Q, K, V, 0.25)
    want = libref.dense_attention(Q, K, V, 0.25, np.ones((S, S), bool))
    np.testing.assert_allclose(got, want, rtol=1e-11, atol=1e-12)


def test_attention_block_causal_with_diag_mask_is_causal_attention(oracle):
    Z, H, S, D, B = 1, 2, 48, 8, 16
    lay = W.layout_causal_blocks(S // B, H)
    Q, K, V = rand(Z, H, S, D, seed=33), rand(Z, H, S, D, seed=34), rand(Z, H, S, D, seed=35)
    got = oracle.attention(lay, B, Q, K, V, 0.3, W.MASK_DIAG_CAUSAL)
    want = libref.dense_attention(Q, K, V, 0.3, np.tril(np.ones((S, S), bool)))
    np.testing.assert_allclose(got, want, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("kind", [W.MASK_NONE, W.MASK_DENSE, W.MASK_DIAG_CAUSAL])
def test_attention_random_layout_matches_masked_dense(oracle, kind):
    Z, H, S, D, B = 2, 2, 48, 8, 8
    lay = random_layout(H, S // B, 0.3, 36)
    mask = W.random_mask(S, 0.6, 37) if kind == W.MASK_DENSE else None
    Q, K, V = rand(Z, H, S, D, seed=38), rand(Z, H, S, D, seed=39), rand(Z, H, S, D, seed=40)
    M = libref.expand_mask(lay, B).astype(bool) & libref.keep_mask(S, B, kind, mask)[None]
    got = oracle.attention(lay, B, Q, K, V, 0.7, kind, mask)
    want = libref.dense_attention(Q, K, V, 0.7, M[None])
    np.testing.assert_allclose(got, want, rtol=1e-11, atol=1e-12)


def test_attention_zero_query_gives_mean_of_values(oracle):
    Z, H, S, D, B = 1, 2, 40, 6, 8
    lay = random_layout(H, S // B, 0.5, 41)
    Q = np.zeros((Z, H, S, D), np.float32)
    K, V = rand(Z, H, S, D, seed=42), rand(Z, H, S, D, seed=43)
    got = oracle.attention(lay, B, Q, K, V, 1.0)
    M = libref.expand_mask(lay, B).astype(np.float64)  # [H, S, S]
    cnt = M.sum(-1, keepdims=True)
    want = np.where(cnt > 0, np.matmul(M, V[0].astype(np.float64)) / np.maximum(cnt, 1), 0.0)
    np.testing.assert_allclose(got[0], want, rtol=1e-12, atol=1e-13)


def test_attention_unit_values_give_ones(oracle):
    Z, H, S, D, B = 1, 1, 32, 4, 8
    lay = random_layout(H, S // B, 0.5, 44)
    Q, K = rand(Z, H, S, D, seed=45), rand(Z, H, S, D, seed=46)
    V = np.ones((Z, H, S, D), np.float32)
    got = oracle.attention(lay, B, Q, K, V, 1.0)
    rows = libref.expand_mask(lay, B)[0].any(-1)
    np.testing.assert_allclose(got[0, 0][rows], 1.0, rtol=1e-13)
    assert np.all(got[0, 0][~rows] == 0.0)


# the rows' log-sum-exp of the kept scaled scores (the softmax normaliser)

@pytest.mark.parametrize("kind", [W.MASK_NONE, W.MASK_DENSE, W.MASK_DIAG_CAUSAL])
def test_attention_lse_is_scipy_logsumexp_of_masked_scores(oracle, kind):
    from scipy.special import logsumexp
    Z, H, S, D, B = 2, 2, 48, 8, 8
    lay = random_layout(H, S // B, 0.35, 60)
    mask = W.random_mask(S, 0.6, 61) if kind == W.MASK_DENSE else None
    Q, K = rand(Z, H, S, D, seed=62), rand(Z, H, S, D, seed=63)
    M = libref.expand_mask(lay, B).astype(bool) & libref.keep_mask(S, B, kind, mask)[None]  # [H, S, S]
    s = 0.45 * np.einsum("zhrd,zhcd->zhrc", Q.astype(np.float64), K.astype(np.float64))
    want = logsumexp(np.where(M[None], s, -np.inf), axis=-1)  # -inf for empty rows
    got = oracle.attention_lse(lay, B, Q, K, 0.45, kind, mask)
    empty = ~M.any(-1)
    assert empty.any()  # the random layout has an empty block-row
    assert np.all(np.isneginf(got[:, empty]))
    np.testing.assert_allclose(got[:, ~empty], want[:, ~empty], rtol=1e-12, atol=1e-12)


def test_attention_lse_zero_query_is_log_of_count(oracle):
    # every kept score is 0: lse = log |R|
    Z, H, S, D, B = 1, 2, 40, 6, 8
    lay = random_layout(H, S // B, 0.5, 64)
    Q = np.zeros((Z, H, S, D), np.float32)
    K = rand(Z, H, S, D, seed=65)
    cnt = libref.expand_mask(lay, B).sum(-1)  # [H, S]
    got = oracle.attention_lse(lay, B, Q, K, 1.0)[0]
    np.testing.assert_allclose(got[cnt > 0], np.log(cnt[cnt > 0]), rtol=1e-14)
    assert np.all(np.isneginf(got[cnt == 0]))


def test_attention_lse_selection_matches_full(oracle):
    Z, H, S, D, B = 2, 2, 32, 8, 16
    lay = random_layout(H, S // B, 0.6, 66)
    Q, K = rand(Z, H, S, D, seed=67), rand(Z, H, S, D, seed=68)
    full = oracle.attention_lse(lay, B, Q, K, 0.3, W.MASK_DIAG_CAUSAL).reshape(-1)
    sel = np.array([0, 5, 17, 33, 64, 127], np.int64)
    got = oracle.attention_lse(lay, B, Q, K, 0.3, W.MASK_DIAG_CAUSAL, sel=sel)
    np.testing.assert_array_equal(got, full[sel])


@pytest.mark.parametrize("kind", [W.MASK_NONE, W.MASK_DENSE, W.MASK_DIAG_CAUSAL])
def test_attention_equals_sdd_softmax_dsd_chain(oracle, kind):
    # the page's chain: SDD output reduced by the block softmax, then DSD with V
    Z, H, S, D, B = 2, 3, 32, 8, 4
    lay = random_layout(H, S // B, 0.35, 47)
    mask = W.random_mask(S, 0.6, 48) if kind == W.MASK_DENSE else None
    Q, K, V = rand(Z, H, S, D, seed=49), rand(Z, H, S, D, seed=50), rand(Z, H, S, D, seed=51)
    scores = oracle.sdd(lay, B, Q, K)
    P = oracle.softmax(lay, B, scores.astype(np.float32), 0.45, kind, mask)
    # the chain is evaluated in fp64 throughout: feed P to DSD at full precision
    # by splitting it into two float32 parts (hi + lo)
    hi = P.astype(np.float32)
    lo = (P - hi.astype(np.float64)).astype(np.float32)
    chain = oracle.dsd(lay, B, hi, V) + oracle.dsd(lay, B, lo, V)
    direct = oracle.attention(lay, B, Q, K, V, 0.45, kind, mask)
    # scores were rounded to float32 before the softmax: tolerance covers that
    np.testing.assert_allclose(chain, direct, rtol=1e-5, atol=1e-6)


@pytest.mark.parametrize("kind", [W.MASK_NONE, W.MASK_DENSE, W.MASK_DIAG_CAUSAL])
def test_attention_selection_matches_full(oracle, kind):
    Z, H, S, D, B = 2, 2, 32, 8, 8
    lay = random_layout(H, S // B, 0.5, 52)
    Q, K, V = rand(Z, H, S, D, seed=53), rand(Z, H, S, D, seed=54), rand(Z, H, S, D, seed=55)
    mask = W.random_mask(S, 0.7, 56) if kind == W.MASK_DENSE else None
    full = oracle.attention(lay, B, Q, K, V, 0.5, kind, mask)
    sel = np.array([3, S + 5, 3 * S + 31])
    np.testing.assert_array_equal(oracle.attention(lay, B, Q, K, V, 0.5, kind, mask, sel=sel),
                                  full.reshape(-1, D)[sel])


# ------------------------------------------------------------ backward ----
# The backward functions follow the chain rule applied to the forward
# definitions; they are pinned to the oracle's own forward by central finite
# differences (inputs on a 2^-6 grid, steps of 2^-10: exact in fp32), to
# closed forms, and to the composition of the other oracle functions.

def grid(*shape, seed=0, lo=-2.0, hi=2.0):
    x = np.random.default_rng(seed).uniform(lo, hi, shape)
    return (np.round(x * 64) / 64).astype(np.float32)


def _fd(f, x, eps=2.0 ** -10):
    """Central differences of the scalar f at every element of x (float32)."""
    g = np.zeros(x.shape, np.float64)
    flat, gf = x.reshape(-1), g.reshape(-1)
    for e in range(flat.size):
        keep = flat[e]
        flat[e] = keep + eps
        fp = f(x)
        flat[e] = keep - eps
        fm = f(x)
        flat[e] = keep
        gf[e] = (fp - fm) / (2 * eps)
    return g


@pytest.mark.parametrize("kind", [W.MASK_NONE, W.MASK_DENSE, W.MASK_DIAG_CAUSAL])
def test_softmax_backward_matches_finite_differences(oracle, kind):
    Z, H, nb, B, scale = 1, 2, 3, 4, 0.7
    lay = random_layout(H, nb, 0.6, 21)
    lay[1, 0, 0] = 1
    nnz = int(lay.sum())
    X = grid(Z, nnz, B, B, seed=22)
    dY = grid(Z, nnz, B, B, seed=23)
    mask = (np.random.default_rng(24).random((nb * B, nb * B)) < 0.8).astype(np.uint8) if kind == W.MASK_DENSE else None
    f = lambda x: float(np.sum(oracle.softmax(lay, B, x, scale, kind, mask) * dY))
    want = _fd(f, X)
    Y = oracle.softmax(lay, B, X, scale, kind, mask)
    got = oracle.softmax_backward(lay, B, Y, dY, scale)
    np.testing.assert_allclose(got, want, rtol=1e-4, atol=2e-6)


def test_softmax_backward_constant_gradient_is_zero(oracle):
    # sum_c y_c = 1 on every non-empty row, so a constant dY has no effect
    lay = random_layout(2, 4, 0.5, 25)
    nnz = int(lay.sum())
    Y = oracle.softmax(lay, 8, grid(2, nnz, 8, 8, seed=26), 0.5)
    got = oracle.softmax_backward(lay, 8, Y, np.full(Y.shape, 3.25, np.float32), 0.5)
    np.testing.assert_allclose(got, 0.0, atol=1e-6)


@pytest.mark.parametrize("kind", [W.MASK_NONE, W.MASK_DENSE, W.MASK_DIAG_CAUSAL])
def test_attention_backward_matches_finite_differences(oracle, kind):
    Z, H, nb, B, D, scale = 1, 1, 3, 4, 4, 0.6
    S = nb * B
    lay = np.array([[[1, 0, 1], [0, 0, 0], [1, 1, 1]]], np.uint8)  # block-row 1 empty
    Q, K, V = grid(Z, H, S, D, seed=31), grid(Z, H, S, D, seed=32), grid(Z, H, S, D, seed=33)
    G = grid(Z, H, S, D, seed=34)
    mask = (np.random.default_rng(35).random((S, S)) < 0.7).astype(np.uint8) if kind == W.MASK_DENSE else None
    dQ, dK, dV = oracle.attention_backward(lay, B, Q, K, V, G, scale, kind, mask)
    loss = lambda q, k, v: float(np.sum(oracle.attention(lay, B, q, k, v, scale, kind, mask) * G))
    np.testing.assert_allclose(dQ, _fd(lambda x: loss(x, K, V), Q.copy()), rtol=1e-4, atol=2e-6)
    np.testing.assert_allclose(dK, _fd(lambda x: loss(Q, x, V), K.copy()), rtol=1e-4, atol=2e-6)
    np.testing.assert_allclose(dV, _fd(lambda x: loss(Q, K, x), V.copy()), rtol=1e-4, atol=2e-6)
    # the empty block-row has no gradient into Q
    assert np.all(dQ[0, 0, B:2 * B] == 0)


def test_attention_backward_constant_values_give_no_score_gradient(oracle):
    # V constant over keys: O does not depend on the scores, so dQ = dK = 0
    Z, H, nb, B, D = 1, 2, 4, 8, 8
    S = nb * B
    lay = random_layout(H, nb, 0.5, 36)
    Q, K = grid(Z, H, S, D, seed=37), grid(Z, H, S, D, seed=38)
    V = np.broadcast_to(grid(Z, H, 1, D, seed=39), (Z, H, S, D)).copy()
    dQ, dK, _ = oracle.attention_backward(lay, B, Q, K, V, grid(Z, H, S, D, seed=40), 0.4)
    np.testing.assert_allclose(dQ, 0.0, atol=1e-9)
    np.testing.assert_allclose(dK, 0.0, atol=1e-9)


@pytest.mark.parametrize("kind", [W.MASK_NONE, W.MASK_DIAG_CAUSAL])
def test_attention_backward_equals_unfused_chain(oracle, kind):
    # dV = DSD(P^T, dO), dS = softmax_backward(P, SDD(dO, V)), dQ = DSD(dS, K),
    # dK = DSD(dS^T, Q) with P = softmax(SDD(Q, K)): other oracle functions
    Z, H, nb, B, D, scale = 2, 2, 4, 8, 16, 0.25
    lay = random_layout(H, nb, 0.5, 41)
    S = nb * B
    Q, K, V, G = (grid(Z, H, S, D, seed=s) for s in (42, 43, 44, 45))
    P = oracle.softmax(lay, B, oracle.sdd(lay, B, Q, K), scale, kind)
    dS = oracle.softmax_backward(lay, B, P, oracle.sdd(lay, B, G, V), scale)
    dQ, dK, dV = oracle.attention_backward(lay, B, Q, K, V, G, scale, kind)
    # P and dS pass through fp32 between the chain's steps
    np.testing.assert_allclose(dV, oracle.dsd(lay, B, P, G, trans_a=1), rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(dQ, oracle.dsd(lay, B, dS, K), rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(dK, oracle.dsd(lay, B, dS, Q, trans_a=1), rtol=1e-5, atol=1e-6)


# ------------------------------------------------------ affine geometry ----
# SPLAT / ACSR abstract (NSF PAR record): banded and strided attention layouts
# have rows whose columns follow a formula in the row index.  The pins build
# the same layouts by independent numpy constructions.

def _terms(*ts):
    t = np.zeros((1, 2, 5), np.int32)
    for k, v in enumerate(ts):
        t[0, k] = v
    return np.array([len(ts)], np.int32), t


@pytest.mark.parametrize("nb,w", [(1, 0), (6, 0), (9, 2), (12, 4), (5, 7)])
def test_affine_band_is_numpy_band(oracle, nb, w):
    n, t = _terms((1, -w, 1, 2 * w + 1, 0))
    want = W.layout_band(nb, w)
    assert np.array_equal(oracle.affine_expand(n, t, nb), want)


@pytest.mark.parametrize("nb", [3, 10])
def test_affine_lower_triangle_is_tril(oracle, nb):
    n, t = _terms((1, -(nb - 1), 1, nb, 0))
    assert np.array_equal(oracle.affine_expand(n, t, nb)[0], np.tril(np.ones((nb, nb), np.uint8)))


@pytest.mark.parametrize("nb,local,stride", [(256, 4, 16), (40, 3, 8), (17, 1, 5)])
def test_affine_strided_is_sparse_transformer_fixed(oracle, nb, local, stride):
    # local window (offsets -(local-1) .. 0) plus every stride-th column, causal
    n, t = _terms((1, -(local - 1), 1, local, 0), (0, 0, stride, (nb - 1) // stride + 1, 1))
    assert np.array_equal(oracle.affine_expand(n, t, nb), W.layout_strided_causal(nb, local, stride))


def test_affine_column_terms_causal_and_not(oracle):
    nb = 10
    cols = np.zeros(nb, bool)
    cols[[2, 5, 8]] = True
    n, t = _terms((0, 2, 3, 3, 0))
    assert np.array_equal(oracle.affine_expand(n, t, nb)[0], np.broadcast_to(cols, (nb, nb)).astype(np.uint8))
    n, t = _terms((0, 2, 3, 3, 1))
    want = (np.broadcast_to(cols, (nb, nb)) & (np.arange(nb)[None, :] <= np.arange(nb)[:, None]))
    assert np.array_equal(oracle.affine_expand(n, t, nb)[0], want.astype(np.uint8))
    n, t = _terms()
    assert not oracle.affine_expand(n, t, nb).any()


def test_affine_describable_known_cases(oracle):
    nb = 8
    i, j = np.meshgrid(np.arange(nb), np.arange(nb), indexing="ij")
    assert oracle.affine_describable(W.layout_band(nb, 2)[0])
    assert oracle.affine_describable(W.layout_strided_causal(nb, 2, 4)[0])
    assert oracle.affine_describable(np.zeros((nb, nb), np.uint8))
    assert oracle.affine_describable(np.ones((nb, nb), np.uint8))
    # a band plus one full column
    lay = W.layout_band(nb, 1)[0]
    lay[:, 5] = 1
    assert oracle.affine_describable(lay)
    # parity checkerboard: rows alternate between two column sets
    assert not oracle.affine_describable(((i + j) % 2 == 0).astype(np.uint8))
    # two separate diagonals
    assert not oracle.affine_describable(((j == i) | (j == i + 5)).astype(np.uint8))
    # a band plus one full row
    lay = W.layout_band(nb, 1)[0]
    lay[3, :] = 1
    assert not oracle.affine_describable(lay)
