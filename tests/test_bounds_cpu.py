"""The per-entry bounds of the GPU parity tests (tests/gpu_util.py), checked on
the CPU: a faithful emulation of the kernels' arithmetic (fp32 accumulation,
fp32 exponentials and normalisation, one rounding of P and of the output to the
16-bit type) must pass every bound, and planted mistakes of the kind the
normwise bar alone lets through (a probability leaked into a masked entry, a
small block dropped from a product, a rounding step too many) must fail one.
The emulation is torch on the CPU, the expected values are the oracle's."""

import numpy as np
import pytest
import torch

import libref
from gpu_util import (PROB_TOL, assert_close, attention_acc, gamma, softmax_rel_bound,
                      softmax_zero_positions)
from sparse_attention_layout_gb300 import workloads as W


def _rlayout(H, nb, p, seed):
    lay = (np.random.default_rng(seed).random((H, nb, nb)) < p).astype(np.uint8)
    lay[:, np.arange(nb), np.arange(nb)] = 1
    lay[0, 2, :] = 0
    return lay


def _emulate_scores(lay, B, A, Bm):
    """fp32 scores of the present blocks, [Z, nnz, B, B] (exact inputs)."""
    s = torch.matmul(A.float(), Bm.float().transpose(-1, -2)).double().numpy()
    return libref.dense_to_blocks(lay, B, s)


def _emulate_softmax(lay, B, s32, scale, kind, mask):
    """fp32 softmax of fp32 scores on the layout, in block format (float64 array
    holding fp32 values)."""
    S = lay.shape[1] * B
    Ms = libref.expand_mask(lay, B).astype(bool) & libref.keep_mask(S, B, kind, mask)[None]
    sd = torch.from_numpy(libref.blocks_to_dense(lay, B, s32)).float() * scale
    sd = torch.where(torch.from_numpy(Ms)[None], sd, torch.tensor(float("-inf")))
    m = sd.amax(dim=-1, keepdim=True)
    e = torch.where(torch.isfinite(m), torch.exp(sd - torch.where(torch.isfinite(m), m, torch.zeros_like(m))),
                    torch.zeros_like(sd))
    l = e.sum(dim=-1, keepdim=True)
    p = torch.where(l > 0, e / l, torch.zeros_like(e))
    return libref.dense_to_blocks(lay, B, p.double().numpy())


def _round(x, dtype):
    return torch.from_numpy(np.asarray(x)).to(dtype).double().numpy()


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("kind", [0, 1, 2])
def test_softmax_bounds_accept_rounding_and_catch_a_leak(oracle, dtype, kind):
    B, H, Z, nb = 16, 2, 2, 9
    S = nb * B
    lay = _rlayout(H, nb, 0.4, 3 + kind)
    nnz = int(lay.sum())
    X = W.randn((Z, nnz, B, B), {torch.bfloat16: "bf16", torch.float16: "f16"}[dtype], 5)
    mask = W.random_mask(S, 0.7, 6) if kind == 1 else None
    want = oracle.softmax(lay, B, X, 0.4, kind, mask)
    zeros = softmax_zero_positions(lay, B, Z, kind, mask)
    got = _round(_emulate_softmax(lay, B, X.double().numpy(), 0.4, kind, mask), dtype)
    assert_close(got, want, dtype, "emulated softmax", rel=PROB_TOL[dtype], zeros=zeros)
    if kind != 0:
        # a probability leaked into an entry the mask removes
        bad = got.copy()
        pos = tuple(int(v[0]) for v in np.nonzero(zeros))
        bad[pos] = 1e-3
        with pytest.raises(AssertionError, match="exactly 0"):
            assert_close(bad, want, dtype, "leak", rel=PROB_TOL[dtype], zeros=zeros)
    # one small probability off by 2 % (well inside the normwise 2e-2 bar)
    bad = got.copy()
    idx = np.unravel_index(np.argmin(np.where(want > 0.01 * want.max(), want, np.inf)), want.shape)
    bad[idx] *= 1.02
    with pytest.raises(AssertionError, match="elementwise relative"):
        assert_close(bad, want, dtype, "small entry", rel=PROB_TOL[dtype], zeros=zeros)


@pytest.mark.parametrize("scores_rounded", [False, True])
def test_fused_softmax_bound_accepts_fp32_scores_and_rounded_chain(oracle, scores_rounded):
    dtype = torch.bfloat16
    B, H, Z, nb, K = 16, 2, 1, 8, 64
    lay = _rlayout(H, nb, 0.4, 11)
    A = W.randn((Z, H, nb * B, K), "bf16", 12)
    Bm = W.randn((Z, H, nb * B, K), "bf16", 13)
    s_ref = oracle.sdd(lay, B, A, Bm)
    smag = oracle.sdd(lay, B, A.abs(), Bm.abs())
    want = oracle.softmax(lay, B, s_ref, 0.2, 2)
    s32 = _emulate_scores(lay, B, A, Bm)
    if scores_rounded:
        s32 = _round(s32, dtype)
    got = _round(_emulate_softmax(lay, B, s32, 0.2, 2, None), dtype)
    rel = softmax_rel_bound(lay, B, s_ref, smag, 0.2, K, dtype, scores_rounded)
    assert_close(got, want, dtype, "emulated fused SDD + softmax", rel=rel,
                 zeros=softmax_zero_positions(lay, B, Z, 2))
    if not scores_rounded:
        # the fused bound does not admit a chain that rounds the scores first
        s16 = _round(_emulate_scores(lay, B, A, Bm), dtype)
        chain = _round(_emulate_softmax(lay, B, s16, 0.2, 2, None), dtype)
        with pytest.raises(AssertionError, match="elementwise relative"):
            assert_close(chain, want, dtype, "rounded scores", rel=rel)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_sdd_bound_accepts_fp32_accumulation_and_catches_a_dropped_term(oracle, dtype):
    B, H, Z, nb, K = 16, 2, 2, 6, 48
    lay = _rlayout(H, nb, 0.5, 21)
    code = "f32" if dtype == torch.float32 else "bf16"
    A = W.randn((Z, H, nb * B, K), code, 22)
    Bm = W.randn((Z, H, nb * B, K), code, 23)
    want = oracle.sdd(lay, B, A, Bm)
    mag = oracle.sdd(lay, B, A.abs(), Bm.abs())
    got = _round(_emulate_scores(lay, B, A, Bm), dtype)
    assert_close(got, want, dtype, "emulated SDD", mag=mag, acc=gamma(K))
    # the last product of the contraction dropped
    short = _round(_emulate_scores(lay, B, A[..., :-1], Bm[..., :-1]), dtype)
    with pytest.raises(AssertionError):
        assert_close(short, want, dtype, "dropped term", mag=mag, acc=gamma(K))
    if dtype != torch.float32:
        # a small entry off by 1 % of the largest: inside the normwise 2e-2 bar,
        # outside its own bound
        bad = got.copy()
        idx = np.unravel_index(np.argmin(np.abs(want)), want.shape)
        bad[idx] += 0.01 * np.abs(want).max()
        with pytest.raises(AssertionError, match="forward error bound"):
            assert_close(bad, want, dtype, "small entry", mag=mag, acc=gamma(K))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
def test_attention_bound_accepts_rounded_p_and_catches_a_masked_block(oracle, dtype):
    B, H, Z, nb, D = 16, 2, 1, 8, 64
    S = nb * B
    lay = _rlayout(H, nb, 0.35, 31)
    code = {torch.float32: "f32", torch.bfloat16: "bf16", torch.float16: "f16"}[dtype]
    Q, K, V = (W.randn((Z, H, S, D), code, 32 + k) for k in range(3))
    scale = 1.0 / np.sqrt(D)
    want = oracle.attention(lay, B, Q, K, V, scale, 2)
    mag = oracle.attention(lay, B, Q, K, V.abs(), scale, 2)
    acc = attention_acc(Q, K, scale, dtype, S)

    def emulate(lay_used, kind):
        p = _emulate_softmax(lay_used, B, _emulate_scores(lay_used, B, Q, K), scale, kind, None)
        if dtype != torch.float32:
            p = _round(p, dtype)
        pd = torch.from_numpy(libref.blocks_to_dense(lay_used, B, p)).float()
        return _round((pd @ V.float()).double().numpy(), dtype)

    assert_close(emulate(lay, 2), want, dtype, "emulated attention", mag=mag, acc=acc)
    # rows with nothing kept (block-row 2 of head 0 is empty) are exactly 0
    assert np.all(emulate(lay, 2)[:, 0, 2 * B:3 * B] == 0)
    # one more block attended (present in the layout of the mistake only)
    off = np.argwhere(lay[0] == 0)
    off = off[off[:, 0] != 2][0]
    lay2 = lay.copy()
    lay2[0, off[0], off[1]] = 1
    with pytest.raises(AssertionError):
        assert_close(emulate(lay2, 2), want, dtype, "extra block", mag=mag, acc=acc)
    # the causal mask inside the diagonal blocks ignored
    with pytest.raises(AssertionError):
        assert_close(emulate(lay, 0), want, dtype, "no causal mask", mag=mag, acc=acc)
