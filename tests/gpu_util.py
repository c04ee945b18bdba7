"""Shared helpers of the GPU parity tests.

Every check applies the parity bar to the whole tensor -- normwise
max |g - r| / max |r| <= 1e-5 for fp32 outputs, <= 2e-2 for bf16 / fp16 --
and, on top of it, a bound on each entry:

- probabilities (softmax outputs): elementwise relative error <= a bound
  derived from the output's unit roundoff u (2^-24 fp32, 2^-8 bf16, 2^-11
  fp16), and the entries the oracle defines as 0 (masked inside a present
  block, rows with nothing kept) exactly 0;
- products (SDD, DSD, DDS, attention): |g - r| <= 2 u |r| + acc * mag, where
  mag is the same product evaluated on the operands' absolute values (the
  oracle run on |A|, |B|) and acc the relative error of the fp32 accumulation
  and of any rounded intermediate: the standard forward error bound of a
  dot product, entry by entry.

The elementwise relative error max |g - r| / |r| over |r| > 1e-3 max |r| is
reported in every assertion message.
"""

import numpy as np
import torch

TOL = {torch.float32: 1e-5, torch.bfloat16: 2e-2, torch.float16: 2e-2}
# unit roundoff of each output type (round to nearest)
U = {torch.float32: 2.0 ** -24, torch.bfloat16: 2.0 ** -8, torch.float16: 2.0 ** -11}
# elementwise relative error of a softmax output computed in fp32 from exact
# inputs: one rounding to the output type plus the fp32 exponentials and
# normalisation (< 1e-4); fp32 outputs are held to the 1e-5 parity bar per entry
PROB_TOL = {torch.float32: 1e-5, torch.bfloat16: 2.0 ** -8 + 1e-4, torch.float16: 2.0 ** -11 + 1e-4}
# below these magnitudes an output type is subnormal (fp16) or flushed to zero
# by the fp32 exponentials: there only the absolute error is bounded, by the floor
REL_FLOOR = {torch.float32: 2.0 ** -120, torch.bfloat16: 2.0 ** -120, torch.float16: 2.0 ** -14}
EXP_ERR = 2.0 ** -20  # relative error allowance of one fp32 2^x (hardware ex2 or exp2f / expf)


def gamma(n) -> float:
    """Relative error coefficient of an fp32 sum of n products: (n + 2) * 2^-22,
    four times the textbook n * 2^-24, leaving room for tensor-core adders that
    align their addends before rounding."""
    return (float(n) + 2.0) * 2.0 ** -22


def _np64(x):
    if isinstance(x, torch.Tensor):
        x = x.detach().double().cpu().numpy()
    return np.asarray(x, dtype=np.float64)


def normwise_err(got, want) -> float:
    """max |g - r| / max |r| over the tensor (0 when both are exactly 0)."""
    g, r = _np64(got), _np64(want)
    assert g.shape == r.shape, (g.shape, r.shape)
    assert np.all(np.isfinite(g)), "non-finite output"
    scale = np.max(np.abs(r)) if r.size else 0.0
    diff = np.max(np.abs(g - r)) if r.size else 0.0
    if scale == 0.0:
        return float(diff)
    return float(diff / scale)


def elementwise_err(got, want, floor=1e-3) -> float:
    """max |g - r| / |r| over the entries with |r| > floor * max |r|."""
    g, r = _np64(got), _np64(want)
    if not r.size:
        return 0.0
    big = np.abs(r) > floor * np.max(np.abs(r))
    if not big.any():
        return 0.0
    return float(np.max(np.abs(g[big] - r[big]) / np.abs(r[big])))


def assert_close(got, want, dtype, what="", *, rel=None, zeros=None, mag=None, acc=None):
    """Normwise bar, then the per-entry bounds that are given:
    rel   elementwise relative bound (scalar or array shaped like want) on
          entries above the type's REL_FLOOR; below it |g - r| <= the floor;
    zeros boolean array: positions the oracle defines as 0, checked to be
          exactly 0 in both;
    mag, acc  |g - r| <= 2 u |r| + acc * mag entry by entry (acc scalar or
          broadcastable)."""
    g, r = _np64(got), _np64(want)
    err = normwise_err(g, r)
    ew = elementwise_err(g, r)
    tag = f"{what}: normwise {err:.3e}, elementwise (|r| > 1e-3 max) {ew:.3e}"
    assert err <= TOL[dtype], f"{tag} -- normwise above {TOL[dtype]:.0e}"
    if zeros is not None:
        z = np.broadcast_to(np.asarray(zeros, dtype=bool), r.shape)
        assert np.all(r[z] == 0.0), f"{tag} -- the oracle is not 0 where it defines 0"
        bad = int(np.count_nonzero(g[z] != 0.0))
        assert bad == 0, f"{tag} -- {bad} entries that must be exactly 0 are not"
    if rel is not None:
        bound = np.broadcast_to(np.asarray(rel, dtype=np.float64), r.shape)
        floor = REL_FLOOR[dtype]
        big = np.abs(r) > floor
        d = np.abs(g - r)
        if big.any():
            ratio = d[big] / (bound[big] * np.abs(r[big]))
            worst = float(np.max(ratio))
            assert worst <= 1.0, (f"{tag} -- elementwise relative error {worst:.3f}x its bound "
                                  f"(max bound {float(np.max(bound[big])):.2e})")
        if (~big).any():
            assert float(np.max(d[~big])) <= floor, f"{tag} -- tiny entries off by more than {floor:.1e}"
    if mag is not None:
        m = _np64(mag)
        bound = 2.0 * U[dtype] * np.abs(r) + np.asarray(acc, dtype=np.float64) * m
        d = np.abs(g - r)
        over = d > bound
        if over.any():
            idx = np.unravel_index(int(np.argmax(np.where(over, d - bound, -np.inf))), r.shape)
            raise AssertionError(f"{tag} -- {int(over.sum())} entries above the forward error bound, "
                                 f"e.g. at {idx}: |g - r| = {d[idx]:.3e} > {bound[idx]:.3e} "
                                 f"(r = {r[idx]:.3e}, mag = {m[idx]:.3e})")
    return err


def attention_acc(Q, K, scale, dtype, n_keys, scores_rounded=False):
    """Per-row relative error coefficient of attention O = P V against
    mag = P |V| (both [Z, H, S, D]): returns [Z, H, S, 1].

    The scores s = q . k carry the fp32 accumulation error gamma(D) |q| . |k|
    (bounded by gamma(D) ||q|| ||k|| with Cauchy-Schwarz) and, when the chain
    rounds them to the data type, u |s| <= u ||q|| ||k|| more; a score error
    ds moves ln p_j by at most scale (ds_j + max_i ds_i), and the row's
    exponentials and normalisation add a few EXP_ERR and gamma(n_keys).  P is
    rounded to the data type before P V (16-bit types), and P V accumulates
    n_keys products in fp32."""
    q = Q if isinstance(Q, torch.Tensor) else torch.from_numpy(np.asarray(Q))
    k = K if isinstance(K, torch.Tensor) else torch.from_numpy(np.asarray(K))
    qn = q.double().norm(dim=-1, keepdim=True).cpu().numpy()                          # [Z, H, S, 1]
    kmax = k.double().norm(dim=-1).amax(dim=-1)[..., None, None].cpu().numpy()        # [Z, H, 1, 1]
    D = q.shape[-1]
    us = U[dtype] if (scores_rounded and dtype != torch.float32) else 0.0
    ds = (gamma(D) + us) * qn * kmax
    up = U[dtype] if dtype != torch.float32 else 0.0
    lnp = 2.0 * scale * ds + 4.0 * EXP_ERR + gamma(n_keys)
    rel_p = np.expm1(lnp)
    return (1.0 + up) * rel_p + up + gamma(n_keys)


def softmax_rel_bound(lay, B, scores, smag, scale, K, dtype, scores_rounded):
    """Per-entry relative bound of P = softmax(scale * s) on the layout when
    the scores s (oracle values, [Z, nnz, B, B]) are computed with fp32
    accumulation over K products (error gamma(K) * smag, smag the scores of
    the absolute operands) and, if scores_rounded, rounded to the data type
    before the softmax (error u |s|).  Each row's bound uses the largest score
    error of the row: ln p_j moves by at most scale (ds_j + max_i ds_i)."""
    s = _np64(scores)
    m = _np64(smag)
    us = U[dtype] if (scores_rounded and dtype != torch.float32) else 0.0
    ds = gamma(K) * m + us * np.abs(s)                                  # [Z, nnz, B, B]
    lay = np.asarray(lay)
    hs, is_, _ = np.nonzero(lay)
    # largest error over each row of the whole S x S row (all blocks of the block-row)
    key = hs * lay.shape[1] + is_
    Z = s.shape[0]
    rowmax = np.zeros((Z, lay.shape[0] * lay.shape[1], B))
    np.maximum.at(rowmax, (slice(None), key), ds.max(axis=3))
    row = rowmax[:, key][..., None]                                     # [Z, nnz, B, 1]
    rel_p = np.expm1(scale * (ds + row) + 4.0 * EXP_ERR)
    up = U[dtype]
    return (1.0 + up) * rel_p + PROB_TOL[dtype]


def softmax_zero_positions(lay, B, Z, kind, mask=None):
    """Positions of a block-format softmax output [Z, nnz, B, B] that the
    oracle defines as exactly 0: entries the mask removes inside present
    blocks, and every entry of a row with nothing kept."""
    lay = np.asarray(lay)
    H, nb = lay.shape[0], lay.shape[1]
    S = nb * B
    hs, is_, js = np.nonzero(lay)
    r = np.arange(B)
    keep = np.ones((hs.size, B, B), dtype=bool)
    if kind == 2:
        diag = is_ == js
        keep[diag] = r[None, :, None] >= r[None, None, :]
    elif kind == 1:
        mk = np.asarray(mask, dtype=bool)
        for n, (i, j) in enumerate(zip(is_, js)):
            keep[n] = mk[i * B:(i + 1) * B, j * B:(j + 1) * B]
    # rows with nothing kept anywhere in their block-row
    rowkeep = np.zeros((H * nb, B), dtype=bool)
    np.logical_or.at(rowkeep, hs * nb + is_, keep.any(axis=2))
    alive = rowkeep[hs * nb + is_]                                      # [nnz, B]
    keep &= alive[:, :, None]
    return np.broadcast_to(~keep[None], (Z, hs.size, B, B))


def to_np(t):
    return t.detach().float().cpu().numpy()


def dev(t):
    return t.to("cuda").contiguous()


# ---------------------------------------------------------- softmax backward --

def row_reduce(lay, B, M):
    """Sum of M over each query row's blocks, broadcast back onto the block
    format: M [Z, nnz, B, B] -> [Z, nnz, B, 1] (the blocks of one block-row
    are consecutive ids, CSR order)."""
    cnt = np.asarray(lay).reshape(-1, lay.shape[2]).sum(axis=1).astype(np.int64)
    ptr = np.concatenate([[0], np.cumsum(cnt)])
    out = np.zeros(M.shape[:3] + (1,), np.float64)
    for k in np.nonzero(cnt)[0]:
        a, b = ptr[k], ptr[k + 1]
        out[:, a:b] = M[:, a:b].sum(axis=(1, 3))[:, None, :, None]
    return out


def check_softmax_backward_elementwise(lay, B, Y, dY, got, want, scale, dtype, what):
    """Every entry of dX = scale * y * (g - d), d = rowsum(y .* g), within the
    forward error bound of an fp32 evaluation: the dot product of a row of n
    entries is off by at most n 2^-23 sum|y g|; scale * y * (g - d) adds three
    fp32 roundings (2^-21 of scale |y| (|g| + |d|)); the stored value one
    rounding of the output type (U) plus, for fp16, its subnormal spacing
    2^-24.  dX is exactly 0 wherever Y is 0."""
    y, g = _np64(Y), _np64(dY)
    n = row_reduce(lay, B, np.ones_like(y))
    A = row_reduce(lay, B, np.abs(y * g))
    d = np.abs(row_reduce(lay, B, y * g))
    r = _np64(want)
    bound = (U[dtype] * np.abs(r)
             + (1 + U[dtype]) * scale * np.abs(y) * (n * 2.0 ** -23 * A + 2.0 ** -21 * (np.abs(g) + d))
             + (2.0 ** -24 if dtype == torch.float16 else 0.0))
    x = _np64(got)
    err = np.abs(x - r)
    bad = err > bound
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} entries out of bound, worst excess "
                           f"{float((err - bound).max()):.3e}")
    assert (x[y == 0] == 0).all(), f"{what}: nonzero gradient where Y is 0"
