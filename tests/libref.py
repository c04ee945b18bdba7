"""Library-routine restatements used to pin the oracle.

Each helper reaches the block-sparse result through numpy / scipy dense
routines (np.kron expansion of the layout, np.matmul, scipy.special.softmax)
on inputs where the block-sparse operation reduces to a dense one.  None of it
reuses the oracle's loops, and none of it is used by the CUDA path.
"""

import numpy as np
from scipy.special import softmax as sp_softmax


def block_coords(layout):
    """(h, i, j) of every present block in block-id order (row-major rank)."""
    h, i, j = np.nonzero(np.asarray(layout))
    return h, i, j


def expand_mask(layout, B):
    """[H, S, S] 0/1 element mask from the [H, nb, nb] block layout."""
    lay = np.asarray(layout, dtype=np.uint8)
    return np.stack([np.kron(lay[h], np.ones((B, B), dtype=np.uint8)) for h in range(lay.shape[0])])


def blocks_to_dense(layout, B, X):
    """X [Z, nnz, B, B] -> dense [Z, H, S, S] with zeros outside the blocks."""
    lay = np.asarray(layout)
    H, nb = lay.shape[0], lay.shape[1]
    Z = X.shape[0]
    out = np.zeros((Z, H, nb * B, nb * B), dtype=np.float64)
    hs, is_, js = block_coords(lay)
    for n, (h, i, j) in enumerate(zip(hs, is_, js)):
        out[:, h, i * B:(i + 1) * B, j * B:(j + 1) * B] = X[:, n]
    return out


def dense_to_blocks(layout, B, Dn):
    """Dense [Z, H, S, S] -> [Z, nnz, B, B] sampled on the layout."""
    hs, is_, js = block_coords(layout)
    return np.stack([Dn[:, h, i * B:(i + 1) * B, j * B:(j + 1) * B]
                     for h, i, j in zip(hs, is_, js)], axis=1)


def keep_mask(S, B, kind, mask=None):
    if kind == 0:
        return np.ones((S, S), dtype=bool)
    if kind == 1:
        return np.asarray(mask, dtype=bool)
    r = np.arange(S)[:, None]
    c = np.arange(S)[None, :]
    return (r // B != c // B) | (c <= r)


def masked_softmax(scores, M):
    """Row softmax of `scores` over entries where M is true; rows with no
    true entry give zeros.  scores, M: [..., S, S]."""
    s = np.where(M, scores, -np.inf)
    empty = ~M.any(axis=-1, keepdims=True)
    s = np.where(empty, 0.0, s)
    p = sp_softmax(s, axis=-1)
    return np.where(M & ~empty, p, 0.0)


def dense_attention(Q, K, V, scale, M):
    """softmax(scale Q K^T restricted to M) V with numpy matmul / scipy softmax."""
    Q, K, V = (np.asarray(t, dtype=np.float64) for t in (Q, K, V))
    s = scale * np.matmul(Q, np.swapaxes(K, -1, -2))
    return np.matmul(masked_softmax(s, M), V)
