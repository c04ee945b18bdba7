"""Seeded synthetic inputs: block layouts and dense tensors.

This module draws random numbers and builds 0/1 block layouts. It holds none
of the arithmetic of the block-sparse operations themselves, so both the CUDA
path and the fp64 CPU oracle may be fed from it.

The layouts follow the sparse multi-head-attention patterns named in the SPLAT
abstract ("SPLAT: A framework for optimised GPU code-generation for SParse
reguLar ATtention", NSF PAR record of D. Jain et al., abstract): banded /
sliding window, global rows and columns, random blocks and strided columns,
at moderate densities.  A layout is a uint8 array of shape [H, nb, nb] with
values 0/1; entry (h, i, j) = 1 means the B x B block at block-row i and
block-column j of head h is present ("question on blocksparse", openai/triton
issue 117, answer on the layout being a tensor of 0s and 1s with 16/32/64/128
blocks).
"""

from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

MASK_NONE = 0
MASK_DENSE = 1
MASK_DIAG_CAUSAL = 2


# --------------------------------------------------------------------------
# layout patterns
# --------------------------------------------------------------------------

def layout_random_diag(nb: int, density: float, H: int = 1, seed: int = 0) -> np.ndarray:
    """Each block present with probability `density`; diagonal blocks forced on."""
    rng = np.random.default_rng(seed)
    lay = (rng.random((H, nb, nb)) < density).astype(np.uint8)
    idx = np.arange(nb)
    lay[:, idx, idx] = 1
    return lay


def layout_bigbird(nb: int, H: int, window: int = 3, n_global: int = 2,
                   n_random: int = 3, seed: int = 0) -> np.ndarray:
    """BigBird-style: sliding window of `window` blocks centred on the diagonal,
    the first `n_global` block-rows and block-columns full, and `n_random` extra
    blocks per non-global row drawn (without replacement) from the row's
    remaining blocks.  Drawn independently per head."""
    rng = np.random.default_rng(seed)
    half = window // 2
    lay = np.zeros((H, nb, nb), dtype=np.uint8)
    for h in range(H):
        for i in range(nb):
            lo, hi = max(0, i - half), min(nb, i + half + 1)
            lay[h, i, lo:hi] = 1
        lay[h, :n_global, :] = 1
        lay[h, :, :n_global] = 1
        for i in range(n_global, nb):
            off = np.flatnonzero(lay[h, i] == 0)
            k = min(n_random, off.size)
            if k:
                lay[h, i, rng.choice(off, size=k, replace=False)] = 1
    return lay


def layout_band(nb: int, half_width_blocks: int, H: int = 1) -> np.ndarray:
    """Block band |i - j| <= half_width_blocks, identical for every head."""
    i = np.arange(nb)[:, None]
    j = np.arange(nb)[None, :]
    one = (np.abs(i - j) <= half_width_blocks).astype(np.uint8)
    return np.broadcast_to(one, (H, nb, nb)).copy()


def layout_uniform(nb: int, density: float, H: int = 1, seed: int = 0) -> np.ndarray:
    """Exactly round(density * nb^2) blocks per head, chosen uniformly without
    replacement."""
    rng = np.random.default_rng(seed)
    k = int(round(density * nb * nb))
    lay = np.zeros((H, nb * nb), dtype=np.uint8)
    for h in range(H):
        lay[h, rng.choice(nb * nb, size=k, replace=False)] = 1
    return lay.reshape(H, nb, nb)


def layout_strided_causal(nb: int, local_blocks: int, stride: int, H: int = 1) -> np.ndarray:
    """Sparse-Transformer 'fixed' pattern, causal at block level: block (i, j)
    present when j <= i and (i - j < local_blocks or j % stride == 0)."""
    i = np.arange(nb)[:, None]
    j = np.arange(nb)[None, :]
    one = ((j <= i) & (((i - j) < local_blocks) | (j % stride == 0))).astype(np.uint8)
    return np.broadcast_to(one, (H, nb, nb)).copy()


def layout_causal_blocks(nb: int, H: int = 1) -> np.ndarray:
    """Lower block-triangular layout (j <= i)."""
    one = np.tril(np.ones((nb, nb), dtype=np.uint8))
    return np.broadcast_to(one, (H, nb, nb)).copy()


# --------------------------------------------------------------------------
# tensors
# --------------------------------------------------------------------------

_TORCH_DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


def torch_dtype(name: str) -> torch.dtype:
    return _TORCH_DTYPES[name]


def randn(shape, dtype: str, seed: int) -> torch.Tensor:
    """N(0, 1) drawn in fp32 on the CPU from a seeded generator, then rounded
    to `dtype`.  Returns a CPU tensor."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    return torch.randn(*shape, generator=g, dtype=torch.float32).to(_TORCH_DTYPES[dtype])


def uniform(shape, dtype: str, seed: int, lo: float = -1.0, hi: float = 1.0) -> torch.Tensor:
    """U(lo, hi) drawn in fp32 on the CPU, then rounded to `dtype`."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    x = torch.rand(*shape, generator=g, dtype=torch.float32)
    return (x * (hi - lo) + lo).to(_TORCH_DTYPES[dtype])


def random_mask(S: int, p_keep: float, seed: int) -> np.ndarray:
    """Dense uint8 keep-mask [S, S] (1 = keep), Bernoulli(p_keep)."""
    rng = np.random.default_rng(seed)
    return (rng.random((S, S)) < p_keep).astype(np.uint8)


# --------------------------------------------------------------------------
# the five workloads
# --------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class AttentionWorkload:
    name: str
    Z: int
    H: int
    S: int
    D: int
    B: int
    dtype: str
    mask_kind: int
    scale: float
    index: int  # 1-based workload number, used to derive seeds

    @property
    def nb(self) -> int:
        return self.S // self.B

    def layout(self) -> np.ndarray:
        nb, H = self.nb, self.H
        if self.name == "tiny":
            return layout_random_diag(nb, 0.30, H=H, seed=self.index)
        if self.name == "bigbird":
            return layout_bigbird(nb, H, window=3, n_global=2, n_random=3, seed=self.index)
        if self.name == "band":
            return layout_band(nb, half_width_blocks=512 // self.B, H=H)
        if self.name == "strided":
            return layout_strided_causal(nb, local_blocks=256 // self.B, stride=16, H=H)
        raise KeyError(self.name)

    def qkv(self, shard: int = 0):
        """Q, K, V of the workload; `shard` selects an independent draw (one per
        rank when several GPUs each process their own batch)."""
        shape = (self.Z, self.H, self.S, self.D)
        base = 1000 + 10 * self.index + 7919 * shard
        return (randn(shape, self.dtype, base + 0),
                randn(shape, self.dtype, base + 1),
                randn(shape, self.dtype, base + 2))


TINY = AttentionWorkload("tiny", 1, 1, 256, 64, 16, "f32", MASK_NONE, 1.0 / 8.0, 1)
BIGBIRD = AttentionWorkload("bigbird", 2, 12, 4096, 64, 64, "f32", MASK_DIAG_CAUSAL, 1.0 / 8.0, 2)
BAND = AttentionWorkload("band", 4, 16, 8192, 128, 128, "bf16", MASK_NONE, 1.0 / math.sqrt(128), 3)
STRIDED = AttentionWorkload("strided", 1, 32, 16384, 128, 64, "bf16", MASK_DIAG_CAUSAL,
                            1.0 / math.sqrt(128), 5)

ATTENTION_WORKLOADS = {w.name: w for w in (TINY, BIGBIRD, BAND, STRIDED)}


@dataclasses.dataclass(frozen=True)
class SpmmWorkload:
    """General block-sparse spMM: a sparse S x S operand (block B) against a
    dense operand; DSD takes the dense operand as [S, N], DDS as [N, S]."""
    S: int = 8192
    N: int = 4096
    B: int = 32
    dtype: str = "bf16"
    index: int = 4

    def _salt(self, density: float) -> int:
        # the block size enters the seeds only for the other block sizes, so the
        # 32-wide workload keeps its original draws
        return int(round(density * 100)) + (0 if self.B == 32 else 1000 * self.B)

    def layout(self, density: float) -> np.ndarray:
        return layout_uniform(self.S // self.B, density, H=1, seed=self.index * 100 + self._salt(density))

    def sparse_values(self, nnz: int, density: float) -> torch.Tensor:
        return uniform((1, nnz, self.B, self.B), self.dtype, 4000 + self._salt(density))

    def dense_dsd(self, density: float) -> torch.Tensor:
        return uniform((1, 1, self.S, self.N), self.dtype, 4100 + self._salt(density))

    def dense_dds(self, density: float) -> torch.Tensor:
        return uniform((1, 1, self.N, self.S), self.dtype, 4200 + self._salt(density))


SPMM = SpmmWorkload()
SPMM_DENSITIES = (0.10, 0.25, 0.50)
# the same spMM shapes at the other block sizes (8192 x 8192 sparse operand,
# 4096-wide dense operand), densities 10 % and 50 %
SPMM_BLOCKS = {b: SpmmWorkload(B=b) for b in (16, 32, 64, 128)}
SPMM_BLOCK_DENSITIES = (0.10, 0.50)
