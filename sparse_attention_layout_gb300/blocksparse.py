"""Block-sparse matmul and softmax objects in the shape of the API the source
issue describes ("question on blocksparse", openai/triton issue 117): a
matmul built from a 0/1 layout, a block size and a mode -- 'sdd' (sparse =
dense x dense, sampled), 'dsd' (dense = sparse x dense) or 'dds' (dense =
dense x sparse) -- and a softmax built from a layout and a block size that
reduces the rows of the SDD output; dense keep-masks may be passed.

Each object compiles its layout once (``bsp.bsp_layout_compile``) and is
differentiable through torch autograd.  Every forward and backward step is a
call into the CUDA library; the gradients of each mode are the other two modes
with the operands' orientations flipped:

    sdd  C = op(A) op(B) on the layout:  dop(A) = dC op(B)^T  (dsd),
                                         dop(B) = op(A)^T dC  (dds)
    dsd  C = op(S) op(B):                dS = dC op(B)^T on the layout (sdd),
                                         dop(B) = op(S)^T dC  (dsd)
    dds  C = op(A) op(S):                dop(A) = dC op(S)^T  (dds),
                                         dS = op(A)^T dC on the layout (sdd)
    softmax  Y = softmax(scale X):       dX = scale Y (dY - rowsum(Y dY))

Shapes: dense operands [Z, H, rows, cols] (contiguous), block-sparse ones
[Z, nnz, block, block] with the layout's blocks in row-major (h, i, j) order.
"""

from __future__ import annotations

import numpy as np
import torch

from . import bsp

MODES = ("sdd", "dsd", "dds")


def _np_layout(layout) -> np.ndarray:
    if isinstance(layout, torch.Tensor):
        layout = layout.detach().to("cpu").numpy()
    lay = np.ascontiguousarray(layout, dtype=np.uint8)
    if lay.ndim == 2:
        lay = lay[None]
    return lay


def _c(t):
    return t if t.is_contiguous() else t.contiguous()


# ------------------------------------------------------------------ matmul --

def _sdd(L, a, b, ta, tb):
    return bsp.bsp_sdd(L, _c(a), _c(b), trans_a=ta, trans_b=tb)


def _dsd(L, s, b, ta, tb):
    return bsp.bsp_dsd(L, _c(s), _c(b), trans_a=ta, trans_b=tb)


def _dds(L, a, s, ta, tb):
    return bsp.bsp_dds(L, _c(a), _c(s), trans_a=ta, trans_b=tb)


class _Matmul(torch.autograd.Function):
    @staticmethod
    def forward(ctx, a, b, L, mode, ta, tb):
        ctx.L, ctx.mode, ctx.ta, ctx.tb = L, mode, ta, tb
        ctx.save_for_backward(a, b)
        if mode == "sdd":
            return _sdd(L, a, b, ta, tb)
        if mode == "dsd":
            return _dsd(L, a, b, ta, tb)
        return _dds(L, a, b, ta, tb)

    @staticmethod
    def backward(ctx, dc):
        a, b = ctx.saved_tensors
        L, mode, ta, tb = ctx.L, ctx.mode, ctx.ta, ctx.tb
        dc = _c(dc)
        da = db = None
        if mode == "sdd":
            # a, b dense; dc block-sparse
            if ctx.needs_input_grad[0]:
                da = _dds(L, b, dc, tb, 1) if ta else _dsd(L, dc, b, 0, 1 - tb)
            if ctx.needs_input_grad[1]:
                db = _dsd(L, dc, a, 1, ta) if tb else _dds(L, a, dc, 1 - ta, 0)
        elif mode == "dsd":
            # a block-sparse, b dense; dc dense [S, N]
            if ctx.needs_input_grad[0]:
                da = _sdd(L, b, dc, tb, 1) if ta else _sdd(L, dc, b, 0, 1 - tb)
            if ctx.needs_input_grad[1]:
                db = _dds(L, dc, a, 1, ta) if tb else _dsd(L, a, dc, 1 - ta, 0)
        else:
            # a dense, b block-sparse; dc dense [M, S]
            if ctx.needs_input_grad[0]:
                da = _dsd(L, b, dc, tb, 1) if ta else _dds(L, dc, b, 0, 1 - tb)
            if ctx.needs_input_grad[1]:
                db = _sdd(L, dc, a, 1, ta) if tb else _sdd(L, a, dc, 1 - ta, 0)
        return da, db, None, None, None, None


class matmul:
    """Block-sparse matrix product on a fixed layout.

    layout: 0/1 array [H, nb, nb] (or [nb, nb] for one head); block: 16, 32,
    64 or 128; mode: 'sdd', 'dsd' or 'dds' (any case); trans_a / trans_b use
    the transpose of the first / second operand.  Calling the object with
    (a, b) returns the product (block-sparse for 'sdd', dense otherwise)."""

    def __init__(self, layout, block: int, mode: str, trans_a: bool = False, trans_b: bool = False):
        mode = mode.lower()
        if mode not in MODES:
            raise ValueError(f"mode must be one of {MODES}, got {mode!r}")
        self.layout = _np_layout(layout)
        self.block = int(block)
        self.mode = mode
        self.trans_a, self.trans_b = int(bool(trans_a)), int(bool(trans_b))
        self.L = bsp.bsp_layout_compile(self.layout, self.block)

    def __call__(self, a, b):
        return _Matmul.apply(a, b, self.L, self.mode, self.trans_a, self.trans_b)


# ----------------------------------------------------------------- softmax --

class _Softmax(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, L, scale, kind, mask):
        y = bsp.bsp_softmax(L, _c(x), None, scale, kind, mask)
        ctx.L, ctx.scale = L, scale
        ctx.save_for_backward(y)
        return y

    @staticmethod
    def backward(ctx, dy):
        (y,) = ctx.saved_tensors
        return bsp.bsp_softmax_backward(ctx.L, y, _c(dy), None, ctx.scale), None, None, None, None


class softmax:
    """Row softmax over the blocks of an SDD output, on a fixed layout.

    Calling the object with x [Z, nnz, block, block] returns softmax(scale x)
    over each row's present entries.  attn_mask: optional dense keep-mask
    [S, S] (uint8 or bool, 1 = keep, on the device); diagonal_causal: keep only
    columns <= row inside the diagonal blocks.  Masked entries, and rows with
    nothing kept, give 0."""

    def __init__(self, layout, block: int):
        self.layout = _np_layout(layout)
        self.block = int(block)
        self.L = bsp.bsp_layout_compile(self.layout, self.block)

    def __call__(self, x, scale: float = 1.0, attn_mask=None, diagonal_causal: bool = False):
        if attn_mask is not None and diagonal_causal:
            raise ValueError("pass either a dense mask or diagonal_causal")
        kind = bsp.MASK_NONE
        mask = None
        if attn_mask is not None:
            kind = bsp.MASK_DENSE
            mask = _c(attn_mask.to(torch.uint8))
        elif diagonal_causal:
            kind = bsp.MASK_DIAG_CAUSAL
        return _Softmax.apply(x, self.L, float(scale), kind, mask)
