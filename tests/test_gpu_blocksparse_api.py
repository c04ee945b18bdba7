"""The blocksparse module (matmul in its three modes, softmax; the API shape
of "question on blocksparse", openai/triton issue 117): forward results and
autograd gradients against a dense float64 torch reference on the CPU, whose
gradients come from torch's own autograd (so the mode-to-mode gradient
mapping of the module is checked independently).  Tolerances: normwise 1e-5
for fp32, 2e-2 for bf16."""

import numpy as np
import pytest
import torch

from gpu_util import normwise_err

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-5, torch.bfloat16: 2e-2}


@pytest.fixture(scope="module")
def bs():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from sparse_attention_layout_gb300 import build
    build.build()
    from sparse_attention_layout_gb300 import blocksparse
    return blocksparse


def rlayout(H, nb, p, seed):
    lay = (np.random.default_rng(seed).random((H, nb, nb)) < p).astype(np.uint8)
    lay[:, np.arange(nb), np.arange(nb)] = 1  # every row and column has a block
    return lay


def to_dense(lay, B, X):
    """[Z, nnz, B, B] -> [Z, H, S, S] (zeros outside the layout)."""
    H, nb, _ = lay.shape
    Z = X.shape[0]
    D = torch.zeros(Z, H, nb * B, nb * B, dtype=X.dtype)
    for n, (h, i, j) in enumerate(zip(*np.nonzero(lay))):
        D[:, h, i * B:(i + 1) * B, j * B:(j + 1) * B] = X[:, n]
    return D


def to_blocks(lay, B, D):
    return torch.stack([D[:, h, i * B:(i + 1) * B, j * B:(j + 1) * B] for h, i, j in zip(*np.nonzero(lay))], 1)


def mask_of(lay, B):
    return torch.from_numpy(np.kron(lay, np.ones((B, B), np.uint8))).double()


def op(x, t):
    return x.transpose(-1, -2) if t else x


def close(got, want, dtype, what):
    err = normwise_err(got.detach().float().cpu().numpy(), want.detach().numpy())
    assert err <= TOL[dtype], f"{what}: normwise error {err:.3e}"


@pytest.mark.parametrize("mode", ["sdd", "dsd", "dds"])
@pytest.mark.parametrize("trans", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_matmul_forward_and_gradients(bs, mode, trans, dt):
    dtype = {"f32": torch.float32, "bf16": torch.bfloat16}[dt]
    ta, tb = trans
    B, nb, H, Z, K = 32, 5, 2, 2, 48
    S = nb * B
    lay = rlayout(H, nb, 0.4, 7 + 3 * ta + tb)
    g = torch.Generator().manual_seed(11)

    def rnd(*shape):
        return torch.randn(*shape, generator=g).to(dtype)

    nnz = int(lay.sum())
    M = mask_of(lay, B)
    if mode == "sdd":
        a, b = rnd(Z, H, *((K, S) if ta else (S, K))), rnd(Z, H, *((S, K) if tb else (K, S)))
    elif mode == "dsd":
        a, b = rnd(Z, nnz, B, B), rnd(Z, H, *((K, S) if tb else (S, K)))
    else:
        a, b = rnd(Z, H, *((S, K) if ta else (K, S))), rnd(Z, nnz, B, B)
    # reference: float64 dense, gradients by torch autograd
    ar, br = a.double().requires_grad_(), b.double().requires_grad_()
    if mode == "sdd":
        cr = to_blocks(lay, B, (op(ar, ta) @ op(br, tb)) * M)
    elif mode == "dsd":
        cr = op(to_dense(lay, B, ar), ta) @ op(br, tb)
    else:
        cr = op(ar, ta) @ op(to_dense(lay, B, br), tb)
    gc = rnd(*cr.shape)
    (cr * gc.double()).sum().backward()
    # the module on the GPU
    mm = bs.matmul(lay, B, mode, trans_a=bool(ta), trans_b=bool(tb))
    ag, bg = a.cuda().requires_grad_(), b.cuda().requires_grad_()
    c = mm(ag, bg)
    c.backward(gc.cuda())
    torch.cuda.synchronize()
    what = f"{mode} trans={trans} {dt}"
    close(c, cr, dtype, what + " forward")
    close(ag.grad, ar.grad, dtype, what + " grad a")
    close(bg.grad, br.grad, dtype, what + " grad b")


@pytest.mark.parametrize("kind", ["none", "dense", "diag"])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_softmax_forward_and_gradient(bs, kind, dt):
    dtype = {"f32": torch.float32, "bf16": torch.bfloat16}[dt]
    B, nb, H, Z, scale = 32, 6, 2, 2, 0.4
    S = nb * B
    lay = rlayout(H, nb, 0.4, 21)
    g = torch.Generator().manual_seed(12)
    x = torch.randn(Z, int(lay.sum()), B, B, generator=g).to(dtype)
    keep = mask_of(lay, B).bool()
    dense_mask = None
    if kind == "dense":
        dense_mask = torch.rand(S, S, generator=g) < 0.8
        dense_mask[torch.arange(S), torch.arange(S)] = True  # no row left empty
        keep = keep & dense_mask
    elif kind == "diag":
        blk = torch.arange(S) // B
        same = blk[:, None] == blk[None, :]
        keep = keep & (~same | (torch.arange(S)[None, :] <= torch.arange(S)[:, None]))
    xr = x.double().requires_grad_()
    logits = (scale * to_dense(lay, B, xr)).masked_fill(~keep, float("-inf"))
    yr = to_blocks(lay, B, torch.softmax(logits, dim=-1))
    gy = torch.randn(yr.shape, generator=g).to(dtype)
    (yr * gy.double()).sum().backward()
    sm = bs.softmax(lay, B)
    xg = x.cuda().requires_grad_()
    y = sm(xg, scale=scale, attn_mask=None if dense_mask is None else dense_mask.cuda(),
           diagonal_causal=kind == "diag")
    y.backward(gy.cuda())
    torch.cuda.synchronize()
    close(y, yr, dtype, f"softmax {kind} {dt} forward")
    close(xg.grad, xr.grad, dtype, f"softmax {kind} {dt} grad")


def test_attention_through_the_module(bs):
    # SDD -> softmax -> DSD built from the module, gradients for Q, K, V
    B, nb, H, Z, D, scale = 64, 4, 2, 1, 64, 0.125
    S = nb * B
    lay = rlayout(H, nb, 0.5, 31)
    g = torch.Generator().manual_seed(13)
    q, k, v = (torch.randn(Z, H, S, D, generator=g) for _ in range(3))
    sdd = bs.matmul(lay, B, "sdd", trans_b=True)
    sm = bs.softmax(lay, B)
    dsd = bs.matmul(lay, B, "dsd")
    qg, kg, vg = (t.cuda().requires_grad_() for t in (q, k, v))
    o = dsd(sm(sdd(qg, kg), scale=scale), vg)
    go = torch.randn(o.shape, generator=g)
    o.backward(go.cuda())
    qr, kr, vr = (t.double().requires_grad_() for t in (q, k, v))
    logits = (scale * qr @ kr.transpose(-1, -2)).masked_fill(mask_of(lay, B) == 0, float("-inf"))
    orf = torch.softmax(logits, -1) @ vr
    (orf * go.double()).sum().backward()
    torch.cuda.synchronize()
    for got, want, name in ((o, orf, "O"), (qg.grad, qr.grad, "dQ"), (kg.grad, kr.grad, "dK"), (vg.grad, vr.grad, "dV")):
        close(got, want, torch.float32, f"module attention {name}")
