"""GPU parity of the backward pass through the C ABI against the fp64 oracle:
the block-sparse softmax backward (every block size and dtype, in place and
not), the attention backward (dQ, dK, dV; block sizes, dtypes, head sizes,
mask kinds, tensor-core and CUDA-core paths of the forward ops it chains) and
the torch autograd wrapper.

Tolerance (normwise): 1e-5 for fp32 outputs; 2e-2 for bf16 / fp16 softmax
backward outputs and 3e-2 for bf16 / fp16 attention gradients, whose chain
rounds four intermediates (P, dP, dX and the output) to the 16-bit type
(each a relative 2^-9 for bf16) and subtracts a row mean from dP."""

import numpy as np
import pytest
import torch

from gpu_util import TOL, check_softmax_backward_elementwise, dev, normwise_err, to_np
from sparse_attention_layout_gb300 import workloads as W

pytestmark = pytest.mark.gpu

DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}
GRAD_TOL = {torch.float32: 1e-5, torch.bfloat16: 3e-2, torch.float16: 3e-2}


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


def rlayout(H, nb, p, seed):
    lay = (np.random.default_rng(seed).random((H, nb, nb)) < p).astype(np.uint8)
    lay[:, np.arange(nb), np.arange(nb)] = 1
    if nb > 3:
        lay[0, 2, :] = 0   # an empty block-row
    return lay


def randn(shape, dtype, seed):
    return W.randn(shape, {torch.float32: "f32", torch.bfloat16: "bf16", torch.float16: "f16"}[dtype], seed)


def check(got, want, tol, what):
    err = normwise_err(to_np(got), want)
    assert err <= tol, f"{what}: normwise error {err:.3e} > {tol:.0e}"


@pytest.mark.parametrize("B", [16, 32, 64, 128])
@pytest.mark.parametrize("dt", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("in_place", [False, True])
def test_softmax_backward(bsp, oracle, B, dt, in_place):
    dtype = DTYPES[dt]
    Z, H, scale = 2, 2, 0.3
    nb = max(3, 512 // B)
    lay = rlayout(H, nb, 0.3, 60 + B)
    L = bsp.bsp_layout_compile(lay, B)
    # Y: a softmax output (rows sum to 1, zeros at masked entries)
    Y = bsp.bsp_softmax(L, dev(randn((Z, L.nnz, B, B), dtype, 61)), None, 0.5, W.MASK_DIAG_CAUSAL)
    dY = dev(randn((Z, L.nnz, B, B), dtype, 62))
    want = oracle.softmax_backward(lay, B, Y, dY, scale)
    got = bsp.bsp_softmax_backward(L, Y, dY, dY if in_place else None, scale)
    torch.cuda.synchronize()
    check(got, want, TOL[dtype], f"softmax backward B={B} {dt} in_place={in_place}")


@pytest.mark.parametrize("B", [16, 32, 64, 128])
@pytest.mark.parametrize("dt", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("kind", [0, 1, 2])
def test_attention_backward(bsp, oracle, path, B, dt, D, kind):
    dtype = DTYPES[dt]
    Z, H, scale = 2, 2, 1.0 / np.sqrt(D)
    nb = max(4, 384 // B)  # >= 4: block-row 2 is empty
    S = nb * B
    lay = rlayout(H, nb, 0.4, 70 + B)
    L = bsp.bsp_layout_compile(lay, B)
    Q, K, V, G = (randn((Z, H, S, D), dtype, s) for s in (71, 72, 73, 74))
    mask = W.random_mask(S, 0.7, 75) if kind == W.MASK_DENSE else None
    dmask = None if mask is None else torch.from_numpy(mask).cuda()
    dQ, dK, dV = bsp.attention_backward(L, dev(Q), dev(K), dev(V), dev(G), scale, kind, dmask)
    torch.cuda.synchronize()
    wQ, wK, wV = oracle.attention_backward(lay, B, Q, K, V, G, scale, kind, mask)
    tol = GRAD_TOL[dtype]
    check(dV, wV, tol, f"dV B={B} {dt} D={D} kind={kind} {path}")
    check(dQ, wQ, tol, f"dQ B={B} {dt} D={D} kind={kind} {path}")
    check(dK, wK, tol, f"dK B={B} {dt} D={D} kind={kind} {path}")
    # the empty block-row gets no query gradient
    assert (dQ[0, 0, 2 * B:3 * B] == 0).all()


@pytest.mark.parametrize("B", [64, 128])
@pytest.mark.parametrize("D", [32, 96])
@pytest.mark.parametrize("kind", [0, 1, 2])
@pytest.mark.parametrize("with_stats", [False, True])
def test_attention_backward_other_head_sizes(bsp, oracle, B, D, kind, with_stats):
    # head sizes outside the fused forward's (64, 128): the recomputing backward
    # takes its chain (fused dP + softmax backward on the tensor cores), the
    # backward from O and lse the one-pass P + dX kernel and a DSD for dQ
    dtype = torch.bfloat16
    Z, H, scale = 2, 2, 1.0 / np.sqrt(D)
    nb = max(4, 384 // B)
    S = nb * B
    lay = rlayout(H, nb, 0.4, 60 + B)
    L = bsp.bsp_layout_compile(lay, B)
    Q, K, V, G = (randn((Z, H, S, D), dtype, s) for s in (61, 62, 63, 64))
    mask = W.random_mask(S, 0.7, 65) if kind == W.MASK_DENSE else None
    dmask = None if mask is None else torch.from_numpy(mask).cuda()
    q, k, v, g = dev(Q), dev(K), dev(V), dev(G)
    if with_stats:
        O, lse = bsp.bsp_attention_lse(L, q, k, v, None, None, scale, kind, dmask)
        dQ, dK, dV = bsp.attention_backward_lse(L, q, k, v, O, g, lse, scale, kind, dmask)
    else:
        dQ, dK, dV = bsp.attention_backward(L, q, k, v, g, scale, kind, dmask)
    torch.cuda.synchronize()
    assert bsp.bsp_status_check(L) == 0
    wQ, wK, wV = oracle.attention_backward(lay, B, Q, K, V, G, scale, kind, mask)
    tol = GRAD_TOL[dtype]
    what = f"B={B} D={D} kind={kind} stats={with_stats}"
    check(dV, wV, tol, f"dV {what}")
    check(dQ, wQ, tol, f"dQ {what}")
    check(dK, wK, tol, f"dK {what}")
    assert (dQ[0, 0, 2 * B:3 * B] == 0).all()


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_autograd_wrapper(bsp, oracle, dt):
    dtype = DTYPES[dt]
    Z, H, B, D, scale = 1, 3, 64, 64, 0.125
    nb = 6
    S = nb * B
    lay = W.layout_strided_causal(nb, local_blocks=2, stride=3, H=H)
    L = bsp.bsp_layout_compile(lay, B)
    Q, K, V, G = (randn((Z, H, S, D), dtype, s) for s in (81, 82, 83, 84))
    q, k, v = (dev(t).requires_grad_() for t in (Q, K, V))
    out = bsp.block_sparse_attention(L, q, k, v, scale, W.MASK_DIAG_CAUSAL)
    out.backward(dev(G))
    torch.cuda.synchronize()
    check(out, oracle.attention(lay, B, Q, K, V, scale, W.MASK_DIAG_CAUSAL), TOL[dtype], f"autograd forward {dt}")
    wQ, wK, wV = oracle.attention_backward(lay, B, Q, K, V, G, scale, W.MASK_DIAG_CAUSAL)
    for got, want, name in ((q.grad, wQ, "dQ"), (k.grad, wK, "dK"), (v.grad, wV, "dV")):
        check(got, want, GRAD_TOL[dtype], f"autograd {name} {dt}")


def test_backward_empty_layout_and_zero_batch(bsp):
    lay = np.zeros((2, 4, 4), np.uint8)
    L = bsp.bsp_layout_compile(lay, 32)
    Q = torch.randn(1, 2, 128, 64, device="cuda", dtype=torch.bfloat16)
    dQ, dK, dV = bsp.attention_backward(L, Q, Q, Q, Q, 0.1)
    torch.cuda.synchronize()
    assert all((t == 0).all() for t in (dQ, dK, dV))
    E = torch.empty(0, 2, 128, 64, device="cuda", dtype=torch.bfloat16)
    dQ, dK, dV = bsp.attention_backward(bsp.bsp_layout_compile(np.ones((2, 4, 4), np.uint8), 32), E, E, E, E, 0.1)
    assert dQ.shape == E.shape


@pytest.mark.parametrize("B,dt,nb", [(128, "bf16", 16), (64, "f32", 24), (32, "f16", 48)])
def test_softmax_backward_long_rows(bsp, oracle, B, dt, nb):
    """Rows longer than the register-resident limit (160 vectors of 16 bytes
    a row for 16-bit types, 320 for fp32) take the two-pass path."""
    dtype = DTYPES[dt]
    scale = 0.2
    lay = np.ones((1, nb, nb), np.uint8)
    L = bsp.bsp_layout_compile(lay, B)
    elt = torch.tensor([], dtype=dtype).element_size()
    assert nb * B * elt // 16 > 160 * elt // 2
    Y = bsp.bsp_softmax(L, dev(randn((1, L.nnz, B, B), dtype, 91)), None, 0.4)
    dY = dev(randn((1, L.nnz, B, B), dtype, 92))
    got = bsp.bsp_softmax_backward(L, Y, dY, None, scale)
    torch.cuda.synchronize()
    check(got, oracle.softmax_backward(lay, B, Y, dY, scale), TOL[dtype], f"long rows B={B} {dt}")


# ------------------------------------------ softmax backward: kernel paths ----

def eye_plus_row(nb, i):
    lay = np.eye(nb, dtype=np.uint8)[None].copy()
    lay[0, i, :] = 1
    return lay


def band_plus_row(nb, w, i):
    lay = W.layout_band(nb, w)
    lay[0, i, :] = 1
    return lay


def cyclic_band(nb, w):
    d = (np.arange(nb)[None, :] - np.arange(nb)[:, None]) % nb
    return ((d <= w) | (d >= nb - w)).astype(np.uint8)[None]


# (B, dtype, layout, kernel): the backward runs on the chunk kernel when the
# layout has a row past 160 vectors of 16 bytes and the largest chunk of the
# softmax's list is at most 48 KB per array, else on the one-warp-per-row
# kernel, launched for 3 blocks per SM (fp32, or rows averaging more than 128
# vectors) or 4
SMB_CASES = {
    # rows of 1..24 blocks of 64 bf16: 8, 16 and 32 lanes a row in registers,
    # and rows past 160 vectors (one warp a row, eight rows a chunk)
    "lanes_8_16_32_and_long_bf16": (64, "bf16", lambda: W.layout_causal_blocks(24), "chunk"),
    # the same for fp32 (4 elements a vector, 10 vectors a lane): rows of
    # 1..48 blocks of 32
    "lanes_8_16_32_and_long_f32": (32, "f32", lambda: W.layout_causal_blocks(48), "chunk"),
    # a bf16 row of 100 blocks of 64 (12.5 KB): two rows a chunk, two warps
    # a row
    "two_warps_a_row": (64, "bf16", lambda: eye_plus_row(100, 50), "chunk"),
    # one fp32 row of 600 blocks of 16 (37.5 KB): one row a chunk, four warps
    "four_warps_a_row": (16, "f32", lambda: eye_plus_row(600, 300), "chunk"),
    # rows of 5 to 9 blocks of 128 bf16 (at most 144 vectors, 124 on
    # average): every row in the row kernel's registers, 4 blocks per SM
    "row_kernel_registers_4": (128, "bf16", lambda: W.layout_band(16, 4), "rows4"),
    # every row 9 blocks of 128 bf16 (144 vectors): 3 blocks per SM
    "row_kernel_registers_3": (128, "bf16", lambda: cyclic_band(16, 4), "rows3"),
    # fp32 rows of up to 7 blocks of 32: 3 blocks per SM
    "row_kernel_registers_f32": (32, "f32", lambda: W.layout_band(32, 3), "rows3"),
    # fp16, a row of 200 blocks of 128 (50 KB): the row kernel (its
    # register path for the diagonal rows, two passes for the long row)
    "row_kernel_fallback": (128, "f16", lambda: eye_plus_row(200, 7), "rows4"),
    # the same long row over a band of 9 blocks a row (159 vectors on
    # average): two passes at 3 blocks per SM
    "row_kernel_fallback_3": (128, "f16", lambda: band_plus_row(200, 4, 7), "rows3"),
    # a row longer than the largest chunk (66.5 KB): the row kernel
    "row_kernel_unchunked": (128, "bf16", lambda: eye_plus_row(260, 0), "rows4"),
}


@pytest.mark.parametrize("case", list(SMB_CASES))
def test_softmax_backward_kernel_paths(bsp, oracle, case):
    B, dt, mk, kernel = SMB_CASES[case]
    dtype = DTYPES[dt]
    scale = 0.35
    lay = mk()
    L = bsp.bsp_layout_compile(lay, B)
    elt = torch.tensor([], dtype=dtype).element_size()
    ch = L.softmax_chunks(elt)
    R = ch["items"][:, 3] >> 16
    rows_blocks = ch["items"][:, 2]
    vec_per_row = rows_blocks * B * elt // 16
    on_chunks = ch["fits"] and ch["max_bytes"] <= 48 * 1024 and vec_per_row.max() > 160
    assert on_chunks == (kernel == "chunk"), (case, ch["fits"], ch["max_bytes"])
    if not on_chunks:
        mean_vec = L.nnz * B * elt // 16 // (lay.shape[0] * lay.shape[1])
        assert kernel == ("rows3" if elt == 4 or mean_vec > 128 else "rows4"), (case, mean_vec)
    if case.startswith("lanes"):
        regs = 40 * elt // 16  # vectors a lane holds
        for lo, hi in ((0, 8 * regs), (8 * regs, 16 * regs), (16 * regs, 32 * regs), (32 * regs, 1 << 30)):
            assert ((vec_per_row > lo) & (vec_per_row <= hi)).any(), (case, lo, hi)
    if case == "two_warps_a_row":
        assert (R == 2).any() and (vec_per_row[R == 2] > 160).all()
    if case == "four_warps_a_row":
        assert (R == 1).any()
    Z = 2 if L.nnz * B * B <= 4 << 20 else 1
    Y = bsp.bsp_softmax(L, dev(randn((Z, L.nnz, B, B), dtype, 95)), None, 0.7)
    dY = dev(randn((Z, L.nnz, B, B), dtype, 96))
    got = bsp.bsp_softmax_backward(L, Y, dY, None, scale)
    torch.cuda.synchronize()
    assert bsp.bsp_status_check(L) == 0
    want = oracle.softmax_backward(lay, B, Y, dY, scale)
    check_softmax_backward_elementwise(lay, B, Y, dY, got, want, scale, dtype, case)
    # in place (dX = dY): the same bytes
    dY2 = dY.clone()
    bsp.bsp_softmax_backward(L, Y, dY2, dY2, scale)
    torch.cuda.synchronize()
    assert torch.equal(dY2, got)


# ------------------------------------------- forward lse + backward_lse ----

def lse_bound(Q, K, scale, n_keys):
    """|lse_gpu - lse_oracle| per row: the score error of an fp32 accumulation
    of D products, scale * gamma(D) * |q| * max|k| (Cauchy-Schwarz), plus the
    relative error of a sum of n_keys exponentials (2^-22 each, 2^-24 per
    addition with a factor 4 for tensor-core adders), plus the rounding of
    the logarithm and the final products (2^-22 of |lse| and an absolute
    2^-22)."""
    from gpu_util import gamma
    q = Q.double().norm(dim=-1)                      # [Z, H, S]
    kmax = K.double().norm(dim=-1).amax(dim=-1, keepdim=True)
    return (scale * gamma(Q.shape[-1]) * q * kmax + (n_keys + 4) * 2.0 ** -22).numpy()


@pytest.mark.parametrize("B", [16, 64, 128])
@pytest.mark.parametrize("dt", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("kind", [0, 1, 2])
def test_attention_lse(bsp, oracle, path, B, dt, D, kind):
    # the forward's O is the plain forward's, byte for byte; lse matches the
    # oracle's log-sum-exp row by row (-inf exactly for rows with nothing kept)
    dtype = DTYPES[dt]
    Z, H, scale = 2, 2, 1.0 / np.sqrt(D)
    nb = max(4, 384 // B) + 1
    S = nb * B
    lay = rlayout(H, nb, 0.35, 110 + B)
    mask = W.random_mask(S, 0.7, 111) if kind == W.MASK_DENSE else None
    dmask = None if mask is None else torch.from_numpy(mask).cuda()
    Q, K, V = (randn((Z, H, S, D), dtype, s) for s in (112, 113, 114))
    q, k, v = dev(Q), dev(K), dev(V)
    L = bsp.bsp_layout_compile(lay, B)
    O, lse = bsp.bsp_attention_lse(L, q, k, v, None, None, scale, kind, dmask)
    O0 = bsp.bsp_attention(L, q, k, v, None, scale, kind, dmask)
    torch.cuda.synchronize()
    assert bsp.bsp_status_check(L) == 0
    assert torch.equal(O, O0), "bsp_attention_lse's O differs from bsp_attention's"
    want = oracle.attention_lse(lay, B, Q, K, scale, kind, mask)
    got = lse.cpu().double().numpy()
    empty = np.isneginf(want)
    assert empty.any()
    assert np.all(np.isneginf(got[empty])), "rows with nothing kept must have lse = -inf"
    err = np.abs(got[~empty] - want[~empty])
    bound = lse_bound(Q, K, scale, S)[~empty] + 2.0 ** -22 * np.abs(want[~empty])
    worst = np.argmax(err - bound)
    assert np.all(err <= bound), f"lse B={B} {dt} D={D} kind={kind} {path}: error {err[worst]:.3e} > {bound[worst]:.3e}"


@pytest.mark.parametrize("B", [16, 32, 64, 128])
@pytest.mark.parametrize("dt", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("kind", [0, 1, 2])
def test_attention_backward_lse(bsp, oracle, path, B, dt, D, kind):
    # gradients from the forward's O and lse: the oracle's, within the same
    # tolerance as the recomputing chain
    dtype = DTYPES[dt]
    Z, H, scale = 2, 2, 1.0 / np.sqrt(D)
    nb = max(4, 384 // B)  # >= 4: block-row 2 is empty
    S = nb * B
    lay = rlayout(H, nb, 0.4, 70 + B)
    L = bsp.bsp_layout_compile(lay, B)
    Q, K, V, G = (randn((Z, H, S, D), dtype, s) for s in (71, 72, 73, 74))
    mask = W.random_mask(S, 0.7, 75) if kind == W.MASK_DENSE else None
    dmask = None if mask is None else torch.from_numpy(mask).cuda()
    q, k, v, g = dev(Q), dev(K), dev(V), dev(G)
    O, lse = bsp.bsp_attention_lse(L, q, k, v, None, None, scale, kind, dmask)
    dQ, dK, dV = bsp.attention_backward_lse(L, q, k, v, O, g, lse, scale, kind, dmask)
    torch.cuda.synchronize()
    assert bsp.bsp_status_check(L) == 0
    wQ, wK, wV = oracle.attention_backward(lay, B, Q, K, V, G, scale, kind, mask)
    tol = GRAD_TOL[dtype]
    check(dV, wV, tol, f"dV (lse) B={B} {dt} D={D} kind={kind} {path}")
    check(dQ, wQ, tol, f"dQ (lse) B={B} {dt} D={D} kind={kind} {path}")
    check(dK, wK, tol, f"dK (lse) B={B} {dt} D={D} kind={kind} {path}")
    assert (dQ[0, 0, 2 * B:3 * B] == 0).all()


@pytest.mark.parametrize("dt", ["bf16", "f16"])
@pytest.mark.parametrize("kind", [0, 1, 2])
def test_attention_backward_lse_partial_row_tile(bsp, oracle, dt, kind):
    # blocks of 64 and an odd block count: the last row tile holds one block-row
    # and rows past the sequence end; the one-pass kernel that also accumulates
    # dQ (head size 128) writes only the rows inside the sequence
    dtype = DTYPES[dt]
    B, nb, D, Z, H = 64, 7, 128, 3, 2
    S, scale = nb * B, 1.0 / np.sqrt(D)
    lay = rlayout(H, nb, 0.45, 90 + kind)
    lay[:, nb - 1, :] = 0
    lay[0, nb - 1, nb - 1] = 1  # head 0: the last block-row keeps its diagonal block only
    L = bsp.bsp_layout_compile(lay, B)
    Q, K, V, G = (randn((Z, H, S, D), dtype, s) for s in (91, 92, 93, 94))
    mask = W.random_mask(S, 0.7, 95) if kind == W.MASK_DENSE else None
    dmask = None if mask is None else torch.from_numpy(mask).cuda()
    q, k, v, g = dev(Q), dev(K), dev(V), dev(G)
    O, lse = bsp.bsp_attention_lse(L, q, k, v, None, None, scale, kind, dmask)
    dQ, dK, dV = bsp.attention_backward_lse(L, q, k, v, O, g, lse, scale, kind, dmask)
    torch.cuda.synchronize()
    assert bsp.bsp_status_check(L) == 0
    wQ, wK, wV = oracle.attention_backward(lay, B, Q, K, V, G, scale, kind, mask)
    tol = GRAD_TOL[dtype]
    check(dV, wV, tol, f"dV (lse, partial tile) {dt} kind={kind}")
    check(dQ, wQ, tol, f"dQ (lse, partial tile) {dt} kind={kind}")
    check(dK, wK, tol, f"dK (lse, partial tile) {dt} kind={kind}")
    assert (dQ[:, 1, (nb - 1) * B:] == 0).all(), "head 1's last block-row keeps nothing: dQ = 0 there"


def test_lse_pair_empty_layout_and_zero_batch(bsp):
    # nothing kept anywhere: O = 0, lse = -inf, every gradient 0; Z = 0: no work
    lay = np.zeros((2, 4, 4), np.uint8)
    L = bsp.bsp_layout_compile(lay, 32)
    Q = torch.randn(1, 2, 128, 64, device="cuda", dtype=torch.bfloat16)
    O, lse = bsp.bsp_attention_lse(L, Q, Q, Q, None, None, 0.1)
    dQ, dK, dV = bsp.attention_backward_lse(L, Q, Q, Q, O, Q, lse, 0.1)
    torch.cuda.synchronize()
    assert (O == 0).all() and torch.isneginf(lse).all()
    assert all((t == 0).all() for t in (dQ, dK, dV))
    E = torch.empty(0, 2, 128, 64, device="cuda", dtype=torch.bfloat16)
    L1 = bsp.bsp_layout_compile(np.ones((2, 4, 4), np.uint8), 32)
    O, lse = bsp.bsp_attention_lse(L1, E, E, E, None, None, 0.1)
    dQ, dK, dV = bsp.attention_backward_lse(L1, E, E, E, O, E, lse, 0.1)
    assert dQ.shape == E.shape and lse.shape == (0, 2, 128)


def test_backward_lse_rejects_missing_statistics(bsp):
    L = bsp.bsp_layout_compile(np.ones((1, 2, 2), np.uint8), 64)
    Q = torch.randn(1, 1, 128, 64, device="cuda", dtype=torch.bfloat16)
    ws = torch.empty(1, 4, 64, 64, device="cuda", dtype=torch.bfloat16)
    f = bsp.lib().bsp_attention_backward_lse
    p = bsp._ptr
    lse = torch.zeros(1, 1, 128, device="cuda")
    # no lse, no O: BSP_ERR_INVALID_ARG; misaligned lse: BSP_ERR_ALIGNMENT
    assert f(L.handle, 1, p(Q), p(Q), p(Q), p(Q), p(Q), None, p(Q), p(Q), p(Q), 1, 64, 0.1, 0, None, p(ws), p(ws),
             None) == -1
    assert f(L.handle, 1, p(Q), p(Q), p(Q), None, p(Q), p(lse), p(Q), p(Q), p(Q), 1, 64, 0.1, 0, None, p(ws), p(ws),
             None) == -1
    bad = bsp.ctypes.c_void_p(lse.data_ptr() + 4)
    assert f(L.handle, 1, p(Q), p(Q), p(Q), p(Q), p(Q), bad, p(Q), p(Q), p(Q), 1, 64, 0.1, 0, None, p(ws), p(ws),
             None) == -3
