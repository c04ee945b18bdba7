"""The kernels' failure paths, provoked on purpose without a fault: a bounded
wait that runs out, and a bounds check that fails.

bsp_diag_wait_limit shortens the wait limit of the handle's tensor-core
kernels and injects one of two failures into the fused attention kernel: the
first Q tile of every CTA is never loaded nor signalled (the Q K^T issuer's
wait runs out), or the K producer sees a block-column outside the layout for
its first step (its bounds check fires before the column becomes a copy
coordinate; an out-of-range copy coordinate would only read the fill value).
Either way every role stops, waits for what it had issued, frees its tensor
memory and returns.  The call must end within a small multiple of the
limit, the status word must hold the right code, and the next call on the
same handle, with the injection off, must match the oracle."""

import time

import numpy as np
import pytest
import torch

from gpu_util import assert_close, attention_acc, to_np
from sparse_attention_layout_gb300 import workloads as W

pytestmark = pytest.mark.gpu

LIMIT_NS = 5_000_000  # 5 ms


@pytest.fixture(scope="module")
def bsp():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from sparse_attention_layout_gb300 import build
    build.build()
    from sparse_attention_layout_gb300 import bsp as m
    return m


def _case():
    B, nb, H, Z, D = 64, 8, 2, 2, 64
    lay = W.layout_strided_causal(nb, local_blocks=3, stride=3, H=H)
    Q, K, V = (W.randn((Z, H, nb * B, D), "bf16", 800 + s) for s in range(3))
    return lay, B, Q, K, V, 1.0 / np.sqrt(D)


@pytest.mark.parametrize("inject,code", [("skip_first_q", -6), ("bad_column", -7)])
def test_attention_failure_path_reports_and_recovers(bsp, oracle, inject, code):
    lay, B, Q, K, V, scale = _case()
    L = bsp.bsp_layout_compile(lay, B)
    q, k, v = (t.cuda() for t in (Q, K, V))
    bits = {"skip_first_q": bsp.INJECT_SKIP_FIRST_Q, "bad_column": bsp.INJECT_BAD_COLUMN}[inject]
    bsp.bsp_diag_wait_limit(L, LIMIT_NS, bits)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    bsp.bsp_attention(L, q, k, v, None, scale, W.MASK_DIAG_CAUSAL)
    status = bsp.bsp_status_check(L)  # synchronises
    elapsed = time.perf_counter() - t0
    assert status == code, f"{inject}: status {status}, expected {code}"
    assert elapsed < 2.0, f"{inject}: the failing call took {elapsed:.2f} s"
    assert bsp.bsp_status_check(L) == 0  # read and cleared
    # the same handle, the default limit, no injection: a correct result
    bsp.bsp_diag_wait_limit(L, 0, 0)
    O = bsp.bsp_attention(L, q, k, v, None, scale, W.MASK_DIAG_CAUSAL)
    torch.cuda.synchronize()
    assert bsp.bsp_status_check(L) == 0
    want = oracle.attention(lay, B, Q, K, V, scale, W.MASK_DIAG_CAUSAL)
    mag = oracle.attention(lay, B, Q, K, V.abs(), scale, W.MASK_DIAG_CAUSAL)
    assert_close(to_np(O), want, torch.bfloat16, f"attention after {inject}", mag=mag,
                 acc=attention_acc(Q, K, scale, torch.bfloat16, lay.shape[1] * B))
    # and the other kernels of the handle still run (SDD, softmax, DSD chain)
    O2 = bsp.attention_unfused(L, q, k, v, scale, W.MASK_DIAG_CAUSAL)
    torch.cuda.synchronize()
    assert bsp.bsp_status_check(L) == 0
    assert_close(to_np(O2), want, torch.bfloat16, f"unfused chain after {inject}")


def test_short_wait_limit_without_injection_is_harmless(bsp, oracle):
    # a 50 ms limit is far above any legal wait of these small launches
    lay, B, Q, K, V, scale = _case()
    L = bsp.bsp_layout_compile(lay, B)
    bsp.bsp_diag_wait_limit(L, 50_000_000, 0)
    q, k, v = (t.cuda() for t in (Q, K, V))
    O = bsp.bsp_attention(L, q, k, v, None, scale, W.MASK_DIAG_CAUSAL)
    P = bsp.bsp_sdd_softmax(L, q, k, None, scale, W.MASK_DIAG_CAUSAL)
    O2 = bsp.bsp_dsd(L, P, v)
    torch.cuda.synchronize()
    assert bsp.bsp_status_check(L) == 0
    want = oracle.attention(lay, B, Q, K, V, scale, W.MASK_DIAG_CAUSAL)
    assert_close(to_np(O), want, torch.bfloat16, "attention, 50 ms limit")
    assert_close(to_np(O2), want, torch.bfloat16, "fused SDD + softmax -> DSD, 50 ms limit")


def test_short_wait_limit_softmax_chunk_kernels(bsp, oracle):
    """The softmax's chunk kernel and the softmax backward's (a layout with a
    row past the backward row kernel's registers) wait on their bulk copies
    with the handle's limit: a 50 ms limit leaves them correct, and the
    backward's row kernel (no waits) on a short-row layout as well."""
    from gpu_util import PROB_TOL, check_softmax_backward_elementwise, softmax_zero_positions
    B, scale = 64, 0.5
    long_rows = W.layout_causal_blocks(24)          # rows of 1..24 blocks of 64 bf16
    short_rows = W.layout_band(24, 2)               # rows of at most 5 blocks
    for lay in (long_rows, short_rows):
        L = bsp.bsp_layout_compile(lay, B)
        bsp.bsp_diag_wait_limit(L, 50_000_000, 0)
        X = W.randn((2, L.nnz, B, B), "bf16", 41)
        Y = bsp.bsp_softmax(L, X.cuda(), None, scale, W.MASK_DIAG_CAUSAL)
        dY = W.randn((2, L.nnz, B, B), "bf16", 42).cuda()
        dX = bsp.bsp_softmax_backward(L, Y, dY, None, scale)
        torch.cuda.synchronize()
        assert bsp.bsp_status_check(L) == 0
        want = oracle.softmax(lay, B, X, scale, W.MASK_DIAG_CAUSAL)
        assert_close(to_np(Y), want, torch.bfloat16, "softmax, 50 ms limit", rel=PROB_TOL[torch.bfloat16],
                     zeros=softmax_zero_positions(lay, B, 2, W.MASK_DIAG_CAUSAL))
        check_softmax_backward_elementwise(lay, B, Y, dY, dX, oracle.softmax_backward(lay, B, Y, dY, scale),
                                           scale, torch.bfloat16, "softmax backward, 50 ms limit")


def test_wait_limit_rejects_unknown_injection(bsp):
    L = bsp.bsp_layout_compile(np.ones((1, 2, 2), np.uint8), 64)
    with pytest.raises(bsp.BspError) as e:
        bsp.bsp_diag_wait_limit(L, 0, 4)
    assert e.value.code == -1
