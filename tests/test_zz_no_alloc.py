"""bsp_softmax_noalloc: the softmax entry point for callers that cannot
allocate device memory (a runtime that owns every byte of the GPU, a plugin
handed only its buffers).  It keeps the layout tables in a fixed device array
the library declares itself instead of a compiled handle.

Checked through the C ABI against the fp64 oracle (elementwise bound, masked
entries exactly 0) and against the existing entry point (bsp_softmax with a
compiled handle, which runs the same kernels on the same tables: identical
bytes), on calls in a row with different layouts, block sizes, dtypes (fp32,
bf16, fp16) and masks, so a call must not depend on what the previous one left
in the shared array; one layout has a row longer than the largest softmax
chunk, which takes the one-warp-per-row kernel.  Collected last (file name) so
that a run stopping at the first failure has already run every other test."""

import ctypes

import numpy as np
import pytest
import torch

from gpu_util import PROB_TOL, assert_close, softmax_zero_positions, to_np
from sparse_attention_layout_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from sparse_attention_layout_gb300 import build
    build.build()
    from sparse_attention_layout_gb300 import bsp
    L = bsp.lib()
    P, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    L.bsp_softmax_noalloc.argtypes = [P, i32, i32, i32, i32, P, P, i32, f32, i32, P, P]
    L.bsp_softmax_noalloc.restype = i32
    return L


def _call(lib, lay, B, code, X, Y, scale, kind, mask):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    lay = np.ascontiguousarray(lay, dtype=np.uint8)
    return lib.bsp_softmax_noalloc(ctypes.c_void_p(lay.ctypes.data), lay.shape[0], lay.shape[1], B, code,
                                   ctypes.c_void_p(X.data_ptr()), ctypes.c_void_p(Y.data_ptr()), X.shape[0],
                                   float(scale), kind,
                                   ctypes.c_void_p(0 if mask is None else mask.data_ptr()), stream)


def _long_row_layout(nb):
    lay = np.eye(nb, dtype=np.uint8)[None].copy()
    lay[0, nb // 2, :] = 1
    return lay


def test_noalloc_softmax_matches_oracle_and_compiled_handle(lib, oracle):
    from sparse_attention_layout_gb300 import bsp
    cases = [  # (layout, block, dtype, mask kind, scale)
        (W.layout_strided_causal(16, local_blocks=4, stride=4, H=3), 64, torch.bfloat16, W.MASK_DIAG_CAUSAL, 0.09),
        (W.layout_random_diag(20, 0.3, H=2, seed=5), 32, torch.float32, W.MASK_DENSE, 0.3),
        # 260 blocks of 128 fp16 in one block-row: 66 560-byte rows, past the
        # 64 KB chunk budget (one warp per row)
        (_long_row_layout(260), 128, torch.float16, W.MASK_DIAG_CAUSAL, 0.5),
        (W.layout_random_diag(12, 0.4, H=2, seed=8), 16, torch.float16, W.MASK_NONE, 0.7),
    ]
    codes = {torch.float32: bsp.F32, torch.bfloat16: bsp.BF16, torch.float16: bsp.F16}
    for lay, B, dtype, kind, scale in cases:
        S = lay.shape[1] * B
        handle = bsp.bsp_layout_compile(lay, B)
        if lay.shape[1] == 260:
            assert not handle.softmax_chunks(2)["fits"]  # the long-row kernel runs
        Z = 2 if S < 8192 else 1
        X = W.randn((Z, handle.nnz, B, B), {torch.float32: "f32", torch.bfloat16: "bf16",
                                            torch.float16: "f16"}[dtype], 40 + B)
        Xd = X.cuda()
        maskh = W.random_mask(S, 0.8, 9) if kind == W.MASK_DENSE else None
        mask = None if maskh is None else torch.from_numpy(maskh).cuda()
        got = torch.full_like(Xd, float("nan"))
        assert _call(lib, lay, B, codes[dtype], Xd, got, scale, kind, mask) == 0
        torch.cuda.synchronize()
        want = oracle.softmax(lay, B, X, scale, kind, maskh)
        assert_close(to_np(got), want, dtype, f"noalloc softmax B={B} {dtype}", rel=PROB_TOL[dtype],
                     zeros=softmax_zero_positions(lay, B, Z, kind, maskh))
        ref = bsp.bsp_softmax(handle, Xd, None, scale, kind, mask)
        torch.cuda.synchronize()
        assert torch.equal(got, ref), f"noalloc softmax B={B} {dtype}: differs from bsp_softmax"


def test_noalloc_rejects_tables_beyond_the_array(lib):
    from sparse_attention_layout_gb300 import bsp
    lay = np.ones((16, 256, 256), np.uint8)  # 1M blocks: the tables alone are > 4 MiB
    X = torch.zeros(1, 1, 16, 16, device="cuda", dtype=torch.bfloat16)
    assert _call(lib, lay, 16, bsp.BF16, X, X, 1.0, W.MASK_NONE, None) == -4  # BSP_ERR_OOM
