"""bsp_softmax_noalloc: the softmax entry point for callers that cannot
allocate device memory (a runtime that owns every byte of the GPU, a plugin
handed only its buffers).  It keeps the layout tables in a fixed device array
the library declares itself instead of a compiled handle.

Checked through the C ABI against the existing entry point (bsp_softmax with a
compiled handle), on two calls in a row with different layouts, block sizes,
dtypes and masks, so the second call must not depend on what the first one
left in the shared array.  Collected last (file name) so that a run stopping
at the first failure has already run every other test."""

import ctypes

import numpy as np
import pytest
import torch

from gpu_util import assert_close, to_np
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


def test_noalloc_softmax_matches_compiled_handle_twice(lib):
    from sparse_attention_layout_gb300 import bsp
    cases = [  # (layout, block, dtype, mask kind, scale)
        (W.layout_strided_causal(16, local_blocks=4, stride=4, H=3), 64, torch.bfloat16, W.MASK_DIAG_CAUSAL, 0.09),
        (W.layout_random_diag(20, 0.3, H=2, seed=5), 32, torch.float32, W.MASK_DENSE, 0.3),
    ]
    codes = {torch.float32: bsp.F32, torch.bfloat16: bsp.BF16}
    for lay, B, dtype, kind, scale in cases:
        S = lay.shape[1] * B
        handle = bsp.bsp_layout_compile(lay, B)
        X = torch.randn(2, handle.nnz, B, B, device="cuda").to(dtype)
        mask = torch.from_numpy(W.random_mask(S, 0.8, 9)).cuda() if kind == W.MASK_DENSE else None
        want = bsp.bsp_softmax(handle, X, None, scale, kind, mask)
        got = torch.full_like(X, float("nan"))
        assert _call(lib, lay, B, codes[dtype], X, got, scale, kind, mask) == 0
        torch.cuda.synchronize()
        assert_close(to_np(got), to_np(want), dtype, f"noalloc softmax B={B} {dtype}")


def test_noalloc_rejects_tables_beyond_the_array(lib):
    from sparse_attention_layout_gb300 import bsp
    lay = np.ones((16, 256, 256), np.uint8)  # 1M blocks: the tables alone are > 4 MiB
    X = torch.zeros(1, 1, 16, 16, device="cuda", dtype=torch.bfloat16)
    assert _call(lib, lay, 16, bsp.BF16, X, X, 1.0, W.MASK_NONE, None) == -4  # BSP_ERR_OOM
