"""The FMA-pipe 2^x used by the fused attention softmax for part of its
columns, held to its stated bound against fp64 exp2: relative error <= 1.1e-4
for x >= -125 (fitted 1.01e-4 plus fp32 rounding), exact powers of two at
integers, and a tiny positive value (<= 2^-124.5) for x < -125 and -inf."""

import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from sparse_attention_layout_gb300 import bsp, build
    build.build()
    L = bsp.lib()
    L.bsp_diag_exp2.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]
    L.bsp_diag_exp2.restype = ctypes.c_int
    return L


def _eval(lib, x: np.ndarray) -> np.ndarray:
    xd = torch.from_numpy(x.astype(np.float32)).cuda()
    yd = torch.full_like(xd, float("nan"))
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.bsp_diag_exp2(ctypes.c_void_p(xd.data_ptr()), ctypes.c_void_p(yd.data_ptr()), x.size, stream) == 0
    torch.cuda.synchronize()
    return yd.cpu().numpy()


def test_relative_error_bound(lib):
    rng = np.random.default_rng(3)
    x = np.concatenate([np.linspace(-125.0, 9.0, 2_000_001), rng.uniform(-30, 8, 1_000_001)]).astype(np.float32)
    y = _eval(lib, x).astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    rel = np.abs(y / ref - 1.0)
    assert rel.max() <= 1.1e-4, (rel.max(), x[rel.argmax()])


def test_integers_exact(lib):
    x = np.arange(-125, 9, dtype=np.float32)
    assert np.array_equal(_eval(lib, x), np.exp2(x.astype(np.float64)).astype(np.float32))


def test_below_range_and_minus_inf(lib):
    x = np.array([-125.5, -126, -200, -1e30, -np.inf, -np.inf, -3.4e38], np.float32)
    y = _eval(lib, x)
    assert np.all(np.isfinite(y)) and np.all(y > 0) and np.all(y <= 2.0 ** -124.5)


def test_odd_length_and_empty(lib):
    x = np.array([0.5, -1.25, 3.0], np.float32)
    assert np.allclose(_eval(lib, x), np.exp2(x.astype(np.float64)), rtol=1.1e-4, atol=0)
    from sparse_attention_layout_gb300 import bsp
    assert bsp.lib().bsp_diag_exp2(None, None, 0, None) == 0
