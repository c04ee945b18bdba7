"""Shared helpers of the GPU parity tests."""

import numpy as np
import torch

TOL = {torch.float32: 1e-5, torch.bfloat16: 2e-2, torch.float16: 2e-2}


def normwise_err(got, want) -> float:
    """max |g - r| / max |r| over the tensor (0 when both are exactly 0)."""
    g = np.asarray(got, dtype=np.float64)
    r = np.asarray(want, dtype=np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    assert np.all(np.isfinite(g)), "non-finite output"
    scale = np.max(np.abs(r)) if r.size else 0.0
    diff = np.max(np.abs(g - r)) if r.size else 0.0
    if scale == 0.0:
        return float(diff)
    return float(diff / scale)


def assert_close(got, want, dtype, what=""):
    err = normwise_err(got, want)
    assert err <= TOL[dtype], f"{what}: normwise error {err:.3e} > {TOL[dtype]:.0e}"
    return err


def to_np(t):
    return t.detach().float().cpu().numpy()


def dev(t):
    return t.to("cuda").contiguous()
