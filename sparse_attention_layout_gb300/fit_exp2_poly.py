"""Coefficients of the cubic behind exp2_poly2 (csrc/tc_common.cuh).

2^f on f in [-1/2, 1/2] by p(f) = 1 + f (c1 + f (c2 + f c3)): p(0) = 1 is
held so that integer arguments give exact powers of two, and c1..c3 minimise
the largest relative error |p(f) - 2^f| / 2^f.  The minimax fit is Lawson's
iteratively reweighted least squares: solve the weighted least-squares fit,
raise the weights where the error is large (w <- w sqrt(e / max e)), repeat.

    python -m sparse_attention_layout_gb300.fit_exp2_poly

prints the float32 coefficients the kernel header holds and their maximum
relative error on a dense grid.
"""
import numpy as np


def fit(points: int = 20001, iterations: int = 200):
    f = np.linspace(-0.5, 0.5, points)
    t = np.exp2(f)
    A = np.stack([f, f ** 2, f ** 3], axis=1)
    w = np.full_like(f, 1.0 / points)
    c = np.zeros(3)
    for _ in range(iterations):
        rel = w / t  # weighted relative residual (p - t) / t, p = 1 + A c
        c, *_ = np.linalg.lstsq(A * rel[:, None], (t - 1.0) * rel, rcond=None)
        e = np.abs((1.0 + A @ c - t) / t)
        w = w * np.sqrt(e / e.max()) + 1e-30
        w /= w.sum()
    c32 = c.astype(np.float32)
    # the error of the float32 coefficients, the polynomial evaluated in fp64
    p = 1.0 + f * (float(c32[0]) + f * (float(c32[1]) + f * float(c32[2])))
    return c32, float(np.max(np.abs(p - t) / t))


if __name__ == "__main__":
    c, err = fit()
    print("c1 = %.9gf, c2 = %.9gf, c3 = %.9gf" % tuple(float(x) for x in c))
    print("max relative error %.3e" % err)
