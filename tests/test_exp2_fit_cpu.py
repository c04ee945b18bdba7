"""The cubic of exp2_poly2 (csrc/tc_common.cuh) is the one its fitting script
produces: the header's float32 coefficients equal fit_exp2_poly.fit()'s, and
their largest relative error against 2^f on [-1/2, 1/2] stays under the
bound the GPU test holds the device function to."""
import os
import re

import numpy as np

from sparse_attention_layout_gb300 import fit_exp2_poly

HDR = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "sparse_attention_layout_gb300",
                   "csrc", "tc_common.cuh")


def header_coefficients():
    src = open(HDR).read()
    m = re.search(r"constexpr float c1 = ([0-9.e+-]+)f, c2 = ([0-9.e+-]+)f, c3 = ([0-9.e+-]+)f;", src)
    assert m, "exp2_poly2's coefficients not found"
    return np.array([float(v) for v in m.groups()], dtype=np.float32)


def test_header_holds_the_fitted_coefficients():
    c, err = fit_exp2_poly.fit()
    assert np.array_equal(header_coefficients(), c), (header_coefficients(), c)
    assert err < 1.02e-4


def test_fit_is_near_minimax():
    # p(f) - 1 = f q(f) with q quadratic, so the relative error is f / 2^f
    # times the error of q against (2^f - 1) / f: the minimax q makes that
    # weighted error reach its maximum with alternating signs at four points
    # (three coefficients), i.e. sign(e) * sign(f) alternates across the
    # extrema of |e| (e itself is 0 at f = 0)
    c = header_coefficients().astype(np.float64)
    f = np.linspace(-0.5, 0.5, 20001)
    e = (1.0 + f * (c[0] + f * (c[1] + f * c[2]))) / np.exp2(f) - 1.0
    emax = np.abs(e).max()
    peaks = [i for i in range(1, len(f) - 1) if abs(e[i]) >= abs(e[i - 1]) and abs(e[i]) >= abs(e[i + 1])]
    peaks = [0] + peaks + [len(f) - 1]
    big = [np.sign(e[i]) * np.sign(f[i]) for i in peaks if abs(e[i]) > 0.97 * emax]
    flips = sum(1 for a, b in zip(big, big[1:]) if a != b)
    assert flips >= 3, (big, emax)
