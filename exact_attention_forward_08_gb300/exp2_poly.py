"""Coefficients of the polynomial 2^f on f in [-1/2, 1/2] used by the
emulated exp2 of the softmax ("FlashAttention-4 wiki", "Core methods":
Cody-Waite range reduction plus a degree-3 Horner polynomial on the FMA
units, the integer part added to the IEEE-754 exponent field).

    2^x = 2^j * 2^f,  j = rint(x),  f = x - j in [-1/2, 1/2]
    2^f ~= ((c3 f + c2) f + c1) f + c0

The coefficients are fitted here by iteratively reweighted least squares that
drives the maximum relative error towards the equioscillating (minimax)
optimum.  Running this module prints them; ``csrc/fa_kernel.cuh`` holds the
printed values and ``tests/test_exp2_poly.py`` checks that the two agree.
"""
from __future__ import annotations

import numpy as np

DEGREE = 3


def fit(degree: int = DEGREE, iters: int = 60) -> np.ndarray:
    """Coefficients c0..c_degree (ascending) minimising the max relative error."""
    f = np.cos(np.linspace(0.0, np.pi, 4001)) * 0.5  # Chebyshev-spaced nodes on [-1/2, 1/2]
    y = np.exp2(f)
    A = np.vander(f, degree + 1, increasing=True) / y[:, None]  # relative-error rows
    w = np.ones_like(f)
    c = None
    for _ in range(iters):
        sw = np.sqrt(w)
        c, *_ = np.linalg.lstsq(A * sw[:, None], sw, rcond=None)
        err = np.abs(A @ c - 1.0)
        w = w * (err / err.max() + 1e-3)  # emphasise the largest errors
        w /= w.mean()
    return c


def max_rel_error(c: np.ndarray) -> float:
    f = np.linspace(-0.5, 0.5, 200001)
    p = np.polyval(c[::-1], f)
    return float(np.max(np.abs(p / np.exp2(f) - 1.0)))


def coefficients_f32() -> list:
    return [float(np.float32(v)) for v in fit()]


if __name__ == "__main__":
    c = fit()
    print("coefficients (c0..c3):", ", ".join(f"{np.float32(v)!r}" for v in c))
    print("max relative error:", max_rel_error(c.astype(np.float32).astype(np.float64)))
