"""The erf approximation the MX quantising epilogues use for GELU
(Abramowitz & Stegun, Handbook of Mathematical Functions, 7.1.26): its stated
bound |error| <= 1.5e-7 holds over a dense grid in float64, and the float32
evaluation order of the kernels (Horner in t, then exp(-z^2)) stays within a
few float32 roundings of it.  The GPU layers that use it are checked against
the oracle's exact-erf GELU in tests/test_gpu_mxfp8.py."""

import numpy as np
from scipy.special import erf

P = 0.3275911
A = (0.254829592, -0.284496736, 1.421413741, -1.453152027, 1.061405429)


def one_minus_erf(z, dt):
    z = z.astype(dt)
    t = dt(1.0) / (dt(P) * z + dt(1.0))
    poly = t * (dt(A[0]) + t * (dt(A[1]) + t * (dt(A[2]) + t * (dt(A[3]) + t * dt(A[4])))))
    return poly * np.exp(-z * z)


def test_stated_bound_float64():
    z = np.linspace(0.0, 8.0, 400001)
    err = np.abs((1.0 - one_minus_erf(z, np.float64)) - erf(z))
    assert err.max() <= 1.5e-7


def test_float32_evaluation_and_gelu():
    v = np.linspace(-12.0, 12.0, 200001)
    e = one_minus_erf(np.abs(v) / np.sqrt(2.0), np.float32).astype(np.float64)
    gelu = np.where(v >= 0, v * (1.0 - 0.5 * e), 0.5 * v * e)
    exact = 0.5 * v * (1.0 + erf(v / np.sqrt(2.0)))
    # 1.5e-7 from the method plus float32 rounding of t, the polynomial and exp
    assert np.max(np.abs(gelu - exact) / np.maximum(np.abs(v), 1.0)) <= 4e-7
    # negative inputs keep their tiny values (no cancellation)
    assert np.all(gelu[v < -5] < 0)
