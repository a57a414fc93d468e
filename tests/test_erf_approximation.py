"""The erf used by the tensor-core GELU epilogue: Abramowitz & Stegun, Handbook of
Mathematical Functions, eq. 7.1.26, erf(x) = 1 - (a1 t + ... + a5 t^5) exp(-x^2),
t = 1/(1 + p x), stated absolute error <= 1.5e-7 for x >= 0. The coefficients below are
the ones the kernel uses (token_routing_gb300/csrc/common.cuh); this checks them against
the published bound, in double and in float32 arithmetic, and the GELU / GELU' built from
them against the exact forms."""
import math

import numpy as np

P = 0.3275911
A = (0.254829592, -0.284496736, 1.421413741, -1.453152027, 1.061405429)


def erf_as(x, dtype):
    x = np.asarray(x, dtype=dtype)
    ax = np.abs(x)
    t = dtype(1) / (dtype(1) + dtype(P) * ax)
    poly = dtype(A[4])
    for a in (A[3], A[2], A[1], A[0]):
        poly = poly * t + dtype(a)
    poly = poly * t
    return np.sign(x) * (dtype(1) - poly * np.exp(-ax * ax))


def test_published_error_bound():
    x = np.linspace(-6, 6, 120001)
    ref = np.array([math.erf(v) for v in x])
    assert np.abs(erf_as(x, np.float64) - ref).max() <= 1.5e-7
    # in float32 the rounding of the steps adds a few ulp of 1.0
    assert np.abs(erf_as(x.astype(np.float32), np.float32) - ref).max() <= 6e-7


def test_gelu_and_derivative_from_one_exponential():
    a = np.linspace(-8, 8, 4001)
    e = np.exp(-a * a / 2)
    Phi = 0.5 + np.copysign(0.5 * erf_as(np.abs(a) / math.sqrt(2), np.float64), a)
    gelu = a * Phi
    dgelu = Phi + a * e / math.sqrt(2 * math.pi)
    Phi_ref = np.array([0.5 * (1 + math.erf(v / math.sqrt(2))) for v in a])
    np.testing.assert_allclose(gelu, a * Phi_ref, atol=1e-6)
    np.testing.assert_allclose(dgelu, Phi_ref + a * np.exp(-a * a / 2) / math.sqrt(2 * math.pi), atol=1e-7)
