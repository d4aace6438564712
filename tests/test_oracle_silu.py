"""Pins of the gate activation phi(z) = z / (1 + e^{-z}) (SiLU) by facts the
mathematics fixes, independent of how the oracle writes it (no GPU)."""

import math

import numpy as np

from oracle import reader as R


def test_silu_zero_and_hand_value():
    assert R.silu(np.float64(0.0)) == 0.0
    # phi(1) = 1 / (1 + 1/e) = e / (e + 1)
    assert abs(R.silu(np.float64(1.0)) - math.e / (math.e + 1.0)) < 1e-15
    # phi(-1) = -1 / (1 + e)
    assert abs(R.silu(np.float64(-1.0)) + 1.0 / (1.0 + math.e)) < 1e-15


def test_silu_odd_part_is_identity():
    # z sigma(z) - (-z) sigma(-z) = z (sigma(z) + sigma(-z)) = z
    z = np.linspace(-30.0, 30.0, 601)
    assert np.allclose(R.silu(z) - R.silu(-z), z, rtol=0, atol=1e-13)


def test_silu_asymptotes():
    big = np.array([20.0, 40.0, 200.0])
    assert np.all(np.abs(R.silu(big) / big - 1.0) < 1e-8)
    neg = -big
    assert np.all(np.abs(R.silu(neg)) < 1e-6)
    assert np.all(R.silu(neg) <= 0.0)
    # far below the fp64 range of e^{-z}: still 0 from below, never NaN
    assert R.silu(np.float64(-1000.0)) == 0.0


def test_silu_minimum():
    # phi has one minimum, where phi'(z) = sigma(z)(1 + z(1 - sigma(z))) = 0,
    # at z* ~ -1.2784645; phi(z*) ~ -0.2784645 (= z* + 1)
    z = np.linspace(-3.0, 0.0, 300001)
    v = R.silu(z)
    i = int(np.argmin(v))
    assert abs(z[i] + 1.2784645) < 1e-5
    assert abs(v[i] - (z[i] + 1.0)) < 1e-5
    assert abs(R.silu_grad(np.float64(z[i]))) < 1e-4
