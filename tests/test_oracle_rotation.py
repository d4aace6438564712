"""Pins of the oracle's rotation and coordinate selection (no GPU)."""

import math

import numpy as np
import pytest
import scipy.linalg

from oracle import reader as R


def test_sylvester_matches_scipy_hadamard():
    # scipy builds the Sylvester matrix by Kronecker doubling: a different route.
    assert np.array_equal(R.sylvester_hadamard(128), scipy.linalg.hadamard(128).astype(float))


def test_rotation_orthogonal_and_preserves_dot_products():
    rng = np.random.default_rng(1)
    Hp = 384
    sigma = np.where(rng.random(Hp) < 0.5, -1, 1).astype(np.int8)
    # R as an explicit matrix: rotate the identity.
    Rm = R.rotate(np.eye(Hp), sigma).T          # column j = R e_j
    assert np.allclose(Rm @ Rm.T, np.eye(Hp), atol=1e-13)
    g = rng.standard_normal(Hp)
    x = rng.standard_normal(Hp)
    assert abs(R.rotate(g, sigma) @ R.rotate(x, sigma) - g @ x) < 1e-12 * (np.abs(g) @ np.abs(x))


def test_rotation_of_unit_vector_closed_form():
    rng = np.random.default_rng(2)
    sigma = np.where(rng.random(256) < 0.5, -1, 1).astype(np.int8)
    for j in (0, 5, 127, 128, 200):
        e = np.zeros(256)
        e[j] = 1.0
        out = R.rotate(e, sigma)
        b, jj = divmod(j, 128)
        expect = np.zeros(256)
        col = scipy.linalg.hadamard(128)[:, jj] * sigma[j] / math.sqrt(128)
        expect[128 * b:128 * (b + 1)] = col
        assert np.allclose(out, expect, atol=1e-15)
    # e_0: every output coordinate of block 0 equals sigma_0 / sqrt(128)
    e0 = np.zeros(256)
    e0[0] = 1
    assert np.allclose(R.rotate(e0, sigma)[:128], sigma[0] / math.sqrt(128))


def test_rotation_blocks_are_independent():
    rng = np.random.default_rng(3)
    sigma = np.where(rng.random(256) < 0.5, -1, 1).astype(np.int8)
    x = rng.standard_normal(256)
    y = x.copy()
    y[128:] = 0
    assert np.allclose(R.rotate(x, sigma)[:128], R.rotate(y, sigma)[:128], atol=1e-15)
    assert np.all(R.rotate(y, sigma)[128:] == 0)


def test_butterfly_fp32_agrees_with_fp64_rotation():
    rng = np.random.default_rng(4)
    sigma = np.where(rng.random(512) < 0.5, -1, 1).astype(np.int8)
    x = rng.standard_normal(512).astype(np.float32)
    x[[3, 77, 300, 450]] *= 20
    mag = R.butterfly_magnitudes_fp32(x, sigma)
    assert mag.dtype == np.float32 and mag.shape == (4, 128)
    exact = np.abs(R.rotate(x.astype(np.float64), sigma)).reshape(4, 128) * math.sqrt(128)
    assert np.allclose(mag, exact, rtol=2e-6, atol=1e-5)


def test_butterfly_is_exact_on_small_integers():
    # small integers: every fp32 butterfly sum is exact, so it must equal H (sigma x)
    rng = np.random.default_rng(5)
    sigma = np.where(rng.random(128) < 0.5, -1, 1).astype(np.int8)
    x = rng.integers(-50, 50, 128).astype(np.float32)
    mag = R.butterfly_magnitudes_fp32(x, sigma)[0]
    ref = np.abs(scipy.linalg.hadamard(128) @ (sigma.astype(np.int64) * x.astype(np.int64)))
    assert np.array_equal(mag.astype(np.int64), ref)


def _brute_select(mag, c):
    out = np.zeros(mag.shape, bool)
    for b in range(mag.shape[0]):
        for i in range(mag.shape[1]):
            beats = sum(1 for j in range(mag.shape[1])
                        if mag[b, j] > mag[b, i] or (mag[b, j] == mag[b, i] and j < i))
            out[b, i] = beats < c
    return out


@pytest.mark.parametrize("c", [1, 80, 127, 128])
def test_selection_brute_force_with_ties(c):
    rng = np.random.default_rng(6)
    mag = rng.integers(0, 20, (3, 128)).astype(np.float32)   # many exact ties
    sel = R.select_coordinates(mag, c)
    assert np.array_equal(sel, _brute_select(mag, c))
    assert np.all(sel.sum(axis=1) == c)


def test_selection_ties_go_to_lower_index():
    mag = np.ones((1, 128), np.float32)
    sel = R.select_coordinates(mag, 80)
    assert sel[0, :80].all() and not sel[0, 80:].any()
