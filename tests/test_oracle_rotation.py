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


def test_screen_selects_on_exact_rotation():
    # the screened set is the c largest |Rx| of the float64 rotation, checked
    # by brute force on rotations that the closed form R e_j pins above
    rng = np.random.default_rng(4)
    sigma = np.where(rng.random(256) < 0.5, -1, 1).astype(np.int8)
    x = rng.standard_normal(256)
    x[[3, 77]] *= 20
    mag = np.abs(R.rotate(x, sigma)).reshape(2, 128)
    assert np.array_equal(R.select_coordinates(mag, 80), _brute_select(mag, 80))


def test_selection_gaps_hand_values():
    mag = np.zeros((3, 128))
    mag[0, :10] = np.arange(10, 0, -1)      # 10, 9, ..., 1 then zeros
    mag[1, :] = 5.0                          # all tied: gap 0
    # block 2 stays zero: no order to protect
    g = R.selection_gaps(mag, 3)
    assert g[0] == (8.0 - 7.0) / 8.0
    assert g[1] == 0.0
    assert np.isinf(g[2])
    assert np.all(np.isinf(R.selection_gaps(mag, 128)))
    # the gap at c = 10 of block 0: (1 - 0) / 1
    assert R.selection_gaps(mag, 10)[0] == 1.0


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
