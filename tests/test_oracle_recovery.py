"""Pins of the oracle's recovery basis U and coefficients b (no GPU)."""

import numpy as np

from oracle import reader as R
from tests.helpers import make_layer


def _projector(U):
    U = U.astype(np.float64)
    return U @ U.T


def test_basis_matches_svd_left_singular_vectors():
    layer = make_layer(H=128, E=8, topk=2, I=64, r=8, seed=1)
    Dall = np.concatenate([layer.d(e) for e in range(8)], axis=1)     # [H][E*I]
    Usvd, svals, _ = np.linalg.svd(Dall, full_matrices=False)
    P_svd = Usvd[:, :8] @ Usvd[:, :8].T
    assert np.linalg.norm(_projector(layer.U) - P_svd, 2) < 5e-3        # fp16 storage
    assert np.allclose(layer.eigenvalues, svals[:8] ** 2, rtol=1e-10)


def test_basis_columns_orthonormal_and_canonical():
    layer = make_layer(H=128, E=8, topk=2, I=64, r=8, seed=2)
    U = layer.U.astype(np.float64)
    assert np.allclose(U.T @ U, np.eye(8), atol=3e-3)
    for j in range(8):
        i = np.argmax(np.abs(U[:, j]))
        assert U[i, j] > 0


def test_eckart_young_residual():
    layer = make_layer(H=128, E=8, topk=2, I=64, r=8, seed=3)
    Dall = np.concatenate([layer.d(e) for e in range(8)], axis=1)
    ev = np.linalg.eigvalsh(Dall @ Dall.T)[::-1]
    U = layer.U.astype(np.float64)
    resid = np.linalg.norm(Dall - U @ (U.T @ Dall)) ** 2
    assert abs(resid - ev[8:].sum()) < 5e-3 * ev.sum()


def test_full_rank_basis_reconstructs_down_columns():
    layer = make_layer(H=128, E=4, topk=2, I=64, r=128, seed=4)
    U = layer.U.astype(np.float64)
    for e in range(2):
        d = layer.d(e)
        b = layer.b(e).astype(np.float64)            # [I][r]
        assert np.allclose(U @ b.T, d, atol=3e-3 * np.abs(d).max())


def test_coefficients_are_projections():
    layer = make_layer(H=128, E=4, topk=2, I=64, r=8, seed=5)
    U16 = layer.U
    for e in range(4):
        b = layer.b(e)
        ref = np.einsum("hr,hi->ir", U16.astype(np.float64), layer.d(e))
        assert np.array_equal(b, ref.astype(np.float16))
