"""Checks of the seeded input generator (no GPU)."""

import numpy as np
import torch

from calibration_free_sparse_gb300 import synthetic as S


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    a = (rng.standard_normal(100000) * 10.0 ** rng.integers(-6, 6, 100000)).astype(np.float32)
    ref = torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(S.f32_to_bf16_bits(a), ref)


def test_weight_recipe():
    G, V, D = S.weights(0, 8, 64, 256)
    assert G.shape == (8, 64, 256) and D.shape == (8, 256, 64) and G.dtype == np.uint16
    g = (G.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    big = np.abs(g) > 6 / np.sqrt(256)
    assert 0.0005 < big.mean() < 0.0016
    assert abs(g[~big].std() * np.sqrt(256) - 1) < 0.02
    G2, _, _ = S.weights(0, 8, 64, 256)
    assert np.array_equal(G, G2)
    G3, _, _ = S.weights(1, 8, 64, 256)
    assert not np.array_equal(G, G3)


def test_activation_outliers():
    x = S.activations(3, 4, 2048)
    big = np.abs(x) > 8
    cols = np.nonzero(big.any(axis=0))[0]
    assert 1 <= len(cols) <= 4


def test_routing():
    ids, w = S.routing(0, 16, 128, 8)
    assert ids.shape == (16, 8) and w.dtype == np.float32
    for t in range(16):
        assert len(set(ids[t].tolist())) == 8
        assert abs(w[t].sum() - 1) < 1e-6
        assert np.all(np.diff(w[t]) <= 0)       # ordered by decreasing logit


def test_signs():
    s = S.signs(0, 2944)
    assert set(np.unique(s).tolist()) == {-1, 1} and s.dtype == np.int8


def test_budget_to_k():
    assert S.budget_to_k(0.178, 6144) == 756
    assert S.budget_to_k(0.128, 6144) == 449
    assert S.QWEN3_235B.k == S.budget_to_k(0.128, 12288)
