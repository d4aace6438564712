"""Pins of the oracle's batch-shared selection (no GPU)."""

import numpy as np
import pytest

from calibration_free_sparse_gb300 import synthetic as S
from oracle import reader as R
from tests.helpers import dense_moe, make_layer, make_tokens


@pytest.fixture(scope="module")
def small():
    return make_layer(H=256, E=8, topk=2, I=64, c=80, r=8, seed=31)


def test_kept_count_rounds_half_up():
    assert R.shared_kept_count(756, 8, 8) == 756
    assert R.shared_kept_count(756, 16, 8) == 1512
    assert R.shared_kept_count(3, 1, 2) == 2          # 1.5 -> 2
    assert R.shared_kept_count(5, 3, 4) == 4          # 3.75 -> 4
    assert R.shared_kept_count(5, 1, 4) == 1          # 1.25 -> 1
    assert R.shared_kept_count(0, 7, 8) == 0


def test_batch_of_one_is_the_per_token_reader(small):
    x, ids, w = make_tokens(small, 1, seed=2)
    for k in (0, 1, 17, 64, small.shape.N):
        sh = R.decode_shared(small, x, ids, w, k)
        one = R.decode_token(small, x[0], ids[0], w[0], k)
        assert sh.K == k
        assert np.array_equal(sh.kept, one.kept)
        assert np.array_equal(sh.tokens[0].kept, one.kept)
        assert np.allclose(sh.tokens[0].y, one.y, rtol=1e-13, atol=1e-13 * np.abs(one.y).max())


def test_all_channels_kept_is_dense_moe_per_token(small):
    x, ids, w = make_tokens(small, 3, seed=4)
    res = R.decode_shared(small, x, ids, w, small.shape.N)
    assert res.K == res.experts.size * small.shape.I
    for t in range(3):
        ref = dense_moe(small, x[t], ids[t], w[t])
        assert np.allclose(res.tokens[t].y, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
        assert not res.tokens[t].y_recovery.any()


def test_selection_by_brute_force():
    layer = make_layer(H=128, E=4, topk=2, I=16, c=80, r=4, seed=7)
    x, ids, w = make_tokens(layer, 3, seed=8)
    k = 5
    res = R.decode_shared(layer, x, ids, w, k)
    I = layer.shape.I
    total = {}
    for t in range(3):
        sc = R.decode_token(layer, x[t], ids[t], w[t], k).score   # the same screen
        for s_ in range(2):
            e = int(ids[t][s_])
            for i in range(I):
                total[e * I + i] = total.get(e * I + i, 0.0) + float(sc[s_][i])
    n_e = len({int(e) for e in ids.reshape(-1)})
    K = int(k * n_e / 2 + 0.5)
    ranked = sorted(total, key=lambda g: (-total[g], g))
    assert res.K == K
    assert list(res.kept) == sorted(ranked[:K])
    for t in range(3):
        mine = sorted(g for g in ranked[:K] if g // I in {int(e) for e in ids[t]})
        assert list(res.tokens[t].kept) == mine


def test_identical_tokens_share_the_per_token_set(small):
    x, ids, w = make_tokens(small, 1, seed=9)
    B = 4
    xb, idb, wb = np.repeat(x, B, 0), np.repeat(ids, B, 0), np.repeat(w, B, 0)
    k = 20
    res = R.decode_shared(small, xb, idb, wb, k)
    one = R.decode_token(small, x[0], ids[0], w[0], k)
    assert res.K == k
    assert np.array_equal(res.kept, one.kept)
    for t in range(B):
        assert np.allclose(res.tokens[t].y, one.y, rtol=1e-12, atol=1e-12 * np.abs(one.y).max())


def test_exact_part_is_dense_moe_restricted_to_the_shared_set(small):
    x, ids, w = make_tokens(small, 3, seed=10)
    res = R.decode_shared(small, x, ids, w, 30)
    I = small.shape.I
    kept = set(int(g) for g in res.kept)
    for t in range(3):
        ref = np.zeros(small.shape.H)
        xx = x[t].astype(np.float64)
        for s_, e in enumerate(ids[t]):
            e = int(e)
            keep = np.array([e * I + i in kept for i in range(I)])
            h = small.g(e) @ xx
            a = (h / (1 + np.exp(-h))) * (small.v(e) @ xx) * keep
            ref += float(w[t][s_]) * (small.d(e) @ a)
        assert np.allclose(res.tokens[t].y_exact, ref, rtol=1e-11, atol=1e-12 * np.abs(ref).max())


def test_skipped_channels_recovered_with_each_tokens_own_estimates(small):
    """Full-rank U makes the recovery exact for the estimates: y_recovery is
    then sum over the token's skipped channels of w p d."""
    layer = make_layer(H=128, E=4, topk=2, I=32, c=80, r=128, seed=12)
    x, ids, w = make_tokens(layer, 2, seed=13)
    res = R.decode_shared(layer, x, ids, w, 10)
    I = layer.shape.I
    kept = set(int(g) for g in res.kept)
    for t in range(2):
        ref = np.zeros(layer.shape.H)
        for s_, e in enumerate(ids[t]):
            e = int(e)
            for i in range(I):
                if e * I + i not in kept:
                    ref += float(w[t][s_]) * res.tokens[t].p[s_, i] * layer.d(e)[:, i]
        # U and b are FP16: agreement to FP16 rounding
        assert np.abs(res.tokens[t].y_recovery - ref).max() <= 2e-3 * np.abs(ref).max()
