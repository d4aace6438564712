"""Pins of the oracle's per-token decode (no GPU)."""

import numpy as np
import pytest

from oracle import reader as R
from tests.helpers import dense_moe, make_layer, make_tokens


@pytest.fixture(scope="module")
def tiny():
    return make_layer(H=256, E=16, topk=2, I=128, c=80, r=8, seed=0)


def test_all_channels_kept_equals_dense_moe(tiny):
    x, ids, w = make_tokens(tiny, 3, seed=1)
    N = tiny.shape.N
    for t in range(3):
        res = R.decode_token(tiny, x[t], ids[t], w[t], N)
        ref = dense_moe(tiny, x[t], ids[t], w[t])
        assert np.allclose(res.y, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
        assert not res.y_recovery.any()


def test_exact_part_equals_dense_moe_restricted_to_kept(tiny):
    x, ids, w = make_tokens(tiny, 2, seed=2)
    k = 32
    for t in range(2):
        res = R.decode_token(tiny, x[t], ids[t], w[t], k)
        # dense computation with the skipped channels' activations zeroed
        ref = np.zeros(tiny.shape.H)
        xx = x[t].astype(np.float64)
        for s, e in enumerate(ids[t]):
            e = int(e)
            keep = np.zeros(tiny.shape.I, bool)
            for g in res.kept:
                if g // tiny.shape.I == e:
                    keep[g % tiny.shape.I] = True
            h = tiny.g(e) @ xx
            a = (h / (1 + np.exp(-h))) * (tiny.v(e) @ xx) * keep
            ref += float(w[t][s]) * (tiny.d(e) @ a)
        assert np.allclose(res.y_exact, ref, rtol=1e-12, atol=1e-13)


def _dequantized_rows(layer, e):
    """Rows whose rotated blocks are exactly alpha * t: R^T (alpha t)."""
    sk = layer.sketch(e)
    sh = layer.shape
    out = []
    for gv in range(2):
        wq = sk.t[gv].astype(np.float64) * np.transpose(sk.alpha[:, gv, :]).astype(np.float64)[..., None]
        wq = wq.reshape(sh.I, sh.Hp)
        # R is orthogonal and block diagonal: R^T u = sigma * (H u) / sqrt(128) per block
        Hm = R.sylvester_hadamard()
        u = wq.reshape(sh.I, sh.nb, 128) @ Hm.T / np.sqrt(128)
        out.append(u.reshape(sh.I, sh.Hp) * layer.sigma.astype(np.float64))
    return out


def test_full_screen_estimate_equals_dot_with_dequantized_rows():
    layer = make_layer(H=256, E=4, topk=2, I=64, c=128, r=8, seed=3)
    x, ids, w = make_tokens(layer, 1, seed=3)
    res = R.decode_token(layer, x[0], ids[0], w[0], 10)
    xp = R.pad_hidden(x[0].astype(np.float64), layer.shape.Hp)
    for s, e in enumerate(ids[0]):
        gq, vq = _dequantized_rows(layer, int(e))
        assert np.allclose(res.ghat[s], gq @ xp, rtol=1e-10, atol=1e-10)
        assert np.allclose(res.vhat[s], vq @ xp, rtol=1e-10, atol=1e-10)


def test_partial_screen_is_projection_onto_selected_rotated_coordinates(tiny):
    x, ids, w = make_tokens(tiny, 1, seed=4)
    res = R.decode_token(tiny, x[0], ids[0], w[0], 10)
    sh = tiny.shape
    xp = R.pad_hidden(x[0].astype(np.float64), sh.Hp)
    # x_c = R^T (mask * R x): the part of x the screen sees
    Rx = R.rotate(xp, tiny.sigma).reshape(sh.nb, 128) * res.mask
    Hm = R.sylvester_hadamard()
    xc = ((Rx @ Hm.T) / np.sqrt(128)).reshape(-1) * tiny.sigma
    assert res.mask.sum() == sh.nb * sh.c
    for s, e in enumerate(ids[0]):
        gq, vq = _dequantized_rows(tiny, int(e))
        assert np.allclose(res.ghat[s], gq @ xc, rtol=1e-10, atol=1e-10)
        assert np.allclose(res.vhat[s], vq @ xc, rtol=1e-10, atol=1e-10)


def test_score_is_norm_of_estimated_output_contribution(tiny):
    x, ids, w = make_tokens(tiny, 1, seed=5)
    res = R.decode_token(tiny, x[0], ids[0], w[0], 10)
    for s, e in enumerate(ids[0]):
        D = tiny.d(int(e))
        contrib = np.linalg.norm(D * (float(w[0][s]) * res.p[s])[None, :], axis=0)
        assert np.allclose(res.score[s], contrib, rtol=1e-6)   # dnorm is stored fp32


def _brute_topk(scores, gids, k):
    keep = []
    for n in range(len(scores)):
        beats = sum(1 for m in range(len(scores))
                    if scores[m] > scores[n] or (scores[m] == scores[n] and gids[m] < gids[n]))
        if beats < k:
            keep.append(gids[n])
    return sorted(keep)


@pytest.mark.parametrize("k", [0, 1, 7, 31, 255, 256])
def test_topk_brute_force(tiny, k):
    x, ids, w = make_tokens(tiny, 1, seed=6)
    res = R.decode_token(tiny, x[0], ids[0], w[0], k)
    gids = [int(e) * 128 + i for e in ids[0] for i in range(128)]
    assert list(res.kept) == _brute_topk(res.score.reshape(-1), gids, k)


def test_topk_ties_resolved_by_lower_channel_id(tiny):
    x, ids, w = make_tokens(tiny, 1, seed=7)
    # equal routing weights and two identical experts' worth of scores via a
    # layer whose weights are duplicated across experts
    lay = R.Layer(tiny.shape, tiny.G.copy(), tiny.V.copy(), tiny.D.copy(), tiny.sigma)
    lay.G[5] = lay.G[9]
    lay.V[5] = lay.V[9]
    lay.D[5] = lay.D[9]
    res = R.decode_token(lay, x[0], np.array([9, 5]), np.array([0.5, 0.5], np.float32), 41)
    sc = res.score
    assert np.array_equal(sc[0], sc[1])
    kept = set(res.kept.tolist())
    # an odd k splits exactly one tied pair: expert 5's copy (lower id) wins it
    split = [i for i in range(128) if ((5 * 128 + i) in kept) != ((9 * 128 + i) in kept)]
    assert len(split) == 1
    assert (5 * 128 + split[0]) in kept
    gids = [9 * 128 + i for i in range(128)] + [5 * 128 + i for i in range(128)]
    assert list(res.kept) == _brute_topk(sc.reshape(-1), gids, 41)


def test_recovery_only_when_nothing_kept(tiny):
    x, ids, w = make_tokens(tiny, 1, seed=8)
    res = R.decode_token(tiny, x[0], ids[0], w[0], 0)
    assert not res.y_exact.any() and res.kept.size == 0
    coef = np.zeros(tiny.shape.r)
    for s, e in enumerate(ids[0]):
        coef += (float(w[0][s]) * res.p[s]) @ tiny.b(int(e)).astype(np.float64)
    assert np.allclose(res.y, tiny.U.astype(np.float64) @ coef)


def test_full_rank_recovery_reproduces_skipped_channels():
    layer = make_layer(H=128, E=4, topk=2, I=64, c=80, r=128, seed=9)
    x, ids, w = make_tokens(layer, 1, seed=9)
    res = R.decode_token(layer, x[0], ids[0], w[0], 20)
    kept = set(res.kept.tolist())
    ref = np.zeros(128)
    for s, e in enumerate(ids[0]):
        e = int(e)
        for i in range(64):
            if e * 64 + i not in kept:
                ref += float(w[0][s]) * res.p[s, i] * layer.d(e)[:, i]
    assert np.linalg.norm(res.y_recovery - ref) < 5e-3 * np.linalg.norm(ref)


def test_decode_batch_is_per_token(tiny):
    x, ids, w = make_tokens(tiny, 3, seed=10)
    out = R.decode(tiny, x, ids, w, 16)
    for t in range(3):
        one = R.decode_token(tiny, x[t], ids[t], w[t], 16)
        assert np.array_equal(out[t].kept, one.kept)
        assert np.array_equal(out[t].y, one.y)


def test_padded_hidden_layer():
    layer = make_layer(H=200, E=4, topk=2, I=64, c=80, r=8, seed=11)
    assert layer.shape.Hp == 256
    x, ids, w = make_tokens(layer, 1, seed=11)
    res = R.decode_token(layer, x[0], ids[0], w[0], layer.shape.N)
    ref = dense_moe(layer, x[0], ids[0], w[0])
    assert np.allclose(res.y, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
