"""Pins of the oracle's full-screen ranking by the expected squared output
error of skipping a channel (no GPU): on a layer whose rotated rows are
exactly ternary the ranking key is the actual squared error that skipping
leaves in the output; on a random layer the rho-based variance matches the
screen's actual error on average; k = N is the dense MoE."""

import numpy as np
import pytest

from calibration_free_sparse_gb300 import synthetic as S
from oracle import reader as R
from tests.helpers import dense_moe, make_layer, make_tokens


def exact_sketch_layer(H=256, E=4, topk=2, I=64, r=8, seed=5, noise=0.0):
    """Gate and up rows sigma * (H_128 t) 2^-9 per block: their rotated
    blocks are exactly sqrt(128) 2^-9 t (ternary t), and every entry is an
    integer of at most 128 times 2^-9, exact in BF16.  noise > 0 adds
    N(0, (noise 2^-9)^2) to every entry: small sketch errors."""
    rng = np.random.default_rng(seed)
    shape = R.Shape(H=H, E=E, topk=topk, I=I, c=128, r=r)
    sigma = S.signs(seed, shape.Hp)
    Hm = R.sylvester_hadamard(128)
    rows = []
    for _ in range(2):
        t = rng.choice([-1, 0, 1], size=(E, I, shape.nb, 128), p=[0.3, 0.4, 0.3])
        w = np.einsum("kc,eibc->eibk", Hm, t).reshape(E, I, shape.Hp) * 2.0 ** -9
        w = w * sigma.astype(np.float64)[None, None, :]
        if noise:
            w = w + noise * 2.0 ** -9 * rng.standard_normal(w.shape)
        rows.append(S.f32_to_bf16_bits(w[..., :H].astype(np.float32)))
    _, _, D = S.weights(seed, E, I, H)
    layer = R.Layer(shape, rows[0], rows[1], D, sigma)
    for e in range(E if not noise else 0):   # exact: the sketch reproduces the rows
        for gv, W in ((0, layer.g(e)), (1, layer.v(e))):
            Wr = R.rotate(R.pad_hidden(W, shape.Hp), sigma).reshape(I, shape.nb, 128)
            assert np.allclose(np.abs(Wr)[Wr != 0], np.sqrt(128) * 2.0 ** -9, rtol=1e-12)
    return layer


def test_needs_the_full_screen():
    layer = make_layer(H=256, E=4, topk=2, I=64, c=80, r=8, seed=1)
    x, ids, w = make_tokens(layer, 1, seed=1)
    with pytest.raises(ValueError):
        R.expected_skip_error(layer, x[0], ids[0], w[0])


def test_exact_sketch_key_is_the_skip_error():
    layer = exact_sketch_layer()
    x, ids, w = make_tokens(layer, 2, seed=3)
    for t in range(2):
        sc, err = R.expected_skip_error(layer, x[t], ids[t], w[t])
        xx = x[t].astype(np.float64)
        U = layer.U.astype(np.float64)
        actual = np.zeros_like(err)
        for s_, e in enumerate(int(v) for v in ids[t]):
            a = R.silu(layer.g(e) @ xx) * (layer.v(e) @ xx)
            Db = U @ layer.b(e).astype(np.float64).T            # [H][I]: U b_j
            res = a[None, :] * layer.d(e) - sc.p[s_][None, :] * Db
            actual[s_] = float(w[t][s_]) ** 2 * (res * res).sum(axis=0)
        # FP16 alpha, U and b: agreement to about 1e-3 of the largest key
        assert np.abs(err - actual).max() <= 2e-3 * actual.max()
        # and the ranking is the ranking by the actual error where they differ clearly
        big = actual.reshape(-1) > 0.05 * actual.max()
        order = np.argsort(-err.reshape(-1)[big], kind="stable")
        assert np.all(np.diff(actual.reshape(-1)[big][order]) <= 2e-3 * actual.max())


def test_rho_variance_matches_the_screen_error_on_average():
    layer = make_layer(H=512, E=2, topk=2, I=256, c=128, r=8, seed=7)
    x, ids, w = make_tokens(layer, 1, seed=9)
    xx = x[0].astype(np.float64)
    sh = layer.shape
    Rx = R.rotate(R.pad_hidden(xx, sh.Hp), layer.sigma).reshape(sh.nb, 128)
    rn2 = (Rx * Rx).sum(axis=1)
    sc = R.screen_token(layer, x[0], ids[0], w[0])
    for s_, e in enumerate(int(v) for v in ids[0]):
        rho = layer.sketch(e).rho.astype(np.float64)
        for gv, (W, est) in enumerate(((layer.g(e), sc.ghat[s_]), (layer.v(e), sc.vhat[s_]))):
            emp = np.mean((W @ xx - est) ** 2)
            pred = np.mean(rn2 @ rho[:, gv, :])
            assert 0.7 < emp / pred < 1.4, (e, gv, emp / pred)


def test_all_channels_kept_is_dense_moe():
    layer = make_layer(H=256, E=4, topk=2, I=64, c=128, r=8, seed=11)
    x, ids, w = make_tokens(layer, 2, seed=12)
    for t in range(2):
        res = R.decode_token_rho(layer, x[t], ids[t], w[t], layer.shape.N)
        ref = dense_moe(layer, x[t], ids[t], w[t])
        assert np.allclose(res.y, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_selection_is_the_top_k_of_the_key():
    layer = make_layer(H=256, E=4, topk=2, I=32, c=128, r=8, seed=13)
    x, ids, w = make_tokens(layer, 1, seed=14)
    k = 11
    res = R.decode_token_rho(layer, x[0], ids[0], w[0], k)
    I = layer.shape.I
    keys = {int(e) * I + i: float(res.score[s_][i]) for s_, e in enumerate(ids[0]) for i in range(I)}
    best = sorted(keys, key=lambda g: (-keys[g], g))[:k]
    assert list(res.kept) == sorted(best)


def test_key_is_the_expected_error_under_the_rho_error_model():
    """Monte Carlo of the definition: with the true activations drawn around
    the estimates with the rho-based variances, the mean squared norm of what
    skipping leaves, w (a d - p U b), computed from the stored U and b,
    matches the key where first order holds.  Three groups of channels: both
    estimates well determined (the p^2 term dominates), the up estimate near
    zero (the up variance dominates) and the gate estimate near zero (the gate
    variance through phi' dominates)."""
    rng = np.random.default_rng(21)
    layer = exact_sketch_layer(E=2, I=256, seed=17, noise=0.15)
    x, ids, w = make_tokens(layer, 1, seed=18)
    sh = layer.shape
    sc, err = R.expected_skip_error(layer, x[0], ids[0], w[0])
    Rx = R.rotate(R.pad_hidden(x[0].astype(np.float64), sh.Hp), layer.sigma).reshape(sh.nb, 128)
    rn2 = (Rx * Rx).sum(axis=1)
    U = layer.U.astype(np.float64)
    groups = {"determined": 0, "up near zero": 0, "gate near zero": 0}
    for s_, e in enumerate(int(v) for v in ids[0]):
        rho = layer.sketch(e).rho.astype(np.float64)
        sd_g, sd_v = np.sqrt(rn2 @ rho[:, 0, :]), np.sqrt(rn2 @ rho[:, 1, :])
        Db = U @ layer.b(e).astype(np.float64).T
        for i in range(sh.I):
            g, v = sc.ghat[s_][i], sc.vhat[s_][i]
            small_g, small_v = sd_g[i] < 0.05 * abs(g), sd_v[i] < 0.05 * abs(v)
            if small_g and small_v:
                grp = "determined"
            elif small_g and abs(v) < 2 * sd_v[i]:
                grp = "up near zero"
            elif small_v and abs(g) < 2 * sd_g[i] and sd_g[i] < 0.1:
                grp = "gate near zero"
            else:
                continue
            a = R.silu(g + sd_g[i] * rng.standard_normal(40000)) * (v + sd_v[i] * rng.standard_normal(40000))
            res = a[:, None] * layer.d(e)[:, i][None, :] - sc.p[s_][i] * Db[:, i][None, :]
            mc = float(w[0][s_]) ** 2 * np.mean((res * res).sum(axis=1))
            assert abs(mc - err[s_][i]) <= 0.05 * mc + 1e-12, (grp, e, i, mc, err[s_][i])
            groups[grp] += 1
    assert all(n >= 2 for n in groups.values()), groups
