"""Pins of the oracle's layer stack (no GPU): the normalised input, the
residual carry and, with every channel kept, a stack of textbook gated-MoE
blocks."""

import numpy as np
import pytest

from calibration_free_sparse_gb300 import synthetic as S
from oracle import reader as R
from tests.helpers import dense_moe, make_layer


@pytest.fixture(scope="module")
def layers():
    return [make_layer(H=256, E=8, topk=2, I=64, c=80, r=8, seed=20 + l) for l in range(3)]


def routing_stack(L, B, E, topk, seed):
    ids, w = zip(*(S.routing(seed + l, B, E, topk) for l in range(L)))
    return np.stack(ids), np.stack(w)


def test_normalised_input_has_unit_rms_and_ignores_scale():
    h = S.activations(5, 4, 384).astype(np.float64)
    x = R.rms_normalise(h)
    ms = np.mean(h * h, axis=-1)
    # mean(x^2) = ms / (ms + eps): one up to the epsilon
    assert np.allclose(np.mean(x * x, axis=-1), ms / (ms + R.RMS_EPS), rtol=1e-14)
    # scale invariant up to the epsilon's share eps / mean(h^2)
    assert np.allclose(R.rms_normalise(37.0 * h), x, rtol=2 * R.RMS_EPS / ms.min())
    # direction kept: x is a positive multiple of h
    assert np.all(np.sign(x) == np.sign(h))
    # a zero residual stays finite
    assert np.all(R.rms_normalise(np.zeros((1, 8))) == 0.0)


def test_stack_with_all_channels_kept_is_a_stack_of_dense_moe_blocks(layers):
    B = 2
    sh = layers[0].shape
    h0 = S.activations(9, B, sh.H)
    ids, w = routing_stack(len(layers), B, sh.E, sh.topk, seed=40)
    res, h_out = R.decode_stack(layers, h0, ids, w, sh.N)
    h = h0.astype(np.float64)
    for l, layer in enumerate(layers):
        for t in range(B):
            # the layer input, normalised by a different route: norm / sqrt(H)
            ht = h[t]
            rms = np.sqrt(ht @ ht / sh.H + R.RMS_EPS)
            xt = (ht / rms).astype(np.float32)
            ref = dense_moe(layer, xt, ids[l, t], w[l, t])
            assert np.allclose(res[l][t].y, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
        h = h + np.stack([r.y for r in res[l]])
    assert np.array_equal(h_out, h)


def test_residual_carries_every_layer_output(layers):
    B = 3
    sh = layers[0].shape
    h0 = S.activations(11, B, sh.H)
    ids, w = routing_stack(len(layers), B, sh.E, sh.topk, seed=50)
    k = 40
    res, h_out = R.decode_stack(layers, h0, ids, w, k)
    total = h0.astype(np.float64) + sum(np.stack([r.y for r in rl]) for rl in res)
    assert np.allclose(h_out, total, rtol=1e-13, atol=1e-13)
    # layer l's input is the residual after layers 0 .. l-1: re-deriving the
    # second layer from the first layer's output gives the same kept sets
    h1 = h0.astype(np.float64) + np.stack([r.y for r in res[0]])
    x1 = R.rms_normalise(h1).astype(np.float32)
    again = R.decode(layers[1], x1, ids[1], w[1], k)
    for t in range(B):
        assert np.array_equal(again[t].kept, res[1][t].kept)


def test_single_layer_stack_is_the_layer_on_the_normalised_input(layers):
    B = 2
    sh = layers[0].shape
    h0 = 3.0 * S.activations(13, B, sh.H)
    ids, w = routing_stack(1, B, sh.E, sh.topk, seed=60)
    res, h_out = R.decode_stack(layers[:1], h0, ids, w, 24)
    x = R.rms_normalise(h0).astype(np.float32)
    direct = R.decode(layers[0], x, ids[0], w[0], 24)
    for t in range(B):
        assert np.array_equal(direct[t].y, res[0][t].y)
    with pytest.raises(AssertionError):   # the raw residual is not the input
        raw = R.decode(layers[0], h0.astype(np.float32), ids[0], w[0], 24)
        for t in range(B):
            assert np.array_equal(raw[t].y, res[0][t].y)
