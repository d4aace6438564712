"""Shared test helpers: seeded layers for the oracle (no method arithmetic)."""

import numpy as np

from calibration_free_sparse_gb300 import synthetic as S
from oracle import reader as R


def make_layer(H, E, topk, I, c=80, r=8, seed=0):
    shape = R.Shape(H=H, E=E, topk=topk, I=I, c=c, r=r)
    G, V, D = S.weights(seed, E, I, H)
    sigma = S.signs(seed, shape.Hp)
    return R.Layer(shape, G, V, D, sigma)


def make_tokens(layer, B, seed=0):
    sh = layer.shape
    x = S.activations(seed, B, sh.H)
    ids, w = S.routing(seed, B, sh.E, sh.topk)
    return x, ids, w


def dense_moe(layer, x, ids, w):
    """Textbook gated MoE output sum_e w_e D_e (phi(G_e x) * (V_e x)), fp64."""
    out = np.zeros(layer.shape.H)
    x = x.astype(np.float64)
    for e, we in zip(ids, w):
        G = layer.g(int(e))
        V = layer.v(int(e))
        D = layer.d(int(e))
        h = G @ x
        out += float(we) * (D @ ((h / (1 + np.exp(-h))) * (V @ x)))
    return out
