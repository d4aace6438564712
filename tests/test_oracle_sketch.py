"""Pins of the oracle's ternary sketch, packing and down norms (no GPU)."""

import numpy as np
import pytest

from oracle import reader as R


def test_constant_magnitude_block_is_exactly_ternary():
    rng = np.random.default_rng(0)
    signs = np.where(rng.random((5, 128)) < 0.5, -1.0, 1.0)
    w = 0.375 * signs                        # |w| = m everywhere: Delta = 0.7 m < m
    t, a, rho = R.ternarize(w)
    assert np.array_equal(t, signs.astype(np.int8))
    assert np.all(a == np.float16(0.375)) and np.all(rho == 0)


def test_two_level_block_hand_computed():
    # 64 entries of +-2 and 64 of +-0.5: mean|w| = 1.25, Delta = 0.875,
    # support = the +-2 entries, alpha = 2, rho = (64 * 0.25) / 128 = 0.125
    rng = np.random.default_rng(1)
    s = np.where(rng.random(128) < 0.5, -1.0, 1.0)
    mag = np.array([2.0] * 64 + [0.5] * 64)
    perm = rng.permutation(128)
    w = (s * mag)[perm]
    t, a, rho = R.ternarize(w[None])
    expect_t = np.where(np.abs(w) > 1, np.sign(w), 0).astype(np.int8)
    assert np.array_equal(t[0], expect_t)
    assert a[0] == np.float16(2.0) and rho[0] == np.float16(0.125)


def test_zero_block():
    t, a, rho = R.ternarize(np.zeros((2, 128)))
    assert not t.any() and not a.any() and not rho.any()


def test_alpha_is_least_squares_for_its_support():
    rng = np.random.default_rng(2)
    w = rng.standard_normal((50, 128))
    t, a, rho = R.ternarize(w)
    tf = t.astype(float)
    # unrounded alpha minimises sum (w - alpha t)^2 over alpha for the fixed support
    alpha = (np.abs(w) * (t != 0)).sum(1) / (t != 0).sum(1)
    err = lambda al: ((w - al[:, None] * tf) ** 2).sum(1)  # noqa: E731
    for eps in (1e-3, -1e-3):
        assert np.all(err(alpha) <= err(alpha + eps))
    assert np.allclose(a.astype(float), alpha, rtol=1e-3)
    # stored rho is the mean squared residual with the stored fp16 alpha
    res = ((w - a.astype(float)[:, None] * tf) ** 2).mean(1)
    assert np.allclose(rho.astype(float), res, rtol=1e-3)


def test_twn_support_fraction_gaussian():
    # For Gaussian blocks the TWN threshold 0.7 E|w| keeps P(|z| > 0.7*0.798) ~ 0.576
    rng = np.random.default_rng(3)
    t, _, _ = R.ternarize(rng.standard_normal((4000, 128)))
    frac = (t != 0).mean()
    assert abs(frac - 0.576) < 0.01


def test_pack_bit_positions():
    t = np.array([1, -1, 0, 1, 0, 0, -1, 0], np.int8)
    p = R.pack_codes(t)
    assert p.shape == (32,)                               # padded to one sector
    assert p[0] == (0b01 | 0b11 << 2 | 0b00 << 4 | 0b01 << 6)
    assert p[1] == (0b11 << 4)
    assert not p[2:].any()


@pytest.mark.parametrize("I", [4, 64, 128, 768, 2880])
def test_pack_roundtrip_and_stride(I):
    rng = np.random.default_rng(I)
    t = rng.integers(-1, 2, (3, I)).astype(np.int8)
    p = R.pack_codes(t)
    assert p.shape[-1] == R.run_stride(I) and p.shape[-1] % 32 == 0
    assert np.array_equal(R.unpack_codes(p, I), t)


def test_sketch_layout_matches_definition():
    rng = np.random.default_rng(4)
    I, H = 64, 256
    G = rng.standard_normal((I, H))
    V = rng.standard_normal((I, H))
    sigma = np.where(rng.random(H) < 0.5, -1, 1).astype(np.int8)
    sk = R.sketch_expert(G, V, sigma, H)
    packed = sk.packed()                                   # [nb][128][2][S]
    assert packed.shape == (2, 128, 2, 32)
    # coordinate c of block b, gate run: trits of channel i
    Gr = R.rotate(G, sigma).reshape(I, 2, 128)
    t, a, _ = R.ternarize(Gr)
    for b in range(2):
        for c in (0, 17, 127):
            assert np.array_equal(R.unpack_codes(packed[b, c, 0], I), t[:, b, c])
        assert np.array_equal(sk.alpha[b, 0], a[:, b])


def test_down_norms_match_library_norm():
    rng = np.random.default_rng(5)
    D = rng.standard_normal((300, 40))
    assert np.allclose(R.down_norms(D), np.linalg.norm(D, axis=0).astype(np.float32))


def test_bf16_decode():
    bits = np.array([0x3F80, 0xBF80, 0x0000, 0x4049, 0x0001], np.uint16)
    vals = R.bf16_bits_to_f64(bits)
    assert vals[0] == 1.0 and vals[1] == -1.0 and vals[2] == 0.0
    assert vals[3] == 3.140625
    assert vals[4] == 2.0 ** -133
