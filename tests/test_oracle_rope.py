"""Pins of the oracle's rotary position embedding (pre-RoPE key quantization).

"O Seu Cache KV Nao Tem um Problema de Bits. Tem um Problema de Geometria",
section "Embebedos Rotatorios Complicam as Chaves": RoPE turns pairs of
channels by an angle set by each token's position; keys are quantized before
the rotation and rotated after dequantization (section "O Que Fazer Com
Isso", item 2).  The oracle's reading: pairs (2i, 2i+1), angle t * theta_i,
theta_i = base^(-2i/dim), position = index in the sequence.  Each pin below
catches a different plausible mistake: a wrong pair layout or frequency (the
complex-exponential form and the worked values), a sign error (norms are kept
by either sign, but the worked values and the complex form are not), a wrong
position (identity at 0, the relative-position property), and rows past a
sequence's end being touched.
"""
import math

import numpy as np
import pytest

import oracle


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def test_position_zero_is_identity():
    x = _rand((2, 3, 5, 64), 0)
    y = oracle.rope(x, [5, 5], 10000.0)
    np.testing.assert_array_equal(y[:, :, 0], x[:, :, 0])


def test_worked_values_single_pair():
    # dim 2: theta_0 = base^0 = 1, so the token at position t turns by t radians
    x = np.zeros((1, 1, 4, 2))
    x[0, 0, :, 0] = 1.0
    y = oracle.rope(x, [4], 10000.0)[0, 0]
    for t in range(4):
        assert y[t, 0] == pytest.approx(math.cos(t), abs=1e-15)
        assert y[t, 1] == pytest.approx(math.sin(t), abs=1e-15)


def test_worked_values_last_pair_frequency():
    # dim 8, base 100: pair 3 turns by t * 100^(-6/8) = t / 31.6227766...
    x = np.zeros((1, 1, 11, 8))
    x[0, 0, :, 7] = 1.0  # second channel of pair 3
    y = oracle.rope(x, [11], 100.0)[0, 0]
    a = 10 * 100.0 ** (-0.75)
    assert y[10, 6] == pytest.approx(-math.sin(a), abs=1e-15)
    assert y[10, 7] == pytest.approx(math.cos(a), abs=1e-15)
    np.testing.assert_array_equal(y[:, :6], 0.0)


def test_matches_complex_exponential_form():
    """Independent restatement: pair i as the complex number x_2i + i x_2i+1,
    multiplied by exp(i t theta_i)."""
    B, H, T, D = 2, 2, 300, 128
    base = 10000.0
    x = _rand((B, H, T, D), 1) * 3.0
    y = oracle.rope(x, [T, T], base)
    z = x[..., 0::2] + 1j * x[..., 1::2]
    theta = base ** (-np.arange(D // 2) * 2.0 / D)
    rot = z * np.exp(1j * np.arange(T)[:, None] * theta[None, :])
    np.testing.assert_allclose(y[..., 0::2], rot.real, rtol=0, atol=1e-12)
    np.testing.assert_allclose(y[..., 1::2], rot.imag, rtol=0, atol=1e-12)


def test_keeps_pair_norms():
    x = _rand((1, 4, 200, 64), 2)
    y = oracle.rope(x, [200], 500000.0)
    np.testing.assert_allclose(y[..., 0::2] ** 2 + y[..., 1::2] ** 2, x[..., 0::2] ** 2 + x[..., 1::2] ** 2,
                               rtol=1e-12)


def test_scores_depend_only_on_relative_position():
    """R(p) q . R(t) k = q . R(t - p) k: a query at position p against a key at
    t gives the score of an unrotated query against the key at t - p."""
    D = 64
    q = _rand(D, 3)
    k = _rand(D, 4)
    base = 10000.0
    T = 900

    def rotated(v, t):
        x = np.zeros((1, 1, T, D))
        x[0, 0, t] = v
        return oracle.rope(x, [T], base)[0, 0, t]

    for p, t in ((5, 17), (100, 300), (0, 899), (640, 641)):
        assert rotated(q, p) @ rotated(k, t) == pytest.approx(q @ rotated(k, t - p), rel=1e-10, abs=1e-10)


def test_rows_past_the_length_are_untouched():
    x = _rand((2, 1, 50, 32), 5)
    y = oracle.rope(x, [20, 0], 10000.0)
    np.testing.assert_array_equal(y[0, :, 20:], x[0, :, 20:])
    np.testing.assert_array_equal(y[1], x[1])
    assert not np.array_equal(y[0, :, 1:20], x[0, :, 1:20])


def test_rope_spreads_a_fixed_outlier_channel():
    """The page's mechanism: a key channel that is large at every token is
    turned into its pair partner as the position grows, so after RoPE the
    partner channel inherits the outlier range (per-channel groups of
    post-RoPE keys then see a wide range in both channels)."""
    T, D = 512, 64
    x = _rand((1, 1, T, D), 6)
    x[..., 0] += 20.0  # fixed outlier channel 0 (pair 0 turns by t radians)
    y = oracle.rope(x, [T], 10000.0)
    assert np.ptp(x[0, 0, :, 1]) < 10.0
    assert np.ptp(y[0, 0, :, 1]) > 35.0  # the partner now swings over about +-20
