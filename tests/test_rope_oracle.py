"""Pins of the RoPE-realignment oracle (oracle/rope.py) against facts that do
not come from its own formula."""
import math

import numpy as np
import pytest

from oracle import rope


def _rope_abs(x, p, theta=10000.0):
    """Absolute rotary embedding at position p, written independently as a
    complex multiplication: pair i is the complex number x[i] + j x[i + d/2]
    turned by exp(j p theta^(-2i/d))."""
    d = x.shape[-1]
    z = x[..., : d // 2] + 1j * x[..., d // 2:]
    w = np.exp(1j * p * theta ** (-2.0 * np.arange(d // 2) / d))
    z = z * w
    return np.concatenate([z.real, z.imag], axis=-1)


@pytest.mark.parametrize("d", [4, 64, 128])
def test_realign_moves_absolute_rope(d):
    # a key embedded at position n and moved by delta equals the key embedded at n + delta
    rng = np.random.default_rng(d)
    k = rng.standard_normal((5, d))
    for n, delta in [(0, 7), (100, -37), (4096, 123456), (31, 0)]:
        got = rope.realign(_rope_abs(k, n), delta)
        np.testing.assert_allclose(got, _rope_abs(k, n + delta), rtol=0, atol=1e-9)


def test_composition_inverse_and_norms():
    rng = np.random.default_rng(3)
    k = rng.standard_normal((7, 128))
    np.testing.assert_allclose(rope.realign(rope.realign(k, 300), -300), k, atol=1e-12)
    np.testing.assert_allclose(rope.realign(rope.realign(k, 11), 29), rope.realign(k, 40), atol=1e-12)
    r = rope.realign(k, 98765)
    pair = lambda x: x[:, :64] ** 2 + x[:, 64:] ** 2
    np.testing.assert_allclose(pair(r), pair(k), rtol=1e-12)


def test_scores_depend_on_relative_position_only():
    # moving a query and a key by the same delta leaves their dot product
    rng = np.random.default_rng(5)
    q, k = rng.standard_normal(64), rng.standard_normal(64)
    base = float(np.dot(q, k))
    for delta in (1, 17, -5000, 2 ** 20):
        assert abs(float(np.dot(rope.realign(q, delta), rope.realign(k, delta))) - base) < 1e-9


def test_special_angles_by_hand():
    # d = 4: pairs (0, 2) and (1, 3); theta^(-2*1/4) = theta^(-1/2).
    # theta = 4 / pi^2 makes pair 1 turn by exactly pi/2 per position.
    theta = 4.0 / math.pi ** 2
    k = np.array([1.0, 2.0, 3.0, 5.0])
    r = rope.realign(k, 1, theta)
    # pair 1 (2, 5) turned by 90 degrees -> (-5, 2); pair 0 (1, 3) by 1 radian
    np.testing.assert_allclose(r[[1, 3]], [-5.0, 2.0], atol=1e-12)
    np.testing.assert_allclose(r[[0, 2]], [math.cos(1) - 3 * math.sin(1), 3 * math.cos(1) + math.sin(1)],
                               atol=1e-12)
    # two positions: pair 1 turns by pi -> negated
    np.testing.assert_allclose(rope.realign(k, 2, theta)[[1, 3]], [-2.0, -5.0], atol=1e-12)
    # delta 0 is the identity
    np.testing.assert_array_equal(rope.realign(k, 0), k)


def _pair_scales(x, d):
    """Per-channel scales large enough for any rotation of a pair: the
    largest pair norm of each frequency over 440 (so no result saturates)."""
    h = d // 2
    pn = np.sqrt(x[:, :h] ** 2 + x[:, h:] ** 2).max(axis=0) / 440.0
    return np.concatenate([pn, pn]).astype(np.float32)


def test_fp8_realign_zero_delta_keeps_every_value():
    from oracle import fp8
    rng = np.random.default_rng(1)
    d = 128
    s = rng.uniform(2.0 ** -10, 2.0, d).astype(np.float32)
    codes = rng.integers(0, 256, (64, d)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x7E              # no NaN codes in a page
    out = rope.realign_fp8(codes, s, 0)
    # the same values (x*1 - y*0 may turn a negative zero into +0)
    assert np.array_equal(fp8.decode(out), fp8.decode(codes))
    assert np.array_equal(out[codes != 0x80], codes[codes != 0x80])


@pytest.mark.parametrize("delta", [1, -7, 4097, 123457])
def test_fp8_realign_within_half_an_e4m3_step_of_the_exact_rotation(delta):
    from oracle import fp8
    rng = np.random.default_rng(delta & 0xFFFF)
    d = 128
    x = rng.standard_normal((300, d)) * 2.0
    s = _pair_scales(x, d)
    codes = fp8.quantize(x, s)
    got = fp8.dequantize(rope.realign_fp8(codes, s, delta), s)
    exact = realign_ref = rope.realign(fp8.dequantize(codes, s), delta)
    a = np.abs(exact) / s
    step = np.where(a >= 2.0 ** -6, 2.0 ** (np.floor(np.log2(np.maximum(a, 1e-300))) - 3), 2.0 ** -9) * s
    assert np.all(np.abs(got - realign_ref) <= 0.5 * step * (1 + 1e-5) + 1e-12)


def test_fp8_realign_saturates_like_a_write():
    from oracle import fp8
    d = 8
    s = np.array([1.0, 1.0, 1.0, 1.0, 2.0 ** -4, 1.0, 1.0, 1.0], np.float32)
    codes = fp8.quantize(np.array([[448.0, 0, 0, 0, 0, 0, 0, 0]]), s)
    # frequency 0 of d = 8 turns by delta radians: a quarter turn moves 448
    # from channel 0 into channel 4, whose range is only 448 / 16
    delta = 11        # 11 rad = 1.75 turns, close to a quarter turn back
    out = fp8.dequantize(rope.realign_fp8(codes, s, delta, theta=10000.0), s)
    ang = rope.angles(d, delta)[0]
    assert abs(out[0, 4]) == 448.0 * 2.0 ** -4 and np.sign(out[0, 4]) == np.sign(448.0 * np.sin(ang))
