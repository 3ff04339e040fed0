"""Pins of the FP8 (E4M3) oracle (oracle/fp8.py) against the format's own
definition, torch's float8_e4m3fn conversions and hand-derived values."""
import numpy as np
import pytest
import torch

from oracle import fp8


def test_decode_hand_values():
    # sign | exponent (bias 7) | mantissa
    cases = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6,
             0x38: 1.0, 0x39: 1.125, 0x3F: 1.875, 0x40: 2.0, 0x7E: 448.0,
             0x77: 240.0, 0xB8: -1.0, 0xFE: -448.0}
    for c, v in cases.items():
        assert fp8.decode([c])[0] == v, hex(c)
    assert np.signbit(fp8.decode([0x80])[0]) and fp8.decode([0x80])[0] == 0.0
    nan = np.isnan(fp8.decode(np.arange(256, dtype=np.uint8)))
    assert nan.sum() == 2 and nan[0x7F] and nan[0xFF]


def test_every_code_matches_torch():
    c = np.arange(256, dtype=np.uint8)
    ours = fp8.decode(c)
    ref = torch.from_numpy(c).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])
    assert np.array_equal(np.signbit(ours[ok]), np.signbit(ref[ok]))


def test_encode_matches_torch_inside_the_range():
    # torch rounds to nearest even as well; above 448 it gives NaN where the
    # saturating conversion gives 448, so compare inside the range only
    rng = np.random.default_rng(7)
    x = np.concatenate([rng.standard_normal(50000) * 40, rng.standard_normal(20000) * 2.0 ** -8,
                        rng.uniform(-448, 448, 20000)]).astype(np.float32)
    # every midpoint between neighbouring codes, and a hair either side
    pos = fp8.decode(np.arange(127, dtype=np.uint8))
    mid = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    x = np.concatenate([x, mid, -mid, np.nextafter(mid, np.float32(0)), np.nextafter(mid, np.float32(500))])
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(fp8.encode(x.astype(np.float64)), ref)


def test_round_trip_of_all_finite_codes():
    c = np.array([i for i in range(256) if i not in (0x7F, 0xFF)], dtype=np.uint8)
    assert np.array_equal(fp8.encode(fp8.decode(c)), c)


@pytest.mark.parametrize("x,code", [
    (1.0625, 0x38),                # halfway 1 .. 1.125: even mantissa (1.0)
    (1.1875, 0x3A),                # halfway 1.125 .. 1.25: even mantissa (1.25)
    (2.0 ** -10, 0x00),            # halfway 0 .. 2^-9
    (3 * 2.0 ** -10, 0x02),        # halfway 2^-9 .. 2^-8
    (-3 * 2.0 ** -10, 0x82),
    (1.06251, 0x39),
    (400.0, 0x7C),                 # step 32 in [256, 512): halfway 384 .. 416 -> 384 (even)
    (416.0, 0x7D),
    (432.0, 0x7E),                 # halfway 416 .. 448 -> 448 (even)
    (448.0, 0x7E), (463.9, 0x7E), (464.0, 0x7E), (1e6, 0x7E), (np.inf, 0x7E),
    (-1e6, 0xFE), (-np.inf, 0xFE), (-1e-9, 0x80), (-0.0, 0x80), (0.0, 0x00),
])
def test_ties_saturation_and_sign(x, code):
    assert fp8.encode([x])[0] == code


def test_nan_maps_to_nan_code():
    assert fp8.encode([np.nan])[0] == 0x7F


def test_half_ulp_error_bound_and_monotone():
    rng = np.random.default_rng(3)
    x = np.sort(np.concatenate([rng.uniform(-448, 448, 40000), rng.uniform(-2 ** -6, 2 ** -6, 40000)]))
    y = fp8.decode(fp8.encode(x))
    err = np.abs(y - x)
    normal = np.abs(x) >= 2.0 ** -6
    # normal range: 3 mantissa bits -> half an ulp is 2^-4 of the binade's base
    assert np.all(err[normal] <= 2.0 ** -4 * 2.0 ** np.floor(np.log2(np.abs(x[normal]))))
    assert np.all(err[~normal] <= 2.0 ** -10)
    assert np.all(np.diff(y) >= 0)


def test_quantize_uses_fp32_reciprocal_and_product():
    # power-of-two scales are exact: the codes are those of x / s
    x = np.array([0.3, -7.25, 100.0, 2.0 ** -12], dtype=np.float32).astype(np.float64)
    s = np.array([0.25, 2.0, 0.5, 2.0 ** -8])
    assert np.array_equal(fp8.quantize(x, s), fp8.encode(x / s))
    # a scale whose reciprocal is not exact: 1/3 in fp32 is 0.3333333432...,
    # so 3 * r rounds up to exactly 1 in fp32 (code 0x38), as it does in
    # float64 arithmetic of the fp32 values
    r = np.float32(1.0) / np.float32(3.0)
    assert float(r) != 1.0 / 3.0
    assert fp8.quantize(np.array([3.0]), np.array([3.0]))[0] == fp8.encode([float(np.float32(3.0) * r)])[0]
    # x * r in fp32 versus exact x / s: pick x where the two sides of a
    # midpoint differ -- the fp32 product decides
    xs = np.float32(np.linspace(1, 400, 200001, dtype=np.float32))
    sc = np.full_like(xs, 3.0, dtype=np.float64)
    q32 = fp8.quantize(xs.astype(np.float64), sc)
    q64 = fp8.encode(xs.astype(np.float64) / 3.0)
    diff = np.nonzero(q32 != q64)[0]
    for i in diff[:20]:
        p = np.float32(xs[i]) * r
        assert q32[i] == fp8.encode([float(p)])[0]
    # dequantize is decode times scale
    c = np.arange(0, 127, 5, dtype=np.uint8)
    assert np.array_equal(fp8.dequantize(c, 0.5), fp8.decode(c) * 0.5)
