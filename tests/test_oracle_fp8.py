"""Pins of the e4m3 quantiser of the oracle (OCP FP8 E4M3: bias 7, 3
mantissa bits, no infinities, S.1111.111 NaN, max 448, subnormals of 2^-9)
against the format's definition, not against the function itself."""
import numpy as np
import pytest

from oracle import fp8 as F


def test_format_landmarks():
    v = F.e4m3_values()
    assert v[0x7E] == 448.0 and v[0xFE] == -448.0
    assert v[0x08] == 2.0 ** -6              # smallest normal
    assert v[0x01] == 2.0 ** -9              # smallest subnormal
    assert v[0x07] == 7 * 2.0 ** -9          # largest subnormal
    assert v[0x38] == 1.0 and v[0x39] == 1.125
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF])
    assert np.isfinite(np.delete(v, [0x7F, 0xFF])).all()


def test_every_finite_code_round_trips():
    v = F.e4m3_values()
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)])
    assert np.array_equal(F.quantize_codes(v[codes]), codes.astype(np.uint8))


def test_midpoints_round_to_the_even_code_and_neighbours_to_their_side():
    v = F.e4m3_values()
    for c in range(0x7E):                     # adjacent positive values v[c] < v[c+1]
        lo, hi = v[c], v[c + 1]
        mid = (lo + hi) / 2
        even = c if c % 2 == 0 else c + 1
        assert F.quantize_codes([mid])[0] == even
        assert F.quantize_codes([-mid])[0] == (even | 0x80)
        eps = (hi - lo) * 1e-6
        assert F.quantize_codes([mid - eps])[0] == c
        assert F.quantize_codes([mid + eps])[0] == c + 1


def test_saturation_and_signed_zero():
    assert list(F.quantize_codes([448.0, 448.5, 1e9, -1e9])) == [0x7E, 0x7E, 0x7E, 0xFE]
    assert list(F.quantize_codes([0.0, -0.0, 2.0 ** -11, -(2.0 ** -11)])) == [0x00, 0x80, 0x00, 0x80]


@pytest.mark.parametrize("amax", [448.0, 1.75, 1.7500001, 1.0, 3.0, 5.3, 0.01, 1e-5, 300.0, 449.0, 1e4])
def test_power_of_two_scale(amax):
    k = F.pow2_scale_exponent(amax)
    assert amax * 2.0 ** k <= 448.0 < amax * 2.0 ** (k + 1)
    assert F.pow2_scale_exponent(0.0) == 0


def test_scale_exponent_stays_in_fp32_normal_range():
    """The scale 2^k is an fp32 number: for amax below 2^-119 the largest k
    with amax * 2^k <= 448 would exceed 127, so k stops at 127."""
    assert F.pow2_scale_exponent(2.0 ** -119) == 127          # (1.0 <= 1.75) -> 8 + 119
    assert F.pow2_scale_exponent(1.9 * 2.0 ** -120) == 127    # (1.9 > 1.75) -> 7 + 120
    assert F.pow2_scale_exponent(2.0 ** -126) == 127
    assert F.pow2_scale_exponent(2.0 ** -133) == 127          # a bf16 subnormal
    assert F.pow2_scale_exponent(2.0 ** -118) == 126
    codes, k = F.quantize_tensor(np.full(4, 2.0 ** -126))
    assert k == 127 and list(codes) == [0x40] * 4              # 2^-126 * 2^127 = 2.0 = code 0x40


def test_dequantized_tensor_error_within_half_ulp():
    rng = np.random.default_rng(0)
    x = rng.standard_normal(10000) * 3
    y = F.dequantized_tensor(x)
    k = F.pow2_scale_exponent(np.abs(x).max())
    xs, ys = x * 2.0 ** k, y * 2.0 ** k
    # half an ulp of e4m3 at |xs|: 2^(floor(log2|xs|) - 4) for normals, 2^-10 below 2^-6
    e = np.floor(np.log2(np.maximum(np.abs(xs), 2.0 ** -6)))
    assert (np.abs(ys - xs) <= 2.0 ** (e - 4) + 1e-15).all()
