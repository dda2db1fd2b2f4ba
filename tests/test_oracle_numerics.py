"""Pins of the oracle's scalar numerics against IEEE-754 rules and closed forms."""

import numpy as np
import pytest

from oracle.numerics import (FLT_MAX, hdr_forward_exact, hdr_inverse_exact,
                             round_storage, sanitize)


def _all_positive_finite_fp16():
    bits = np.arange(0, 0x7C00, dtype=np.uint16)
    return bits.view(np.float16)


def test_fp16_rounding_is_identity_on_representable_values():
    h = _all_positive_finite_fp16()
    back = round_storage(h.astype(np.float64), "fp16")
    assert np.array_equal(back.view(np.uint16), h.view(np.uint16))
    neg = round_storage(-h.astype(np.float64), "fp16")
    assert np.array_equal(neg.view(np.uint16), h.view(np.uint16) | 0x8000)


def test_fp16_rounding_midpoints_follow_round_to_nearest_even():
    # Consecutive fp16 values a < b; their midpoint is exact in float64.
    h = _all_positive_finite_fp16()
    a = h[:-1].astype(np.float64)
    b = h[1:].astype(np.float64)
    mid = (a + b) / 2
    got = round_storage(mid, "fp16").view(np.uint16)
    abits = h[:-1].view(np.uint16)
    bbits = h[1:].view(np.uint16)
    even = np.where(abits % 2 == 0, abits, bbits)
    assert np.array_equal(got, even)
    up = round_storage(mid + (b - a) * 1e-6, "fp16").view(np.uint16)
    down = round_storage(mid - (b - a) * 1e-6, "fp16").view(np.uint16)
    assert np.array_equal(up, bbits)
    assert np.array_equal(down, abits)


def test_fp16_rounding_special_cases():
    cases = {
        65504.0: 0x7BFF,          # largest finite
        65519.99: 0x7BFF,         # below the overflow midpoint
        65520.0: 0x7C00,          # the midpoint to 2^16 rounds to +Inf
        2.0 ** -24: 0x0001,       # smallest subnormal
        2.0 ** -25: 0x0000,       # tie between 0 and 2^-24 -> even (0)
        1.5 * 2.0 ** -25: 0x0001,
        -0.0: 0x8000,
        1.0 + 2.0 ** -11: 0x3C00,  # tie -> even mantissa (1.0)
        1.0 + 2.0 ** -11 + 2.0 ** -40: 0x3C01,  # just above the tie: no double rounding
    }
    for value, bits in cases.items():
        got = round_storage(np.array([value]), "fp16").view(np.uint16)[0]
        assert got == bits, (value, hex(got), hex(bits))
    assert np.isnan(round_storage(np.array([np.nan]), "fp16")[0])


def test_fp32_rounding_ties_to_even():
    one = np.float64(1.0)
    ulp = 2.0 ** -23
    assert round_storage(np.array([one + ulp / 2]), "fp32")[0] == np.float32(1.0)
    assert round_storage(np.array([one + 1.5 * ulp]), "fp32")[0] == np.float32(1.0 + 2 * ulp)


@pytest.mark.parametrize("lo,hi", [(0.0, 1.0), (-1.0, 1.0), (0.0, float(FLT_MAX))])
def test_sanitize_enumerated_cases(lo, hi):
    tiny = np.float32(1e-40)  # subnormal
    inputs = np.array([np.nan, np.inf, -np.inf, 0.0, -0.0, tiny, -tiny,
                       0.5, -0.5, 2.0, -2.0, FLT_MAX, -FLT_MAX], np.float32)
    out = sanitize(inputs, lo, hi)
    assert out.dtype == np.float32
    assert not np.isnan(out).any()
    assert (out >= lo).all() and (out <= hi).all()
    expected = []
    for v in inputs:
        if np.isnan(v):
            v = np.float32(0.0)
        if v < lo:
            v = np.float32(lo)
        elif v > hi:
            v = np.float32(hi)
        expected.append(v)
    assert np.array_equal(out.view(np.uint32), np.array(expected, np.float32).view(np.uint32))
    # in-range values (including -0.0 and subnormals) pass through bit for bit
    inside = (inputs >= lo) & (inputs <= hi)
    assert np.array_equal(out[inside].view(np.uint32), inputs[inside].view(np.uint32))


def test_hdr_transfer_closed_forms():
    x = np.array([0.0, 1.0, 3.0, 7.0, 15.0, 2.0 ** 20 - 1], np.float64)
    assert np.allclose(hdr_forward_exact(x), [0, 1, 2, 3, 4, 20], rtol=0, atol=1e-15 * 20)
    assert hdr_forward_exact(np.float32(0.0)) == 0.0
    y = np.array([0.0, 1.0, 2.0, 3.0, 10.0])
    assert np.allclose(hdr_inverse_exact(y), [0, 1, 3, 7, 1023], rtol=1e-15)


def test_hdr_transfer_round_trip_and_monotone():
    x = np.logspace(-30, 38, 20001).astype(np.float32).astype(np.float64)
    f = hdr_forward_exact(x)
    assert (np.diff(f) >= 0).all()
    back = hdr_inverse_exact(f)
    assert np.allclose(back, x, rtol=4 * 2.0 ** -52 * 64, atol=0)
    # small x: F(x) ~ x / ln 2 (derivative at 0)
    small = np.array([1e-20, 1e-12], np.float64)
    assert np.allclose(hdr_forward_exact(small), small / np.log(2.0), rtol=1e-12)
