"""Pins of the oracle's number formats: bf16 rounding, E4M3 encode/decode and
the E8M0 (MX) scale exponent.

Each value is checked against something other than the oracle's own code:
the closed forms of the OCP E4M3 / MX definitions, brute force over every
code, and PyTorch's independent float8_e4m3fn / bfloat16 conversions.
"""
import math

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _e4m3_closed_form(code: int) -> float:
    s, e, m = code >> 7, (code >> 3) & 15, code & 7
    if e == 15 and m == 7:
        return math.nan
    mag = m * 2.0 ** -9 if e == 0 else (8 + m) * 2.0 ** (e - 10)
    return -mag if s else mag


def test_e4m3_decode_all_codes_match_torch_and_closed_form():
    torch_vals = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    for c in range(256):
        v = oracle.e4m3_decode(c)
        cf = _e4m3_closed_form(c)
        if math.isnan(cf):
            assert math.isnan(v) and math.isnan(torch_vals[c]) and c in (0x7F, 0xFF)
            continue
        assert v == cf == torch_vals[c], hex(c)
        assert math.copysign(1.0, v) == math.copysign(1.0, cf)


def test_e4m3_defining_points():
    # largest finite, smallest subnormal, smallest normal, one, 2^8
    assert oracle.e4m3_decode(0x7E) == 448.0
    assert oracle.e4m3_decode(0x01) == 2.0 ** -9
    assert oracle.e4m3_decode(0x08) == 2.0 ** -6
    assert oracle.e4m3_decode(0x38) == 1.0
    assert oracle.e4m3_decode(0x78) == 256.0
    assert oracle.e4m3_decode(0xFE) == -448.0


def test_e4m3_round_trip_every_finite_code():
    for c in range(256):
        if c & 0x7F == 0x7F:
            continue
        assert oracle.e4m3_encode(oracle.e4m3_decode(c)) == c, hex(c)


def test_e4m3_midpoints_round_to_even_code():
    finite = [c for c in range(0x7F)]
    for lo, hi in zip(finite[:-1], finite[1:]):
        mid = 0.5 * (oracle.e4m3_decode(lo) + oracle.e4m3_decode(hi))
        want = lo if lo % 2 == 0 else hi
        assert oracle.e4m3_encode(mid) == want
        assert oracle.e4m3_encode(-mid) == want | 0x80
        # just off the midpoint the nearest code wins
        assert oracle.e4m3_encode(mid * (1 - 1e-12)) == lo
        assert oracle.e4m3_encode(mid * (1 + 1e-12)) == hi


def test_e4m3_saturates_and_keeps_nan():
    for v in (448.0, 449.0, 464.0, 480.0, 1e6, 1e300, math.inf):
        assert oracle.e4m3_encode(v) == 0x7E
        assert oracle.e4m3_encode(-v) == 0xFE
    assert oracle.e4m3_encode(math.nan) & 0x7F == 0x7F
    assert oracle.e4m3_encode(0.0) == 0x00
    assert oracle.e4m3_encode(-0.0) == 0x80
    # below half the smallest subnormal -> zero; at exactly half -> zero (even)
    assert oracle.e4m3_encode(2.0 ** -10) == 0x00
    assert oracle.e4m3_encode(2.0 ** -10 * 1.0001) == 0x01


def test_e4m3_encode_matches_torch_on_dense_grid():
    rng = np.random.default_rng(7)
    vals = np.concatenate([
        rng.uniform(-463.0, 463.0, 3000),
        rng.standard_normal(3000) * 2.0 ** rng.integers(-12, 8, 3000),
    ]).astype(np.float32)
    want = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(float(v)) for v in vals], dtype=np.uint8)
    np.testing.assert_array_equal(got, want)


def test_bf16_round_matches_torch():
    rng = np.random.default_rng(11)
    vals = np.concatenate([
        rng.standard_normal(5000).astype(np.float32) * np.float32(2.0) ** rng.integers(-140, 120, 5000),
        np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 2.0 ** -133, 2.0 ** -134, 3 * 2.0 ** -135,
                  3.3895313892515355e38, 3.3961776e38, -0.0, 0.0], dtype=np.float32),
    ])
    want = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.bf16_round(float(v)) for v in vals], dtype=np.uint16)
    np.testing.assert_array_equal(got, want)


def test_bf16_ties_and_overflow():
    assert oracle.bf16_round(1 + 2 ** -8) == 0x3F80          # tie -> even (1.0)
    assert oracle.bf16_round(1 + 3 * 2 ** -8) == 0x3F82      # tie -> even (1 + 2^-6)
    assert oracle.bf16_round(2.0 ** 128 * (1 - 2 ** -9)) == 0x7F80   # rounds past the max -> inf
    assert oracle.bf16_round(2.0 ** 128 * (1 - 2 ** -8)) == 0x7F7F   # the largest finite bf16
    for b in (0x0001, 0x3F80, 0xC2F7, 0x7F7F, 0x8000):
        assert oracle.bf16_round(oracle.bf16_decode(b)) == b


@pytest.mark.parametrize("k", [-100, -20, -9, -1, 0, 1, 5, 8, 100])
def test_mx_scale_exponent_closed_form(k):
    # floor(log2(amax)) - 8 over the whole binade [2^k, 2^(k+1))
    for f in (1.0, 1.0000001, 1.5, 1.9, 1.9999999):
        assert oracle.mx_scale_exp(f * 2.0 ** k) == k - 8


def test_mx_scale_exponent_clamps():
    assert oracle.mx_scale_exp(0.0) == -127
    assert oracle.mx_scale_exp(2.0 ** -119) == -127
    assert oracle.mx_scale_exp(2.0 ** -130) == -127
    assert oracle.mx_scale_exp(2.0 ** -118) == -126
    assert oracle.mx_scale_exp(2.0 ** 200) == 127
