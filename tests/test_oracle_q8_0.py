"""Pins for the oracle's q8_0 encoder (LeatEngine, "Run": q8_0 KV cache in about
half the memory of f16; Leone, "What ships": q8 KV storage).

Encoding: blocks of 32 values along head_dim, fp32 scale d = amax / 127 by IEEE
division, stored as f16 (ties to even), codes round(x / d) half away from zero.
Pinned to hand-derived blocks (golden file), to exact rational arithmetic, to
numpy's IEEE fp32 division, and to the error bound |x - d q| <= d/2."""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle as O
from conftest import GOLDEN


def _golden():
    with open(os.path.join(GOLDEN, "q8_0_blocks.json")) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _golden(), ids=lambda c: c["name"])
def test_golden_blocks(case):
    x = np.zeros(32, np.float32)
    x[:len(case["x"])] = case["x"]
    codes, sb, _ = O.q8_0_encode_block(x)
    want = np.zeros(32, np.int8)
    want[:len(case["codes"])] = case["codes"]
    np.testing.assert_array_equal(codes, want, err_msg=case["note"])
    assert sb == int(case["scale_bits"], 16), case["note"]


def _fl32(r: Fraction) -> float:
    """Round a rational to the nearest fp32, ties to even (normal range)."""
    if r == 0:
        return 0.0
    sign = -1 if r < 0 else 1
    a = abs(r)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    ulp = Fraction(2) ** (e - 23)
    n = a / ulp
    whole = n.numerator // n.denominator
    rem = n - whole
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and whole % 2):
        whole += 1
    return sign * float(whole * ulp)


def _encode_exact(x):
    amax = max(abs(Fraction(float(v))) for v in x)
    d = _fl32(amax / 127)
    codes = []
    for v in x:
        if d == 0:
            codes.append(0)
            continue
        y = Fraction(_fl32(Fraction(float(v)) / Fraction(d)))
        c = (abs(y) + Fraction(1, 2)).__floor__()
        codes.append(int(-c if y < 0 else c))
    return np.array(codes, np.int8), d


def test_matches_exact_rational_encoding():
    rng = np.random.default_rng(11)
    for trial in range(60):
        x = rng.standard_normal(32).astype(np.float32) * np.float32(10.0 ** rng.uniform(-3, 3))
        if trial % 3 == 0:  # plant exact ties x/d = k + 1/2 for a power-of-two scale
            x = (rng.integers(-126, 127, 32) + 0.5).astype(np.float32)
            x[0] = 127.0
        codes, sb, d = O.q8_0_encode_block(x)
        want_codes, want_d = _encode_exact(x)
        np.testing.assert_array_equal(codes, want_codes)
        assert d == want_d
        assert sb == O.f16_from_f32(want_d)


def test_matches_numpy_fp32_division():
    rng = np.random.default_rng(12)
    x = rng.standard_normal((4000, 32)).astype(np.float32)
    codes, scales = O.q8_0_encode(x)
    amax = np.abs(x).max(axis=1)
    d = amax / np.float32(127.0)                 # IEEE fp32 division
    y = x / d[:, None]                           # IEEE fp32 division
    ref = np.where(y < 0, -np.floor(-y.astype(np.float64) + 0.5),
                   np.floor(y.astype(np.float64) + 0.5)).astype(np.int8)
    np.testing.assert_array_equal(codes, ref)
    np.testing.assert_array_equal(scales[:, 0], d.astype(np.float16).view(np.uint16))


def test_error_bound_and_range():
    rng = np.random.default_rng(13)
    x = (rng.standard_normal((2000, 32)) * rng.uniform(1e-3, 1e3, (2000, 1))).astype(np.float32)
    codes, _ = O.q8_0_encode(x)
    d = (np.abs(x).max(axis=1).astype(np.float64) / 127.0).astype(np.float32).astype(np.float64)
    err = np.abs(x.astype(np.float64) - d[:, None] * codes)
    # |x - d q| <= d/2 up to the rounding of x/d to fp32 (relative 2^-24 of |x/d| <= 127.5)
    assert np.all(err <= d[:, None] * (0.5 + 128 * 2.0 ** -24))
    assert codes.min() >= -127 and codes.max() <= 127
    # the element holding amax maps to +-127 exactly
    idx = np.abs(x).argmax(axis=1)
    np.testing.assert_array_equal(np.abs(codes[np.arange(2000), idx]), 127)


def test_all_equal_block():
    for v in (3.0, -7.25, 1e-20, 6.0e4):
        codes, sb, d = O.q8_0_encode_block(np.full(32, v, np.float32))
        assert np.all(codes == (127 if v > 0 else -127))


def test_block_bytes_about_half_of_f16():
    # 32 values: 32 int8 codes + one 2-byte f16 scale = 34 bytes, against 64 bytes of f16
    assert (32 * 1 + 2) / (32 * 2) == pytest.approx(0.53125)
    codes, scales = O.q8_0_encode(np.ones((5, 128), np.float32))
    assert codes.nbytes + scales.nbytes == 5 * 4 * 34
