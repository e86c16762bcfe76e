"""Pins for the oracle's bfloat16 rounding and widening (the stored form of
BF16 KV: tinyllm, "The repository currently provides": BF16/F32 KV caching).

bfloat16 is the high half of a binary32, rounded to nearest with ties to
even.  Pinned to hand-derived cases (tests/golden/bf16_rounding.json), to an
exact rational computation of round-to-nearest-even on 8 significant bits,
to torch's own fp32 -> bfloat16 conversion on the CPU, and (widening) to the
definition "the value of the binary32 whose high half is the pattern" for
every one of the 65,536 patterns."""
import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle as O
from conftest import GOLDEN


def _golden():
    with open(os.path.join(GOLDEN, "bf16_rounding.json")) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _golden(), ids=lambda c: c["x"])
def test_hand_derived_cases(case):
    assert O.bf16_from_f32(float(case["x"])) == int(case["bits"], 16), case["why"]


def test_widening_every_pattern_is_the_high_half_of_a_binary32():
    bits = np.arange(65536, dtype=np.uint32)
    as_f32 = (bits << 16).view(np.float32).astype(np.float64)
    got = np.array([O.bf16_to_f64(int(b)) for b in bits])
    nan = np.isnan(as_f32)
    assert np.array_equal(np.isnan(got), nan)
    np.testing.assert_array_equal(got[~nan], as_f32[~nan])


def _rne8(x: float) -> float:
    """Round-to-nearest-even of a finite fp32 x to 8 significant bits, exactly
    (normal range only), with Python rationals."""
    if x == 0:
        return x
    a = Fraction(abs(x))
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    ulp = Fraction(2) ** (e - 7)
    n = a / ulp
    whole = n.numerator // n.denominator
    rem = n - whole
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and whole % 2 == 1):
        whole += 1
    r = float(whole * ulp)
    return -r if x < 0 else r


def test_exact_rational_rounding():
    rng = np.random.default_rng(3)
    xs = np.concatenate([rng.standard_normal(3000) * 10.0 ** rng.integers(-30, 30, 3000),
                         np.float32(1.0) + np.arange(1, 512) * np.float32(2.0 ** -16)])
    for x in xs.astype(np.float32):
        want = _rne8(float(x))
        assert O.bf16_to_f64(O.bf16_from_f32(float(x))) == want, float(x)


def test_torch_cpu_conversion_agrees():
    rng = np.random.default_rng(4)
    raw = rng.integers(0, 2**32, 20000, dtype=np.uint64).astype(np.uint32)
    xs = raw.view(np.float32)
    xs = xs[np.isfinite(xs)]
    mids = ((rng.integers(0, 2**16, 5000, dtype=np.uint32) << 16) | 0x8000).view(np.float32)
    xs = np.concatenate([xs, mids[np.isfinite(mids)]])  # exact ties
    ours = O.bf16_encode(xs)
    theirs = torch.from_numpy(xs).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, theirs)
