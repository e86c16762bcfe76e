"""Pins for the oracle's binary16 conversions (f16 KV storage: Leone, "What
ships"; LeatEngine, "Run").

The oracle rounds fp32 -> f16 with its own routine written from the format
definition.  It is pinned to: hand-derived patterns at every rounding boundary
(golden file), exact rational arithmetic, numpy's float16 conversion, and GCC's
_Float16 conversion, over every tie of the binary16 grid and a random sample of
all fp32 bit patterns."""
import json
import os
import subprocess
import tempfile
from fractions import Fraction

import numpy as np
import pytest

import oracle as O
from conftest import GOLDEN


def _golden():
    with open(os.path.join(GOLDEN, "f16_rounding.json")) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _golden(), ids=lambda c: c["x"])
def test_golden_f16_patterns(case):
    x = float.fromhex(case["x"]) if "0x" in case["x"] else float(case["x"])
    assert O.f16_from_f32(x) == int(case["bits"], 16), case["note"]


def _f16_rne_exact(x: float) -> int:
    """binary16 bits of fp32 x by exact rational arithmetic: enumerate the two
    neighbouring representable values and pick the nearer, ties to even."""
    if x != x:
        raise ValueError
    sign = 0x8000 if np.signbit(x) else 0
    a = Fraction(abs(x))
    if a == 0:
        return sign
    # all non-negative finite binary16 values are k * 2^-24 * 2^max(e,0)... walk the grid:
    # value(bits) for bits in [0, 0x7c00) is increasing; binary search on it.
    def val(b):
        e, f = b >> 10, b & 0x3FF
        return Fraction(f, 1 << 24) if e == 0 else Fraction(1024 + f, 1 << 10) * Fraction(2) ** (e - 15)
    lo, hi = 0, 0x7BFF
    if a >= val(0x7BFF):
        # above the largest finite value: overflow threshold is the midpoint 65520
        return sign | (0x7C00 if a >= Fraction(65520) else 0x7BFF)
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if val(mid) <= a:
            lo = mid
        else:
            hi = mid
    dlo, dhi = a - val(lo), val(hi) - a
    if dlo < dhi:
        return sign | lo
    if dhi < dlo:
        return sign | hi
    return sign | (lo if lo % 2 == 0 else hi)


def _tie_values():
    """fp32 values on, just below and just above every binary16 rounding midpoint,
    over the normal and subnormal range, both signs."""
    out = []
    for e in range(-26, 16):
        for frac in range(0, 1024, 7):
            base = (1024 + frac) * 2.0 ** (e - 10)  # a value on the f16-like grid
            mid = base + 2.0 ** (e - 11)
            for v in (mid, np.nextafter(np.float32(mid), np.float32(0)),
                      np.nextafter(np.float32(mid), np.float32(np.inf))):
                v32 = np.float32(v)
                if np.isfinite(v32):
                    out += [float(v32), -float(v32)]
    for k in range(0, 1024, 3):  # subnormal midpoints (k + 1/2) * 2^-24
        mid = (k + 0.5) * 2.0 ** -24
        out += [mid, -mid, float(np.nextafter(np.float32(mid), np.float32(1)))]
    return np.array(out, np.float32)


def test_matches_exact_rational_rounding_on_ties():
    xs = _tie_values()
    got = O.f16_encode(xs)
    sample = np.random.default_rng(7).choice(xs.size, 3000, replace=False)
    for i in sample:
        assert got[i] == _f16_rne_exact(float(xs[i])), float(xs[i])


def test_matches_numpy_float16_on_ties_and_random_bits():
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 2**32, size=400_000, dtype=np.uint64).astype(np.uint32)
    xs = np.concatenate([_tie_values(), bits.view(np.float32)])
    xs = xs[~np.isnan(xs)]
    with np.errstate(over="ignore"):
        ref = xs.astype(np.float16).view(np.uint16)
    np.testing.assert_array_equal(O.f16_encode(xs), ref)


def test_matches_gcc_float16():
    src = r"""
    #include <stdio.h>
    #include <stdint.h>
    #include <string.h>
    int main(void) {
      uint32_t u; float f; _Float16 h; uint16_t b;
      while (scanf("%u", &u) == 1) { memcpy(&f, &u, 4); h = (_Float16)f; memcpy(&b, &h, 2);
        printf("%u\n", (unsigned)b); }
      return 0;
    }"""
    with tempfile.TemporaryDirectory() as tmp:
        c = os.path.join(tmp, "h.c")
        exe = os.path.join(tmp, "h")
        with open(c, "w") as f:
            f.write(src)
        r = subprocess.run(["gcc", "-O0", c, "-o", exe], capture_output=True)
        if r.returncode != 0:
            pytest.skip("gcc has no _Float16 on this target")
        xs = _tie_values()[::5]
        rng = np.random.default_rng(2)
        xs = np.concatenate([xs, rng.standard_normal(2000).astype(np.float32) * 1000])
        inp = "\n".join(str(int(u)) for u in xs.view(np.uint32))
        out = subprocess.run([exe], input=inp, capture_output=True, text=True, check=True).stdout
        ref = np.array([int(v) for v in out.split()], np.uint16)
    np.testing.assert_array_equal(O.f16_encode(xs), ref)


def test_widening_is_exact_for_every_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = O.f16_decode(bits)
    nan = np.isnan(ref)
    np.testing.assert_array_equal(np.isnan(got), nan)
    np.testing.assert_array_equal(got[~nan], ref[~nan])
    # and signs of zeros
    assert np.signbit(got[0x8000]) and not np.signbit(got[0])


def test_round_trip_of_representable_values():
    bits = np.arange(0x7C00, dtype=np.uint16)
    vals = bits.view(np.float16).astype(np.float32)
    np.testing.assert_array_equal(O.f16_encode(vals), bits)
    np.testing.assert_array_equal(O.f16_encode(-vals), bits | 0x8000)
