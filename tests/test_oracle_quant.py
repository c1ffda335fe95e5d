"""Pins of the oracle's INT2 quantiser, float16 rounding and 2-bit packing.

Each check ties the oracle to something other than itself: an exact rational
re-derivation of float16 rounding, hand-derived worked examples
(tests/golden), and the closed-form error bound of a uniform quantiser.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import qwm_oracle as O


# ---------------------------------------------------------------- float16 RNE

def _exact_f16(x: Fraction) -> float:
    """Nearest float16 to an exact rational, ties to even; inf beyond the range."""
    if x == 0:
        return 0.0
    sign = -1 if x < 0 else 1
    a = abs(x)
    e = 0
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, -14)                      # subnormals share the spacing 2^-24
    spacing = Fraction(2) ** (e - 10)
    q, rem = divmod(a, spacing)
    half = spacing / 2
    if rem > half or (rem == half and q % 2 == 1):
        q += 1
    v = q * spacing
    if v >= 65520 or (v > 65504):
        return sign * float("inf")
    return sign * float(v)


def test_f16_conversion_is_round_to_nearest_even():
    rng = np.random.default_rng(7)
    vals = list(rng.standard_normal(3000).astype(np.float32) * np.float32(100))
    vals += list((rng.standard_normal(500) * 1e-6).astype(np.float32))       # subnormal range
    vals += list((rng.uniform(6e4, 7e4, 200)).astype(np.float32))            # overflow edge
    # exact midpoints between neighbouring float16 values
    h = rng.integers(0, 0x7BFF, 500).astype(np.uint16).view(np.float16)
    nxt = (h.view(np.uint16) + 1).view(np.float16)
    mids = (h.astype(np.float64) + nxt.astype(np.float64)) / 2
    vals += list(mids.astype(np.float32))
    for v in vals:
        with np.errstate(over="ignore"):
            got = float(np.asarray(v, np.float32).astype(np.float16))
        assert got == _exact_f16(Fraction(float(v))), v


def test_f16_saturate():
    h, sat = O.f16_saturate(np.array([7e4, -7e4, 65504.0, 1.0], np.float32))
    assert h.tolist() == [65504.0, -65504.0, 65504.0, 1.0]
    assert sat.tolist() == [True, True, False, False]


# ------------------------------------------------------------- worked examples

def _golden(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


@pytest.mark.parametrize("name", ["int2_group_0_to_31.json", "int2_group_half_ties.json"])
def test_quantiser_worked_examples(golden_dir, name):
    g = _golden(golden_dir, name)
    x = np.array(g["x"], np.float32)
    zero, scale, codes, sat = O.quantize_int2(x[None, :])
    assert float(zero[0]) == g["zero"]
    assert float(scale[0]) == g["scale"]
    assert codes[0].tolist() == g["codes"]
    assert not sat.any()
    if "packed_hex" in g:
        assert O.pack_codes(codes[0]).tobytes().hex() == g["packed_hex"]


def test_pack_roundtrip_and_bit_order():
    rng = np.random.default_rng(1)
    c = rng.integers(0, 4, (50, 128)).astype(np.uint8)
    p = O.pack_codes(c)
    assert p.shape == (50, 32)
    assert (O.unpack_codes(p) == c).all()
    # channel c lands in bits 2*(c%4) of byte c//4
    one = np.zeros(8, np.uint8)
    one[5] = 3
    assert O.pack_codes(one).tolist() == [0, 3 << 2]


# ------------------------------------------------------------------ error bound

def _groups(rng, n):
    """Groups of 32 float32 values of many shapes: wide, narrow, constant,
    far from zero, tiny, with repeated values."""
    out = []
    for i in range(n):
        kind = i % 6
        if kind == 0:
            x = rng.standard_normal(32) * 10 ** rng.uniform(-3, 3)
        elif kind == 1:
            x = 1000.0 + rng.uniform(0, 0.1, 32)                  # narrow, far from 0
        elif kind == 2:
            x = np.full(32, rng.standard_normal())                # constant
        elif kind == 3:
            x = rng.standard_normal(32) * 1e-6                    # float16 subnormal params
        elif kind == 4:
            x = rng.integers(-3, 4, 32).astype(np.float64) * 0.25
        else:
            x = rng.standard_normal(32) * 300 + rng.standard_normal() * 3000
        out.append(x)
    return np.asarray(out).astype(np.float32)


def _check_bound(x, zero, scale, codes):
    xh = O.dequantize(zero, scale, codes)
    x64 = x.astype(np.float64)
    z = zero.astype(np.float64)[:, None]
    s = scale.astype(np.float64)[:, None]
    slack = np.maximum.reduce([np.zeros_like(z), z - x64.min(1, keepdims=True),
                               x64.max(1, keepdims=True) - (z + 3 * s)])
    tol = np.maximum(s / 2, slack) + 2.0 ** -20 * (np.abs(x64) + np.abs(z) + 3 * s)
    return np.abs(x64 - xh) <= tol


def test_codes_in_range_and_dequant_error_bound():
    rng = np.random.default_rng(3)
    x = _groups(rng, 3000)
    zero, scale, codes, sat = O.quantize_int2(x)
    assert codes.dtype == np.uint8 and codes.max() <= 3
    assert not sat.any()
    assert _check_bound(x, zero, scale, codes).all()
    # constant groups store scale 0 and code 0 and reproduce f16(value)
    const = (x.max(1) == x.min(1))
    assert const.any()
    assert (scale[const] == 0).all() and (codes[const] == 0).all()


def test_bound_catches_truncation_instead_of_rounding(monkeypatch):
    """A quantiser that truncates instead of rounding breaks the bound: the
    bound is tight enough to catch the most plausible quantiser mistake."""
    rng = np.random.default_rng(4)
    x = _groups(rng, 600)
    monkeypatch.setattr(O.np, "rint", np.floor)
    zero, scale, codes, _ = O.quantize_int2(x)
    monkeypatch.undo()
    assert not _check_bound(x, zero, scale, codes).all()


def test_scale_division_single_rounding():
    """f16(f32(R/3)) equals the float16 nearest to the exact R/3: rounding the
    quotient to float32 first never lands on a float16 midpoint."""
    rng = np.random.default_rng(5)
    R = np.abs(rng.standard_normal(4000) * 10 ** rng.uniform(-6, 4, 4000)).astype(np.float32)
    for r in R[:1500]:
        via32 = float((np.float32(r) / np.float32(3)).astype(np.float16))
        exact = _exact_f16(Fraction(float(r)) / 3)
        assert via32 == exact
