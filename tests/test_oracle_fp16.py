"""Pins of the oracle's FP16 arithmetic and activation (CPU only).

What fixes the expected values:
 - IEEE 754 binary16 conversion, checked against numpy's own float16
   conversion (a separate implementation) on every binary16 pattern and on
   the float32 values where rounding is decided (ties, neighbours of ties,
   the subnormal range, the overflow threshold) plus random bit patterns.
 - "Profiling neural material inference", "Bad versus good activation": the
   max form and the branchy per-lane form are the same operation, with the
   slope written half(0.01).
"""
import numpy as np
import pytest

ALL16 = np.arange(65536, dtype=np.uint32).astype(np.uint16)


def _is_nan16(h):
    return ((h & 0x7C00) == 0x7C00) & ((h & 0x3FF) != 0)


def test_f16_to_f32_all_patterns(orc):
    got = orc.f16_to_f32_array(ALL16)
    ref = ALL16.view(np.float16).astype(np.float32)
    nan = _is_nan16(ALL16)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_f16_roundtrip_all_patterns(orc):
    back = orc.f32_to_f16_array(orc.f16_to_f32_array(ALL16))
    nan = _is_nan16(ALL16)
    assert np.array_equal(back[~nan], ALL16[~nan])
    assert _is_nan16(back[nan]).all()


def _decision_points():
    """float32 values where binary16 rounding is decided."""
    h = ALL16[~_is_nan16(ALL16) & ((ALL16 & 0x7C00) != 0x7C00)]
    v = np.unique(np.abs(h.view(np.float16).astype(np.float64)))
    mids = (v[:-1] + v[1:]) / 2.0                 # exact ties, representable in float32
    pts = [v, mids, np.array([65504.0, 65519.0, 65520.0, 65535.0, 65536.0, 1e6,
                              2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26, 2.0 ** -26,
                              2.0 ** -14, 2.0 ** -14 - 2.0 ** -25])]
    x = np.concatenate(pts).astype(np.float32)
    assert np.array_equal(x.astype(np.float64)[:len(v) + len(mids)],
                          np.concatenate([v, mids]))   # ties survived the cast
    up = np.nextafter(x, np.float32(np.inf))
    dn = np.nextafter(x, np.float32(0))
    x = np.concatenate([x, up, dn])
    return np.concatenate([x, -x])


def test_f32_to_f16_rounding_points(orc):
    x = _decision_points()
    got = orc.f32_to_f16_array(x)
    ref = x.astype(np.float16).view(np.uint16)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(float(x[i]), hex(got[i]), hex(ref[i])) for i in bad[:10]]


def test_f32_to_f16_random_bits(orc):
    rng = np.random.default_rng(12345)
    bits = rng.integers(0, 2 ** 32, size=2_000_000, dtype=np.uint64).astype(np.uint32)
    # also concentrate on the binary16 range (exponents 100..143)
    exps = rng.integers(100, 144, size=2_000_000, dtype=np.uint64).astype(np.uint32)
    mant = rng.integers(0, 2 ** 23, size=2_000_000, dtype=np.uint64).astype(np.uint32)
    sign = rng.integers(0, 2, size=2_000_000, dtype=np.uint64).astype(np.uint32)
    bits2 = (sign << 31) | (exps << 23) | mant
    x = np.concatenate([bits, bits2]).view(np.float32)
    got = orc.f32_to_f16_array(x)
    with np.errstate(over="ignore", invalid="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    nan = np.isnan(x)
    assert _is_nan16(got[nan]).all()
    assert np.array_equal(got[~nan], ref[~nan])


def test_slope_is_half_of_0_01(orc):
    # value = max(value, value * half(0.01)): the slope is the FP16 value
    # nearest 0.01, 1311 * 2^-17.
    s = orc.slope_f16()
    assert s == 0x211F
    assert orc.f16_to_f32(s) == 1311 * 2.0 ** -17 == 0.01000213623046875
    assert s == int(np.float16(0.01).view(np.uint16))


def test_activation_forms_agree_on_every_pattern(orc):
    # The page's two activations (max form, branchy per-lane form) agree on
    # all 65,536 FP16 patterns; NaN inputs give NaN in both.
    a = orc.leaky_max_array(ALL16)
    b = orc.leaky_branchy_array(ALL16)
    nan = _is_nan16(ALL16)
    assert np.array_equal(a[~nan], b[~nan])
    assert _is_nan16(a[nan]).all() and _is_nan16(b[nan]).all()


def test_activation_closed_form(orc):
    # Non-negative values pass through; negative ones become the FP16 product
    # with half(0.01), computed here by numpy's float16 arithmetic.
    a = orc.leaky_max_array(ALL16)
    h = ALL16.view(np.float16)
    finite = np.isfinite(h)
    neg = finite & (h < 0)
    pos = finite & ~(h < 0)
    assert np.array_equal(a[pos], ALL16[pos])          # includes +0 and -0
    prod = (h[neg] * np.float16(0.01)).view(np.uint16)
    assert np.array_equal(a[neg], prod)
    assert orc.leaky_max(0xBC00) == 0xA11F             # -1 -> -half(0.01)
    assert orc.leaky_max(0x8000) == 0x8000             # -0 stays -0
    assert orc.leaky_max(0xFC00) == 0xFC00             # -inf * 0.01 = -inf
