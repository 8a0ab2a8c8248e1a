"""The split-f16 operand scheme of the tensor-core kernels, checked on the host
in exact (float64) arithmetic.

Every fp32 operand v of a tcgen05 kind::f16 product is carried as two f16
parts: hi = v rounded to f16, lo = the remainder v - hi rounded to f16.  The
kernels form the remainder in fp32 (one mixed-precision FMA of the f16 hi, or
a conversion of hi back to fp32 and a subtraction; both give v - hi exactly),
and the error budget of the tensor-core paths rests on three facts checked
here with numpy's IEEE round-to-nearest float16 and float32:

  * v - hi is exact in fp32 (so both kernel forms give the same lo);
  * |v - hi - lo| <= 2^-24 for |v| <= 1 (the sines and cosines of E), i.e.
    fp32's own rounding of a unit-modulus value, and <= 2^-23 |v| for
    1/4 <= |v| <= 1; for the weights, scaled by a power of two below 2^15,
    <= 2^-22 |v|;
  * a product a b of such values taken as hi*hi + hi*lo + lo*hi (the grid
    kernels) is within 3 * 2^-24 of a b, and with lo*lo as well (the coil
    kernel at arbitrary coordinates) within 2 * 2^-24 + 2^-48.
"""

import numpy as np

F16, F32 = np.float16, np.float32


def split(v):
    v = np.asarray(v, dtype=F32)
    hi = v.astype(F16)
    rem = v - hi.astype(F32)                  # fp32 subtraction, as in the kernels
    lo = rem.astype(F16)
    return hi, rem, lo


def unit_values(n=1 << 20, seed=0):
    rng = np.random.default_rng(seed)
    v = rng.uniform(-1.0, 1.0, n).astype(F32)
    # magnitudes spread over many binades, down into f16's subnormal range
    w = (rng.uniform(-1.0, 1.0, n) * np.exp2(-rng.integers(0, 40, n))).astype(F32)
    edges = np.array([0.0, -0.0, 1.0, -1.0, np.nextafter(F32(1), F32(0)), 2.0 ** -14,
                      2.0 ** -15, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26, 0.5 + 2.0 ** -12,
                      0.5 + 2.0 ** -13, 1 - 2.0 ** -12, 1 - 2.0 ** -11 - 2.0 ** -24,
                      np.float32(np.sin(1.0))], dtype=F32)
    return np.concatenate([v, w, edges, -edges])


def test_remainder_is_exact_in_fp32():
    v = unit_values()
    hi, rem, _ = split(v)
    exact = v.astype(np.float64) - hi.astype(np.float64)
    assert np.array_equal(rem.astype(np.float64), exact)


def test_two_parts_within_fp32_rounding_of_a_unit_value():
    v = unit_values()
    hi, _, lo = split(v)
    err = np.abs(v.astype(np.float64) - hi.astype(np.float64) - lo.astype(np.float64))
    assert err.max() <= 2.0 ** -24
    big = np.abs(v) >= 0.25
    assert np.all(err[big] <= 2.0 ** -23 * np.abs(v[big].astype(np.float64)))
    # hi alone would be 2^-12 off: the low part is what carries fp32 precision
    assert np.abs(v.astype(np.float64) - hi.astype(np.float64)).max() > 2.0 ** -13


def test_split_products():
    rng = np.random.default_rng(1)
    a = rng.uniform(-1.0, 1.0, 1 << 20).astype(F32)
    b = rng.uniform(-1.0, 1.0, 1 << 20).astype(F32)
    ah, _, al = split(a)
    bh, _, bl = split(b)
    ah, al, bh, bl = (x.astype(np.float64) for x in (ah, al, bh, bl))
    ab = a.astype(np.float64) * b.astype(np.float64)
    three = ah * bh + ah * bl + al * bh
    four = three + al * bl
    assert np.abs(ab - three).max() <= 3 * 2.0 ** -24
    assert np.abs(ab - four).max() <= 2 * 2.0 ** -24 + 2.0 ** -48
    # the dropped lo*lo term itself: at most 2^-24 (|lo| <= 2^-12 each)
    assert np.abs(al * bl).max() <= 2.0 ** -24


def test_parts_of_a_scaled_weight():
    """The weights are scaled by a power of two 2^k so that the largest is
    just below 2^15 (f16 reaches 65504; small weights stay clear of its
    subnormals) before the
    split; the scaling and its inverse are exact, and every part pair is
    within 2^-22 of the weight relative to itself (2^-25 absolute where the
    remainder is an f16 subnormal)."""
    rng = np.random.default_rng(2)
    w = (rng.standard_normal(1 << 16) * 1e-6).astype(F32)
    top = int(np.floor(np.log2(np.abs(w).max()))) + 1      # max |w| < 2^top
    k = 15 - top
    ws = (w * F32(2.0 ** k)).astype(F32)
    assert np.abs(ws).max() < 2.0 ** 15
    assert np.array_equal(ws.astype(np.float64) * 2.0 ** -k, w.astype(np.float64))
    hi, _, lo = split(ws)
    v = ws.astype(np.float64)
    err = np.abs(v - hi.astype(np.float64) - lo.astype(np.float64))
    assert np.all(err <= np.maximum(2.0 ** -22 * np.abs(v), 2.0 ** -25))
    assert np.abs(hi.astype(np.float64)).max() < 65504.0     # no f16 overflow
