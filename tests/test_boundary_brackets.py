"""The boundary kernel's fp32 fast path, checked on the CPU.

The kernel rounds each output (y = x w r, h' = (sqrt(n-1) h + y) / sqrt(n),
z = h' w r2) to bf16 from plain fp32 arithmetic whenever two fp32 numbers
that bracket the exact value round to the same bf16 number, and recomputes
the element exactly otherwise. These tests replay that decision with IEEE
float32 arithmetic in numpy, on random and on deliberately near-midpoint
inputs, and check the claim it rests on: a closed bracket's bf16 number is
the exact value's correctly rounded bf16 number (the reference is the fp64
value rounded directly to bf16, `oracle.bf16.round_bf16`). They also check
that brackets close for nearly every ordinary element, so the exact path
stays rare.

The brackets replayed here:
- y and z: ends fl(ab * s_lo) and fl(ab * s_hi), where ab is the exact
  product of two bf16 values and s_lo, s_hi = fl(r_hi (1 -+ 2^-21)),
  r_hi = fl32(r);
- h': v = fl(fl(cm_hi h + y) c_hi) with ends fl(v -+ m c_bnd), where
  m = fl(|h| cm_hi + |y|) and c_bnd = c_hi 2^-20 (each fl(a b + c) one
  rounding, as a fused multiply-add).
"""
import numpy as np
import pytest

from oracle import bf16 as obf

F32 = np.float32


def bf16_bits_of_f32(x):
    """bf16 bits of float32 values rounded to nearest, ties to even."""
    b = np.asarray(x, dtype=F32).view(np.uint32).astype(np.uint64)
    return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)


def fma32(a, b, c):
    """fl32(a * b + c): a * b of two float32 values is exact in float64; the
    float64 sum can round before the float32 rounding, which moves the result
    by at most one float32 ulp in rare cases, far inside the brackets' margins."""
    a64 = np.asarray(a, dtype=F32).astype(np.float64)
    b64 = np.asarray(b, dtype=F32).astype(np.float64)
    return (a64 * b64 + np.asarray(c, dtype=F32).astype(np.float64)).astype(F32)


def random_bf16(rng, n, lo_exp, hi_exp):
    """bf16 values (as float64) with random sign, significand and exponent."""
    v = rng.standard_normal(n) * np.exp2(rng.uniform(lo_exp, hi_exp, n))
    return obf.round_bf16(v)


def decided(ref, err):
    """Cases whose fp64 reference rounds the same at both ends of its own error."""
    return np.equal(obf.round_bf16(ref - err), obf.round_bf16(ref + err))


def scaled_bracket(a, b, r):
    ab = (a * b).astype(F32)  # exact: 8 x 8 significant bits
    r_hi = r.astype(F32)
    s_lo = (r_hi * F32(1.0 - 2.0 ** -21)).astype(F32)
    s_hi = (r_hi * F32(1.0 + 2.0 ** -21)).astype(F32)
    lo = bf16_bits_of_f32(ab * s_lo)
    hi = bf16_bits_of_f32(ab * s_hi)
    return lo, hi


def residual_bracket(h, y, n):
    cm, c = np.sqrt(n - 1.0), 1.0 / np.sqrt(float(n))
    cm_hi, c_hi = F32(cm), F32(c)
    c_bnd = F32(np.ldexp(np.float64(c_hi), -20))
    v = (fma32(cm_hi, h, y) * c_hi).astype(F32)
    m = fma32(np.abs(h), cm_hi, np.abs(y))
    lo = bf16_bits_of_f32(fma32(m, -c_bnd, v))
    hi = bf16_bits_of_f32(fma32(m, c_bnd, v))
    ref = (cm * h + y) * c
    err = 8 * 2.0 ** -53 * (np.abs(cm * h) + np.abs(y)) * c  # the fp64 reference's own error, generously
    return lo, hi, ref, err


def test_scaled_bracket_random():
    rng = np.random.default_rng(1)
    n = 1_000_000
    a = random_bf16(rng, n, -30, 30)
    b = obf.round_bf16(1.0 + 0.02 * rng.standard_normal(n))  # norm weights
    r = np.exp2(rng.uniform(-12, 12, n))                      # 1/sqrt(mean + eps)
    lo, hi = scaled_bracket(a, b, r)
    closed = lo == hi
    exact = obf.encode(a * b * r)
    assert np.array_equal(hi[closed], exact[closed])
    assert closed.mean() > 0.999, closed.mean()


def test_scaled_bracket_near_midpoints():
    # a * b * r placed within 2^-18 (relative) of a bf16 rounding midpoint:
    # most brackets stay open; every one that closes must still be right
    rng = np.random.default_rng(2)
    n = 1_000_000
    a = random_bf16(rng, n, -8, 8)
    b = obf.round_bf16(1.0 + 0.02 * rng.standard_normal(n))
    t = random_bf16(rng, n, -8, 8)
    t = np.where(t == 0, 1.0, t)
    _, ex = np.frexp(t)
    mid = t + np.copysign(np.ldexp(1.0, ex - 9), t)  # half a bf16 step above |t|
    r = np.abs(mid / (a * b)) * (1.0 + rng.uniform(-2.0 ** -18, 2.0 ** -18, n))
    ok = np.isfinite(r) & (r > 0)
    a, b, r = a[ok], b[ok], r[ok]
    lo, hi = scaled_bracket(a, b, r)
    closed = lo == hi
    exact = obf.encode(a * b * r)
    assert np.array_equal(hi[closed], exact[closed])
    assert 0.5 < closed.mean() < 1.0  # both kinds occur


@pytest.mark.parametrize("n", [2, 5, 10, 17, 20, 40, 60, 100])
def test_residual_bracket_random(n):
    rng = np.random.default_rng(n)
    m = 500_000
    h = random_bf16(rng, m, -6, 6)
    y = random_bf16(rng, m, -6, 6)
    lo, hi, ref, err = residual_bracket(h, y, n)
    use = (lo == hi) & decided(ref, err)
    assert np.array_equal(hi[use], obf.encode(ref[use]))
    assert (lo == hi).mean() > 0.998, (lo == hi).mean()


@pytest.mark.parametrize("n", [2, 5, 10, 17, 100])
def test_residual_bracket_near_cancellation(n):
    # y the bf16 rounding of -sqrt(n-1) h times (1 + d) with |d| <= 2^-6: the
    # sum keeps a handful of significant bits, where plain fp32 would be wrong
    rng = np.random.default_rng(100 + n)
    m = 500_000
    h = random_bf16(rng, m, -6, 6)
    y = obf.round_bf16(-np.sqrt(n - 1.0) * h * (1.0 + rng.uniform(-2.0 ** -6, 2.0 ** -6, m)))
    lo, hi, ref, err = residual_bracket(h, y, n)
    use = (lo == hi) & decided(ref, err)
    assert np.array_equal(hi[use], obf.encode(ref[use]))
    assert (lo != hi).any()  # the exact path is needed here
    if n in (2, 5, 10, 17):
        # n - 1 a perfect square: some pairs cancel exactly, and a zero result
        # never closes (its ends have opposite signs) but goes to the exact path
        zero = ref == 0
        assert zero.any()
        assert not (lo == hi)[zero & (h != 0)].any()


# ---------------------------------------------------------------- per-pair checks
# The decode routing kernel with eight tokens keeps the earlier per-element
# checks: v = fl(ab r_hi) with the interval fl(v -+ fl(|v| 2^-21)) for y and
# z, and v = fl(fl(cm_hi h + y) c_hi) with fl(v -+ e), e = fl(fl(fl(|fl(cm_hi
# h)| + |y|) c_hi) 2^-20), for h'.

def scaled_interval(a, b, r):
    ab = (a * b).astype(F32)
    v = (ab * r.astype(F32)).astype(F32)
    e = (np.abs(v) * F32(2.0 ** -21)).astype(F32)
    return bf16_bits_of_f32(v - e), bf16_bits_of_f32(v + e), bf16_bits_of_f32(v)


def residual_interval(h, y, n):
    cm, c = np.sqrt(n - 1.0), 1.0 / np.sqrt(float(n))
    cm_hi, c_hi = F32(cm), F32(c)
    ch = (cm_hi * h.astype(F32)).astype(F32)
    v = (fma32(cm_hi, h, y) * c_hi).astype(F32)
    e = (((np.abs(ch) + np.abs(y).astype(F32)).astype(F32) * c_hi).astype(F32) * F32(2.0 ** -20)).astype(F32)
    ref = (cm * h + y) * c
    err = 8 * 2.0 ** -53 * (np.abs(cm * h) + np.abs(y)) * c
    return bf16_bits_of_f32(v - e), bf16_bits_of_f32(v + e), bf16_bits_of_f32(v), ref, err


def test_per_pair_scaled_check():
    rng = np.random.default_rng(7)
    n = 1_000_000
    a = random_bf16(rng, n, -8, 8)
    b = obf.round_bf16(1.0 + 0.02 * rng.standard_normal(n))
    t = random_bf16(rng, n, -8, 8)
    t = np.where(t == 0, 1.0, t)
    _, ex = np.frexp(t)
    mid = t + np.copysign(np.ldexp(1.0, ex - 9), t)
    near = np.abs(mid / (a * b)) * (1.0 + rng.uniform(-2.0 ** -18, 2.0 ** -18, n))
    r = np.where(rng.random(n) < 0.5, near, np.exp2(rng.uniform(-12, 12, n)))
    ok = np.isfinite(r) & (r > 0)
    a, b, r = a[ok], b[ok], r[ok]
    lo, hi, val = scaled_interval(a, b, r)
    closed = lo == hi
    assert np.array_equal(val[closed], obf.encode(a * b * r)[closed])


@pytest.mark.parametrize("n", [5, 20, 100])
def test_per_pair_residual_check(n):
    rng = np.random.default_rng(200 + n)
    m = 500_000
    h = random_bf16(rng, m, -6, 6)
    d = rng.uniform(-2.0 ** -6, 2.0 ** -6, m)
    y = np.where(rng.random(m) < 0.5, obf.round_bf16(-np.sqrt(n - 1.0) * h * (1.0 + d)), random_bf16(rng, m, -6, 6))
    lo, hi, val, ref, err = residual_interval(h, y, n)
    use = (lo == hi) & decided(ref, err)
    assert np.array_equal(val[use], obf.encode(ref[use]))
