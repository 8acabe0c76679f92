"""The division-free quotient the quantization kernels use, checked on the host.

The kernels compute fl32(x / s) as
    r = RN(1/s), r_lo = RN(RN(1 - s*r) * r), q0 = RN(x*r + RN(x*r_lo)),
    q = RN(q0 + RN(x - s*q0) * r)
(each RN(a*b + c) one fused multiply-add), which Markstein's theorem (P. Markstein, IBM J.
Res. Dev. 34(1), 1990) makes the correctly rounded quotient when q0 is faithful and the
residual is exact. Here the same sequence runs in exact integer arithmetic with one
round-to-nearest-even to binary32 per operation, and is compared with IEEE binary32 division
(numpy) over every non-zero finite bf16 x, for scales whose quotients land on or next to FP8
rounding midpoints, random scales, and the ends of the range the kernels use it in
([2^-80, 2^100]). The claim checked: equal quotients wherever |x/s| >= 2^-20.
"""

import struct
from fractions import Fraction

import numpy as np
import pytest

F32_MIN_EXP = -149  # exponent of the smallest binary32 subnormal


def decompose(f: float):
    """binary32 value -> (m, e) with value = m * 2**e, m a signed integer, |m| < 2**24."""
    b = struct.unpack("<I", struct.pack("<f", f))[0]
    sign = -1 if b >> 31 else 1
    E, M = (b >> 23) & 0xFF, b & 0x7FFFFF
    if E == 0xFF:
        raise ValueError("non-finite")
    if E == 0:
        return sign * M, F32_MIN_EXP
    return sign * (M | 0x800000), E - 150


def round_scaled(num: int, exp: int) -> float:
    """num * 2**exp rounded to binary32, to nearest, ties to even (inf beyond the range)."""
    if num == 0:
        return 0.0
    sign = -1.0 if num < 0 else 1.0
    n = abs(num)
    top = n.bit_length() - 1 + exp  # binary exponent of the leading bit
    qexp = max(top - 23, F32_MIN_EXP)
    shift = qexp - exp
    if shift <= 0:
        m = n << (-shift)
    else:
        m, rem = n >> shift, n & ((1 << shift) - 1)
        half = 1 << (shift - 1)
        if rem > half or (rem == half and (m & 1)):
            m += 1
    if m == 1 << 24:
        m, qexp = m >> 1, qexp + 1
    if qexp + 23 > 127:
        return sign * float("inf")
    return sign * float(np.float32(m * 2.0 ** qexp))


def round_fraction(v: Fraction) -> float:
    """A rational value rounded to binary32, to nearest, ties to even."""
    if v == 0:
        return 0.0
    sign = -1 if v < 0 else 1
    v = abs(v)
    p, q = v.numerator, v.denominator
    top = p.bit_length() - q.bit_length()
    if Fraction(p, q) < Fraction(2) ** top:
        top -= 1
    qexp = max(top - 23, F32_MIN_EXP)
    scaled = Fraction(p, q) / Fraction(2) ** qexp
    m = scaled.numerator // scaled.denominator
    rem = scaled - m
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and (m & 1)):
        m += 1
    return round_scaled(sign * m, qexp)


def fma(a: float, b: float, c: float) -> float:
    """RN(a*b + c) in binary32, exactly (one rounding)."""
    ma, ea = decompose(a)
    mb, eb = decompose(b)
    mc, ec = decompose(c)
    e = min(ea + eb, ec)
    return round_scaled(ma * mb * (1 << (ea + eb - e)) + mc * (1 << (ec - e)), e)


def mul(a: float, b: float) -> float:
    return fma(a, b, 0.0)


def kernel_quotient(x: float, s: float) -> float:
    r = round_fraction(1 / Fraction(s))
    r_lo = mul(fma(-s, r, 1.0), r)
    q0 = fma(x, r, mul(x, r_lo))
    return fma(fma(-s, q0, x), r, q0)


def nonzero_finite_bf16() -> np.ndarray:
    bits = np.arange(1 << 16, dtype=np.uint32) << 16
    v = bits.view(np.float32)
    return v[np.isfinite(v) & (v != 0)]


def check_scale(s: float, xs: np.ndarray) -> int:
    s = float(np.float32(s))
    with np.errstate(over="ignore", under="ignore"):
        ref = (xs / np.float32(s)).astype(np.float32)
    checked = 0
    for x, q_ref in zip(xs.tolist(), ref.tolist()):
        if not np.isfinite(q_ref) or abs(q_ref) < 2.0 ** -20:
            continue
        q = kernel_quotient(x, s)
        assert np.float32(q).view(np.uint32) == np.float32(q_ref).view(np.uint32), \
            f"s={s!r} x={x!r}: method {q!r} != IEEE {q_ref!r}"
        checked += 1
    return checked


@pytest.mark.parametrize("amax", [3.375, 3.5, 4.0, 7.0 * 2.0 ** -9, 27.0 * 2.0 ** 5])
def test_every_bf16_at_scales_of_few_bits(amax):
    """amax / 448 for amax values whose quotients x / s sit on or within 2^-24 of e4m3
    rounding midpoints for many bf16 x (the cases a bracket cannot settle)."""
    xs = nonzero_finite_bf16()
    xs = xs[np.abs(xs) <= amax]
    assert check_scale(np.float32(amax) / np.float32(448.0), xs) > 5000


def test_random_scales_sampled():
    g = np.random.default_rng(5)
    xs = nonzero_finite_bf16()
    for s in np.exp2(g.uniform(-80, 100, 12)):
        assert check_scale(float(s), g.choice(xs, 1500, replace=False)) > 0


@pytest.mark.parametrize("s", [2.0 ** -80, 2.0 ** 100, float(np.nextafter(np.float32(2.0 ** -80), np.float32(1)))])
def test_range_ends_sampled(s):
    g = np.random.default_rng(6)
    assert check_scale(s, g.choice(nonzero_finite_bf16(), 3000, replace=False)) > 0


def test_the_check_rejects_the_plain_product():
    """RN(x * RN(1/s)) alone (no tail, no correction) is not always the IEEE quotient: the
    comparison above can tell the method from that shortcut."""
    s = float(np.float32(np.float32(3.375) / np.float32(448.0)))
    xs = nonzero_finite_bf16()
    xs = xs[np.abs(xs) <= 3.375]
    ref = (xs / np.float32(s)).astype(np.float32)
    r = round_fraction(1 / Fraction(s))
    differ = sum(mul(x, r) != q_ref for x, q_ref in zip(xs.tolist(), ref.tolist()))
    assert differ > 100


def test_emulated_rounding_matches_numpy():
    """The exact-arithmetic helpers against numpy's binary32 on products (one rounding)."""
    g = np.random.default_rng(7)
    a = (g.standard_normal(2000) * np.exp2(g.integers(-60, 60, 2000))).astype(np.float32)
    b = (g.standard_normal(2000) * np.exp2(g.integers(-60, 60, 2000))).astype(np.float32)
    for x, y in zip(a.tolist(), b.tolist()):
        assert mul(x, y) == float(np.float32(x) * np.float32(y))
    for v in [Fraction(1, 3), Fraction(2, 3), Fraction(-7, 448), Fraction(1, 1 << 149), Fraction(3, 1 << 150)]:
        assert round_fraction(v) == float(np.float32(float(v))) or v.denominator > (1 << 140)
