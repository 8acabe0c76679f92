"""Pins for the oracle's wider rows: float8_e5m2, the static activation scale, the
general exact product and the weight-only (up-converted) linear.

Sources of truth, as in test_oracle_pins.py: the format definition (golden values),
torch's own float8_e5m2 conversion, exact rational arithmetic (fractions) on small
inputs, identities the method implies, and planted mistakes that must be caught.
"""

import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import fp8_oracle as O
from test_oracle_pins import (all_bf16_as_f32, f32_neighbourhoods, is_correctly_rounded_bf16,
                              is_correctly_rounded_f32)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def torch_e5m2(x_f32: np.ndarray) -> np.ndarray:
    """torch's fp32 -> float8_e5m2 (RNE, overflows to inf) after clamping to +-57344."""
    x = np.clip(np.asarray(x_f32, np.float32), -57344.0, 57344.0)
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.float8_e5m2).view(torch.uint8).numpy()


def frac_value(code: int, fmt: str) -> Fraction:
    return Fraction(O._decode_code(code) if fmt == "e4m3" else O._decode_code_e5m2(code))


def frac_nearest(v: Fraction, negative: bool, fmt: str) -> int:
    """Nearest finite code by exhaustive scan, ties to the even code, sign from `negative`."""
    top = 0x7E if fmt == "e4m3" else 0x7B
    base = 0x80 if negative else 0x00
    best, best_d = None, None
    for c in range(base, base + top + 1):
        d = abs(frac_value(c, fmt) - v)
        if best_d is None or d < best_d or (d == best_d and c % 2 == 0):
            best, best_d = c, d
    return best


def e5m2_boundary_points() -> np.ndarray:
    pos = O.E5M2_DECODE[:0x7C]
    mids = (pos[:-1] + pos[1:]) / 2
    extra = np.array([61440.0, 65536.0, 1e6, 3e38], np.float64)
    return f32_neighbourhoods(np.concatenate([pos, mids, extra]).astype(np.float32))


# ---------------------------------------------------------------------------
# reusable checks (mutants below reuse them)
# ---------------------------------------------------------------------------

def check_decode_e5m2(table) -> None:
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e5m2).double().numpy()
    ours = np.asarray(table, np.float64)
    assert np.array_equal(np.isnan(ref), np.isnan(ours))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], ours[ok])
    assert np.array_equal(np.signbit(ref[ok]), np.signbit(ours[ok]))


def check_encode_e5m2(encode, x) -> None:
    got, want = encode(x), torch_e5m2(x)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, f"{bad.size} mismatches, first x={x[bad[:5]]} got={got[bad[:5]]} want={want[bad[:5]]}"


def check_exact_dot_values(fn, A, pa, B, pb) -> None:
    S = fn(A, pa, B, pb)
    for m in range(A.shape[0]):
        for n in range(B.shape[0]):
            exact = sum(Fraction(float(A[m, k])) * Fraction(float(B[n, k])) for k in range(A.shape[1]))
            assert Fraction(float(S[m, n])) == Fraction(float(exact)), (m, n)  # exact, rounded once


def check_linear_bruteforce(y, a, qw, s_w, bias, fmt_a, fmt_w, s_a) -> None:
    """y against the definition: q = nearest(fp32(a / s_a)); exact sum; one bf16 rounding."""
    M, K = a.shape
    N = qw.shape[0]
    sw = np.broadcast_to(np.asarray(s_w, np.float32), (N,))
    for m in range(M):
        qrow = []
        for k in range(K):
            quot = np.float32(a[m, k]) / np.float32(s_a)
            qrow.append(frac_nearest(Fraction(float(quot)), bool(np.signbit(quot)), fmt_a))
        for n in range(N):
            S = sum(frac_value(qrow[k], fmt_a) * frac_value(int(qw[n, k]), fmt_w) for k in range(K))
            exact = Fraction(float(np.float32(s_a))) * Fraction(float(sw[n])) * S
            if bias is not None:
                exact += Fraction(float(bias[n]))
            assert is_correctly_rounded_bf16(float(y[m, n]), exact), (m, n)


def check_weight_only_bruteforce(y, a, qw, s_w, bias, fmt_w) -> None:
    N = qw.shape[0]
    sw = np.broadcast_to(np.asarray(s_w, np.float32), (N,))
    for m in range(a.shape[0]):
        for n in range(N):
            S = sum(Fraction(float(a[m, k])) * frac_value(int(qw[n, k]), fmt_w) for k in range(a.shape[1]))
            exact = Fraction(float(sw[n])) * S + (Fraction(float(bias[n])) if bias is not None else 0)
            assert is_correctly_rounded_bf16(float(y[m, n]), exact), (m, n)


def bf16(x):
    return torch.from_numpy(np.asarray(x, np.float32)).bfloat16().float().numpy()


def tiny(seed, M=3, N=5, K=9, mag=1.0):
    g = np.random.default_rng(seed)
    a = bf16(g.standard_normal((M, K)) * 3 * mag)
    w = bf16(g.standard_normal((N, K)) * g.uniform(0.01, 0.1, (N, 1)))
    bias = bf16(g.standard_normal(N))
    return a, w, bias


# ---------------------------------------------------------------------------
# e5m2 format
# ---------------------------------------------------------------------------

def test_e5m2_golden_values():
    with open(os.path.join(GOLDEN, "e5m2_values.txt")) as f:
        rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    assert len(rows) >= 15
    for code, val in rows:
        c, v = int(code, 16), float(val)
        if math.isnan(v):
            assert math.isnan(O.E5M2_DECODE[c])
        else:
            assert O.E5M2_DECODE[c] == v and math.copysign(1, O.E5M2_DECODE[c]) == math.copysign(1, v)


def test_e5m2_decode_vs_torch():
    check_decode_e5m2(O.E5M2_DECODE)


def test_e5m2_encode_all_bf16_vs_torch():
    check_encode_e5m2(O.e5m2_encode, all_bf16_as_f32())


def test_e5m2_encode_boundaries_vs_torch():
    check_encode_e5m2(O.e5m2_encode, e5m2_boundary_points())


def test_e5m2_encode_random_fp32_vs_torch():
    g = np.random.default_rng(21)
    bits = g.integers(0, 1 << 32, size=1_000_000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    dense = (g.standard_normal(500_000) * np.exp2(g.integers(-19, 17, 500_000))).astype(np.float32)
    check_encode_e5m2(O.e5m2_encode, np.concatenate([x, dense]))


def test_e5m2_roundtrip_all_finite_codes():
    codes = np.array([c for c in range(256) if (c & 0x7F) <= 0x7B], np.uint8)
    assert np.array_equal(O.e5m2_encode(O.e5m2_decode(codes).astype(np.float32)), codes)


def test_e5m2_encode_bruteforce_fractions():
    g = np.random.default_rng(22)
    x = np.concatenate([(g.standard_normal(200) * np.exp2(g.integers(-20, 17, 200))).astype(np.float32),
                        e5m2_boundary_points()[::1499]])
    for xi, ci in zip(x, O.e5m2_encode(x)):
        assert ci == frac_nearest(Fraction(float(xi)), bool(np.signbit(xi)), "e5m2"), xi


def test_e5m2_saturates_never_inf_and_keeps_zero_sign():
    x = np.array([57344, 57345, 61439, 61440, 65536, 1e30, -1e30, -0.0, 0.0, -1e-30, 2.0 ** -17], np.float32)
    assert list(O.e5m2_encode(x)) == [0x7B, 0x7B, 0x7B, 0x7B, 0x7B, 0x7B, 0xFB, 0x80, 0x00, 0x80, 0x00]


def test_encode_dispatch():
    x = np.linspace(-500, 500, 1001).astype(np.float32)
    assert np.array_equal(O.encode(x, "e4m3"), O.e4m3_encode(x))
    assert np.array_equal(O.encode(x, "e5m2"), O.e5m2_encode(x))
    assert np.array_equal(O.decode(np.arange(256), "e5m2"), O.E5M2_DECODE, equal_nan=True)


# ---------------------------------------------------------------------------
# e5m2 scale and quantization
# ---------------------------------------------------------------------------

def test_e5m2_scale_is_correctly_rounded_quotient_for_every_bf16_amax():
    b = all_bf16_as_f32()
    amaxes = np.unique(np.abs(b[b >= 0]))
    s = O.scale_from_amax(amaxes, "e5m2")
    for a, si in zip(amaxes[::7], s[::7]):
        if a == 0:
            assert si == 1.0
        else:
            assert is_correctly_rounded_f32(si, Fraction(float(a)) / 57344), (a, si)


def test_e5m2_amax_element_maps_to_max_code():
    g = np.random.default_rng(23)
    for mag in (1e-30, 1e-3, 1.0, 3e5, 1e30):
        x = bf16(g.standard_normal((13, 29)) * mag)
        q, s = O.quantize_per_tensor(x, "e5m2")
        i = np.unravel_index(np.argmax(np.abs(x)), x.shape)
        assert q[i] == (0xFB if x[i] < 0 else 0x7B)
        assert np.all((q & 0x7F) <= 0x7B)
        qr, _ = O.quantize_per_row(x, "e5m2")
        for r in range(x.shape[0]):
            j = np.argmax(np.abs(x[r]))
            assert qr[r, j] == (0xFB if x[r, j] < 0 else 0x7B)


# ---------------------------------------------------------------------------
# general exact product
# ---------------------------------------------------------------------------

def _codes(g, shape, fmt):
    top = 0x7E if fmt == "e4m3" else 0x7B
    c = g.integers(0, top + 1, shape).astype(np.uint8)
    return c | (g.integers(0, 2, shape).astype(np.uint8) << 7)


@pytest.mark.parametrize("fa,fw", [("e5m2", "e5m2"), ("e4m3", "e5m2"), ("e5m2", "e4m3"), ("e4m3", "e4m3")])
def test_exact_dot_all_format_pairs_vs_fractions(fa, fw):
    g = np.random.default_rng(24)
    qa, qw = _codes(g, (3, 41), fa), _codes(g, (4, 41), fw)
    S = O.exact_dot(qa, qw, fa, fw)
    for m in range(3):
        for n in range(4):
            exact = sum(frac_value(int(qa[m, k]), fa) * frac_value(int(qw[n, k]), fw) for k in range(41))
            assert Fraction(float(S[m, n])) == Fraction(float(exact))


def test_exact_dot_values_extreme_ranges_vs_fractions():
    """Magnitudes spanning 2**-130 .. 2**120: a single float64 matmul loses the small terms."""
    g = np.random.default_rng(25)
    A = bf16(g.standard_normal((2, 24)) * np.exp2(g.integers(-120, 110, (2, 24))))
    qw = _codes(g, (3, 24), "e5m2")
    B = O.e5m2_decode(qw)
    check_exact_dot_values(O.exact_dot_values, A.astype(np.float64), 8, B, 3)
    plain = A.astype(np.float64) @ B.T
    S = O.exact_dot_values(A.astype(np.float64), 8, B, 3)
    # the inputs are chosen so that plain float64 summation is not exact somewhere
    exact = [[sum(Fraction(float(A[m, k])) * Fraction(float(B[n, k])) for k in range(24)) for n in range(3)]
             for m in range(2)]
    assert any(Fraction(float(plain[m, n])) != exact[m][n] for m in range(2) for n in range(3))
    assert all(Fraction(float(S[m, n])) == Fraction(float(exact[m][n])) for m in range(2) for n in range(3))


def test_exact_dot_general_equals_single_matmul_for_e4m3():
    g = np.random.default_rng(26)
    qa, qw = _codes(g, (5, 700), "e4m3"), _codes(g, (6, 700), "e4m3")
    S1 = O.exact_dot(qa, qw)
    S2 = O.exact_dot_values(O.e4m3_decode(qa), 4, O.e4m3_decode(qw), 4)
    assert np.array_equal(S1, S2)


def test_exact_dot_values_cancellation_keeps_tiny_remainder():
    # 57344 * 57344 - 57344 * 57344 + 2**-16 * 2**-16 = 2**-32 exactly
    A = np.array([[57344.0, 57344.0, 2.0 ** -16]])
    B = np.array([[57344.0, -57344.0, 2.0 ** -16]])
    assert O.exact_dot_values(A, 3, B, 3)[0, 0] == 2.0 ** -32


# ---------------------------------------------------------------------------
# static activation scale
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_static_scale_equal_to_dynamic_reproduces_dynamic(fmt):
    a, w, bias = tiny(27, M=4, N=6, K=33)
    qw, s_w = O.quantize_per_row(w, fmt)
    y_dyn, qa_dyn, s_dyn = O.linear(a, qw, s_w, bias, fmt_a=fmt, fmt_w=fmt)
    y_st, qa_st, s_st = O.linear(a, qw, s_w, bias, fmt_a=fmt, fmt_w=fmt, s_a=s_dyn)
    assert s_st == s_dyn and np.array_equal(qa_st, qa_dyn) and np.array_equal(y_st, y_dyn)


@pytest.mark.parametrize("fmt_a,fmt_w", [("e4m3", "e4m3"), ("e5m2", "e5m2"), ("e4m3", "e5m2")])
def test_static_linear_bruteforce_with_saturation(fmt_a, fmt_w):
    a, w, bias = tiny(28, M=3, N=4, K=11)
    qw, s_w = O.quantize_per_tensor(w, fmt_w)
    s_a = np.float32(O.amax(a) / O.fp8_max(fmt_a) / 4)  # a calibrated scale 4x too small: saturation
    y, qa, s = O.linear(a, qw, s_w, bias, fmt_a=fmt_a, fmt_w=fmt_w, s_a=s_a)
    top = 0x7E if fmt_a == "e4m3" else 0x7B
    assert s == s_a and np.any((qa & 0x7F) == top)
    big = np.abs(a) > np.float32(s_a) * np.float32(O.fp8_max(fmt_a)) * 1.01
    assert np.all((qa[big] & 0x7F) == top)
    check_linear_bruteforce(y, a, qw, s_w, bias, fmt_a, fmt_w, s_a)


# ---------------------------------------------------------------------------
# weight-only (up-converted) linear
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("channelwise", [False, True])
def test_weight_only_bruteforce(fmt, channelwise):
    a, w, bias = tiny(29, M=3, N=4, K=13)
    qw, s_w = O.quantize_per_row(w, fmt) if channelwise else O.quantize_per_tensor(w, fmt)
    check_weight_only_bruteforce(O.linear_weight_only(a, qw, s_w, bias, fmt), a, qw, s_w, bias, fmt)
    check_weight_only_bruteforce(O.linear_weight_only(a, qw, s_w, None, fmt), a, qw, s_w, None, fmt)


def test_weight_only_identity_weights_return_scaled_activations():
    """W = I (code 1.0): Y = bf16(s_w * a), a textbook case of the up-conversion."""
    g = np.random.default_rng(30)
    a = bf16(g.standard_normal((4, 16)) * np.exp2(g.integers(-30, 30, (4, 16))))
    for fmt, one in (("e4m3", 0x38), ("e5m2", 0x3C)):
        qw = np.where(np.eye(16, dtype=bool), np.uint8(one), np.uint8(0))
        y = O.linear_weight_only(a, qw, np.float32(0.75), None, fmt)
        assert np.array_equal(y, O.bf16_round(a.astype(np.float64) * 0.75))


def test_weight_only_equals_bf16_linear_of_upconverted_weights():
    """Up-converting (decode * s_w in float64, exact) and running the plain product agrees."""
    a, w, bias = tiny(31, M=5, N=7, K=64)
    qw, s_w = O.quantize_per_row(w)
    y = O.linear_weight_only(a, qw, s_w, bias)
    W = O.e4m3_decode(qw) * s_w.astype(np.float64)[:, None]
    y2 = O.bf16_round(a.astype(np.float64) @ W.T + bias)
    assert np.all(np.abs(y - y2) <= O.ulp_bf16(y2))


def test_weight_only_tolerance_bounds_fp32_accumulation():
    g = np.random.default_rng(32)
    a = bf16(g.standard_normal((3, 1024)))
    qw, s_w = O.quantize_per_tensor(bf16(g.standard_normal((5, 1024)) * 0.02))
    y = O.linear_weight_only(a, qw, s_w)
    W = O.e4m3_decode(qw).astype(np.float32)
    acc = np.zeros((3, 5), np.float32)
    for k in range(1024):
        acc = (acc + a[:, k:k + 1] * W[:, k][None, :]).astype(np.float32)
    y32 = bf16(acc * np.float32(s_w))
    tol = O.tolerance_weight_only(a, qw, s_w, y)
    assert np.all(np.abs(y32.astype(np.float64) - y) <= tol)


# ---------------------------------------------------------------------------
# planted mistakes in the wider rows
# ---------------------------------------------------------------------------

def _mutant_e5m2_bias16():
    t = O.E5M2_DECODE.copy()
    return np.where(np.isfinite(t), t / 2, t)


def _mutant_e5m2_saturate_low(x):
    code = O.e5m2_encode(x)
    return np.where((code & 0x7F) == 0x7B, (code & 0x80) | np.uint8(0x7A), code)


def _mutant_e5m2_ties_up(x):
    x = np.asarray(x, np.float32)
    mag = np.abs(x).astype(np.float64)
    pos = O._POSITIVE_E5M2
    hi = np.minimum(np.searchsorted(pos, mag, side="left"), 0x7B)
    lo = np.maximum(hi - 1, 0)
    code = np.where(mag < (pos[lo] + pos[hi]) * 0.5, lo, hi).astype(np.uint8)
    return code | (np.signbit(x).astype(np.uint8) << 7)


def _mutant_exact_dot_one_matmul(A, pa, B, pb):
    return np.asarray(A, np.float64) @ np.asarray(B, np.float64).T


def _mutant_exact_dot_no_cross_terms(A, pa, B, pb):
    # splits each operand at magnitude 1 but forgets the large x small window pairs
    A, B = np.asarray(A, np.float64), np.asarray(B, np.float64)
    Al, As = np.where(np.abs(A) >= 1, A, 0), np.where(np.abs(A) < 1, A, 0)
    Bl, Bs = np.where(np.abs(B) >= 1, B, 0), np.where(np.abs(B) < 1, B, 0)
    return O.exact_dot_values(Al, pa, Bl, pb) + O.exact_dot_values(As, pa, Bs, pb)


@pytest.mark.parametrize("name", ["e5m2_bias", "e5m2_saturate", "e5m2_ties", "dot_one_matmul",
                                  "dot_no_cross_terms", "static_ignored", "weight_only_no_scale"])
def test_planted_mistake_in_wider_rows_is_caught(name):
    g = np.random.default_rng(33)
    A = bf16(g.standard_normal((2, 24)) * np.exp2(g.integers(-120, 110, (2, 24)))).astype(np.float64)
    B = O.e5m2_decode(_codes(g, (3, 24), "e5m2"))
    with pytest.raises(AssertionError):
        if name == "e5m2_bias":
            check_decode_e5m2(_mutant_e5m2_bias16())
        elif name == "e5m2_saturate":
            check_encode_e5m2(_mutant_e5m2_saturate_low, all_bf16_as_f32())
        elif name == "e5m2_ties":
            check_encode_e5m2(_mutant_e5m2_ties_up, all_bf16_as_f32())
        elif name == "dot_one_matmul":
            check_exact_dot_values(_mutant_exact_dot_one_matmul, A, 8, B, 3)
        elif name == "dot_no_cross_terms":
            check_exact_dot_values(_mutant_exact_dot_no_cross_terms, A, 8, B, 3)
        elif name == "static_ignored":
            a, w, bias = tiny(34, M=2, N=3, K=7)
            qw, s_w = O.quantize_per_tensor(w)
            s_a = np.float32(O.amax(a) / 448 / 3)
            y, _, _ = O.linear(a, qw, s_w, bias)  # dynamic instead of the given static scale
            check_linear_bruteforce(y, a, qw, s_w, bias, "e4m3", "e4m3", s_a)
        elif name == "weight_only_no_scale":
            a, w, bias = tiny(35, M=2, N=3, K=7)
            qw, s_w = O.quantize_per_tensor(w)
            y = O.linear_weight_only(a, qw, np.float32(1.0), bias)
            check_weight_only_bruteforce(y, a, qw, s_w, bias, "e4m3")
