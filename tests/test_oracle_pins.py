"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each pin compares the oracle with an independent source of truth: the
e4m3fn/bf16 format definitions (golden values), library conversions (torch,
ml_dtypes) that round by their own bit-level code, exact rational arithmetic
(fractions) on small inputs, invariants the method implies, and the page-1
memory numbers. The last test plants mistakes in copies of oracle functions and
checks that a pin catches each one.
"""

import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import fp8_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------------------
# independent references
# ---------------------------------------------------------------------------

def torch_e4m3(x_f32: np.ndarray) -> np.ndarray:
    """torch's fp32 -> float8_e4m3fn (RNE, non-saturating) after clamping to +-448."""
    x = np.clip(np.asarray(x_f32, np.float32), -448.0, 448.0)
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def all_bf16_as_f32() -> np.ndarray:
    bits = torch.arange(0, 1 << 16, dtype=torch.int32).to(torch.int16)
    x = bits.view(torch.bfloat16).float().numpy()
    return x[np.isfinite(x)]


def f32_neighbourhoods(centres: np.ndarray, radius: int = 16) -> np.ndarray:
    """All fp32 values within `radius` ulps of each centre (both signs)."""
    c = np.asarray(centres, np.float32)
    bits = c.view(np.uint32).astype(np.int64)
    offs = np.arange(-radius, radius + 1, dtype=np.int64)
    nb = (bits[:, None] + offs[None, :]).reshape(-1)
    nb = nb[(nb >= 0) & (nb < 0x7F800000)].astype(np.uint32)
    v = nb.view(np.float32)
    return np.concatenate([v, -v])


def e4m3_boundary_points() -> np.ndarray:
    """fp32 values around every e4m3fn value and every midpoint between neighbours (0..448),
    plus the saturation region."""
    pos = np.array([O._decode_code(c) for c in range(0x7F)], np.float64)
    mids = (pos[:-1] + pos[1:]) / 2
    extra = np.array([464.0, 480.0, 512.0, 1e4, 3e38], np.float64)
    return f32_neighbourhoods(np.concatenate([pos, mids, extra]).astype(np.float32))


def frac_nearest_e4m3(v: Fraction, negative: bool) -> int:
    """Nearest finite e4m3fn code to v by exhaustive scan, ties to even code,
    sign bit from `negative` (so zero results keep the input's sign)."""
    best, best_d = None, None
    base = 0x80 if negative else 0x00
    for c in range(base, base + 0x7F):
        d = abs(Fraction(O._decode_code(c)) - v)
        if best_d is None or d < best_d or (d == best_d and c % 2 == 0):
            best, best_d = c, d
    return best


def is_correctly_rounded_f32(f: np.float32, exact: Fraction) -> bool:
    """f is the round-to-nearest-even fp32 value of `exact`."""
    f = np.float32(f)
    lo = np.nextafter(f, np.float32(-np.inf))
    hi = np.nextafter(f, np.float32(np.inf))
    d = abs(Fraction(float(f)) - exact)
    for g in (lo, hi):
        dg = abs(Fraction(float(g)) - exact)
        if dg < d:
            return False
        if dg == d and (int(np.float32(f).view(np.uint32)) & 1):
            return False
    return True


def bf16_neighbours(y: float):
    b = torch.tensor([y], dtype=torch.float32).to(torch.bfloat16).view(torch.int16).item() & 0xFFFF
    out = []
    for nb in (b - 1, b + 1):
        t = torch.tensor([nb & 0xFFFF], dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
        v = t.float().item()
        if math.isfinite(v):
            out.append(v)
    return out, b


def is_correctly_rounded_bf16(y: float, exact: Fraction) -> bool:
    nbs, bits = bf16_neighbours(y)
    d = abs(Fraction(y) - exact)
    for g in nbs:
        dg = abs(Fraction(g) - exact)
        if dg < d or (dg == d and (bits & 1)):
            return False
    return True


# ---------------------------------------------------------------------------
# reusable pin checks (the planted-mistake test calls them with mutants)
# ---------------------------------------------------------------------------

def check_decode(decode_table) -> None:
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    ours = np.asarray(decode_table, np.float64)
    assert np.array_equal(np.isnan(ref), np.isnan(ours))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], ours[ok])
    assert np.array_equal(np.signbit(ref[ok]), np.signbit(ours[ok]))


def check_encode_vs_torch(encode, x: np.ndarray) -> None:
    got = encode(x)
    want = torch_e4m3(x)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, f"{bad.size} mismatches, first x={x[bad[:5]]} got={got[bad[:5]]} want={want[bad[:5]]}"


def check_scale_exact(scale_fn, amaxes: np.ndarray) -> None:
    s = scale_fn(amaxes)
    for a, si in zip(amaxes, s):
        if a == 0:
            assert si == 1.0
            continue
        assert is_correctly_rounded_f32(si, Fraction(float(a)) / 448), (a, si)


def check_quantize_bruteforce(quantize, x: np.ndarray) -> None:
    q, s = quantize(x)
    for xi, qi in zip(x.reshape(-1), q.reshape(-1)):
        quot = np.float32(xi) / np.float32(s)
        assert is_correctly_rounded_f32(quot, Fraction(float(xi)) / Fraction(float(s)))
        want = frac_nearest_e4m3(Fraction(float(quot)), bool(np.signbit(quot)))
        assert qi == want, (xi, s, quot, qi, want)


def check_scaled_mm_bruteforce(scaled_mm, qa, s_a, qw, s_w, bias) -> None:
    y = scaled_mm(qa, s_a, qw, s_w, bias)
    M, K = qa.shape
    N = qw.shape[0]
    sw = np.broadcast_to(np.asarray(s_w, np.float32), (N,))
    for m in range(M):
        for n in range(N):
            S = sum(Fraction(O._decode_code(int(qa[m, k]))) * Fraction(O._decode_code(int(qw[n, k])))
                    for k in range(K))
            exact = Fraction(float(np.float32(s_a))) * Fraction(float(sw[n])) * S
            if bias is not None:
                exact += Fraction(float(bias[n]))
            assert is_correctly_rounded_bf16(float(y[m, n]), exact), (m, n, float(y[m, n]), float(exact))


def tiny_linear_inputs(seed=7, M=3, N=5, K=7, channelwise=True):
    g = np.random.default_rng(seed)
    a = torch.from_numpy(g.standard_normal((M, K)).astype(np.float32) * 3).bfloat16().float().numpy()
    w = torch.from_numpy(g.standard_normal((N, K)).astype(np.float32)
                         * g.uniform(0.01, 0.1, (N, 1)).astype(np.float32)).bfloat16().float().numpy()
    bias = torch.from_numpy(g.standard_normal(N).astype(np.float32)).bfloat16().float().numpy()
    qa, s_a = O.quantize_per_tensor(a)
    qw, s_w = O.quantize_per_row(w) if channelwise else O.quantize_per_tensor(w)
    return qa, s_a, qw, s_w, bias


# ---------------------------------------------------------------------------
# format
# ---------------------------------------------------------------------------

def test_decode_golden_values():
    with open(os.path.join(GOLDEN, "e4m3fn_values.txt")) as f:
        rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    assert len(rows) >= 15
    for code, val in rows:
        c = int(code, 16)
        v = float(val)
        if math.isnan(v):
            assert math.isnan(O.E4M3_DECODE[c])
        else:
            assert O.E4M3_DECODE[c] == v and math.copysign(1, O.E4M3_DECODE[c]) == math.copysign(1, v)


def test_decode_table_vs_torch():
    check_decode(O.E4M3_DECODE)


def test_decode_table_vs_ml_dtypes():
    ml = pytest.importorskip("ml_dtypes")
    ref = np.arange(256, dtype=np.uint8).view(ml.float8_e4m3fn).astype(np.float64)
    ok = ~np.isnan(ref)
    assert np.array_equal(np.isnan(ref), np.isnan(O.E4M3_DECODE))
    assert np.array_equal(ref[ok], O.E4M3_DECODE[ok])


def test_encode_all_bf16_vs_torch():
    check_encode_vs_torch(O.e4m3_encode, all_bf16_as_f32())


def test_encode_boundaries_vs_torch():
    check_encode_vs_torch(O.e4m3_encode, e4m3_boundary_points())


def test_encode_random_fp32_vs_torch_and_ml_dtypes():
    g = np.random.default_rng(1)
    bits = g.integers(0, 1 << 32, size=2_000_000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    # also dense coverage of the e4m3 range (exponents -12..9)
    dense = (g.standard_normal(1_000_000) * np.exp2(g.integers(-12, 10, 1_000_000))).astype(np.float32)
    x = np.concatenate([x, dense])
    check_encode_vs_torch(O.e4m3_encode, x)
    ml = pytest.importorskip("ml_dtypes")
    ref = np.clip(x, -448, 448).astype(ml.float8_e4m3fn).view(np.uint8)
    assert np.array_equal(O.e4m3_encode(x), ref)


def test_encode_roundtrip_all_finite_codes():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    vals = O.e4m3_decode(codes).astype(np.float32)
    assert np.array_equal(O.e4m3_encode(vals), codes)


def test_encode_bruteforce_fractions():
    g = np.random.default_rng(2)
    x = np.concatenate([
        (g.standard_normal(300) * np.exp2(g.integers(-14, 10, 300))).astype(np.float32),
        e4m3_boundary_points()[::997],
    ])
    got = O.e4m3_encode(x)
    for xi, gi in zip(x, got):
        assert gi == frac_nearest_e4m3(Fraction(float(xi)), bool(np.signbit(xi))), xi


def test_encode_saturates_and_keeps_zero_sign():
    x = np.array([448, 449, 464, 1e30, -1e30, -0.0, 0.0, -1e-30, 1e-30], np.float32)
    assert list(O.e4m3_encode(x)) == [0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0x80, 0x00, 0x80, 0x00]


# ---------------------------------------------------------------------------
# bf16 rounding of the output
# ---------------------------------------------------------------------------

def test_bf16_round_vs_torch_on_fp32_values():
    g = np.random.default_rng(3)
    bits = g.integers(0, 1 << 32, size=1_000_000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[np.isfinite(x) & (np.abs(x) < 3.0e38)]
    # bf16 midpoints exactly: bf16 value + half its spacing (exact in fp32)
    b = all_bf16_as_f32()
    b = b[np.abs(b) < 3.0e38]
    mids = (b.astype(np.float64) + O.ulp_bf16(b) / 2).astype(np.float32)
    x = np.concatenate([x, mids, b])
    want = torch.from_numpy(x).bfloat16().float().numpy()
    assert np.array_equal(O.bf16_round(x.astype(np.float64)), want)


def test_bf16_round_bruteforce_fractions():
    g = np.random.default_rng(4)
    v = g.standard_normal(400) * np.exp2(g.integers(-140, 40, 400).astype(np.float64))
    r = O.bf16_round(v)
    for vi, ri in zip(v, r):
        assert is_correctly_rounded_bf16(float(ri), Fraction(float(vi))), vi


# ---------------------------------------------------------------------------
# scale
# ---------------------------------------------------------------------------

def test_scale_is_correctly_rounded_quotient_for_every_bf16_amax():
    b = all_bf16_as_f32()
    amaxes = np.unique(np.abs(b[b >= 0]))
    check_scale_exact(O.scale_from_amax, amaxes)


def test_scale_of_zero_tensor_is_one_and_codes_zero():
    q, s = O.quantize_per_tensor(np.array([[0.0, -0.0, 0.0]], np.float32))
    assert s == 1.0 and list(q[0]) == [0x00, 0x80, 0x00]
    q, s = O.quantize_per_row(np.zeros((3, 4), np.float32))
    assert np.all(s == 1.0) and np.all(q == 0)


def test_amax_element_maps_to_448():
    g = np.random.default_rng(5)
    for mag in (1e-30, 1e-3, 1.0, 3e5, 1e30):
        x = torch.from_numpy((g.standard_normal((17, 33)) * mag).astype(np.float32)).bfloat16().float().numpy()
        q, s = O.quantize_per_tensor(x)
        i = np.unravel_index(np.argmax(np.abs(x)), x.shape)
        assert q[i] == (0xFE if x[i] < 0 else 0x7E)
        assert np.all((q & 0x7F) <= 0x7E)
        qr, sr = O.quantize_per_row(x)
        for r in range(x.shape[0]):
            j = np.argmax(np.abs(x[r]))
            assert qr[r, j] == (0xFE if x[r, j] < 0 else 0x7E)


def test_quantize_bruteforce_fractions():
    g = np.random.default_rng(6)
    for mag in (1.0, 1e-38, 2e4):
        x = torch.from_numpy((g.standard_normal((4, 9)) * mag).astype(np.float32)).bfloat16().float().numpy()
        x[1, 3] *= 50  # an outlier channel element
        check_quantize_bruteforce(O.quantize_per_tensor, x)


# ---------------------------------------------------------------------------
# product and epilogue
# ---------------------------------------------------------------------------

def test_exact_dot_vs_fractions():
    g = np.random.default_rng(8)
    qa = g.integers(0, 256, (4, 37)).astype(np.uint8)
    qw = g.integers(0, 256, (6, 37)).astype(np.uint8)
    qa[(qa & 0x7F) == 0x7F] = 0x12
    qw[(qw & 0x7F) == 0x7F] = 0x34
    S = O.exact_dot(qa, qw)
    for m in range(4):
        for n in range(6):
            ref = sum(Fraction(O._decode_code(int(qa[m, k]))) * Fraction(O._decode_code(int(qw[n, k])))
                      for k in range(37))
            assert Fraction(S[m, n]) == ref


def test_exact_dot_extreme_magnitudes_exact():
    # K terms of 448*448 mixed with 2**-18 terms: float32 accumulation would lose them
    K = 4096
    qa = np.full((1, K), 0x7E, np.uint8)
    qw = np.full((1, K), 0x7E, np.uint8)
    qa[0, 1::2] = 0x01
    qw[0, 1::2] = 0x81
    S = O.exact_dot(qa, qw)[0, 0]
    assert Fraction(S) == Fraction(448 * 448) * (K // 2) - Fraction(1, 2 ** 18) * (K // 2)


@pytest.mark.parametrize("channelwise", [False, True])
def test_scaled_mm_bruteforce_fractions(channelwise):
    qa, s_a, qw, s_w, bias = tiny_linear_inputs(channelwise=channelwise)
    check_scaled_mm_bruteforce(O.scaled_mm, qa, s_a, qw, s_w, bias)
    check_scaled_mm_bruteforce(O.scaled_mm, qa, s_a, qw, s_w, None)


def test_channelwise_rescale_after_gemm_identity():
    """(s_a A)(s_w,n W_n)^T == s_a s_w,n (A W_n^T): scale the dequantized operands first."""
    qa, s_a, qw, s_w, bias = tiny_linear_inputs(seed=9, M=6, N=11, K=64)
    y = O.scaled_mm(qa, s_a, qw, s_w, bias)
    A = O.e4m3_decode(qa) * np.float64(s_a)
    W = O.e4m3_decode(qw) * s_w.astype(np.float64)[:, None]
    y2 = O.bf16_round(A @ W.T + bias.astype(np.float64))
    tol = O.ulp_bf16(y2)
    assert np.all(np.abs(y.astype(np.float64) - y2) <= tol)


def test_channelwise_with_equal_scales_equals_per_tensor():
    qa, s_a, qw, _, bias = tiny_linear_inputs(seed=10, M=5, N=9, K=40)
    s = np.float32(0.0123)
    y1 = O.scaled_mm(qa, s_a, qw, s, bias)
    y2 = O.scaled_mm(qa, s_a, qw, np.full(9, s, np.float32), bias)
    assert np.array_equal(y1, y2)


def test_linear_of_zero_activations_is_bias():
    w = np.ones((3, 8), np.float32)
    qw, s_w = O.quantize_per_tensor(w)
    bias = np.array([0.5, -2.0, 0.0], np.float32)
    y, qa, s_a = O.linear(np.zeros((2, 8), np.float32), qw, s_w, bias)
    assert s_a == 1.0 and np.all(qa == 0)
    assert np.array_equal(y, np.tile(bias, (2, 1)))


def test_empty_shapes():
    qa, s = O.quantize_per_tensor(np.zeros((0, 5), np.float32))
    assert qa.shape == (0, 5) and s == 1.0
    qw, sw = O.quantize_per_row(np.zeros((4, 0), np.float32))
    assert qw.shape == (4, 0) and np.all(sw == 1.0)
    y = O.scaled_mm(np.zeros((3, 0), np.uint8), 1.0, np.zeros((4, 0), np.uint8), sw,
                    np.array([1, 2, 3, 4], np.float32))
    assert np.array_equal(y, np.tile(np.array([1, 2, 3, 4], np.float32), (3, 1)))


def test_tolerance_bounds_fp32_accumulation():
    """A float32 left-to-right accumulation stays inside the tolerance; a 3-ulp shift does not."""
    g = np.random.default_rng(11)
    a = torch.from_numpy(g.standard_normal((4, 512)).astype(np.float32)).bfloat16().float().numpy()
    w = torch.from_numpy((g.standard_normal((8, 512)) * 0.02).astype(np.float32)).bfloat16().float().numpy()
    qa, s_a = O.quantize_per_tensor(a)
    qw, s_w = O.quantize_per_tensor(w)
    y = O.scaled_mm(qa, s_a, qw, s_w)
    A = O.e4m3_decode(qa).astype(np.float32)
    W = O.e4m3_decode(qw).astype(np.float32)
    acc = np.zeros((4, 8), np.float32)
    for k in range(512):
        acc = (acc + A[:, k:k + 1] * W[:, k][None, :]).astype(np.float32)
    y32 = torch.from_numpy((acc * np.float32(s_a) * np.float32(s_w)).astype(np.float32)).bfloat16().float().numpy()
    tol = O.tolerance(qa, s_a, qw, s_w, y)
    assert np.all(np.abs(y32.astype(np.float64) - y) <= tol)
    assert np.any(np.abs(y.astype(np.float64) * (1 + 3 * 2.0 ** -8) - y) > tol)


# ---------------------------------------------------------------------------
# the page-1 memory numbers pin the FP8 weight storage layout
# ---------------------------------------------------------------------------

def test_weight_memory_golden():
    """bf16 - fp8 weight memory of OpenHermes-2.5-Mistral-7B equals the linears' savings.

    FP8 storage per weight tensor [N, K]: N rows of ld = round_up(K, 16) bytes plus one
    fp32 scale (per-tensor). Every Mistral-7B K is a multiple of 16, so padding adds 0.
    """
    from fp8_w8a8_quantized_dynamic_gb300 import min_ld
    vals, linears, layers = {}, [], 0
    with open(os.path.join(GOLDEN, "mistral7b_weight_memory.txt")) as f:
        for line in f:
            p = line.split()
            if not p or p[0].startswith("#"):
                continue
            if p[0] == "linear":
                linears.append((int(p[2]), int(p[3])))
            elif p[0] == "layers":
                layers = int(p[1])
            else:
                vals[p[0]] = float(p[1])
    saved = layers * sum(2 * N * K - (N * min_ld(K) + 4) for K, N in linears)
    assert abs(saved / 2 ** 30 - (vals["bf16_gib"] - vals["fp8_gib"])) < 1e-4


# ---------------------------------------------------------------------------
# planted mistakes: each mutant of an oracle function must fail one pin
# ---------------------------------------------------------------------------

def _mutant_encode_ties_away(x):
    x = np.asarray(x, np.float32)
    mag = np.abs(x).astype(np.float64)
    pos = O._POSITIVE
    hi = np.minimum(np.searchsorted(pos, mag, side="left"), 0x7E)
    lo = np.maximum(hi - 1, 0)
    mid = (pos[lo] + pos[hi]) * 0.5
    code = np.where(mag < mid, lo, hi).astype(np.uint8)  # ties go up (away from zero)
    return code | (np.signbit(x).astype(np.uint8) << 7)


def _mutant_encode_truncate(x):
    x = np.asarray(x, np.float32)
    mag = np.abs(x).astype(np.float64)
    idx = np.minimum(np.searchsorted(O._POSITIVE, mag, side="right") - 1, 0x7E).astype(np.uint8)
    return idx | (np.signbit(x).astype(np.uint8) << 7)


def _mutant_encode_no_saturation(x):
    x = np.asarray(x, np.float32)
    code = O.e4m3_encode(x)
    return np.where(np.abs(x) > 464, np.uint8(0x7F) | (code & 0x80), code)


def _mutant_scaled_mm_rows_swapped(qa, s_a, qw, s_w, bias=None):
    return O.scaled_mm(qa, s_a, qw[::-1], s_w, bias)


def _mutant_scaled_mm_no_bias(qa, s_a, qw, s_w, bias=None):
    return O.scaled_mm(qa, s_a, qw, s_w, None)


def _mutant_scaled_mm_scale_reversed(qa, s_a, qw, s_w, bias=None):
    sw = np.asarray(s_w)
    return O.scaled_mm(qa, s_a, qw, sw[::-1] if sw.ndim else sw, bias)


def _mutant_scaled_mm_f32_sum(qa, s_a, qw, s_w, bias=None):
    S = (O.e4m3_decode(qa).astype(np.float32) @ O.e4m3_decode(qw).astype(np.float32).T)
    y = S.astype(np.float64) * np.float64(s_a) * np.asarray(s_w, np.float64)
    if bias is not None:
        y = y + bias
    return O.bf16_round(y.astype(np.float32).astype(np.float64))


def _mutant_decode_bias8():
    t = O.E4M3_DECODE.copy()
    return np.where(np.isnan(t), t, t * 2)  # exponent bias 6 instead of 7


@pytest.mark.parametrize("name", ["ties_away", "truncate", "no_saturation", "decode_bias",
                                  "scale_int8", "rows_swapped", "no_bias", "scale_reversed",
                                  "bf16_truncate"])
def test_planted_mistake_is_caught(name):
    with pytest.raises(AssertionError):
        if name == "ties_away":
            check_encode_vs_torch(_mutant_encode_ties_away, all_bf16_as_f32())
        elif name == "truncate":
            check_encode_vs_torch(_mutant_encode_truncate, all_bf16_as_f32())
        elif name == "no_saturation":
            check_encode_vs_torch(_mutant_encode_no_saturation, all_bf16_as_f32())
        elif name == "decode_bias":
            check_decode(_mutant_decode_bias8())
        elif name == "scale_int8":
            check_scale_exact(lambda a: (np.asarray(a, np.float32) / np.float32(127)).astype(np.float32),
                              np.array([1.0, 3.5, 448.0], np.float32))
        elif name in ("rows_swapped", "no_bias", "scale_reversed"):
            fn = {"rows_swapped": _mutant_scaled_mm_rows_swapped, "no_bias": _mutant_scaled_mm_no_bias,
                  "scale_reversed": _mutant_scaled_mm_scale_reversed}[name]
            check_scaled_mm_bruteforce(fn, *tiny_linear_inputs(seed=12))
        elif name == "bf16_truncate":
            v = np.random.default_rng(13).standard_normal(200)
            r = (np.trunc(v / O.ulp_bf16(v)) * O.ulp_bf16(v)).astype(np.float32)
            for vi, ri in zip(v, r):
                assert is_correctly_rounded_bf16(float(ri), Fraction(float(vi)))
