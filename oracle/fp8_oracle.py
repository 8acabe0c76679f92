"""CPU oracle for the FP8 (e4m3fn) W8A8 linear with dynamic per-tensor activation scale.

TEST INFRASTRUCTURE. Only tests/, __graft_entry__.smoke() and the CPU-baseline
leg of bench.py may import this module. The product path (the CUDA library and
its Python binding) never imports, links or calls it, and it shares no code,
table or constant generator with that path.

What is computed, and where the pages fix it:

* Weights and activations are both quantized to torch.float8_e4m3fn at run
  time ("Prototype FP8Linear W8A8 runtime quantization", opening paragraph;
  "Fp8 Quantization Support", opening paragraph: fp8 means e4m3fn).
* Quantization is symmetric (no zero point) with one scale per tensor
  ("Fp8 Quantization Support", example recipe: num_bits 8, type float,
  symmetric true, strategy tensor, for weights and input activations).
* The channelwise variant keeps one weight scale per output channel and
  applies it after the GEMM ("[Kernel] Implement fallback for FP8 channelwise
  using torch._scaled_mm", description: the rescale runs after the scaled mm).
* The pages do not print the scale formula, the rounding mode or the
  saturation rule. Readings taken here: scale = amax / 448 in fp32 (448 is the
  largest finite e4m3fn value), quotient x / scale by IEEE fp32 division,
  round-to-nearest-even to e4m3fn, saturation to +-448, sign of zero kept,
  scale := 1 when amax == 0.

Exactness of the product (why a float64 matmul is the definition, not an
approximation): every e4m3fn value is an integer multiple of 2**-9 with
magnitude <= 448, so every product of two codes is an integer multiple of
2**-18 below 2**17.62. A sum of K such products is an integer multiple of
2**-18 below K * 2**17.62; for K <= 2**17 that integer is below 2**53, so every
partial sum of any summation order is exactly representable in float64 and the
float64 matmul returns the exact sum.

Wider rows, same definitions:

* float8_e5m2 (1 sign bit, 5 exponent bits with bias 15, 2 mantissa bits,
  largest finite value 57344) as the other FP8 format ("Fp8 Quantization
  Support", opening paragraph: e5m2 named as a future extension of the
  quantization arguments). Scale = amax / 57344 for that format; every other
  step is unchanged.
* A static (calibrated) activation scale instead of the dynamic one ("Fp8
  Quantization Support", example recipe: input_activations quantized per
  tensor, scales produced by the oneshot calibration run): q = fp8(x / s_a)
  with the given s_a.
* Weight-only FP8: weights stored as FP8, activations kept in bf16 ("Prototype
  FP8Linear W8A8 runtime quantization": below compute capability 9.0 the
  weights are up-converted to the original dtype, saving memory but no
  compute). Reading taken here: every FP8 code is exactly representable in
  bf16, so the up-conversion is exact and the weight scale is applied to the
  output, Y = bf16(s_w[n] * sum_k a[m, k] * w[n, k] (+ bias[n])), the same
  rescale identity as the channelwise case.

Products that involve e5m2 or bf16 operands span too many binary orders of
magnitude for one float64 matmul to be exact; exact_dot_values splits the
operands into exponent bands whose pairwise matmuls are exact and adds the
band results as Python integers (see its docstring).

Parity pins for every function here live in tests/test_oracle_pins.py.
"""

from __future__ import annotations

import math
from typing import Optional, Tuple

import numpy as np

E4M3_MAX = 448.0          # largest finite e4m3fn value (code 0x7E)
BF16_MIN_EXP = -126       # smallest normal bf16 exponent
BF16_SUB_QUANTUM_EXP = -133  # bf16 subnormal spacing 2**-133 (7 stored mantissa bits)


# ---------------------------------------------------------------------------
# e4m3fn format (the dtype named by "Prototype FP8Linear W8A8 runtime
# quantization" and "Fp8 Quantization Support")
# ---------------------------------------------------------------------------

def _decode_code(c: int) -> float:
    """Value of one e4m3fn code from the format definition.

    1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; exponent field 0 is
    subnormal (m * 2**-9); exponent 15 with mantissa 7 is NaN; there is no
    infinity, so exponent 15 with mantissa 0..6 are ordinary normals (up to 448).
    """
    sign = -1.0 if (c >> 7) & 1 else 1.0
    e = (c >> 3) & 0xF
    m = c & 0x7
    if e == 0xF and m == 0x7:
        return math.nan
    if e == 0:
        return sign * m * 2.0 ** -9
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


E4M3_DECODE = np.array([_decode_code(c) for c in range(256)], dtype=np.float64)
E4M3_DECODE.setflags(write=False)

# the 127 non-negative finite codes 0x00..0x7E, ascending in value (0 .. 448)
_POSITIVE = E4M3_DECODE[:0x7F].copy()
assert np.all(np.diff(_POSITIVE) > 0)


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """e4m3fn codes (uint8) -> float64 values."""
    return E4M3_DECODE[np.asarray(codes, dtype=np.uint8)]


def e4m3_encode(x: np.ndarray) -> np.ndarray:
    """float32 -> e4m3fn code, saturating, round to nearest, ties to even.

    Table search: the two finite magnitudes that bracket |x| are found by
    binary search; |x| is compared with their midpoint exactly (the midpoint of
    two e4m3fn values has 5 significant bits, exact in float64). Below the
    midpoint -> lower, above -> upper, equal -> the code with an even mantissa
    (even code). |x| >= 448 gives 448 (saturation). The sign bit is copied from
    x, so -0 and negative values that round to zero give 0x80. NaN gives 0x7F
    (NaN input is outside the layer's contract).
    """
    x = np.asarray(x, dtype=np.float32)
    mag = np.abs(x).astype(np.float64)
    hi = np.searchsorted(_POSITIVE, mag, side="left")      # first code with value >= |x|
    hi = np.minimum(hi, 0x7E)                                # saturate above 448
    lo = np.maximum(hi - 1, 0)
    mid = (_POSITIVE[lo] + _POSITIVE[hi]) * 0.5
    tie_pick = np.where(hi % 2 == 0, hi, lo)
    code = np.where(mag < mid, lo, np.where(mag > mid, hi, tie_pick)).astype(np.uint8)
    code = np.where(np.isnan(mag), np.uint8(0x7F), code)
    return code | (np.signbit(x).astype(np.uint8) << 7)


# ---------------------------------------------------------------------------
# e5m2 format ("Fp8 Quantization Support": the other FP8 dtype, torch.float8_e5m2)
# ---------------------------------------------------------------------------

E5M2_MAX = 57344.0        # largest finite e5m2 value (code 0x7B)


def _decode_code_e5m2(c: int) -> float:
    """Value of one e5m2 code from the format definition.

    1 sign bit, 5 exponent bits (bias 15), 2 mantissa bits; exponent field 0 is
    subnormal (m * 2**-16); exponent 31 is infinity (mantissa 0) or NaN.
    """
    sign = -1.0 if (c >> 7) & 1 else 1.0
    e = (c >> 2) & 0x1F
    m = c & 0x3
    if e == 0x1F:
        return sign * math.inf if m == 0 else math.nan
    if e == 0:
        return sign * m * 2.0 ** -16
    return sign * (1.0 + m / 4.0) * 2.0 ** (e - 15)


E5M2_DECODE = np.array([_decode_code_e5m2(c) for c in range(256)], dtype=np.float64)
E5M2_DECODE.setflags(write=False)

# the 124 non-negative finite codes 0x00..0x7B, ascending in value (0 .. 57344)
_POSITIVE_E5M2 = E5M2_DECODE[:0x7C].copy()
assert np.all(np.diff(_POSITIVE_E5M2) > 0)


def e5m2_decode(codes: np.ndarray) -> np.ndarray:
    """e5m2 codes (uint8) -> float64 values."""
    return E5M2_DECODE[np.asarray(codes, dtype=np.uint8)]


def _encode_table(x: np.ndarray, positive: np.ndarray, nan_code: int) -> np.ndarray:
    """Round float32 to the nearest value of an ascending table of non-negative finite
    format values (code == table index), ties to the even code, saturating at the
    last entry, sign bit copied from x. Same method as e4m3_encode."""
    x = np.asarray(x, dtype=np.float32)
    mag = np.abs(x).astype(np.float64)
    top = len(positive) - 1
    hi = np.minimum(np.searchsorted(positive, mag, side="left"), top)
    lo = np.maximum(hi - 1, 0)
    mid = (positive[lo] + positive[hi]) * 0.5
    tie_pick = np.where(hi % 2 == 0, hi, lo)
    code = np.where(mag < mid, lo, np.where(mag > mid, hi, tie_pick)).astype(np.uint8)
    code = np.where(np.isnan(mag), np.uint8(nan_code), code)
    return code | (np.signbit(x).astype(np.uint8) << 7)


def e5m2_encode(x: np.ndarray) -> np.ndarray:
    """float32 -> e5m2 code, saturating to +-57344 (never infinity), round to nearest,
    ties to even. The midpoint of two e5m2 values has 4 significant bits (exact)."""
    return _encode_table(x, _POSITIVE_E5M2, 0x7F)


# format name -> (decode table, largest finite value, encoder, significant bits)
FORMATS = {
    "e4m3": (E4M3_DECODE, E4M3_MAX, None, 4),
    "e5m2": (E5M2_DECODE, E5M2_MAX, e5m2_encode, 3),
}


def fp8_max(fmt: str = "e4m3") -> float:
    return FORMATS[fmt][1]


def decode(codes: np.ndarray, fmt: str = "e4m3") -> np.ndarray:
    """FP8 codes of format `fmt` -> float64 values."""
    return FORMATS[fmt][0][np.asarray(codes, dtype=np.uint8)]


def encode(x: np.ndarray, fmt: str = "e4m3") -> np.ndarray:
    """float32 -> FP8 code of format `fmt` (saturating RNE, ties to even)."""
    return e4m3_encode(x) if fmt == "e4m3" else FORMATS[fmt][2](x)


# ---------------------------------------------------------------------------
# bf16 output rounding
# ---------------------------------------------------------------------------

def _bf16_quantum(v: np.ndarray) -> np.ndarray:
    """Spacing of bf16 values around |v| (2**-133 in the subnormal range)."""
    _, e = np.frexp(np.asarray(v, dtype=np.float64))  # v = m * 2**e, 0.5 <= |m| < 1
    return np.ldexp(1.0, np.maximum(e - 8, BF16_SUB_QUANTUM_EXP))


def bf16_round(v: np.ndarray) -> np.ndarray:
    """float64 -> nearest bf16 (ties to even), returned as float32 (exact)."""
    v = np.asarray(v, dtype=np.float64)
    q = _bf16_quantum(v)
    return (np.rint(v / q) * q).astype(np.float32)  # v/q is exact: q is a power of two


def ulp_bf16(y: np.ndarray) -> np.ndarray:
    """Spacing of bf16 values at |y| (2**-133 at zero and in the subnormal range)."""
    return _bf16_quantum(y)


# ---------------------------------------------------------------------------
# Dynamic / per-tensor and per-channel quantization
# ---------------------------------------------------------------------------

def amax(x: np.ndarray) -> np.float32:
    """max |x| over the whole tensor (0 for an empty tensor). Exact."""
    x = np.asarray(x, dtype=np.float32)
    return np.float32(np.max(np.abs(x))) if x.size else np.float32(0.0)


def scale_from_amax(a: np.ndarray, fmt: str = "e4m3") -> np.ndarray:
    """scale = amax / 448 (57344 for e5m2) by IEEE fp32 division; 1.0 where amax == 0
    (or the quotient underflows)."""
    a = np.asarray(a, dtype=np.float32)
    s = (a / np.float32(fp8_max(fmt))).astype(np.float32)
    return np.where(s == 0, np.float32(1.0), s).astype(np.float32)


def quantize_with_scale(x: np.ndarray, s, fmt: str = "e4m3") -> np.ndarray:
    """q = fp8(fp32(x / s)): fp32 quotient, then one saturating RNE rounding to the format.

    With a static (calibrated) s this is the whole activation quantization: values
    beyond s * 448 (s * 57344) saturate."""
    x = np.asarray(x, dtype=np.float32)
    with np.errstate(over="ignore"):  # an fp32 quotient may overflow to inf; it then saturates
        q = (x / np.asarray(s, dtype=np.float32)).astype(np.float32)
    return encode(q, fmt)


def quantize_per_tensor(x: np.ndarray, fmt: str = "e4m3") -> Tuple[np.ndarray, np.float32]:
    """Dynamic per-tensor quantization ("Prototype FP8Linear W8A8 runtime quantization").

    Returns (codes uint8 of x's shape, fp32 scale) with x ~= decode(codes) * scale.
    """
    s = np.float32(scale_from_amax(amax(x), fmt))
    return quantize_with_scale(x, s, fmt), s


def quantize_per_row(x: np.ndarray, fmt: str = "e4m3") -> Tuple[np.ndarray, np.ndarray]:
    """Per-output-channel weight quantization: one scale per row of W [N, K]
    ("[Kernel] Implement fallback for FP8 channelwise using torch._scaled_mm").
    """
    x = np.asarray(x, dtype=np.float32)
    row_amax = np.max(np.abs(x), axis=1) if x.shape[1] else np.zeros(x.shape[0], np.float32)
    s = scale_from_amax(row_amax, fmt)
    return quantize_with_scale(x, s[:, None], fmt), s


# ---------------------------------------------------------------------------
# Scaled GEMM + rescale epilogue
# ---------------------------------------------------------------------------

def _exponent(v: np.ndarray) -> np.ndarray:
    """Binary exponent E with 2**E <= |v| < 2**(E+1) (meaningless where v == 0)."""
    return np.frexp(v)[1].astype(np.int64) - 1


def _bands(X: np.ndarray, width: int):
    """Split X into arrays that each keep the entries whose binary exponent lies in one
    window [start, start + width) (zero elsewhere); yields (X_band, start)."""
    nz = X != 0
    if not nz.any():
        return
    E = _exponent(X)
    lo, hi = int(E[nz].min()), int(E[nz].max())
    for start in range(lo, hi + 1, width):
        sel = nz & (E >= start) & (E < start + width)
        if sel.any():
            yield np.where(sel, X, 0.0), start


def _exponent_span(X: np.ndarray) -> int:
    nz = X != 0
    if not nz.any():
        return 1
    E = _exponent(X[nz])
    return int(E.max() - E.min() + 1)


def exact_dot_values(A: np.ndarray, pa: int, B: np.ndarray, pb: int) -> np.ndarray:
    """S[m, n] = sum_k A[m, k] * B[n, k], exact, then rounded once to float64.

    A holds floats with at most `pa` significant bits, B with at most `pb` (e4m3: 4,
    e5m2: 3, bf16: 8). An entry with binary exponent E is an integer multiple of
    2**(E - p + 1). Inside an exponent window [s, s + W) the entries are multiples of
    2**(s - p + 1) below 2**(s + W), i.e. integers below 2**(W + p - 1) in that unit. For
    a window pair the K products and every partial sum are then integers below
    2**(kbits + Wa + Wb + pa + pb - 2) (K < 2**kbits) in the pair's unit, so the float64
    matmul of the two windowed matrices is exact when Wa + Wb <= 55 - pa - pb - kbits.
    The window results are scaled to the smallest unit, converted to Python integers
    (exact), added as integers and converted back with one rounding.
    """
    A = np.asarray(A, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    M, K = A.shape
    N = B.shape[0]
    assert B.shape[1] == K
    out = np.zeros((M, N), np.float64)
    if M == 0 or N == 0 or K == 0:
        return out
    kbits = int(K).bit_length()
    budget = 55 - pa - pb - kbits
    assert budget >= 2, "K too large for exact window products"
    span_a, span_b = _exponent_span(A), _exponent_span(B)
    # window widths with Wa + Wb == budget minimizing the number of window pairs
    wa = min(range(1, budget), key=lambda w: -(-span_a // w) * -(-span_b // (budget - w)))
    wb = budget - wa
    parts = []
    for Xa, sa in _bands(A, wa):
        for Xb, sb in _bands(B, wb):
            parts.append((Xa @ Xb.T, (sa - pa + 1) + (sb - pb + 1)))
    if not parts:
        return out
    umin = min(u for _, u in parts)
    to_int = np.frompyfunc(int, 1, 1)
    total = None
    for P, _ in parts:
        ints = to_int(np.ldexp(P, -umin))  # P is a multiple of 2**umin: integral, exact
        total = ints if total is None else total + ints
    as_float = np.frompyfunc(float, 1, 1)  # Python int -> float rounds to nearest even
    return np.ldexp(as_float(total).astype(np.float64), umin)


def exact_dot(qa: np.ndarray, qw: np.ndarray, fmt_a: str = "e4m3", fmt_w: str = "e4m3") -> np.ndarray:
    """S[m, n] = sum_k decode(qa[m, k]) * decode(qw[n, k]).

    e4m3 x e4m3: one float64 matmul, exact (module docstring). Any e5m2 operand:
    exact_dot_values (exact, rounded once to float64).
    """
    qa = np.asarray(qa, dtype=np.uint8)
    qw = np.asarray(qw, dtype=np.uint8)
    assert qa.shape[1] == qw.shape[1] <= 2 ** 17
    if fmt_a == "e4m3" and fmt_w == "e4m3":
        return e4m3_decode(qa) @ e4m3_decode(qw).T
    return exact_dot_values(decode(qa, fmt_a), FORMATS[fmt_a][3], decode(qw, fmt_w), FORMATS[fmt_w][3])


def _epilogue(S: np.ndarray, s_a, s_w, bias, return_f64: bool):
    scale = np.float64(np.float32(s_a)) * np.asarray(s_w, dtype=np.float32).astype(np.float64)
    y = S * scale  # broadcasts a vector over columns n
    if bias is not None:
        y = y + np.asarray(bias, dtype=np.float32).astype(np.float64)
    yb = bf16_round(y)
    return (yb, y) if return_f64 else yb


def scaled_mm(qa: np.ndarray, s_a, qw: np.ndarray, s_w, bias: Optional[np.ndarray] = None,
              return_f64: bool = False, fmt_a: str = "e4m3", fmt_w: str = "e4m3"):
    """Y = bf16( s_a * s_w[n] * S[m, n] (+ bias[n]) ), S the exact product.

    s_w is a scalar (per-tensor) or a vector [N] (channelwise); the channelwise
    scale multiplies output column n after the GEMM, which equals scaling row n
    of W first: (s_a A)(s_w,n W_n)^T = s_a s_w,n (A W_n^T) ("[Kernel] Implement
    fallback for FP8 channelwise using torch._scaled_mm", description). The
    scale product s_a * s_w of two fp32 numbers is exact in float64; the rest is
    float64 and one final round-to-nearest-even to bf16.
    """
    return _epilogue(exact_dot(qa, qw, fmt_a, fmt_w), s_a, s_w, bias, return_f64)


def linear(a: np.ndarray, qw: np.ndarray, s_w, bias: Optional[np.ndarray] = None,
           fmt_a: str = "e4m3", fmt_w: str = "e4m3", s_a=None):
    """W8A8 linear with per-tensor activation quantization.

    a: bf16 values as float32 [M, K]; qw, s_w from quantize_per_tensor or
    quantize_per_row of W [N, K]. s_a None: dynamic scale amax(a) / max(fmt_a);
    otherwise the given static (calibrated) scale is used as is. Returns
    (Y bf16-as-float32 [M, N], qa, s_a).
    """
    if s_a is None:
        qa, s_a = quantize_per_tensor(a, fmt_a)
    else:
        s_a = np.float32(s_a)
        qa = quantize_with_scale(a, s_a, fmt_a)
    return scaled_mm(qa, s_a, qw, s_w, bias, fmt_a=fmt_a, fmt_w=fmt_w), qa, s_a


def linear_weight_only(a: np.ndarray, qw: np.ndarray, s_w, bias: Optional[np.ndarray] = None,
                       fmt_w: str = "e4m3", return_f64: bool = False):
    """Weight-only FP8 linear: Y = bf16( s_w[n] * sum_k a[m, k] * decode(qw[n, k]) (+ bias[n]) ).

    a stays bf16 (values as float32); the FP8 weights are up-converted exactly and the
    weight scale multiplies the output ("Prototype FP8Linear W8A8 runtime
    quantization": the up-conversion path below compute capability 9.0).
    """
    S = exact_dot_values(np.asarray(a, np.float32).astype(np.float64), 8, decode(qw, fmt_w), FORMATS[fmt_w][3])
    return _epilogue(S, np.float32(1.0), s_w, bias, return_f64)


def tolerance(qa: np.ndarray, s_a, qw: np.ndarray, s_w, y_ref: np.ndarray,
              fmt_a: str = "e4m3", fmt_w: str = "e4m3") -> np.ndarray:
    """Allowed |y_gpu - y_ref|: one bf16 ulp of y_ref plus K * 2**-23 * sum_k |s_a qa_k * s_w qw_k|.

    The second term bounds fp32 accumulation in any order (twice the classic
    (K-1) * 2**-24 worst-case bound of recursive summation).
    """
    abs_a = np.abs(decode(qa, fmt_a)) * np.float64(np.float32(s_a))
    return _tolerance(abs_a, np.abs(decode(qw, fmt_w)), s_w, y_ref)


def tolerance_weight_only(a: np.ndarray, qw: np.ndarray, s_w, y_ref: np.ndarray, fmt_w: str = "e4m3"):
    """Same bound for the weight-only product (bf16 activations, FP8 weights)."""
    return _tolerance(np.abs(np.asarray(a, np.float32).astype(np.float64)), np.abs(decode(qw, fmt_w)), s_w, y_ref)


def _tolerance(abs_a: np.ndarray, abs_wq: np.ndarray, s_w, y_ref: np.ndarray) -> np.ndarray:
    K = abs_a.shape[1]
    sw = np.asarray(s_w, dtype=np.float32).astype(np.float64)
    abs_w = abs_wq * (sw[:, None] if sw.ndim else sw)
    return ulp_bf16(y_ref) + K * 2.0 ** -23 * (abs_a @ abs_w.T)
