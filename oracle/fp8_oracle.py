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


def scale_from_amax(a: np.ndarray) -> np.ndarray:
    """scale = amax / 448 by IEEE fp32 division; 1.0 where amax == 0 (or the quotient underflows)."""
    a = np.asarray(a, dtype=np.float32)
    s = (a / np.float32(E4M3_MAX)).astype(np.float32)
    return np.where(s == 0, np.float32(1.0), s).astype(np.float32)


def quantize_with_scale(x: np.ndarray, s) -> np.ndarray:
    """q = e4m3(fp32(x / s)): fp32 quotient, then one RNE rounding to e4m3fn."""
    x = np.asarray(x, dtype=np.float32)
    return e4m3_encode((x / np.asarray(s, dtype=np.float32)).astype(np.float32))


def quantize_per_tensor(x: np.ndarray) -> Tuple[np.ndarray, np.float32]:
    """Dynamic per-tensor quantization ("Prototype FP8Linear W8A8 runtime quantization").

    Returns (codes uint8 of x's shape, fp32 scale) with x ~= decode(codes) * scale.
    """
    s = np.float32(scale_from_amax(amax(x)))
    return quantize_with_scale(x, s), s


def quantize_per_row(x: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Per-output-channel weight quantization: one scale per row of W [N, K]
    ("[Kernel] Implement fallback for FP8 channelwise using torch._scaled_mm").
    """
    x = np.asarray(x, dtype=np.float32)
    row_amax = np.max(np.abs(x), axis=1) if x.shape[1] else np.zeros(x.shape[0], np.float32)
    s = scale_from_amax(row_amax)
    return quantize_with_scale(x, s[:, None]), s


# ---------------------------------------------------------------------------
# Scaled GEMM + rescale epilogue
# ---------------------------------------------------------------------------

def exact_dot(qa: np.ndarray, qw: np.ndarray) -> np.ndarray:
    """S[m, n] = sum_k decode(qa[m, k]) * decode(qw[n, k]), exact in float64 (module docstring)."""
    qa = np.asarray(qa, dtype=np.uint8)
    qw = np.asarray(qw, dtype=np.uint8)
    assert qa.shape[1] == qw.shape[1] <= 2 ** 17
    return e4m3_decode(qa) @ e4m3_decode(qw).T


def scaled_mm(qa: np.ndarray, s_a, qw: np.ndarray, s_w, bias: Optional[np.ndarray] = None,
              return_f64: bool = False):
    """Y = bf16( s_a * s_w[n] * S[m, n] (+ bias[n]) ), S the exact product.

    s_w is a scalar (per-tensor) or a vector [N] (channelwise); the channelwise
    scale multiplies output column n after the GEMM, which equals scaling row n
    of W first: (s_a A)(s_w,n W_n)^T = s_a s_w,n (A W_n^T) ("[Kernel] Implement
    fallback for FP8 channelwise using torch._scaled_mm", description). The
    scale product s_a * s_w of two fp32 numbers is exact in float64; the rest is
    float64 and one final round-to-nearest-even to bf16.
    """
    S = exact_dot(qa, qw)
    scale = np.float64(np.float32(s_a)) * np.asarray(s_w, dtype=np.float32).astype(np.float64)
    y = S * scale  # broadcasts a vector over columns n
    if bias is not None:
        y = y + np.asarray(bias, dtype=np.float32).astype(np.float64)
    yb = bf16_round(y)
    return (yb, y) if return_f64 else yb


def linear(a: np.ndarray, qw: np.ndarray, s_w, bias: Optional[np.ndarray] = None):
    """W8A8 linear with dynamic per-tensor activation quantization.

    a: bf16 values as float32 [M, K]; qw, s_w from quantize_per_tensor or
    quantize_per_row of W [N, K]. Returns (Y bf16-as-float32 [M, N], qa, s_a).
    """
    qa, s_a = quantize_per_tensor(a)
    return scaled_mm(qa, s_a, qw, s_w, bias), qa, s_a


def tolerance(qa: np.ndarray, s_a, qw: np.ndarray, s_w, y_ref: np.ndarray) -> np.ndarray:
    """Allowed |y_gpu - y_ref|: one bf16 ulp of y_ref plus K * 2**-23 * sum_k |s_a qa_k * s_w qw_k|.

    The second term bounds fp32 accumulation in any order (twice the classic
    (K-1) * 2**-24 worst-case bound of recursive summation).
    """
    K = np.asarray(qa).shape[1]
    abs_a = np.abs(e4m3_decode(qa)) * np.float64(np.float32(s_a))
    sw = np.asarray(s_w, dtype=np.float32).astype(np.float64)
    abs_w = np.abs(e4m3_decode(qw)) * (sw[:, None] if sw.ndim else sw)
    return ulp_bf16(y_ref) + K * 2.0 ** -23 * (abs_a @ abs_w.T)
