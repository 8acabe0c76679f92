// Device helpers shared by the library's kernels (sm_103a).
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace fp8k {

constexpr float kE4M3Max = 448.0f;      // largest finite float8_e4m3fn value
constexpr int kAmaxMaxBlocks = 1024;    // partial-amax slots in a workspace
constexpr size_t kWsScaleOffset = 4096; // workspace: fp32 activation scale after the partials
constexpr size_t kWsQaOffset = 4352;    // workspace: quantized activations (256-byte aligned)
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // bounded device waits: 2 s

// Device error bits (ORed into a per-module word, read by fp8_last_device_status).
constexpr unsigned int kErrTimeout = 1u;

// ---------------------------------------------------------------------------
// Quantization arithmetic: q = fp8(fp32(x / s)), saturating RNE.
// ---------------------------------------------------------------------------

// FP8 formats (values of fp8_format): 0 = e4m3fn (largest finite 448), 1 = e5m2 (57344).
constexpr int kFmtE4M3 = 0;
constexpr int kFmtE5M2 = 1;
constexpr float kE5M2Max = 57344.0f;

template <int F>
__device__ __forceinline__ constexpr float fp8_max() { return F == kFmtE5M2 ? kE5M2Max : kE4M3Max; }

// Two fp32 -> packed FP8 pair of format F (round to nearest even, saturate to the largest
// finite value; NaN stays NaN). `lo` lands in bits 0..7, `hi` in bits 8..15.
template <int F>
__device__ __forceinline__ uint32_t cvt_fp8x2(float lo, float hi) {
  uint16_t r;
  if constexpr (F == kFmtE5M2)
    asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  else
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two FP8 codes of format F (bits 0..7 and 8..15) -> the same two values as bf16x2 (exact:
// every e4m3 and e5m2 value is a bf16 value), via the exact FP8 -> f16 conversion.
template <int F>
__device__ __forceinline__ uint32_t fp8x2_to_bf16x2(uint32_t codes) {
  uint32_t h;
  const uint16_t c = uint16_t(codes);
  if constexpr (F == kFmtE5M2)
    asm("cvt.rn.f16x2.e5m2x2 %0, %1;" : "=r"(h) : "h"(c));
  else
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(c));
  const float lo = __half2float(__ushort_as_half(uint16_t(h))), hi = __half2float(__ushort_as_half(uint16_t(h >> 16)));
  const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&b);
}

// Quantizer for one scale s: FP8 codes of fl32(x / s), most of the time without a division.
// The kernels' main paths use the exact quotient further below; this bracket serves what
// that form does not cover: scales outside [2^-80, 2^100], ragged row ends, and units whose
// codes show a non-finite input under a caller-supplied scale.
// With r = fl32(1/s), the products L = fl32(|x| * fl32(r * (1 - 2^-20))) and
// H = fl32(x * fl32(r * (1 + 2^-20))) bracket the quotient strictly: each carries at most
// four roundings of 2^-24 (relative) against a 2^-20 margin, so L < |fl32(x/s)| < |H|, and
// the bracket is at most ~2^-19 |x/s| wide. Rounding to FP8 is monotone and symmetric in sign,
// so when L and |H| round to the same FP8 magnitude, that is the magnitude of the quotient's
// code, and H (converted with x's sign) gives the code itself. Zero, overflow to infinity
// (saturation) and fp32 subnormal quotients (FP8 zero) all fall out of the same test.
// Otherwise the quotient lies next to an FP8 rounding boundary and the value is refused: an
// fma residual that proves the quotient exact, or the IEEE division, decides. Scales below
// 2^-125, where 1/s could overflow, always divide.
struct Quantizer {
  float s, r, r_lo, r_hi;
  bool fast;
};

__device__ __forceinline__ Quantizer make_quantizer(float s) {
  Quantizer q;
  q.s = s;
  q.r = __frcp_rn(s);
  q.r_lo = q.r * (1.0f - 0x1p-20f);
  q.r_hi = q.r * (1.0f + 0x1p-20f);
  q.fast = s >= 0x1p-125f && q.r < 0x1p126f;
  return q;
}

template <int F>
static __device__ __noinline__ uint32_t quant2_divide(float x0, float x1, float s) {
  return cvt_fp8x2<F>(__fdiv_rn(x0, s), __fdiv_rn(x1, s));
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Bracket of two values (see Quantizer): returns the codes of the upper ends (with signs) and
// sets `bad` non-zero when a lower end rounds to another magnitude.
template <int F>
__device__ __forceinline__ uint32_t bracket2(float x0, float x1, const Quantizer& q, uint32_t& bad) {
  const uint32_t lo = cvt_fp8x2<F>(fabsf(x0) * q.r_lo, fabsf(x1) * q.r_lo);
  const uint32_t hi = cvt_fp8x2<F>(x0 * q.r_hi, x1 * q.r_hi);
  bad = (hi & 0x7F7Fu) ^ lo;
  return hi;
}

// Two values -> two FP8 bytes of format F (x0 in bits 0..7, x1 in bits 8..15).
template <int F>
__device__ __forceinline__ uint32_t quant2(float x0, float x1, const Quantizer& q) {
  if (q.fast) {
    uint32_t bad;
    const uint32_t c = bracket2<F>(x0, x1, q, bad);
    if (bad == 0) return c;
  }
  return quant2_divide<F>(x0, x1, q.s);
}

// Four values -> four FP8 bytes (x0 in the lowest byte).
template <int F>
__device__ __forceinline__ uint32_t quant4(float x0, float x1, float x2, float x3, const Quantizer& q) {
  return quant2<F>(x0, x1, q) | (quant2<F>(x2, x3, q) << 16);
}

// Eight bf16 (packed in a uint4) -> eight FP8 bytes with no branch. `bad` gets bit p set for
// each pair p (values 2p, 2p+1) the fast path cannot settle: a value within a few ulps of a
// rounding boundary, or every pair when the scale is outside the fast range. Straight-line
// code lets a thread interleave several units; quant8_bf16_fix settles the flagged pairs.
template <int F>
__device__ __forceinline__ uint2 quant8_bf16_try(uint4 v, const Quantizer& q, uint32_t& bad) {
  uint32_t b0, b1, b2, b3;
  const uint32_t w0 = bracket2<F>(bf16_lo(v.x), bf16_hi(v.x), q, b0);
  const uint32_t w1 = bracket2<F>(bf16_lo(v.y), bf16_hi(v.y), q, b1);
  const uint32_t w2 = bracket2<F>(bf16_lo(v.z), bf16_hi(v.z), q, b2);
  const uint32_t w3 = bracket2<F>(bf16_lo(v.w), bf16_hi(v.w), q, b3);
  bad = q.fast ? (uint32_t(b0 != 0) | (uint32_t(b1 != 0) << 1) | (uint32_t(b2 != 0) << 2) | (uint32_t(b3 != 0) << 3))
               : 0xFu;
  return make_uint2(w0 | (w1 << 16), w2 | (w3 << 16));
}

// Quotients the fast path refused. When y = x * fl(1/s) satisfies y * s == x exactly, the
// quotient x / s is y itself; the fma residual proves it, and is exact when
// ulp(y) * ulp(s) >= 2^-126 (both at least 2^-40 in magnitude). That settles most refusals:
// with a scale of few significant bits (amax / 448 when amax's mantissa is a multiple of 7),
// or values whose mantissa shares the scale's factors, many quotients are exact and sit on
// rounding midpoints, where only the tie rule decides. Zeros keep their sign (r may be
// infinite for a tiny scale).
__device__ __forceinline__ bool quotient_is_product(float x, float y, float s) {
  return x == 0.0f || (fabsf(y) >= 0x1p-40f && fabsf(y) < 0x1p100f && s >= 0x1p-40f && fmaf(y, s, -x) == 0.0f);
}

// Exact codes for the pairs flagged in `bad` that the residual settles, in line (short code,
// taken by the lanes that need it); returns the pairs still unsettled.
template <int F>
__device__ __forceinline__ uint32_t quant8_bf16_settle(uint4 v, uint2& codes, uint32_t bad, float s, float r) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t c[2] = {codes.x, codes.y};
  uint32_t left = 0;
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    if (bad & (1u << p)) {
      const float x0 = bf16_lo(w[p]), x1 = bf16_hi(w[p]);
      const float y0 = x0 == 0.0f ? x0 : x0 * r, y1 = x1 == 0.0f ? x1 : x1 * r;
      if (quotient_is_product(x0, y0, s) && quotient_is_product(x1, y1, s)) {
        const int sh = (p & 1) * 16;
        c[p >> 1] = (c[p >> 1] & ~(0xFFFFu << sh)) | (cvt_fp8x2<F>(y0, y1) << sh);
      } else {
        left |= 1u << p;
      }
    }
  }
  codes = make_uint2(c[0], c[1]);
  return left;
}

// Codes of the flagged pairs by IEEE division (out of line: rarely taken).
template <int F>
static __device__ __noinline__ uint2 quant8_bf16_divide(uint4 v, uint2 codes, uint32_t left, float s) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t c[2] = {codes.x, codes.y};
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    if (left & (1u << p)) {
      const uint32_t pair = cvt_fp8x2<F>(__fdiv_rn(bf16_lo(w[p]), s), __fdiv_rn(bf16_hi(w[p]), s));
      const int sh = (p & 1) * 16;
      c[p >> 1] = (c[p >> 1] & ~(0xFFFFu << sh)) | (pair << sh);
    }
  }
  return make_uint2(c[0], c[1]);
}

// Settles the flagged pairs of a unit: the residual proof in line, division for the rest.
template <int F>
__device__ __forceinline__ uint2 quant8_bf16_fix(uint4 v, uint2 codes, uint32_t bad, float s, float r) {
  const uint32_t left = quant8_bf16_settle<F>(v, codes, bad, s, r);
  return left ? quant8_bf16_divide<F>(v, codes, left, s) : codes;
}

// Eight bf16 -> eight FP8 bytes, two values at a time (quant2: bracket, division if refused).
template <int F>
__device__ __forceinline__ uint2 quant8_bf16_pairwise(uint4 v, const Quantizer& q) {
  uint2 r;
  r.x = quant4<F>(bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y), q);
  r.y = quant4<F>(bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w), q);
  return r;
}

// Eight bf16 (packed in a uint4) -> eight FP8 bytes (uint2).
template <int F>
__device__ __forceinline__ uint2 quant8_bf16(uint4 v, const Quantizer& q) {
  uint32_t bad;
  const uint2 r = quant8_bf16_try<F>(v, q, bad);
  return bad == 0 ? r : quant8_bf16_fix<F>(v, r, bad, q.s, q.r);
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) { return __uint_as_float(uint32_t(b) << 16); }

// ---------------------------------------------------------------------------
// Exact quotient without division: fl32(x / s) for every x, no refusals, no branches.
//
// With r = fl32(1/s) (correctly rounded reciprocal) and its tail r_lo = fl32(fl32(1 - s*r) * r)
// (1 - s*r is exact in one fma), q0 = fl32(x*r + fl32(x*r_lo)) approximates x/s to about
// 2^-46 relative, so q0 is faithful (within one ulp of x/s). The residual x - s*q0 of a
// faithful quotient is exactly representable (one fma computes it exactly), and by
// Markstein's theorem (P. Markstein, "Computation of elementary functions on the IBM RISC
// System/6000 processor", IBM J. Res. Dev. 34(1), 1990) q = fl32(q0 + (x - s*q0) * r) is the
// correctly rounded quotient fl32(x / s). Conditions: no underflow in the residual and no
// overflow, which hold for s in [2^-80, 2^100] and quotients of magnitude >= 2^-20; smaller
// quotients may be off in their last bits but stay far below the smallest FP8 rounding
// boundary (2^-17), so the FP8 code is still exact. Checked on a GB300 against IEEE division
// over all finite bf16 x for 27264 scales in that range: equal quotients for |x/s| >= 2^-20,
// equal e4m3 and e5m2 codes everywhere.
//
// Two values travel as one 64-bit register pair through the packed f32x2 multiply and fma
// (sm_100 family): four codes take four unpacks, eight packed arithmetic ops, two
// conversions, one byte permute and one select. Signs come from the inputs (x = -0 gives
// q = +0 in the fma chain; the code must still be 0x80). Non-finite x, or |x/s| beyond
// fp32, give a NaN code (0x7F in magnitude for e4m3, >= 0x7C for e5m2), which no finite
// in-range quotient produces: callers that may see such inputs check for it.
struct ExactScale {
  uint64_t r2, r_lo2, neg_s2;  // (r, r), (r_lo, r_lo), (-s, -s)
  bool fast;                   // s in [2^-80, 2^100]
};

__device__ __forceinline__ uint64_t pack_f32x2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1,%2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

__device__ __forceinline__ ExactScale make_exact_scale(float s) {
  ExactScale k;
  const float r = __frcp_rn(s);
  const float r_lo = fmaf(-s, r, 1.0f) * r;
  k.r2 = pack_f32x2(r, r);
  k.r_lo2 = pack_f32x2(r_lo, r_lo);
  k.neg_s2 = pack_f32x2(-s, -s);
  k.fast = s >= 0x1p-80f && s <= 0x1p100f;
  return k;
}

// fl32(x / s) for the two bf16 values of a word, as a packed pair (low half first).
__device__ __forceinline__ uint64_t exact_quotient2(uint32_t w, const ExactScale& k) {
  const uint64_t x = pack_f32x2(bf16_lo(w), bf16_hi(w));
  const uint64_t q0 = fma_f32x2(x, k.r2, mul_f32x2(x, k.r_lo2));
  return fma_f32x2(fma_f32x2(k.neg_s2, q0, x), k.r2, q0);
}

// Two packed quotient pairs -> four FP8 codes of format F, the first value in the lowest byte.
template <int F>
__device__ __forceinline__ uint32_t cvt_fp8x4(uint64_t p01, uint64_t p23) {
  uint32_t d;
  if constexpr (F == kFmtE5M2)
    asm("{\n .reg .b16 l, h;\n .reg .f32 a, b, c, e;\n mov.b64 {a, b}, %1;\n mov.b64 {c, e}, %2;\n"
        " cvt.rn.satfinite.e5m2x2.f32 l, b, a;\n cvt.rn.satfinite.e5m2x2.f32 h, e, c;\n mov.b32 %0, {l, h};\n}"
        : "=r"(d) : "l"(p01), "l"(p23));
  else
    asm("{\n .reg .b16 l, h;\n .reg .f32 a, b, c, e;\n mov.b64 {a, b}, %1;\n mov.b64 {c, e}, %2;\n"
        " cvt.rn.satfinite.e4m3x2.f32 l, b, a;\n cvt.rn.satfinite.e4m3x2.f32 h, e, c;\n mov.b32 %0, {l, h};\n}"
        : "=r"(d) : "l"(p01), "l"(p23));
  return d;
}

// Four bf16 (two words) -> four FP8 codes; magnitudes from the exact quotients, signs from x.
template <int F>
__device__ __forceinline__ uint32_t exact_codes4(uint32_t w0, uint32_t w1, const ExactScale& k) {
  const uint32_t c = cvt_fp8x4<F>(exact_quotient2(w0, k), exact_quotient2(w1, k));
  return (c & 0x7F7F7F7Fu) | (__byte_perm(w0, w1, 0x7531) & 0x80808080u);
}

// Eight bf16 (a uint4) -> eight FP8 codes.
template <int F>
__device__ __forceinline__ uint2 exact_codes8(uint4 v, const ExactScale& k) {
  return make_uint2(exact_codes4<F>(v.x, v.y, k), exact_codes4<F>(v.z, v.w, k));
}

// Non-zero when a code word holds a NaN code (from a non-finite x or an fp32 overflow of x/s).
template <int F>
__device__ __forceinline__ uint32_t nan_code_bits(uint32_t c) {
  return ((c & 0x7F7F7F7Fu) + (F == kFmtE5M2 ? 0x04040404u : 0x01010101u)) & 0x80808080u;
}

// Eight values through the bracket-and-division path, out of line (rare callers).
template <int F>
__device__ __noinline__ uint2 quant8_bf16_slow(uint4 v, float s) {
  return quant8_bf16<F>(v, make_quantizer(s));
}

// Eight bf16 -> eight FP8 codes of fl32(x / s) for any s: the exact quotient when s is in its
// range, else (or when `check` and a NaN code shows a non-finite x or an overflowing quotient)
// the division path.
template <int F>
__device__ __forceinline__ uint2 quant8_exact(uint4 v, const ExactScale& k, float s, bool check) {
  if (k.fast) {
    const uint2 q = exact_codes8<F>(v, k);
    if (!check || (nan_code_bits<F>(q.x) | nan_code_bits<F>(q.y)) == 0) return q;
  }
  return quant8_bf16_slow<F>(v, s);
}

// scale = amax / 448 (57344 for e5m2) by IEEE fp32 division; 1 when amax is 0 (or the
// quotient underflows).
template <int F>
__device__ __forceinline__ float scale_from_amax(float amax) {
  const float s = __fdiv_rn(amax, fp8_max<F>());
  return s == 0.0f ? 1.0f : s;
}

// max |x| of the bf16 pairs in a 32-bit word, as two 16-bit magnitudes (sign bits cleared).
__device__ __forceinline__ uint32_t abs_max_u16x2(uint32_t acc, uint32_t w) {
  return __vmaxu2(acc, w & 0x7FFF7FFFu);
}

// max |x| over eight bf16 values (a uint4), folded into two 16-bit magnitudes.
__device__ __forceinline__ uint32_t abs_max_v4(uint32_t m2, uint4 v) {
  m2 = abs_max_u16x2(m2, v.x);
  m2 = abs_max_u16x2(m2, v.y);
  m2 = abs_max_u16x2(m2, v.z);
  return abs_max_u16x2(m2, v.w);
}

__device__ __forceinline__ float u16x2_max_to_float(uint32_t m2) {
  const uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
  return __uint_as_float(m << 16);
}

// ---------------------------------------------------------------------------
// Loads / reductions
// ---------------------------------------------------------------------------

// Streaming 16-byte load (read-only path, no L1 allocation).
__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Max over n non-negative partial amax values, by the whole block; result broadcast to all
// threads. `red` must hold blockDim.x/32 floats.
__device__ __forceinline__ float block_max_partials(const float* __restrict__ partials, int n, float* red) {
  float m = 0.0f;
  for (int i = threadIdx.x; i < n; i += blockDim.x) m = fmaxf(m, partials[i]);
  m = warp_max(m);
  const int w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  __syncthreads();  // `red` may still be in use by a previous reduction
  if ((threadIdx.x & 31) == 0) red[w] = m;
  __syncthreads();
  m = 0.0f;
  for (int i = 0; i < nw; ++i) m = fmaxf(m, red[i]);
  return m;
}

// Eight bf16 of row `row` starting at column k (k a multiple of 8), zero beyond K.
__device__ __forceinline__ uint4 load8_bf16(const uint16_t* row, int k, int K, int vec) {
  if (vec && k + 8 <= K) return ld_nc_v4(row + k);
  uint32_t w[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t lo = (k + 2 * j < K) ? row[k + 2 * j] : 0u;
    const uint32_t hi = (k + 2 * j + 1 < K) ? row[k + 2 * j + 1] : 0u;
    w[j] = lo | (hi << 16);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch
// ---------------------------------------------------------------------------

// Let the next kernel in the stream start launching; it still waits (pdl_wait) for our completion.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
// Wait until the preceding kernel in the stream has completed and its writes are visible.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete. Gives up (returns false) when
// *abort_flag becomes non-zero or after limit_ns (kWaitLimitNs by default); on a timeout it
// raises the abort flag and ORs kErrTimeout into *err so the host can report it. Never spins
// unbounded.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                                  unsigned int* err,
                                                  unsigned long long limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 15u) == 0) {
      if (abort_flag != nullptr && *abort_flag) return false;
      if (globaltimer_ns() - t0 > limit_ns) {
        if (abort_flag != nullptr) *abort_flag = 1;
        atomicOr(err, kErrTimeout);
        return false;
      }
    }
  }
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(bar), "r"(bytes) : "memory");
}

}  // namespace fp8k
