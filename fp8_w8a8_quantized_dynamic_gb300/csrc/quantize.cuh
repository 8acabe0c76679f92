// FP8 quantization kernels: amax reduction and the saturating RNE cast.
//
// Per-tensor scale ("Prototype FP8Linear W8A8 runtime quantization": weights and
// activations are quantized at run time; "Fp8 Quantization Support": symmetric,
// strategy "tensor"): s = amax / 448, q = e4m3(x / s). The format is a template
// parameter: e5m2 ("Fp8 Quantization Support", the other FP8 dtype) divides amax by
// 57344 instead. A static (calibrated) activation scale skips the amax pass.
// Per-output-channel scale ("[Kernel] Implement fallback for FP8 channelwise using
// torch._scaled_mm"): one s per row of W.
//
// The per-tensor amax is a two-step reduction with no atomics and no state that must
// start at zero: amax_partials_kernel writes one partial maximum per CTA into the
// workspace; every consumer CTA (the cast kernel, the GEMV) reduces those partials
// itself. Max is exact and order-free, so every CTA derives the identical scale.
#pragma once

#include "device_common.cuh"

namespace fp8k {

constexpr int kQuantThreads = 256;
// Resident cast CTAs per SM the register budget must allow (loads in flight keep HBM busy).
constexpr int kCastBlocksPerSM = 8;

// Cached 16-byte load (the row is read again shortly after).
__device__ __forceinline__ uint4 ld_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

// Block-wide max of a non-negative float; the result is valid in thread 0.
__device__ __forceinline__ float block_max_to_thread0(float v, float* red) {
  v = warp_max(v);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int i = 1; i < (int)(blockDim.x >> 5); ++i) v = fmaxf(v, red[i]);
  }
  return v;
}

// Max |x| over this thread's grid-stride share of a bf16 matrix [rows, cols] with row stride
// ld (elements), as two packed bf16 magnitudes. contiguous != 0: ld == cols and the base is
// 16-byte aligned (flat 16-byte loads). vec != 0: base 16-byte aligned and ld % 8 == 0.
__device__ __forceinline__ uint32_t amax_share(const uint16_t* __restrict__ a, int64_t rows, int64_t cols,
                                               int64_t ld, int contiguous, int vec) {
  uint32_t m2 = 0;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (contiguous) {
    const int64_t n = rows * cols;
    const int64_t n8 = n >> 3;
    const uint4* v = reinterpret_cast<const uint4*>(a);
    int64_t i = tid;
    for (; i + 3 * stride < n8; i += 4 * stride) {
      const uint4 v0 = ld_nc_v4(v + i), v1 = ld_nc_v4(v + i + stride);
      const uint4 v2 = ld_nc_v4(v + i + 2 * stride), v3 = ld_nc_v4(v + i + 3 * stride);
      m2 = abs_max_v4(abs_max_v4(m2, v0), v1);
      m2 = abs_max_v4(abs_max_v4(m2, v2), v3);
    }
    for (; i < n8; i += stride) m2 = abs_max_v4(m2, ld_nc_v4(v + i));
    if (blockIdx.x == 0)
      for (int64_t j = (n8 << 3) + threadIdx.x; j < n; j += blockDim.x) m2 = abs_max_u16x2(m2, a[j]);
  } else {
    const int64_t upr = (cols + 7) >> 3;  // 8-element units per row
    const int64_t units = rows * upr;
    for (int64_t u = tid; u < units; u += stride) {
      const int64_t r = u / upr;
      const int64_t c = (u - r * upr) << 3;
      const uint16_t* src = a + r * ld + c;
      if (vec && c + 8 <= cols) {
        m2 = abs_max_v4(m2, ld_nc_v4(src));
      } else {
        for (int j = 0; j < 8 && c + j < cols; ++j) m2 = abs_max_u16x2(m2, src[j]);
      }
    }
  }
  return m2;
}

// Partial max |x| over a bf16 matrix (see amax_share); writes partials[blockIdx.x].
// `pdl` lets the next kernel launch early (activations only).
__global__ void __launch_bounds__(kQuantThreads)
amax_partials_kernel(const uint16_t* __restrict__ a, int64_t rows, int64_t cols, int64_t ld,
                     int contiguous, int vec, float* __restrict__ partials, int pdl) {
  __shared__ float red[kQuantThreads / 32];
  if (pdl) pdl_trigger();
  pdl_wait();
  const uint32_t m2 = amax_share(a, rows, cols, ld, contiguous, vec);
  const float m = block_max_to_thread0(u16x2_max_to_float(m2), red);
  if (threadIdx.x == 0) partials[blockIdx.x] = m;
}

// Quantize 16 consecutive elements of one row (columns c .. c+15) into 16 FP8 bytes;
// columns >= cols give 0x00.
template <int F>
__device__ __forceinline__ uint4 quant16_row(const uint16_t* __restrict__ src, int64_t c, int64_t cols,
                                             bool vec, const Quantizer& s) {
  uint4 out;
  if (vec && c + 16 <= cols) {
    // pair by pair, each pair's rare division in its own branch: measured faster here than
    // the unit-wide form, which costs registers (occupancy) in this memory-bound loop
    const uint2 q0 = quant8_bf16_pairwise<F>(ld_v4(src), s);
    const uint2 q1 = quant8_bf16_pairwise<F>(ld_v4(src + 8), s);
    out = make_uint4(q0.x, q0.y, q1.x, q1.y);
  } else {
    float x[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) x[j] = (c + j < cols) ? bf16_bits_to_float(src[j]) : 0.0f;
    out.x = quant4<F>(x[0], x[1], x[2], x[3], s);
    out.y = quant4<F>(x[4], x[5], x[6], x[7], s);
    out.z = quant4<F>(x[8], x[9], x[10], x[11], s);
    out.w = quant4<F>(x[12], x[13], x[14], x[15], s);
  }
  return out;
}

// Sixteen values of one row starting at column c (c + 16 <= cols, 16-byte aligned source) by
// the exact quotient. kCheck: the scale does not bound the inputs (a caller-supplied scale),
// so a NaN code (non-finite x, or x / s beyond fp32) sends the unit to quant16_row, which
// saturates or keeps the NaN as the definition says.
template <int F, bool kCheck>
__device__ __forceinline__ uint4 quant16_exact(const uint16_t* __restrict__ src, const ExactScale& k, float s) {
  const uint4 v0 = ld_v4(src), v1 = ld_v4(src + 8);
  uint4 o = make_uint4(exact_codes4<F>(v0.x, v0.y, k), exact_codes4<F>(v0.z, v0.w, k),
                       exact_codes4<F>(v1.x, v1.y, k), exact_codes4<F>(v1.z, v1.w, k));
  if (kCheck && (nan_code_bits<F>(o.x) | nan_code_bits<F>(o.y) | nan_code_bits<F>(o.z) | nan_code_bits<F>(o.w)))
    o = quant16_row<F>(src, 0, 16, true, make_quantizer(s));
  return o;
}

// q[r, 0:ldq) = fp8(A[r, 0:cols) / s) with zero bytes for columns >= cols. Dynamic scale
// (partials != null): s = scale_from_amax(max of the n_partials partials). Static scale
// (partials == null): s = *s_static. CTA 0 stores s to *s_out unless s_out is null.
// For s in the exact quotient's range every 16-byte unit is quantized branch-free, the flat
// loop when both matrices are gap-free (ld == ldq == cols); ragged row ends, unaligned rows
// and scales outside that range take quant16_row (bracket, then division).
template <typename Idx, int F, bool kCheck>
__device__ __forceinline__ void cast_rows(const uint16_t* __restrict__ a, int64_t rows, int64_t cols, int64_t ld,
                                          int vec, float sc, uint8_t* __restrict__ q, int64_t ldq) {
  const ExactScale k = make_exact_scale(sc);
  const Idx upr = static_cast<Idx>(ldq >> 4);  // 16-byte output units per row
  const Idx units = static_cast<Idx>(rows) * upr;
  const Idx stride = static_cast<Idx>(gridDim.x) * blockDim.x;
  const Idx first = static_cast<Idx>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (k.fast && vec && ld == cols && ldq == cols) {
    uint4* dst = reinterpret_cast<uint4*>(q);
    for (Idx u = first; u < units; u += stride) dst[u] = quant16_exact<F, kCheck>(a + (int64_t(u) << 4), k, sc);
    return;
  }
  for (Idx u = first; u < units; u += stride) {
    const Idx r = u / upr;
    const int64_t c = static_cast<int64_t>(u - r * upr) << 4;
    const uint16_t* src = a + (int64_t)r * ld + c;
    *reinterpret_cast<uint4*>(q + (int64_t)r * ldq + c) =
        k.fast && vec && c + 16 <= cols ? quant16_exact<F, kCheck>(src, k, sc)
                                        : quant16_row<F>(src, c, cols, vec != 0, make_quantizer(sc));
  }
}

template <typename Idx, int F>
__global__ void __launch_bounds__(kQuantThreads, kCastBlocksPerSM)
cast_kernel(const uint16_t* __restrict__ a, int64_t rows, int64_t cols, int64_t ld, int vec,
            const float* __restrict__ partials, int n_partials, const float* __restrict__ s_static,
            float* __restrict__ s_out, uint8_t* __restrict__ q, int64_t ldq, int pdl) {
  __shared__ float red[kQuantThreads / 32];
  if (pdl) pdl_trigger();
  pdl_wait();
  const float sc = partials ? scale_from_amax<F>(block_max_partials(partials, n_partials, red)) : *s_static;
  if (s_out != nullptr && blockIdx.x == 0 && threadIdx.x == 0) *s_out = sc;
  // a dynamic scale bounds every |x| by amax, so x / s <= ~448 and no input is non-finite
  // (a non-finite amax gives a scale outside the exact range)
  if (partials)
    cast_rows<Idx, F, false>(a, rows, cols, ld, vec, sc, q, ldq);
  else
    cast_rows<Idx, F, true>(a, rows, cols, ld, vec, sc, q, ldq);
}

// Per-row (output channel) weight quantization: CTA per row, s_w[r] = amax(W[r,:]) / 448
// (57344 for e5m2). The row is read twice; the second read hits L1/L2.
template <int F>
__global__ void __launch_bounds__(kQuantThreads)
quantize_rows_kernel(const uint16_t* __restrict__ w, int64_t N, int64_t K, int64_t ld, int vec,
                     uint8_t* __restrict__ q, int64_t ldq, float* __restrict__ s_w) {
  __shared__ float red[kQuantThreads / 32];
  __shared__ float s_sh;
  pdl_wait();
  for (int64_t r = blockIdx.x; r < N; r += gridDim.x) {
    const uint16_t* row = w + r * ld;
    uint32_t m2 = 0;
    if (vec) {
      const int64_t k8 = K >> 3;
      for (int64_t i = threadIdx.x; i < k8; i += blockDim.x) m2 = abs_max_v4(m2, ld_v4(row + (i << 3)));
      for (int64_t j = (k8 << 3) + threadIdx.x; j < K; j += blockDim.x) m2 = abs_max_u16x2(m2, row[j]);
    } else {
      for (int64_t j = threadIdx.x; j < K; j += blockDim.x) m2 = abs_max_u16x2(m2, row[j]);
    }
    const float m = block_max_to_thread0(u16x2_max_to_float(m2), red);
    if (threadIdx.x == 0) {
      s_sh = scale_from_amax<F>(m);
      s_w[r] = s_sh;
    }
    __syncthreads();
    const float sr = s_sh;
    const ExactScale k = make_exact_scale(sr);  // |W[r, :]| <= amax: no input check needed
    for (int64_t c = (int64_t)threadIdx.x << 4; c < ldq; c += (int64_t)blockDim.x << 4)
      *reinterpret_cast<uint4*>(q + r * ldq + c) = k.fast && vec && c + 16 <= K
                                                       ? quant16_exact<F, false>(row + c, k, sr)
                                                       : quant16_row<F>(row + c, c, K, vec != 0, make_quantizer(sr));
    __syncthreads();  // s_sh and red are reused by the next row
  }
}

// Weight-only up-conversion ("Prototype FP8Linear W8A8 runtime quantization": without FP8
// tensor cores the FP8 weights are up-converted to the original dtype): wb[n, k] =
// bf16(decode(qw[n, k])) for k < K, exact; the weight scale is applied by the GEMM epilogue.
// Columns [K, ldwb) of wb are written as zero. ldwb: multiple of 8 elements.
template <int F>
__global__ void __launch_bounds__(kQuantThreads)
upconvert_kernel(const uint8_t* __restrict__ qw, int64_t N, int64_t K, int64_t ldqw, uint16_t* __restrict__ wb,
                 int64_t ldwb) {
  pdl_trigger();  // the GEMM that follows waits for this kernel before reading wb
  pdl_wait();     // wb may still be read by the previous call's GEMM
  const int64_t upr = ldwb >> 3;  // 8-element (16-byte output) units per row
  const int64_t units = N * upr;
  for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < units; u += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = u / upr;
    const int64_t c = (u - r * upr) << 3;
    uint2 codes = make_uint2(0, 0);
    if (c < K) codes = *reinterpret_cast<const uint2*>(qw + r * ldqw + c);  // ldqw % 16 == 0, c % 8 == 0
    // bytes [K, ldqw) of a quantized row are zero, which up-converts to +0 as required
    uint4 out;
    out.x = fp8x2_to_bf16x2<F>(codes.x);
    out.y = fp8x2_to_bf16x2<F>(codes.x >> 16);
    out.z = fp8x2_to_bf16x2<F>(codes.y);
    out.w = fp8x2_to_bf16x2<F>(codes.y >> 16);
    *reinterpret_cast<uint4*>(wb + r * ldwb + c) = out;
  }
}

// Copy of bf16 A [rows, cols] (any stride) into a 16-byte-aligned buffer with stride ldo
// (a multiple of 8 elements), zero in columns [cols, ldo): the layout TMA needs.
__global__ void __launch_bounds__(kQuantThreads)
copy_rows_bf16_kernel(const uint16_t* __restrict__ a, int64_t rows, int64_t cols, int64_t ld, int vec,
                      uint16_t* __restrict__ out, int64_t ldo, int pdl) {
  if (pdl) pdl_trigger();
  pdl_wait();
  const int64_t upr = ldo >> 3;
  const int64_t units = rows * upr;
  for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < units; u += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = u / upr;
    const int c = int((u - r * upr) << 3);
    *reinterpret_cast<uint4*>(out + r * ldo + c) = load8_bf16(a + r * ld, c, int(cols), vec);
  }
}

// Y[m, :] = bias (or 0) for all m: the K == 0 product.
__global__ void fill_bias_kernel(const uint16_t* __restrict__ bias, uint16_t* __restrict__ y,
                                 int64_t M, int64_t N, int64_t ldy, int pdl) {
  if (pdl) pdl_trigger();
  pdl_wait();
  const int64_t total = M * N;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t m = i / N, n = i - m * N;
    y[m * ldy + n] = bias ? bias[n] : uint16_t(0);
  }
}

}  // namespace fp8k
