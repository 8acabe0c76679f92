// Decode-shape FP8 GEMV: Y[M<=16, N] = bf16(s_a * s_w[n] * sum_k qA[m,k] qW[n,k] (+ bias[n])).
//
// "[WIP] FP8 support": LLM decode runs at sequence length < 16 (the batch), which calls
// for a custom gemv rather than a 16-padded GEMM. The weight matrix is streamed from HBM
// exactly once; everything else is small.
//
// Decomposition. A CTA owns 128 weight rows (8 warps x 16 rows) and one K-slice. The
// K-slices of one row block form a thread-block cluster (up to 8 CTAs); their fp32
// partial sums are combined through distributed shared memory in a fixed order, so the
// result is deterministic and no global scratch is needed.
//
// Tensor-core mapping (mma.sync m16n8k32, e4m3 x e4m3 -> f32): W rows are the MMA's M
// dimension, tokens its N dimension (one n8 tile for M <= 8, two for M <= 16). The sum over
// k is order-free, so the k order inside each 64-byte chunk is permuted such that a lane
// (group g, thread t) feeds both MMAs of the chunk from ONE 16-byte load of W row g
// (bytes 16t..16t+15) and one of row g+8: weights are read with fully used 16-byte loads
// straight into registers. The activation fragment uses the same permutation, which is
// simply row-major [token][k] in shared memory.
//
// Activations: with the dynamic path each CTA quantizes its own K-slice of A into shared
// memory (scale from the partial amax values the amax kernel left in the workspace).
// Weight loads for the first chunks are issued before waiting on the preceding kernel.
#pragma once

#include "device_common.cuh"

namespace fp8k {
namespace gemv {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kRowsPerCta = kWarps * 16;
constexpr int kChunk = 64;        // bytes of K consumed per lane-group step (two k32 MMAs)
constexpr int kUnroll = 4;        // chunks per register group
constexpr int kMaxTokens = 16;
constexpr int kMaxCluster = 8;
constexpr int kMaxSlice = 4096;   // bytes of K per CTA (shared-memory bound)

struct Params {
  const void* a;            // bf16 [M, lda] (dynamic) or e4m3 [M, lda] (pre-quantized)
  int64_t lda;
  const float* partials;    // dynamic: partial amax values
  int n_partials;
  const float* s_a;         // pre-quantized: activation scale (device)
  const uint8_t* qw;        // e4m3 [N, ldqw]
  int64_t ldqw;
  const float* s_w;         // [1] or [N]
  int per_channel;
  const uint16_t* bias;     // bf16 [N] or null
  uint16_t* y;              // bf16 [M, ldy]
  int64_t ldy;
  int M, N, K;
  int kslice;               // bytes of K per CTA, multiple of kChunk
  int act_stride;           // shared-memory row stride of the activation tile (== 64 mod 128)
  int vec_a;                // bf16 A rows allow 16-byte loads
};

__device__ __forceinline__ void mma_e4m3(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint4 lds_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

__device__ __forceinline__ float ld_dsmem_f32(uint32_t local_addr, uint32_t rank) {
  uint32_t remote;
  float v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank));
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
  return v;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}

// One group of kUnroll chunks of W for rows g and g+8 of this warp's 16-row tile.
struct WGroup {
  uint4 lo[kUnroll];  // row g
  uint4 hi[kUnroll];  // row g + 8
};

// Loads chunk u of the group at slice offset kbyte0 + u*kChunk when that offset is < lim.
__device__ __forceinline__ void load_wgroup(WGroup& w, const uint8_t* row_lo, const uint8_t* row_hi,
                                            bool ok_lo, bool ok_hi, int kbyte0, int lim) {
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) {
    const int k = kbyte0 + u * kChunk;
    const bool in_k = k < lim;
    w.lo[u] = (ok_lo && in_k) ? ld_nc_v4(row_lo + k) : make_uint4(0, 0, 0, 0);
    w.hi[u] = (ok_hi && in_k) ? ld_nc_v4(row_hi + k) : make_uint4(0, 0, 0, 0);
  }
}

template <int NT>
__device__ __forceinline__ void mma_wgroup(float (&acc)[NT][4], const WGroup& w, uint32_t act_base,
                                           int act_stride, int chunk0, int nchunks) {
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) {
    if (chunk0 + u < nchunks) {  // warp-uniform
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const uint4 b = lds_v4(act_base + nt * 8 * act_stride + (chunk0 + u) * kChunk);
        mma_e4m3(acc[nt], w.lo[u].x, w.hi[u].x, w.lo[u].y, w.hi[u].y, b.x, b.y);
        mma_e4m3(acc[nt], w.lo[u].z, w.hi[u].z, w.lo[u].w, w.hi[u].w, b.z, b.w);
      }
    }
  }
}

// NT: number of n8 token tiles (1: M <= 8, 2: M <= 16). kDynamic: A is bf16 and is
// quantized here with the scale derived from the partial amax values; otherwise A is
// already e4m3 and s_a is read from memory.
template <int NT, bool kDynamic>
__global__ void __launch_bounds__(kThreads)
gemv_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ float red[kWarps];
  __shared__ float s_a_sh;

  uint8_t* act = smem;  // [NT*8][act_stride] e4m3
  float* part = reinterpret_cast<float*>(smem + NT * 8 * p.act_stride);  // [128][16] fp32 partial sums

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int row_lo = blockIdx.x * kRowsPerCta + warp * 16 + g;
  const int row_hi = row_lo + 8;
  const int k0 = blockIdx.y * p.kslice;
  const int kend16 = (p.K + 15) & ~15;                      // W bytes [K, kend16) are zero
  const int klen = max(0, min(p.kslice, kend16 - k0));
  const int nchunks = (klen + kChunk - 1) / kChunk;

  pdl_trigger();

  // --- weights do not depend on the preceding kernel: start streaming them now
  const uint8_t* wlo = p.qw + (int64_t)row_lo * p.ldqw + k0 + 16 * t;
  const uint8_t* whi = p.qw + (int64_t)row_hi * p.ldqw + k0 + 16 * t;
  const bool ok_lo = row_lo < p.N, ok_hi = row_hi < p.N;
  // a lane's 16-byte load at slice offset x is valid if x < lim: inside the row's K16
  // bytes and inside this CTA's chunks (never prefetch the next slice's bytes)
  const int lim = min(kend16 - k0, nchunks * kChunk) - 16 * t;
  WGroup cur;
  load_wgroup(cur, wlo, whi, ok_lo, ok_hi, 0, lim);

  pdl_wait();

  // --- activation scale
  if constexpr (kDynamic) {
    const float amax = block_max_partials(p.partials, p.n_partials, red);
    if (threadIdx.x == 0) s_a_sh = scale_from_amax(amax);
  } else {
    if (threadIdx.x == 0) s_a_sh = *p.s_a;
  }
  __syncthreads();
  const float s_a = s_a_sh;

  // --- stage this CTA's K-slice of the activations into shared memory as e4m3
  {
    const int span = nchunks * kChunk;
    const int units_per_tok = span >> 3;  // 8 bytes per unit
    const int units = NT * 8 * units_per_tok;
    for (int i = threadIdx.x; i < units; i += kThreads) {
      const int m = i / units_per_tok;
      const int kk = (i - m * units_per_tok) << 3;
      const int k = k0 + kk;
      uint2 q = make_uint2(0, 0);
      if (m < p.M && k < p.K) {
        if constexpr (kDynamic) {
          const uint16_t* src = static_cast<const uint16_t*>(p.a) + (int64_t)m * p.lda + k;
          if (p.vec_a && k + 8 <= p.K) {
            q = quant8_bf16(ld_nc_v4(src), s_a);
          } else {
            float x[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) x[j] = (k + j < p.K) ? bf16_bits_to_float(src[j]) : 0.0f;
            q.x = quant4(x[0], x[1], x[2], x[3], s_a);
            q.y = quant4(x[4], x[5], x[6], x[7], s_a);
          }
        } else {
          // e4m3 rows: ld is a multiple of 16 and bytes [K, ld) are zero
          q = *reinterpret_cast<const uint2*>(static_cast<const uint8_t*>(p.a) + (int64_t)m * p.lda + k);
        }
      }
      *reinterpret_cast<uint2*>(act + m * p.act_stride + kk) = q;
    }
  }
  __syncthreads();

  // --- main loop: stream W, tensor-core dot products against the resident activations
  float acc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.0f;
  const uint32_t act_base = smem_u32(act) + g * p.act_stride + 16 * t;
  for (int c = 0; c < nchunks; c += kUnroll) {
    WGroup nxt;
    const bool more = c + kUnroll < nchunks;
    if (more) load_wgroup(nxt, wlo, whi, ok_lo, ok_hi, (c + kUnroll) * kChunk, lim);
    mma_wgroup<NT>(acc, cur, act_base, p.act_stride, c, nchunks);
    if (more) cur = nxt;
  }

  // --- partial sums -> shared memory: part[row][token]
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int r = warp * 16 + g, col = nt * 8 + 2 * t;
    part[r * kMaxTokens + col] = acc[nt][0];
    part[r * kMaxTokens + col + 1] = acc[nt][1];
    part[(r + 8) * kMaxTokens + col] = acc[nt][2];
    part[(r + 8) * kMaxTokens + col + 1] = acc[nt][3];
  }
  cluster_sync_all();

  // --- split-K reduction across the cluster (fixed order) + epilogue
  const uint32_t rank = cluster_ctarank(), nrank = cluster_nctarank();
  const int rows_per = (kRowsPerCta + nrank - 1) / nrank;
  const int r_begin = rank * rows_per;
  const int r_count = max(0, min(kRowsPerCta, r_begin + rows_per) - r_begin);
  const uint32_t part_base = smem_u32(part);
  for (int i = threadIdx.x; i < r_count * p.M; i += kThreads) {
    const int m = i / r_count;
    const int rl = r_begin + (i - m * r_count);
    const int n = blockIdx.x * kRowsPerCta + rl;
    if (n >= p.N) continue;
    const uint32_t off = (rl * kMaxTokens + m) * 4;
    float sum = 0.0f;
    for (uint32_t q = 0; q < nrank; ++q) sum += ld_dsmem_f32(part_base + off, q);
    const float sw = p.s_w[p.per_channel ? n : 0];
    const float b = p.bias ? bf16_bits_to_float(p.bias[n]) : 0.0f;
    const float yv = fmaf(sum, s_a * sw, b);
    p.y[(int64_t)m * p.ldy + n] = __bfloat16_as_ushort(__float2bfloat16_rn(yv));
  }
  cluster_sync_all();  // peers may still be reading our partials
}

}  // namespace gemv
}  // namespace fp8k
