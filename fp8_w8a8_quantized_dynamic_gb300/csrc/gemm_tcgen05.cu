// Prefill FP8 GEMM for sm_103a on the 5th-generation tensor cores.
//
//   Y[m, n] = bf16( s_a * s_w[n] * sum_k qA[m, k] qW[n, k]  (+ bias[n]) )
//
// The W8A8 product the pages run through torch._scaled_mm / CUTLASS ("Prototype FP8Linear
// W8A8 runtime quantization"; "[Kernel] Implement fallback for FP8 channelwise using
// torch._scaled_mm"), with the channelwise rescale s_a*s_w[n] applied to the fp32
// accumulator in the epilogue: (s_a A)(s_w,n W_n)^T = s_a s_w,n (A W_n^T). qA and qW are
// each e4m3 or e5m2 ("Fp8 Quantization Support"): the operand formats are fields of the
// MMA instruction descriptor, so one kernel serves every pairing.
//
// The same kernel, instantiated with kBf16, runs the weight-only product (bf16 A times the
// up-converted bf16 weights, "Prototype FP8Linear W8A8 runtime quantization") on
// tcgen05.mma kind::f16: a stage still holds 128-byte rows, now of 64 bf16 elements, and
// one MMA still consumes 32 bytes of K (16 elements), so tiles, descriptors and the ring
// are unchanged.
//
// Structure (one CTA per SM, persistent over output tiles of 128 x 256):
//   warp 0      TMA producer: qA tile [128 x 128B] and qW tile [256 x 128B] per stage into a
//               4-stage ring of 128B-swizzled shared memory, completion on an mbarrier.
//   warp 1      TMEM allocator + MMA issuer: tcgen05.mma.cta_group::1.kind::f8f6f4,
//               M=128 N=256 K=32, fp32 accumulators in TMEM, two accumulator buffers of 256
//               columns so the epilogue of tile i overlaps the main loop of tile i+1.
//   warps 2..5  epilogue: tcgen05.ld 32 columns at a time, scale (+bias), bf16, store.
// Ragged M, N and K need no padding: TMA fills out-of-range rows/columns with zeros and
// the epilogue predicates its stores.
//
// Paired mode (kPair, a cluster of two CTAs on row blocks 2i and 2i+1 of the same column
// tile): the 256-row weight tile is shared. Each CTA loads its own qA tile and one half of
// the weight tile, the half multicast into both CTAs' shared memory, so the L2 -> SM traffic
// per tile drops from 48 KB to 32 KB per stage (the single-CTA kernel reads ~19 TB/s from
// L2 at 73 % of its request peak). Each stage's empty barrier then counts the MMA commits of
// both CTAs (a CTA's multicast half overwrites the peer's stage too), and the two CTAs run
// the same tile sequence with the same number of k-blocks.
//
// Every wait is bounded (2 s); on expiry the kernel records an error for the host, drains
// its own outstanding copies and MMAs (again bounded), frees its TMEM and returns.

#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <map>
#include <mutex>

#include "device_common.cuh"
#include "gemm_tcgen05.h"

namespace fp8k {
namespace gemm {

__device__ unsigned int g_gemm_error;

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 128;  // bytes of K per stage: one 128-byte swizzle row (128 FP8 / 64 bf16 elements)
constexpr int kStages = 4;
constexpr int kAccBufs = 2;
constexpr int kTmemCols = kAccBufs * BN;  // 512: the whole tensor memory of the SM
constexpr int kThreads = 192;
constexpr int kEpiThreads = 128;
constexpr uint32_t kABytes = BM * BK;
constexpr uint32_t kBBytes = BN * BK;
constexpr uint32_t kStageBytes = kABytes + kBBytes;
constexpr int kMmaK = 32;  // bytes of K of one MMA (32 FP8 elements, kind::f8f6f4; 16 bf16, kind::f16)

struct SharedCtl {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t tfull[kAccBufs];
  uint64_t tempty[kAccBufs];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  float colscale[kAccBufs][BN];
  float colbias[kAccBufs][BN];
};

constexpr size_t kSmemBytes = 1024 /*alignment slack*/ + kStages * kStageBytes + sizeof(SharedCtl);

// Instruction descriptor, kind::f8f6f4: D fp32 (bits 4-5 = 1), A and B format at bits 7-9 and
// 10-12 (e4m3 = 0, e5m2 = 1), both K-major (bits 15, 16 = 0), N >> 3 at bits 17-22, M >> 4 at
// bits 24-28.
constexpr uint32_t kIdescBase = (1u << 4) | (uint32_t(BN >> 3) << 17) | (uint32_t(BM >> 4) << 24);

constexpr uint32_t make_idesc(int fmt_a, int fmt_w) {
  return kIdescBase | (uint32_t(fmt_a) << 7) | (uint32_t(fmt_w) << 10);
}

// kind::f16 with bf16 A and B: the format fields hold BF16 = 1.
constexpr uint32_t kIdescBf16 = kIdescBase | (1u << 7) | (1u << 10);

// Shared-memory matrix descriptor for a K-major operand tile written by TMA with 128-byte
// swizzle: rows of 128 bytes, 8-row swizzle atoms of 1024 bytes (stride byte offset), start
// address >> 4 in bits 0-13, descriptor version 1 at bit 46, swizzle mode 2 (128B) at bits 61-63.
// The leading byte offset is unused for swizzled K-major layouts (set to 1).
__device__ __forceinline__ uint64_t make_sdesc(uint32_t saddr) {
  uint64_t d = 0;
  d |= uint64_t((saddr & 0x3FFFFu) >> 4);
  d |= uint64_t(1) << 16;
  d |= uint64_t(1024 >> 4) << 32;
  d |= uint64_t(1) << 46;
  d |= uint64_t(2) << 61;
  return d;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];"
      :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y) : "memory");
}

template <bool kBf16>
__device__ __forceinline__ void mma_issue(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  if constexpr (kBf16)
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        :: "r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
  else
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}"
        :: "r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" :: "r"(bar) : "memory");
}

// Multicast forms for the paired mode: the copy lands at the same shared-memory offset in
// every CTA of `mask` and completes bytes on the mbarrier at the same offset in each; the
// commit arrives once on that mbarrier in each CTA of `mask`.
__device__ __forceinline__ void tma_load_2d_mc(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y,
                                               uint16_t mask) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.multicast::cluster"
      " [%0], [%1, {%3, %4}], [%2], %5;"
      :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "h"(mask) : "memory");
}

__device__ __forceinline__ void mma_commit_mc(uint32_t bar, uint16_t mask) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
               :: "r"(bar), "h"(mask) : "memory");
}

__device__ __forceinline__ uint32_t pair_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Every thread of both CTAs: barrier inits visible before the first multicast, and no CTA
// leaves while its peer may still write into its shared memory or arrive on its barriers.
__device__ __forceinline__ void pair_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tmem_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Named barrier over the 128 epilogue threads that also ORs a flag across them, so every
// epilogue warp takes the same exit decision.
__device__ __forceinline__ bool epi_bar_any(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, %2, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r) : "r"(uint32_t(v)), "n"(kEpiThreads) : "memory");
  return r != 0;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  return uint32_t(__bfloat16_as_ushort(__float2bfloat16_rn(lo))) |
         (uint32_t(__bfloat16_as_ushort(__float2bfloat16_rn(hi))) << 16);
}

// Tile order: groups of `group_n` column tiles; inside a group the column index runs fastest,
// so the CTAs resident at one time share a few qA row blocks and a W slice that stays in L2
// while the group sweeps all rows: W is read from HBM once, qA once per group.
__device__ __forceinline__ void tile_coords(int tile, const GemmParams& p, int m_units, int& m_idx, int& n_idx) {
  const int per_group = p.group_n * m_units;
  const int gidx = tile / per_group;
  const int r = tile - gidx * per_group;
  const int n_first = gidx * p.group_n;
  const int gn = min(p.group_n, p.n_tiles - n_first);
  m_idx = r / gn;
  n_idx = n_first + (r - m_idx * gn);
}

// kBf16: operands are bf16 (weight-only product) instead of FP8. kPair: clusters of two CTAs
// sharing the weight tile (see the paired mode above).
template <bool kBf16, bool kPair>
__global__ void __launch_bounds__(kThreads, 1)
gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
            const __grid_constant__ GemmParams p) {
  constexpr int kElemsPerStage = kBf16 ? BK / 2 : BK;  // K elements per stage
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);  // 1024-aligned for the 128B swizzle
  SharedCtl* ctl = reinterpret_cast<SharedCtl*>(smem + kStages * kStageBytes);
  const uint32_t smem_base = smem_u32(smem);
  auto a_stage = [&](int s) { return smem_base + s * kStageBytes; };
  auto b_stage = [&](int s) { return smem_base + s * kStageBytes + kABytes; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // work units: tiles, or (paired) vertical tile pairs; rank r of a pair takes row block 2i + r
  const uint32_t rank = kPair ? pair_rank() : 0u;
  const int m_units = kPair ? (p.m_tiles + 1) / 2 : p.m_tiles;
  const int num_tiles = m_units * p.n_tiles;
  const int first_unit = kPair ? int(blockIdx.x >> 1) : int(blockIdx.x);
  const int unit_stride = kPair ? int(gridDim.x >> 1) : int(gridDim.x);
  auto coords = [&](int unit, int& m_idx, int& n_idx) {
    tile_coords(unit, p, m_units, m_idx, n_idx);
    if (kPair) m_idx = 2 * m_idx + int(rank);
  };
  const int num_kb = (p.K + kElemsPerStage - 1) / kElemsPerStage;
  volatile int* abort_flag = &ctl->abort_flag;

  if (threadIdx.x == 0) {
    asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&tmap_a)) : "memory");
    asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&tmap_b)) : "memory");
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&ctl->full[s]), 1);
      mbar_init(smem_u32(&ctl->empty[s]), kPair ? 2 : 1);  // paired: both CTAs' MMAs read the stage
    }
    for (int b = 0; b < kAccBufs; ++b) {
      mbar_init(smem_u32(&ctl->tfull[b]), 1);
      mbar_init(smem_u32(&ctl->tempty[b]), kEpiThreads);
    }
    mbar_init(smem_u32(&ctl->drain), 1);
    ctl->abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_u32(&ctl->tmem_base)), "n"(kTmemCols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tmem_fence_before();
  __syncthreads();
  if (kPair) pair_sync();  // the peer's barriers exist before the first multicast lands there
  tmem_fence_after();
  const uint32_t tmem_base = ctl->tmem_base;

  pdl_trigger();
  pdl_wait();  // qA / s_a come from the preceding kernel; Y may still be read by it

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      uint32_t it = 0;
      bool ok = true;
      for (int tile = first_unit; tile < num_tiles && ok; tile += unit_stride) {
        int m_idx, n_idx;
        coords(tile, m_idx, n_idx);
        for (int kb = 0; kb < num_kb; ++kb, ++it) {
          const int s = it % kStages;
          const uint32_t ph = (it / kStages) & 1u;
          if (!mbar_wait_bounded(smem_u32(&ctl->empty[s]), ph ^ 1u, abort_flag, &g_gemm_error)) { ok = false; break; }
          const uint32_t fb = smem_u32(&ctl->full[s]);
          mbar_arrive_expect_tx(fb, kStageBytes);
          tma_load_2d(a_stage(s), &tmap_a, fb, kb * kElemsPerStage, m_idx * BM);
          if (kPair)  // this CTA's half of the weight tile, into both CTAs
            tma_load_2d_mc(b_stage(s) + rank * (kBBytes / 2), &tmap_b, fb, kb * kElemsPerStage,
                           n_idx * BN + int(rank) * (BN / 2), uint16_t(0x3));
          else
            tma_load_2d(b_stage(s), &tmap_b, fb, kb * kElemsPerStage, n_idx * BN);
        }
      }
      if (!ok) {
        // drain: the last fill of every stage must land before the CTA's memory is released
        const uint32_t first = it > (uint32_t)kStages ? it - kStages : 0u;
        for (uint32_t j = first; j < it; ++j)
          mbar_wait_bounded(smem_u32(&ctl->full[j % kStages]), (j / kStages) & 1u, nullptr, &g_gemm_error);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      uint32_t it = 0, acc_it = 0;
      bool ok = true;
      for (int tile = first_unit; tile < num_tiles && ok; tile += unit_stride, ++acc_it) {
        const int ab = acc_it % kAccBufs;
        const uint32_t aph = (acc_it / kAccBufs) & 1u;
        if (!mbar_wait_bounded(smem_u32(&ctl->tempty[ab]), aph ^ 1u, abort_flag, &g_gemm_error)) { ok = false; break; }
        tmem_fence_after();
        const uint32_t d_tmem = tmem_base + ab * BN;
        for (int kb = 0; kb < num_kb; ++kb, ++it) {
          const int s = it % kStages;
          const uint32_t ph = (it / kStages) & 1u;
          if (!mbar_wait_bounded(smem_u32(&ctl->full[s]), ph, abort_flag, &g_gemm_error)) { ok = false; break; }
          tmem_fence_after();
          const uint64_t adesc = make_sdesc(a_stage(s));
          const uint64_t bdesc = make_sdesc(b_stage(s));
#pragma unroll
          for (int kk = 0; kk < BK / kMmaK; ++kk) {
            // advance the start address by 32 bytes of K inside the swizzled 128-byte row
            mma_issue<kBf16>(d_tmem, adesc + uint64_t(kk * kMmaK >> 4), bdesc + uint64_t(kk * kMmaK >> 4),
                             p.idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          // frees the stage once these MMAs have read it (in both CTAs' counts when paired)
          if (kPair)
            mma_commit_mc(smem_u32(&ctl->empty[s]), uint16_t(0x3));
          else
            mma_commit(smem_u32(&ctl->empty[s]));
        }
        if (!ok) break;
        mma_commit(smem_u32(&ctl->tfull[ab]));   // accumulator ready for the epilogue
      }
      // all MMAs issued by this thread must finish before TMEM is released
      mma_commit(smem_u32(&ctl->drain));
      mbar_wait_bounded(smem_u32(&ctl->drain), 0, nullptr, &g_gemm_error);
    }
  } else {
    // ---------------- epilogue: warps 2..5 ----------------
    const int q = warp & 3;                    // TMEM lane quarter this warp may access
    const int row_in_tile = q * 32 + lane;
    const int et = threadIdx.x - 64;           // 0..127
    const float s_a = p.s_a ? *p.s_a : 1.0f;
    uint32_t acc_it = 0;
    for (int tile = first_unit; tile < num_tiles; tile += unit_stride, ++acc_it) {
      int m_idx, n_idx;
      coords(tile, m_idx, n_idx);
      const int ab = acc_it % kAccBufs;
      const uint32_t aph = (acc_it / kAccBufs) & 1u;
      // column scales/bias of this tile, double-buffered by accumulator: a warp can only
      // rewrite buffer ab after every epilogue warp passed the barrier of the tile between.
      for (int j = et; j < BN; j += kEpiThreads) {
        const int n = n_idx * BN + j;
        float sc = 0.0f, bb = 0.0f;
        if (n < p.N) {
          sc = s_a * p.s_w[p.per_channel ? n : 0];
          bb = p.bias ? bf16_bits_to_float(p.bias[n]) : 0.0f;
        }
        ctl->colscale[ab][j] = sc;
        ctl->colbias[ab][j] = bb;
      }
      // publishes the column tables; a set abort flag makes all epilogue warps leave together
      if (epi_bar_any(*abort_flag != 0)) break;
      // after a timeout, skip to the next barrier above, which ends the loop uniformly
      // one lane waits and the warp follows its verdict: tcgen05.ld needs a converged warp
      bool ok = lane == 0 ? mbar_wait_bounded(smem_u32(&ctl->tfull[ab]), aph, abort_flag, &g_gemm_error) : true;
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) continue;
      tmem_fence_after();
      const int m = m_idx * BM + row_in_tile;
      uint16_t* yrow = p.y + (int64_t)m * p.ldy;
      const uint32_t tbase = tmem_base + (uint32_t(q * 32) << 16) + ab * BN;
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        const int n0 = n_idx * BN + c * 32;
        if (n0 >= p.N) break;  // warp-uniform
        uint32_t r[32];
        tmem_ld32(tbase + c * 32, r);
        if (m < p.M) {
          const float* cs = &ctl->colscale[ab][c * 32];
          const float* cb = &ctl->colbias[ab][c * 32];
          if (p.y_vec && n0 + 32 <= p.N) {
            uint4* dst = reinterpret_cast<uint4*>(yrow + n0);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              uint32_t w[4];
#pragma unroll
              for (int h = 0; h < 4; ++h) {
                const int j = v * 8 + h * 2;
                w[h] = pack_bf16x2(fmaf(__uint_as_float(r[j]), cs[j], cb[j]),
                                   fmaf(__uint_as_float(r[j + 1]), cs[j + 1], cb[j + 1]));
              }
              dst[v] = make_uint4(w[0], w[1], w[2], w[3]);
            }
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              if (n0 + j < p.N)
                yrow[n0 + j] = __bfloat16_as_ushort(
                    __float2bfloat16_rn(fmaf(__uint_as_float(r[j]), cs[j], cb[j])));
            }
          }
        }
      }
      tmem_fence_before();
      mbar_arrive(smem_u32(&ctl->tempty[ab]));
    }
  }

  __syncwarp();
  tmem_fence_before();
  __syncthreads();
  if (kPair) pair_sync();  // the peer's last multicast copies and commit arrivals are done
  tmem_fence_after();
  if (warp == 1) {
    __syncwarp();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(tmem_base), "n"(kTmemCols) : "memory");
  }
}

}  // namespace gemm
}  // namespace fp8k

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<EncodeTiledFn>(nullptr);
    return reinterpret_cast<EncodeTiledFn>(ptr);
  }();
  return fn;
}

}  // namespace

namespace fp8k {

// 2-D tensor map over a row-major matrix [rows, K] of FP8 bytes or bf16 elements (row stride
// ld bytes), box [box_rows rows x 128 bytes], 128-byte swizzle, zero fill outside the matrix.
static bool make_tensor_map(CUtensorMap* map, const void* base, bool bf16, int64_t rows, int64_t K, int64_t ld,
                            uint32_t box_rows) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {cuuint64_t(K), cuuint64_t(rows)};
  const cuuint64_t strides[1] = {cuuint64_t(ld)};
  const cuuint32_t box[2] = {uint32_t(bf16 ? fp8k::gemm::BK / 2 : fp8k::gemm::BK), box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
             const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_fp8_tensor_map(CUtensorMap* map, const uint8_t* base, int64_t rows, int64_t K, int64_t ld, uint32_t box_rows) {
  return make_tensor_map(map, base, false, rows, K, ld, box_rows);
}

namespace {

// Resident clusters of two for the paired kernel (cached per kernel): clusters must fit in
// one GPC, so GPCs with an odd number of free SMs leave one SM out.
int pair_clusters(const void* kernel, cudaLaunchConfig_t cfg) {
  static std::mutex mu;
  static std::map<const void*, int> cache;
  std::lock_guard<std::mutex> g(mu);
  auto it = cache.find(kernel);
  if (it != cache.end()) return it->second;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(2 * 64);  // any multiple of the cluster size
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  if (std::getenv("FP8W8A8_DEBUG")) std::fprintf(stderr, "fp8w8a8: gemm pairs resident: %d clusters of 2\n", n);
  cache[kernel] = n;
  return n;
}

// Paired (cluster) mode unless FP8W8A8_GEMM_PAIR=0, there is only one row block, or fewer
// than 3/4 of the SMs could run pairs.
bool pair_enabled() {
  static const bool on = [] {
    const char* e = std::getenv("FP8W8A8_GEMM_PAIR");
    return !(e && e[0] == '0');
  }();
  return on;
}

template <bool kBf16>
int launch_kind(const void* a, int64_t lda_bytes, const float* s_a, const void* w, int64_t ldw_bytes,
                const float* s_w, int per_channel, const uint16_t* bias, uint16_t* y, int64_t ldy, int M, int N,
                int K, uint32_t idesc, int num_sms, cudaStream_t stream) {
  using namespace gemm;
  auto single = gemm_kernel<kBf16, false>;
  auto paired = gemm_kernel<kBf16, true>;
  static bool attr_done = false;  // the attribute is per function, set once per process
  if (!attr_done) {
    if (cudaFuncSetAttribute(single, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kSmemBytes)) != cudaSuccess ||
        cudaFuncSetAttribute(paired, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kSmemBytes)) != cudaSuccess ||
        cudaFuncSetAttribute(paired, cudaFuncAttributeNonPortableClusterSizeAllowed, 0) != cudaSuccess)
      return 1;
    attr_done = true;
  }

  GemmParams p;
  p.M = M;
  p.N = N;
  p.K = K;
  p.s_a = s_a;
  p.s_w = s_w;
  p.per_channel = per_channel;
  p.bias = bias;
  p.y = y;
  p.ldy = ldy;
  p.m_tiles = (M + BM - 1) / BM;
  p.n_tiles = (N + BN - 1) / BN;
  p.y_vec = (ldy % 8 == 0) && (reinterpret_cast<uintptr_t>(y) % 16 == 0);
  p.idesc = idesc;

  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  int clusters = 0;
  if (pair_enabled() && p.m_tiles >= 2) {
    clusters = pair_clusters(reinterpret_cast<const void*>(paired), cfg);
    if (2 * clusters < (3 * num_sms) / 4) clusters = 0;
  }
  const bool pair = clusters > 0;
  const int m_units = pair ? (p.m_tiles + 1) / 2 : p.m_tiles;
  // raster: a group of column tiles whose W slice (~26 MB) stays hot in L2 while the group
  // sweeps all rows; qA is then read once per group. Larger hot sets were measured to be
  // evicted by the streaming qA and Y traffic.
  const int64_t slice_budget = int64_t(26) << 20;
  const int64_t w_tile_bytes = int64_t(BN) * ldw_bytes;
  p.group_n = int(std::max<int64_t>(1, std::min<int64_t>(p.n_tiles, slice_budget / w_tile_bytes)));

  CUtensorMap ma, mb;
  if (!make_tensor_map(&ma, a, kBf16, M, K, lda_bytes, BM) ||
      !make_tensor_map(&mb, w, kBf16, N, K, ldw_bytes, pair ? BN / 2 : BN))
    return 2;

  const int units = m_units * p.n_tiles;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  if (pair) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 2;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
    cfg.gridDim = dim3(2 * unsigned(std::min(units, clusters)));
    return cudaLaunchKernelEx(&cfg, paired, ma, mb, p) == cudaSuccess ? 0 : 3;
  }
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(units < num_sms ? units : num_sms);
  return cudaLaunchKernelEx(&cfg, single, ma, mb, p) == cudaSuccess ? 0 : 3;
}

// Shared launch: operands are FP8 (ld in bytes) or bf16 (ld in bytes as well).
int launch_gemm(bool bf16, const void* a, int64_t lda_bytes, const float* s_a, const void* w, int64_t ldw_bytes,
                const float* s_w, int per_channel, const uint16_t* bias, uint16_t* y, int64_t ldy, int M, int N,
                int K, uint32_t idesc, int num_sms, cudaStream_t stream) {
  return bf16 ? launch_kind<true>(a, lda_bytes, s_a, w, ldw_bytes, s_w, per_channel, bias, y, ldy, M, N, K, idesc,
                                  num_sms, stream)
              : launch_kind<false>(a, lda_bytes, s_a, w, ldw_bytes, s_w, per_channel, bias, y, ldy, M, N, K, idesc,
                                   num_sms, stream);
}

}  // namespace

int gemm_launch(const uint8_t* qa, int64_t ldqa, const float* s_a, const uint8_t* qw, int64_t ldqw,
                const float* s_w, int per_channel, const uint16_t* bias, uint16_t* y, int64_t ldy,
                int M, int N, int K, int fmt_a, int fmt_w, int num_sms, cudaStream_t stream) {
  return launch_gemm(false, qa, ldqa, s_a, qw, ldqw, s_w, per_channel, bias, y, ldy, M, N, K,
                     gemm::make_idesc(fmt_a, fmt_w), num_sms, stream);
}

int gemm_bf16_launch(const uint16_t* a, int64_t lda, const uint16_t* w, int64_t ldw, const float* s_w,
                     int per_channel, const uint16_t* bias, uint16_t* y, int64_t ldy, int M, int N, int K,
                     int num_sms, cudaStream_t stream) {
  return launch_gemm(true, a, lda * 2, nullptr, w, ldw * 2, s_w, per_channel, bias, y, ldy, M, N, K,
                     gemm::kIdescBf16, num_sms, stream);
}

unsigned int gemm_read_and_clear_error() {
  unsigned int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, gemm::g_gemm_error, sizeof(v)) != cudaSuccess) return 0;
  cudaMemcpyToSymbol(gemm::g_gemm_error, &zero, sizeof(zero));
  return v;
}

}  // namespace fp8k
