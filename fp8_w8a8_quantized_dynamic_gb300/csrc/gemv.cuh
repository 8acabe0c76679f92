// Decode-shape FP8 GEMV: Y[M<=32, N] = bf16(s_a * s_w[n] * sum_k qA[m,k] qW[n,k] (+ bias[n])).
// qA and qW are e4m3 or e5m2 ("Fp8 Quantization Support", the other FP8 dtype), each
// operand's format a template parameter of the kernel.
//
// "[WIP] FP8 support": LLM decode runs at sequence length < 16 (the batch), which calls
// for a custom gemv rather than a 16-padded GEMM. The weight matrix is streamed from HBM
// exactly once.
//
// Up to 16 tokens, dynamic activation quantization happens inside this kernel: the ranks of
// a cluster together cover all of K, so the maximum of the ranks' max |A| over their
// K-slices, exchanged through distributed shared memory (or every CTA's maximum over all of a
// small A), is the global amax. Every CTA derives the same s_a = amax / 448 and quantizes only
// its own slice while its TMA ring is already filling with weights. A static (calibrated)
// activation scale skips the amax. With pre-quantized activations (fp8_scaled_mm, and
// fp8_linear from 17 tokens on, which quantizes A beforehand) qA and s_a are read instead.
//
// Work split. Rows of W come in blocks of 128; K is split over the S CTAs of a
// thread-block cluster (rank r owns K-range [r*kslice, (r+1)*kslice)). The grid is
// persistent: cluster c processes row blocks c, c + C, c + 2C, ... with C chosen on the
// host so every CTA streams the same number of tiles. Each CTA pushes the fp32 partial sums
// of its row blocks into the shared memory of the ranks that own those rows; one cluster
// barrier publishes them and rank r reduces its share of the rows over all ranks in a fixed
// order (deterministic, no global scratch), applies the scale/bias epilogue and writes Y.
//
// Streaming. Warp 8 is a TMA producer: 2-D tensor-map loads of [128 rows x 128 B] weight
// tiles (128B-swizzled, 16 KB) into an mbarrier ring of up to 12 stages; the first tiles are
// issued from kernel entry, before the wait on the preceding kernel. Up to two n8 token tiles,
// warps 0..7 (16 rows each) read their rows from the tile and run mma.sync m16n8k32 with W
// rows as the MMA's M dimension and tokens as its N dimension. The k order inside each 64-byte
// half-row is permuted so that a lane (group g, thread t) takes one 16-byte load of row g and
// one of row g+8 per half; the activation fragment uses the same permutation, which is plain
// row-major [token][k]. With four token tiles the main loop runs on tcgen05 (kTc, below).
#pragma once

#include "device_common.cuh"
#include "gemv.h"

namespace fp8k {
namespace gemv {

// Device error bits of the GEMV (bounded waits that expired), read by fp8_last_device_status.
__device__ unsigned int g_gemv_error;

// D += W (16 rows x 16 k) * A^T (16 k x 8 tokens), bf16 operands, fp32 accumulate.
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// D += W (16 rows x 32 k, format FW) * A^T (32 k x 8 tokens, format FA), fp32 accumulate.
#define FP8K_MMA_M16N8K32(TW, TA)                                                    \
  asm volatile("mma.sync.aligned.m16n8k32.row.col.f32." TW "." TA ".f32 "          \
               "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"              \
               : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])                      \
               : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1))

template <int FW, int FA>
__device__ __forceinline__ void mma_fp8(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  if constexpr (FW == kFmtE4M3 && FA == kFmtE4M3) FP8K_MMA_M16N8K32("e4m3", "e4m3");
  else if constexpr (FW == kFmtE4M3) FP8K_MMA_M16N8K32("e4m3", "e5m2");
  else if constexpr (FA == kFmtE4M3) FP8K_MMA_M16N8K32("e5m2", "e4m3");
  else FP8K_MMA_M16N8K32("e5m2", "e5m2");
}
#undef FP8K_MMA_M16N8K32

__device__ __forceinline__ uint4 lds_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

__device__ __forceinline__ float4 lds_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
  return v;
}

// Cluster-wide barrier (release/acquire); the non-aligned form tolerates diverged warps.
__device__ __forceinline__ void cluster_sync_all() {
  __syncwarp();
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
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

__device__ __forceinline__ void st_dsmem_v2(uint32_t local_addr, uint32_t rank, float a, float b) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank));
  asm volatile("st.shared::cluster.v2.f32 [%0], {%1,%2};" :: "r"(remote), "f"(a), "f"(b) : "memory");
}

__device__ __forceinline__ float ld_dsmem_f32(uint32_t local_addr, uint32_t rank) {
  uint32_t remote;
  float v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank));
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
  return v;
}

// Split-phase cluster barrier: every thread of every CTA arrives once per phase and waits
// before arriving again.
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release;" ::: "memory"); }
// Arrival that publishes nothing (no release fence): only says "this thread is running".
__device__ __forceinline__ void cluster_arrive_relaxed() { asm volatile("barrier.cluster.arrive.relaxed;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire;" ::: "memory"); }

__device__ __forceinline__ void consumer_bar_sync() {
  asm volatile("bar.sync 1, %0;" :: "n"(kConsumerThreads) : "memory");
}

// Contiguous global -> shared copy of `bytes` (16-byte aligned ends), completing on `bar`.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               :: "r"(dst), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar) : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];"
      :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y) : "memory");
}

// ---- tcgen05 consumer (several token tiles) ----

__device__ __forceinline__ void st_dsmem_v4(uint32_t local_addr, uint32_t rank, float a, float b, float c, float d) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank));
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1,%2,%3,%4};" :: "r"(remote), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}

// Shared-memory descriptor of a K-major operand in the 128-byte swizzle layout: rows of 128
// bytes, 8-row atoms of 1024 bytes (stride byte offset), start address >> 4 in bits 0-13,
// descriptor version 1 at bit 46, swizzle mode 2 (128B) at bits 61-63; the leading byte
// offset is unused for this layout (1).
__device__ __forceinline__ uint64_t tc_sdesc(uint32_t saddr) {
  return uint64_t((saddr & 0x3FFFFu) >> 4) | (uint64_t(1) << 16) | (uint64_t(1024 >> 4) << 32) |
         (uint64_t(1) << 46) | (uint64_t(2) << 61);
}

// D[128 rows x N tokens] (+)= W tile (128 x 32 bytes of K) * A block^T, FP8 operands, fp32 in
// tensor memory; issued by one thread.
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}"
      :: "r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}

// Arrives once on `bar` when every MMA this thread issued before has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" :: "r"(bar)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// N fp32 columns of this thread's tensor-memory lane (warp-collective).
template <int N>
__device__ __forceinline__ void tc_ld(uint32_t taddr, uint32_t (&r)[N]) {
  static_assert(N == 16 || N == 32, "16 or 32 token columns");
  if constexpr (N == 16)
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
  else
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

constexpr int kTcCols = 64;  // tensor memory columns of a tcgen05 GEMV CTA: two accumulators of <= 32

// Loads the 8-element units [i0 + b * kConsumerThreads, b < kRegUnits) of a [rows][upt units]
// bf16 slice starting at column k0 (zero past `units`, past row M and past K) into v.
__device__ __forceinline__ void load_units(uint4 (&v)[kRegUnits], const Params& p, int i0, int units, int upt,
                                           int k0) {
#pragma unroll
  for (int b = 0; b < kRegUnits; ++b) {
    const int i = i0 + b * kConsumerThreads;
    const int m = i / upt, kk = (i - (i / upt) * upt) << 3;
    v[b] = (i < units && m < p.M) ? load8_bf16(p.a + (int64_t)m * p.lda, k0 + kk, p.K, p.vec_a)
                                  : make_uint4(0, 0, 0, 0);
  }
}

__device__ __forceinline__ uint32_t abs_max_units(uint32_t m2, const uint4 (&v)[kRegUnits]) {
#pragma unroll
  for (int b = 0; b < kRegUnits; ++b)
    m2 = abs_max_u16x2(abs_max_u16x2(abs_max_u16x2(abs_max_u16x2(m2, v[b].x), v[b].y), v[b].z), v[b].w);
  return m2;
}

// NT: n8 token tiles (1: M <= 8, 2: M <= 16, 4: M <= 32). kMode: kModeQuantize (A is bf16 and quantized
// here, dynamic scale or the static one when p.s_static is set), kModePrequant (qA and s_a
// given) or kModeBf16 (weight-only: A stays bf16, each weight tile is up-converted to bf16 in
// registers and multiplied with bf16 MMAs; s_a is 1). FA / FW: FP8 formats of the
// activations and the weights.
//
// Start-up order. The producer issues its first p.head_tiles weight tiles at once (they
// never depend on the preceding kernel), then holds the stream until every consumer warp
// has all of its activation loads back: while the weight stream saturates HBM, each
// dependent activation round trip takes several times longer. The dynamic amax is the maximum
// over all of A computed by every CTA (p.cluster_amax == 0, small M*K), or each rank's slice
// maximum exchanged over the cluster through distributed shared memory.
//
// kTc (pre-quantized FP8 activations, two or four token tiles; the host takes it for four):
// the tensor cores' tcgen05 path runs the main loop instead of mma.sync, whose FP8 rate (about
// 38 cycles per m16n8k32 per SM sub-partition, measured on the GB300 through the per-token-tile
// cost) makes four token tiles about twice as slow as the weight stream. Each weight tile is
// the M = 128 operand as TMA left it; the activations arrive by TMA per 128-byte K block as
// [tokens][128 B] in the same 128-byte swizzle and are the N = 8 * NT operand; accumulators
// (two, alternating by row block) live in tensor memory. Warp 0's first lane issues the MMAs
// and commits each stage back to the producer; warps 4..7 read finished accumulators and push
// the partials to their owners.
template <int NT, int kMode, int FA, int FW, bool kTc>
__global__ void __launch_bounds__(kThreads, 1)
gemv_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_a,
            const __grid_constant__ Params p) {
  static_assert(!kTc || (NT >= 2 && kMode == kModePrequant), "tcgen05 path: pre-quantized FP8 activations");
  unsigned int* err = &g_gemv_error;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);

  const uint32_t rank = cluster_ctarank(), nrank = cluster_nctarank();
  const int cluster = blockIdx.x / nrank;
  const int rb_count = (p.row_blocks - cluster + p.num_clusters - 1) / p.num_clusters;  // row blocks of this cluster
  const Layout L = layout(p.stages, p.act_stride, p.act_rows, rb_count);
  const uint32_t ring = base + L.ring, act = base + L.act, part = base + L.part;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + kMaxStages);
  const uint32_t aready = smem_u32(bars + 2 * kMaxStages);
  const uint32_t abar = smem_u32(bars + 2 * kMaxStages + 1);  // bulk copy of A landed

  const int rows_per = (kRows + nrank - 1) / nrank;  // rows of a row block each rank reduces
  const int k0 = int(rank) * p.kslice;
  const int kspan = max(0, min(p.kslice, p.K - k0));
  const int ntiles = (kspan + kTileK - 1) / kTileK;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool cluster_amax = kMode == kModeQuantize && p.s_static == nullptr && p.cluster_amax;
  // FP8 activation byte (token m, slice column kk) of the mma.sync layout
  auto act_at = [&](int m, int kk) -> uint32_t { return act + uint32_t(m * p.act_stride + kk); };

  __shared__ int abort_flag;
  __shared__ uint32_t tmem_sh;
  __shared__ __align__(8) uint64_t tc_bars[5];  // kTc: accumulator full[2], empty[2], drain
  const uint32_t accfull0 = smem_u32(&tc_bars[0]), accempty0 = smem_u32(&tc_bars[2]), drain = smem_u32(&tc_bars[4]);
  __shared__ float s_a_out;
  __shared__ float slice_amax;
  __shared__ float red[kConsumerWarps];
  if (warp == kConsumerWarps && lane == 0)  // fetch the descriptor while the barriers are set up
    asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&tmap_w)) : "memory");
  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, kTc ? 1 : kConsumerWarps);  // kTc: one MMA commit frees a stage
    }
    mbar_init(aready, kConsumerWarps);
    mbar_init(abar, 1);
    if constexpr (kTc) {
      for (int b = 0; b < 2; ++b) {
        mbar_init(accfull0 + 8 * b, 1);
        mbar_init(accempty0 + 8 * b, 4);  // the four reading warps
      }
      mbar_init(drain, 1);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if constexpr (kTc) {
    if (warp == 1) {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                   :: "r"(smem_u32(&tmem_sh)), "n"(kTcCols) : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
  }
  __syncthreads();
  if constexpr (kTc) tc_fence_after();
  pdl_trigger();
  volatile int* ab = &abort_flag;

  if (warp == kConsumerWarps) {
    // ---------------- producer: weights never depend on the preceding kernel ----------------
    cluster_arrive_relaxed();  // phase 1 (start / amax exchange) never waits for the weight stream
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true, held = false;
      for (int r = 0; r < rb_count && ok; ++r) {
        const int rb = cluster + r * p.num_clusters;
        for (int kt = 0; kt < ntiles; ++kt, ++it) {
          if (!held && it == uint32_t(p.head_tiles)) {
            held = true;
            if (!mbar_wait_bounded(aready, 0, ab, err)) { ok = false; break; }
          }
          const int s = it % p.stages;
          const uint32_t ph = (it / p.stages) & 1u;
          if (!mbar_wait_bounded(empty0 + 8 * s, ph ^ 1u, ab, err)) { ok = false; break; }
          mbar_arrive_expect_tx(full0 + 8 * s, kTileBytes);
          tma_load_2d(ring + s * kTileBytes, &tmap_w, full0 + 8 * s, k0 + kt * kTileK, rb * kRows);
        }
      }
      if (!ok) {  // let the copies already issued land before the CTA's memory is released
        const uint32_t first = it > uint32_t(p.stages) ? it - p.stages : 0u;
        for (uint32_t j = first; j < it; ++j)
          mbar_wait_bounded(full0 + 8 * (j % p.stages), (j / p.stages) & 1u, nullptr, err);
      }
    }
    __syncwarp();
    cluster_wait();
  } else {
    // ---------------- consumers ----------------
    // phase 1 of the cluster barrier: the amax exchange (cluster_amax), otherwise only the
    // proof that every CTA of the cluster runs before partials are pushed into its memory
    if (!cluster_amax) cluster_arrive_relaxed();
    pdl_wait();  // A (or qA and s_a) may come from the preceding kernel
    const int span = ntiles * kTileK;  // bytes of K staged per token (zero beyond K)
    // every warp reports once that its activation loads are back, which releases the stream
    auto loads_back = [&]() {
      __syncwarp();
      if (lane == 0) mbar_arrive(aready);
    };
    float s_a;
    if constexpr (kMode == kModeQuantize) {
      if (p.scratch_a != 0) {
        // A (all of it, or this rank's slice) arrives by bulk copies, one per token row, in ring
        // stages the producer will not fill before aready; max and quantization read it there
        const bool full = p.scratch_a == 1;
        const int rowlen = full ? p.K : kspan;  // elements per copied row (a multiple of 8)
        const int col0 = full ? 0 : k0;
        const uint32_t scratch = ring + p.head_tiles * kTileBytes;
        if (threadIdx.x == 0) {
          mbar_arrive_expect_tx(abar, uint32_t(p.M) * uint32_t(rowlen) * 2u);
          for (int m = 0; m < p.M; ++m)
            bulk_load(scratch + uint32_t(m * rowlen) * 2u, p.a + (int64_t)m * p.lda + col0, uint32_t(rowlen) * 2u, abar);
        }
        mbar_wait_bounded(abar, 0, ab, err);
        const int ru = rowlen >> 3;  // 16-byte units per copied row
        if (p.s_static != nullptr) {
          s_a = *p.s_static;
        } else {
          uint32_t m2 = 0;
          for (int i = threadIdx.x; i < p.M * ru; i += kConsumerThreads)
            m2 = abs_max_v4(m2, lds_v4(scratch + uint32_t(i) * 16u));
          float mx = warp_max(u16x2_max_to_float(m2));
          if (lane == 0) red[warp] = mx;
          consumer_bar_sync();
          if (threadIdx.x == 0) {
            for (int w = 1; w < kConsumerWarps; ++w) mx = fmaxf(mx, red[w]);
            slice_amax = mx;
          }
          consumer_bar_sync();
          float amax = slice_amax;
          if (cluster_amax) {
            cluster_arrive();  // phase 1: publish this rank's slice maximum
            cluster_wait();
            float part_max[kMaxCluster];
#pragma unroll
            for (int src = 0; src < kMaxCluster; ++src)
              part_max[src] = src < int(nrank) ? ld_dsmem_f32(smem_u32(&slice_amax), src) : 0.0f;
#pragma unroll
            for (int src = 0; src < kMaxCluster; ++src) amax = fmaxf(amax, part_max[src]);
          }
          s_a = scale_from_amax<FA>(amax);
        }
        const ExactScale kq = make_exact_scale(s_a);
        const bool check = p.s_static != nullptr;  // a given scale does not bound the inputs
        // quantize the slice: kQuantUnroll units per thread per round, all loads first
        const int upt = span >> 3;  // 8-element units per token of this rank's slice
        const int total = p.M * upt;
        const float inv_upt = 1.0f / float(upt);  // unit -> token by float: exact for these sizes
        for (int i0 = threadIdx.x; i0 < total; i0 += kQuantUnroll * kConsumerThreads) {
          uint4 x[kQuantUnroll];
          uint32_t dst[kQuantUnroll];
          bool inside[kQuantUnroll];
#pragma unroll
          for (int j = 0; j < kQuantUnroll; ++j) {
            const int i = i0 + j * kConsumerThreads;
            const int m = int((float(i) + 0.5f) * inv_upt), kk = (i - m * upt) << 3;
            inside[j] = i < total && k0 + kk < p.K;
            dst[j] = i < total ? act_at(m, kk) : 0u;
            x[j] = inside[j] ? lds_v4(scratch + uint32_t(m * rowlen + (full ? k0 : 0) + kk) * 2u)
                             : make_uint4(0, 0, 0, 0);
          }
#pragma unroll
          for (int j = 0; j < kQuantUnroll; ++j) {
            const uint2 q = inside[j] ? quant8_exact<FA>(x[j], kq, s_a, check) : make_uint2(0, 0);
            if (i0 + j * kConsumerThreads < total)
              asm volatile("st.shared.v2.u32 [%0], {%1,%2};" :: "r"(dst[j]), "r"(q.x), "r"(q.y) : "memory");
          }
        }
      } else {
        const int upt = span >> 3;  // 8-element units per token of this rank's slice
        const int units = p.M * upt;
        uint4 v[kRegUnits];  // the first kRegUnits units per thread stay in registers
        load_units(v, p, threadIdx.x, units, upt, k0);
        if (p.s_static != nullptr) {
          s_a = *p.s_static;
        } else {
          uint32_t m2 = abs_max_units(0u, v);
          if (!cluster_amax) {
            // the maximum over all of A, read by every CTA (small M * K)
            const int upt_all = (p.K + 7) >> 3;
            const int units_all = p.M * upt_all;
            for (int i0 = threadIdx.x; i0 < units_all; i0 += kRegUnits * kConsumerThreads) {
              uint4 w[kRegUnits];
              load_units(w, p, i0, units_all, upt_all, 0);
              m2 = abs_max_units(m2, w);
            }
          } else {
            for (int i0 = threadIdx.x + kRegUnits * kConsumerThreads; i0 < units; i0 += kRegUnits * kConsumerThreads) {
              uint4 w[kRegUnits];
              load_units(w, p, i0, units, upt, k0);
              m2 = abs_max_units(m2, w);
            }
          }
          float mx = warp_max(u16x2_max_to_float(m2));
          if (lane == 0) red[warp] = mx;
          consumer_bar_sync();
          if (threadIdx.x == 0) {
            for (int w = 1; w < kConsumerWarps; ++w) mx = fmaxf(mx, red[w]);
            slice_amax = mx;
          }
          consumer_bar_sync();
          float amax = slice_amax;
          if (cluster_amax) {
            cluster_arrive();  // phase 1: publish this rank's slice maximum
            cluster_wait();
            float part_max[kMaxCluster];
#pragma unroll
            for (int src = 0; src < kMaxCluster; ++src)
              part_max[src] = src < int(nrank) ? ld_dsmem_f32(smem_u32(&slice_amax), src) : 0.0f;
#pragma unroll
            for (int src = 0; src < kMaxCluster; ++src) amax = fmaxf(amax, part_max[src]);
          }
          s_a = scale_from_amax<FA>(amax);
        }
        const ExactScale kq = make_exact_scale(s_a);
        const bool check = p.s_static != nullptr;
        // quantize into act[token][k - k0]; units past K and tokens past M are plain zeros
        auto put = [&](int i, const uint4& x) {
          const int m = i / upt, kk = (i - (i / upt) * upt) << 3;
          uint2 q = make_uint2(0, 0);
          if (k0 + kk < p.K) q = quant8_exact<FA>(x, kq, s_a, check);
          asm volatile("st.shared.v2.u32 [%0], {%1,%2};" :: "r"(act_at(m, kk)), "r"(q.x), "r"(q.y) : "memory");
        };
#pragma unroll
        for (int b = 0; b < kRegUnits; ++b) {
          const int i = threadIdx.x + b * kConsumerThreads;
          if (i < units) put(i, v[b]);
        }
        // units beyond the register batch: reload kRegUnits at a time (independent loads)
        for (int i0 = threadIdx.x + kRegUnits * kConsumerThreads; i0 < units; i0 += kRegUnits * kConsumerThreads) {
          uint4 w[kRegUnits];
          load_units(w, p, i0, units, upt, k0);
#pragma unroll
          for (int b = 0; b < kRegUnits; ++b)
            if (i0 + b * kConsumerThreads < units) put(i0 + b * kConsumerThreads, w[b]);
        }
      }
      loads_back();  // every activation load of the prologue has landed (and the scratch is free)
      const int zu = span >> 4;  // 16-byte units per padding token
      for (int i = threadIdx.x; i < (p.act_rows - p.M) * zu; i += kConsumerThreads) {
        const int m = p.M + i / zu;
        const int kk = (i - (i / zu) * zu) << 4;
        asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" :: "r"(act_at(m, kk)), "r"(0u) : "memory");
      }
    } else if constexpr (kMode == kModeBf16) {
      s_a = 1.0f;
      // bf16 activation slice [tokens][span] -> smem (2 bytes an element), zero beyond M and K
      const int upt = span >> 3;  // 8-element units per token
      const int units = p.act_rows * upt;
      for (int i0 = threadIdx.x; i0 < units; i0 += kRegUnits * kConsumerThreads) {
        uint4 v[kRegUnits];
        load_units(v, p, i0, units, upt, k0);
#pragma unroll
        for (int b = 0; b < kRegUnits; ++b) {
          const int i = i0 + b * kConsumerThreads;
          if (i < units) {
            const int m = i / upt, kk = (i - (i / upt) * upt) << 3;
            asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};"
                         :: "r"(act + m * p.act_stride + 2 * kk), "r"(v[b].x), "r"(v[b].y), "r"(v[b].z),
                            "r"(v[b].w) : "memory");
          }
        }
      }
      loads_back();
    } else if constexpr (kTc) {
      s_a = *p.s_a;
      // the qA slice arrives by TMA, one [act_rows tokens x 128 B] box per K block, already in
      // the swizzled layout the MMAs read (zero past M and K)
      if (threadIdx.x == 0) {
        mbar_arrive_expect_tx(abar, uint32_t(ntiles * p.act_rows * kTileK));
        for (int kt = 0; kt < ntiles; ++kt)
          tma_load_2d(act + uint32_t(kt * p.act_rows * kTileK), &tmap_a, abar, k0 + kt * kTileK, 0);
      }
      mbar_wait_bounded(abar, 0, ab, err);
      loads_back();
    } else {
      s_a = *p.s_a;
      // activation slice [tokens][span] of qA -> smem, zero beyond M and K, kRegUnits
      // independent 16-byte loads per thread in flight at a time
      const int upt = span / 16;
      const int units = p.act_rows * upt;
      const int k16 = (p.K + 15) & ~15;
      for (int i0 = threadIdx.x; i0 < units; i0 += kRegUnits * kConsumerThreads) {
        uint4 v[kRegUnits];
#pragma unroll
        for (int b = 0; b < kRegUnits; ++b) {
          const int i = i0 + b * kConsumerThreads;
          const int m = i / upt, kk = (i - (i / upt) * upt) * 16;
          v[b] = make_uint4(0, 0, 0, 0);
          if (i < units && m < p.M && k0 + kk < k16)
            v[b] = *reinterpret_cast<const uint4*>(p.qa + (int64_t)m * p.ldqa + k0 + kk);
        }
#pragma unroll
        for (int b = 0; b < kRegUnits; ++b) {
          const int i = i0 + b * kConsumerThreads;
          if (i < units) {
            const int m = i / upt, kk = (i - (i / upt) * upt) * 16;
            asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};"
                         :: "r"(act_at(m, kk)), "r"(v[b].x), "r"(v[b].y), "r"(v[b].z), "r"(v[b].w) : "memory");
          }
        }
      }
      loads_back();
    }
    if (threadIdx.x == 0) s_a_out = s_a;
    if constexpr (kTc) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // activations -> tensor cores
    consumer_bar_sync();
    if constexpr (kTc) {
      if (!cluster_amax) cluster_wait();  // every CTA of the cluster runs before partials are pushed to it
      const uint32_t tmem = tmem_sh;
      constexpr int N = 8 * NT;
      if (warp == 0) {
        if (lane == 0) {
          // ---------------- MMA issuer ----------------
          // D f32 (bit 4), A = weights (format at bits 7-9), B = activations (10-12), both K-major,
          // N >> 3 at bits 17-22, M >> 4 at bits 24-28
          const uint32_t idesc = (1u << 4) | (uint32_t(FW) << 7) | (uint32_t(FA) << 10) | (uint32_t(N >> 3) << 17) |
                                 (uint32_t(kRows >> 4) << 24);
          uint32_t it = 0;
          bool ok = true;
          for (int r = 0; r < rb_count && ok; ++r) {
            const int b = r & 1;
            if (!mbar_wait_bounded(accempty0 + 8 * b, ((r >> 1) & 1) ^ 1u, ab, err)) break;
            tc_fence_after();
            const uint32_t d = tmem + uint32_t(b * 32);
            for (int kt = 0; kt < ntiles; ++kt, ++it) {
              const int s = it % p.stages;
              const uint32_t ph = (it / p.stages) & 1u;
              if (!mbar_wait_bounded(full0 + 8 * s, ph, ab, err)) { ok = false; break; }
              tc_fence_after();
              const uint64_t adesc = tc_sdesc(ring + s * kTileBytes);
              const uint64_t bdesc = tc_sdesc(act + uint32_t(kt * p.act_rows * 128));
#pragma unroll
              for (int kk = 0; kk < kTileK / 32; ++kk)  // 32 bytes of K per MMA: +2 in the address field
                tc_mma(d, adesc + uint64_t(2 * kk), bdesc + uint64_t(2 * kk), idesc, (kt | kk) != 0 ? 1u : 0u);
              tc_commit(empty0 + 8 * s);  // the stage is free once these MMAs have read it
            }
            if (!ok) break;
            tc_commit(accfull0 + 8 * b);
          }
          // every MMA issued must finish before tensor and shared memory are released
          tc_commit(drain);
          mbar_wait_bounded(drain, 0, nullptr, err);
        }
        __syncwarp();
      } else if (warp >= 4) {
        // ---------------- accumulators -> partials of the owning ranks ----------------
        const int row = (warp & 3) * 32 + lane;  // tensor-memory lane quarter of this warp
        const int owner = row / rows_per;
        for (int r = 0; r < rb_count; ++r) {
          const int b = r & 1;
          bool ok = true;
          if (lane == 0) ok = mbar_wait_bounded(accfull0 + 8 * b, (r >> 1) & 1u, ab, err);
          if (__shfl_sync(0xffffffffu, ok ? 1 : 0, 0) == 0) break;
          tc_fence_after();
          uint32_t v[N];
          tc_ld<N>(tmem + (uint32_t((warp & 3) * 32) << 16) + uint32_t(b * 32), v);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(accempty0 + 8 * b);
          const uint32_t dst = part + r * part_bytes(p.act_rows) +
                               uint32_t((rank * rows_per + (row - owner * rows_per)) * p.act_rows) * 4u;
#pragma unroll
          for (int c = 0; c < N / 4; ++c)
            st_dsmem_v4(dst + 16 * c, owner, __uint_as_float(v[4 * c]), __uint_as_float(v[4 * c + 1]),
                        __uint_as_float(v[4 * c + 2]), __uint_as_float(v[4 * c + 3]));
        }
      }
    } else {
      const int g = lane >> 2, t = lane & 3;
      const uint32_t row_lo = (warp * 16 + g) * kTileK, row_hi = row_lo + 8 * kTileK;
      // this lane's activation fragment: token g, the 16 K of unit (4j + t) of each half-row j
      const uint32_t act_lane = act + g * p.act_stride + (kMode == kModeBf16 ? 32 : 16) * t;
      uint32_t it = 0;
      for (int r = 0; r < rb_count; ++r) {
        float acc[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.0f;
        for (int kt = 0; kt < ntiles; ++kt, ++it) {
          const int s = it % p.stages;
          const uint32_t ph = (it / p.stages) & 1u;
          const bool ok = mbar_wait_bounded(full0 + 8 * s, ph, ab, err);
          if (ok) {
            const uint32_t tile = ring + s * kTileBytes;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              // 16-byte unit (4j + t) of rows g / g+8, at its 128B-swizzled position (row % 8 == g)
              const uint32_t unit = uint32_t(((4 * j + t) ^ g) * 16);
              const uint4 wlo = lds_v4(tile + row_lo + unit);
              const uint4 whi = lds_v4(tile + row_hi + unit);
              if constexpr (kMode == kModeBf16) {
                // 4-byte group i of the unit feeds one k16 MMA: bytes (4i, 4i+1) are its K pair
                // (2t, 2t+1) and bytes (4i+2, 4i+3) its pair (2t+8, 2t+9); the activations use the
                // same order, 8 consecutive bytes of bf16 per MMA
                const uint32_t wl[4] = {wlo.x, wlo.y, wlo.z, wlo.w}, wh[4] = {whi.x, whi.y, whi.z, whi.w};
                uint32_t fa[4][4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  fa[i][0] = fp8x2_to_bf16x2<FW>(wl[i]);
                  fa[i][1] = fp8x2_to_bf16x2<FW>(wh[i]);
                  fa[i][2] = fp8x2_to_bf16x2<FW>(wl[i] >> 16);
                  fa[i][3] = fp8x2_to_bf16x2<FW>(wh[i] >> 16);
                }
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                  const uint32_t boff = act_lane + nt * 8 * p.act_stride + 2 * (kt * kTileK + 64 * j);
                  const uint4 b0 = lds_v4(boff), b1 = lds_v4(boff + 16);
                  mma_bf16(acc[nt], fa[0][0], fa[0][1], fa[0][2], fa[0][3], b0.x, b0.y);
                  mma_bf16(acc[nt], fa[1][0], fa[1][1], fa[1][2], fa[1][3], b0.z, b0.w);
                  mma_bf16(acc[nt], fa[2][0], fa[2][1], fa[2][2], fa[2][3], b1.x, b1.y);
                  mma_bf16(acc[nt], fa[3][0], fa[3][1], fa[3][2], fa[3][3], b1.z, b1.w);
                }
              } else {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                  const uint4 b = lds_v4(act_lane + nt * 8 * p.act_stride + kt * kTileK + 64 * j);
                  mma_fp8<FW, FA>(acc[nt], wlo.x, whi.x, wlo.y, whi.y, b.x, b.y);
                  mma_fp8<FW, FA>(acc[nt], wlo.z, whi.z, wlo.w, whi.w, b.z, b.w);
                }
              }
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(empty0 + 8 * s);
        }
        // push the partials of this row block to the ranks that own their rows:
        // part[r][source rank][row - owner's first row][token] in the owner's shared memory
        if (r == 0 && !cluster_amax) cluster_wait();  // every CTA of the cluster is running
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int row = warp * 16 + g + 8 * h, col = nt * 8 + 2 * t;
            const int owner = row / rows_per;
            const uint32_t dst = part + r * part_bytes(p.act_rows) +
                                 ((rank * rows_per + (row - owner * rows_per)) * p.act_rows + col) * 4;
            st_dsmem_v2(dst, owner, acc[nt][2 * h], acc[nt][2 * h + 1]);
          }
        }
      }
      if (rb_count == 0 && !cluster_amax) cluster_wait();
    }
  }

  // split-K reduction work of this rank: its share of the rows of every row block
  const int r_begin = rank * rows_per;
  const int r_count = max(0, min(kRows, r_begin + rows_per) - r_begin);
  const int q_per_row = (p.M + 3) / 4;  // float4 groups of tokens
  const int items = rb_count * r_count * q_per_row;
  auto item_n = [&](int i, int& q, int& r, int& row) {
    q = i % q_per_row;
    r = i / (q_per_row * r_count);
    row = r_begin + (i / q_per_row) % r_count;
    return (cluster + r * p.num_clusters) * kRows + row;
  };
  // the weight scale and bias of this thread's first output are weights: load them before the
  // barrier so their latency hides behind it
  float sw0 = 0.0f, b0 = 0.0f;
  if (warp < kConsumerWarps && int(threadIdx.x) < items) {
    int q, r, row;
    const int n = item_n(threadIdx.x, q, r, row);
    if (n < p.N) {
      sw0 = p.s_w[p.per_channel ? n : 0];
      b0 = p.bias ? bf16_bits_to_float(p.bias[n]) : 0.0f;
    }
  }

  cluster_sync_all();  // every rank's partials have arrived (and every TMA load is consumed)

  // ---------------- split-K reduction over the cluster + epilogue ----------------
  if (warp < kConsumerWarps) {
    const float s_a = s_a_out;
    for (int i = threadIdx.x; i < items; i += kConsumerThreads) {
      int q, r, row;
      const int n = item_n(i, q, r, row);
      if (n >= p.N) continue;
      const uint32_t off = part + r * part_bytes(p.act_rows) + ((row - r_begin) * p.act_rows + 4 * q) * 4;
      // every source rank's partials are local now; summed in rank order (deterministic)
      float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
      for (uint32_t src = 0; src < nrank; ++src) {
        const float4 v = lds_f4(off + src * rows_per * p.act_rows * 4);
        sum.x += v.x; sum.y += v.y; sum.z += v.z; sum.w += v.w;
      }
      const bool first = i == int(threadIdx.x);
      const float sc = s_a * (first ? sw0 : p.s_w[p.per_channel ? n : 0]);
      const float b = first ? b0 : (p.bias ? bf16_bits_to_float(p.bias[n]) : 0.0f);
      const float vals[4] = {sum.x, sum.y, sum.z, sum.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int m = 4 * q + e;
        if (m < p.M) p.y[(int64_t)m * p.ldy + n] = __bfloat16_as_ushort(__float2bfloat16_rn(fmaf(vals[e], sc, b)));
      }
    }
  }
  // no rank reads another's shared memory after the barrier above, so no second barrier
  // the activation copies into shared memory (TMA boxes of qA, or bulk copies of A) complete
  // on abar: after a wait that gave up they may still be landing, so the issuing thread
  // waits for them (bounded) before the CTA's shared memory is released
  if (threadIdx.x == 0 && ((kTc && kMode == kModePrequant) || (kMode == kModeQuantize && p.scratch_a != 0)))
    mbar_wait_bounded(abar, 0, nullptr, err);
  if constexpr (kTc) {
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(tmem_sh), "n"(kTcCols) : "memory");
  }
}

}  // namespace gemv
}  // namespace fp8k
