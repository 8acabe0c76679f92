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
// Structure (persistent, one CTA per SM, output tiles of 128 x 256 per CTA):
//   warp 0      TMA producer: this CTA's qA tile [128 x 128B] and its part of the qW tile
//               per stage into a ring of 128B-swizzled shared memory, completion on an
//               mbarrier.
//   warp 1      TMEM allocator + MMA issuer: tcgen05.mma kind::f8f6f4, K = 32 per
//               instruction, fp32 accumulators in TMEM, two accumulator buffers of 256
//               columns so the epilogue of tile i overlaps the main loop of tile i+1.
//   warps 2..5  epilogue: tcgen05.ld 32 columns at a time, scale (+bias), bf16, store.
// Ragged M, N and K need no padding: TMA fills out-of-range rows/columns with zeros and
// the epilogue predicates its stores.
//
// Two modes:
//   single   one CTA per 128 x 256 tile, tcgen05.mma.cta_group::1 (M = 128, N = 256),
//            4 stages of 48 KB (A 16 KB + W 32 KB).
//   two-SM   a cluster of two CTAs (a CTA pair) computes a 256 x 256 tile with
//            tcgen05.mma.cta_group::2 (M = 256, N = 256): each CTA holds its own 128 rows
//            of qA and one half (128 rows) of the weight tile, so a stage is 32 KB and the
//            ring is 6 deep. Both CTAs' copies complete on the leader's (rank 0) full
//            barrier; the leader's one elected thread issues the MMAs for the pair, and
//            its commits arrive on both CTAs' barriers. Each CTA's epilogue reads its own
//            tensor memory (the accumulator rows of its A tile). The weight tile crosses
//            from L2 to the SMs once per pair, not once per CTA.
//
// Split-K (one row block, too few column tiles to fill the GPU, a workspace that holds the
// partials): each tile's K blocks are divided among S work units; each unit writes its unscaled
// fp32 partial to the workspace instead of Y, and splitk_reduce_kernel, launched right after
// with programmatic dependent launch, sums the S partials in split order and applies the
// epilogue. The split count comes from a cost model calibrated on a GB300 (plan_splits).
//
// Last wave: when the tiles left after the full waves number at most half of the slots (CTA
// pairs, or CTAs), each of them is computed as 2 units of 128 columns over all of K (4 units of
// 64 on request), so the partial last wave ends sooner. When all tiles fit in half the slots
// (small M) every tile is split that way, into 4 units where they fit, unless K is long enough
// for the K split to win. Those units load their weight rows through a second tensor map with
// the narrower box and issue MMAs with the smaller N.
//
// Every wait is bounded (2 s); on expiry the kernel records an error for the host (with a
// bit naming the wait), stops its peer, drains every copy either CTA issued, frees its
// TMEM and returns.

#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <cstdlib>

#include "device_cache.h"
#include "device_common.cuh"
#include "gemm_tcgen05.h"

namespace fp8k {
namespace gemm {

__device__ unsigned int g_gemm_error;

// Error bits beyond kErrTimeout: which wait gave up (diagnostics for the host).
constexpr unsigned int kSiteEmpty = 0x100u;   // producer waiting for a free stage
constexpr unsigned int kSiteFull = 0x200u;    // MMA issuer waiting for a filled stage
constexpr unsigned int kSiteTempty = 0x400u;  // MMA issuer waiting for a drained accumulator
constexpr unsigned int kSiteTfull = 0x800u;   // epilogue waiting for a finished accumulator
constexpr unsigned int kSiteDrain = 0x1000u;  // exit path: outstanding copies or MMAs

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 128;  // bytes of K per stage: one 128-byte swizzle row (128 FP8 / 64 bf16 elements)
constexpr int kAccBufs = 2;
constexpr int kTmemCols = kAccBufs * BN;  // 512: the whole tensor memory of the SM
constexpr int kThreads = 192;
constexpr int kEpiThreads = 128;
constexpr uint32_t kABytes = BM * BK;
constexpr uint32_t kBBytes = BN * BK;
constexpr int kMmaK = 32;  // bytes of K of one MMA (32 FP8 elements, kind::f8f6f4; 16 bf16, kind::f16)

// Shared-memory ring of each mode: the two-SM CTA holds half of the weight tile per stage.
template <bool kTwo>
struct Ring {
  static constexpr uint32_t stage_bytes = kTwo ? kABytes + kBBytes / 2 : kABytes + kBBytes;
  static constexpr int stages = kTwo ? 6 : 4;
};
constexpr int kMaxStages = 6;
constexpr size_t kRingBytes =
    std::max(size_t(Ring<true>::stages) * Ring<true>::stage_bytes, size_t(Ring<false>::stages) * Ring<false>::stage_bytes);

struct SharedCtl {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t tfull[kAccBufs];
  uint64_t tempty[kAccBufs];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  uint32_t issued[2];  // two-SM: stages each CTA's producer filled (in the leader's block)
  float colscale[kAccBufs][BN];
  float colbias[kAccBufs][BN];
};

constexpr size_t kSmemBytes = 1024 /*alignment slack*/ + kRingBytes + sizeof(SharedCtl);
static_assert(kSmemBytes <= 232448, "ring and control block must fit the 227 KB per-block limit");
static_assert(2 * kSmemBytes > 233472, "two GEMM CTAs must never share an SM (each holds all of TMEM)");

// Instruction descriptor, kind::f8f6f4: D fp32 (bits 4-5 = 1), A and B format at bits 7-9 and
// 10-12 (e4m3 = 0, e5m2 = 1), both K-major (bits 15, 16 = 0), N >> 3 at bits 17-22, M >> 4 at
// bits 24-28.
constexpr uint32_t kIdescBase = (1u << 4) | (uint32_t(BN >> 3) << 17) | (uint32_t(BM >> 4) << 24);

constexpr uint32_t make_idesc(int fmt_a, int fmt_w) {
  return kIdescBase | (uint32_t(fmt_a) << 7) | (uint32_t(fmt_w) << 10);
}

// kind::f16 with bf16 A and B: the format fields hold BF16 = 1.
constexpr uint32_t kIdescBf16 = kIdescBase | (1u << 7) | (1u << 10);

// The same descriptor for an MMA of n columns (a multiple of 16, at most BN).
__host__ __device__ constexpr uint32_t idesc_with_n(uint32_t idesc, int n) {
  return (idesc & ~(0x3Fu << 17)) | (uint32_t(n >> 3) << 17);
}

// The two-SM MMA covers both CTAs' rows: M = 256 in the descriptor.
__host__ __device__ constexpr uint32_t idesc_two_sm(uint32_t idesc) {
  return (idesc & ~(0x1Fu << 24)) | (uint32_t((2 * BM) >> 4) << 24);
}

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

// L2 eviction priorities for the TMA loads and the output stores (createpolicy): the operand
// the raster keeps hot in L2 is loaded evict_last, the one streamed once evict_first.
enum : int { kHintNormal = 0, kHintFirst = 1, kHintLast = 2 };

__device__ __forceinline__ uint64_t l2_policy(int hint) {
  uint64_t p;
  if (hint == kHintLast)
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  else if (hint == kHintFirst)
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  else
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;"
      :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "l"(policy) : "memory");
}

// Two-SM form: the copy lands in this CTA's shared memory and completes its bytes on an
// mbarrier that may be the peer's (here always the leader's).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, uint32_t cluster_bar, int x,
                                                 int y, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;"
      :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(cluster_bar), "r"(x), "r"(y), "l"(policy)
      : "memory");
}

template <bool kBf16, bool kTwo>
__device__ __forceinline__ void mma_issue(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  if constexpr (kTwo && kBf16)
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        :: "r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
  else if constexpr (kTwo)
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}"
        :: "r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
  else if constexpr (kBf16)
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

// Arrives once on `bar` when every MMA this thread issued before has completed; in two-SM
// mode it arrives on the barrier at that offset in both CTAs of the pair.
template <bool kTwo>
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  if constexpr (kTwo)
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
                 :: "r"(bar), "h"(uint16_t(0x3)) : "memory");
  else
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" :: "r"(bar)
                 : "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// A shared-memory address of this CTA, as seen in CTA `rank` of the cluster (shared::cluster).
__device__ __forceinline__ uint32_t map_to_rank(uint32_t a, uint32_t rank) {
  uint32_t d;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(rank));
  return d;
}

__device__ __forceinline__ void st_cluster_u32(uint32_t cluster_addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" :: "r"(cluster_addr), "r"(v) : "memory");
}

__device__ __forceinline__ void arrive_cluster(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" :: "r"(cluster_bar) : "memory");
}

// Accounts for `bytes` that will never arrive on this CTA's barrier (abort path only).
__device__ __forceinline__ void mbar_complete_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.complete_tx.relaxed.cta.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(bytes) : "memory");
}

// Every thread of both CTAs: barrier inits visible before the first remote signal, and no CTA
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

__device__ __forceinline__ void st_global_v4(uint4* p, uint4 v, uint64_t policy) {
  asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;"
               :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "l"(policy) : "memory");
}

// Tile order: groups of `group_n` column tiles; inside a group the column index runs fastest.
// group_n = n_tiles keeps all of W hot in L2 while the row blocks stream past (qA read from
// HBM once); group_n = 1 sweeps all row blocks for one column tile before the next, keeping
// qA hot while W streams once; between the two, a W slice stays hot per group.
__device__ __forceinline__ void tile_coords(int tile, const GemmParams& p, int m_units, int& m_idx, int& n_idx) {
  const int per_group = p.group_n * m_units;
  const int gidx = tile / per_group;
  const int r = tile - gidx * per_group;
  const int n_first = gidx * p.group_n;
  const int gn = min(p.group_n, p.n_tiles - n_first);
  m_idx = r / gn;
  n_idx = n_first + (r - m_idx * gn);
}

// kBf16: operands are bf16 (weight-only product) instead of FP8. kTwo: clusters of two CTAs
// on the two-SM MMA (see the modes above).
template <bool kBf16, bool kTwo>
__global__ void __launch_bounds__(kThreads, 1)
gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
            const __grid_constant__ CUtensorMap tmap_bt, const __grid_constant__ GemmParams p) {
  constexpr int kElemsPerStage = kBf16 ? BK / 2 : BK;  // K elements per stage
  constexpr int kStages = Ring<kTwo>::stages;
  constexpr uint32_t kStageBytes = Ring<kTwo>::stage_bytes;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);  // 1024-aligned for the 128B swizzle
  SharedCtl* ctl = reinterpret_cast<SharedCtl*>(smem + kRingBytes);
  const uint32_t smem_base = smem_u32(smem);
  auto a_stage = [&](int s) { return smem_base + s * kStageBytes; };
  auto b_stage = [&](int s) { return smem_base + s * kStageBytes + kABytes; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // work units: tiles, or (two-SM) vertical tile pairs; rank r of a pair takes row block 2i + r
  const uint32_t rank = kTwo ? cluster_rank() : 0u;
  const bool leader = rank == 0;
  const int m_units = kTwo ? (p.m_tiles + 1) / 2 : p.m_tiles;
  const int S = p.k_splits;  // split-K: work unit = (tile, split); the splits of a tile are adjacent
  // tail: the tiles from p.tail_start on (the last, partial wave) are split by columns into
  // p.tail_split units of BN / tail_split columns each, all of K (tail_split == 1: none)
  const int TS = p.tail_split;
  const int num_tiles = TS > 1 ? p.tail_start + (m_units * p.n_tiles - p.tail_start) * TS : m_units * p.n_tiles * S;
  const int first_unit = kTwo ? int(blockIdx.x >> 1) : int(blockIdx.x);
  const int unit_stride = kTwo ? int(gridDim.x >> 1) : int(gridDim.x);
  // unit -> tile coordinates, K split, first column and column count (BN, or BN / TS in the tail)
  auto coords = [&](int unit, int& m_idx, int& n0, int& ks, int& width) {
    int tu, sub = 0;
    width = BN;
    if (TS > 1 && unit >= p.tail_start) {
      const int v = unit - p.tail_start;
      tu = p.tail_start + v / TS;
      sub = v - (v / TS) * TS;
      width = BN / TS;
      ks = 0;
    } else {
      tu = unit / S;
      ks = unit - tu * S;
    }
    int n_idx;
    tile_coords(tu, p, m_units, m_idx, n_idx);
    if (kTwo) m_idx = 2 * m_idx + int(rank);
    n0 = n_idx * BN + sub * width;
  };
  // bytes one CTA's copies bring into a stage for a unit of `width` columns
  auto stage_bytes_for = [&](int width) { return kABytes + uint32_t(kTwo ? width / 2 : width) * BK; };
  const int num_kb = (p.K + kElemsPerStage - 1) / kElemsPerStage;
  volatile int* abort_flag = &ctl->abort_flag;
  // after a wait gives up: stop the peer CTA as well, so the pair leaves together
  auto fail = [&](unsigned int site) {
    atomicOr(&g_gemm_error, site);
    if (kTwo) st_cluster_u32(map_to_rank(smem_u32(&ctl->abort_flag), rank ^ 1u), 1u);
  };

  if (threadIdx.x == 0) {
    asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&tmap_a)) : "memory");
    asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&tmap_b)) : "memory");
    if (TS > 1) asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&tmap_bt)) : "memory");
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&ctl->full[s]), 1);
      mbar_init(smem_u32(&ctl->empty[s]), 1);  // one commit per stage (two-SM: the leader's, in both CTAs)
    }
    for (int b = 0; b < kAccBufs; ++b) {
      mbar_init(smem_u32(&ctl->tfull[b]), 1);
      // two-SM: the leader's MMA waits until both CTAs' epilogues have drained the buffer
      mbar_init(smem_u32(&ctl->tempty[b]), kTwo ? 2 * kEpiThreads : kEpiThreads);
    }
    mbar_init(smem_u32(&ctl->drain), 1);
    ctl->abort_flag = 0;
    ctl->issued[0] = ctl->issued[1] = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    if (kTwo) {  // one warp of each CTA allocates the pair's tensor memory together
      asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
                   :: "r"(smem_u32(&ctl->tmem_base)), "n"(kTmemCols) : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    } else {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                   :: "r"(smem_u32(&ctl->tmem_base)), "n"(kTmemCols) : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
  }
  tmem_fence_before();
  __syncthreads();
  if (kTwo) pair_sync();  // the peer's barriers exist before the first copy or commit signals them
  tmem_fence_after();
  const uint32_t tmem_base = ctl->tmem_base;

  pdl_trigger();
  pdl_wait();  // qA / s_a come from the preceding kernel; Y may still be read by it

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      const uint64_t pol_a = l2_policy(p.hint_a), pol_b = l2_policy(p.hint_b);
      uint32_t it = 0;
      bool ok = true;
      for (int tile = first_unit, u = 0; tile < num_tiles && ok; tile += unit_stride, ++u) {
        int m_idx, n0, ks, width;
        coords(tile, m_idx, n0, ks, width);
        const CUtensorMap* mapb = width == BN ? &tmap_b : &tmap_bt;
        const uint32_t bytes = stage_bytes_for(width);
        const int kb_begin = ks * p.kb_per_split, kb_end = min(num_kb, kb_begin + p.kb_per_split);
        // serpentine: every other unit of this CTA walks K backwards, so a wave starts on the
        // K blocks the wave before it touched last (still in L2)
        const bool down = p.serpentine && (u & 1);
        for (int j = 0; j < kb_end - kb_begin; ++j, ++it) {
          const int kb = down ? kb_end - 1 - j : kb_begin + j;
          const int s = it % kStages;
          const uint32_t ph = (it / kStages) & 1u;
          if (!mbar_wait_bounded(smem_u32(&ctl->empty[s]), ph ^ 1u, abort_flag, &g_gemm_error)) {
            fail(kSiteEmpty);
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(&ctl->full[s]);
          if (kTwo) {
            // both CTAs' copies complete on the leader's barrier, which expects all of them
            const uint32_t lb = map_to_rank(fb, 0);
            if (leader) mbar_arrive_expect_tx(fb, 2 * bytes);
            tma_load_2d_pair(a_stage(s), &tmap_a, lb, kb * kElemsPerStage, m_idx * BM, pol_a);
            tma_load_2d_pair(b_stage(s), mapb, lb, kb * kElemsPerStage, n0 + int(rank) * (width / 2), pol_b);
          } else {
            mbar_arrive_expect_tx(fb, bytes);
            tma_load_2d(a_stage(s), &tmap_a, fb, kb * kElemsPerStage, m_idx * BM, pol_a);
            tma_load_2d(b_stage(s), mapb, fb, kb * kElemsPerStage, n0, pol_b);
          }
        }
      }
      if (kTwo) {
        // the leader drains the pair's copies after both have stopped (exit path below)
        st_cluster_u32(map_to_rank(smem_u32(&ctl->issued[rank]), 0), it);
      } else if (!ok) {
        // drain: the last fill of every stage must land before the CTA's memory is released
        const uint32_t first = it > (uint32_t)kStages ? it - kStages : 0u;
        for (uint32_t j = first; j < it; ++j)
          if (!mbar_wait_bounded(smem_u32(&ctl->full[j % kStages]), (j / kStages) & 1u, nullptr, &g_gemm_error))
            atomicOr(&g_gemm_error, kSiteDrain);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ---------------- MMA issuer (two-SM: the leader, for both CTAs) ----------------
      const uint32_t idesc = kTwo ? idesc_two_sm(p.idesc) : p.idesc;
      uint32_t it = 0, acc_it = 0;
      bool ok = true;
      for (int tile = first_unit; tile < num_tiles && ok; tile += unit_stride, ++acc_it) {
        const int ab = acc_it % kAccBufs;
        const uint32_t aph = (acc_it / kAccBufs) & 1u;
        if (!mbar_wait_bounded(smem_u32(&ctl->tempty[ab]), aph ^ 1u, abort_flag, &g_gemm_error)) {
          fail(kSiteTempty);
          break;
        }
        tmem_fence_after();
        const uint32_t d_tmem = tmem_base + ab * BN;
        int m_idx, n0, ks, width;
        coords(tile, m_idx, n0, ks, width);
        const uint32_t idesc_u = width == BN ? idesc : idesc_with_n(idesc, width);
        const int kb_begin = ks * p.kb_per_split, kb_end = min(num_kb, kb_begin + p.kb_per_split);
        // the stages arrive in the producer's K order (either direction); the first starts the sum
        for (int j = 0; j < kb_end - kb_begin; ++j, ++it) {
          const int s = it % kStages;
          const uint32_t ph = (it / kStages) & 1u;
          if (!mbar_wait_bounded(smem_u32(&ctl->full[s]), ph, abort_flag, &g_gemm_error)) {
            fail(kSiteFull);
            ok = false;
            break;
          }
          tmem_fence_after();
          const uint64_t adesc = make_sdesc(a_stage(s));
          const uint64_t bdesc = make_sdesc(b_stage(s));
#pragma unroll
          for (int kk = 0; kk < BK / kMmaK; ++kk) {
            // advance the start address by 32 bytes of K inside the swizzled 128-byte row
            mma_issue<kBf16, kTwo>(d_tmem, adesc + uint64_t(kk * kMmaK >> 4), bdesc + uint64_t(kk * kMmaK >> 4),
                                   idesc_u, (j != 0 || kk != 0) ? 1u : 0u);
          }
          mma_commit<kTwo>(smem_u32(&ctl->empty[s]));  // frees the stage once these MMAs have read it
        }
        if (!ok) break;
        mma_commit<kTwo>(smem_u32(&ctl->tfull[ab]));  // accumulator ready for the epilogue(s)
      }
      // all MMAs issued by this thread must finish before TMEM is released
      mma_commit<kTwo>(smem_u32(&ctl->drain));
      if (!mbar_wait_bounded(smem_u32(&ctl->drain), 0, nullptr, &g_gemm_error)) atomicOr(&g_gemm_error, kSiteDrain);
    } else if (lane == 0 && kTwo) {
      // the follower: its tensor memory is written by the leader's MMAs until the drain commit
      if (!mbar_wait_bounded(smem_u32(&ctl->drain), 0, nullptr, &g_gemm_error)) atomicOr(&g_gemm_error, kSiteDrain);
    }
  } else {
    // ---------------- epilogue: warps 2..5 ----------------
    const int q = warp & 3;                    // TMEM lane quarter this warp may access
    const int row_in_tile = q * 32 + lane;
    const int et = threadIdx.x - 64;           // 0..127
    const float s_a = p.s_a ? *p.s_a : 1.0f;
    const uint64_t pol_y = l2_policy(p.hint_y);
    const uint32_t tempty_bar = kTwo ? map_to_rank(smem_u32(&ctl->tempty[0]), 0) : smem_u32(&ctl->tempty[0]);
    uint32_t acc_it = 0;
    for (int tile = first_unit; tile < num_tiles; tile += unit_stride, ++acc_it) {
      int m_idx, col0, ks, width;
      coords(tile, m_idx, col0, ks, width);
      const int ab = acc_it % kAccBufs;
      const uint32_t aph = (acc_it / kAccBufs) & 1u;
      // column scales/bias of this tile, double-buffered by accumulator: a warp can only
      // rewrite buffer ab after every epilogue warp passed the barrier of the tile between.
      for (int j = et; j < width; j += kEpiThreads) {
        const int n = col0 + j;
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
      // one lane per warp waits; after a timeout every warp skips to the barrier above, which
      // then ends the loop uniformly (tcgen05.ld needs a converged warp)
      bool ok = true;
      if (lane == 0 && !mbar_wait_bounded(smem_u32(&ctl->tfull[ab]), aph, abort_flag, &g_gemm_error)) {
        fail(kSiteTfull);
        ok = false;
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (epi_bar_any(!ok)) continue;  // the four warps take the same path
      tmem_fence_after();
      const int m = m_idx * BM + row_in_tile;
      uint16_t* yrow = p.y + (int64_t)m * p.ldy;
      const uint32_t tbase = tmem_base + (uint32_t(q * 32) << 16) + ab * BN;
      if (S > 1) {
        // split-K: this unit's fp32 partial rows go to the workspace (unscaled)
        float* prow = p.part + ((int64_t)ks * p.M + m) * p.ldp;
#pragma unroll 1
        for (int c = 0; c < width / 32; ++c) {
          const int n0 = col0 + c * 32;
          if (n0 >= p.N) break;  // warp-uniform
          uint32_t r[32];
          tmem_ld32(tbase + c * 32, r);
          if (m < p.M) {
            if (n0 + 32 <= p.N) {
              float4* dst = reinterpret_cast<float4*>(prow + n0);
#pragma unroll
              for (int v = 0; v < 8; ++v)
                dst[v] = make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                     __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (n0 + j < p.N) prow[n0 + j] = __uint_as_float(r[j]);
            }
          }
        }
        tmem_fence_before();
        if (kTwo)
          arrive_cluster(tempty_bar + ab * uint32_t(sizeof(uint64_t)));
        else
          mbar_arrive(tempty_bar + ab * uint32_t(sizeof(uint64_t)));
        continue;
      }
#pragma unroll 1
      for (int c = 0; c < width / 32; ++c) {
        const int n0 = col0 + c * 32;
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
              st_global_v4(dst + v, make_uint4(w[0], w[1], w[2], w[3]), pol_y);
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
      if (kTwo)
        arrive_cluster(tempty_bar + ab * uint32_t(sizeof(uint64_t)));
      else
        mbar_arrive(tempty_bar + ab * uint32_t(sizeof(uint64_t)));
    }
  }

  __syncwarp();
  if constexpr (kTwo) {
    // Every copy either producer issued must have landed before either CTA's shared memory
    // is released. Both copies of a stage complete on the leader's barrier; once both
    // producers have stopped (their counts are in the leader's block), the leader accounts
    // for the halves that were never issued and waits for the rest.
    __syncthreads();
    pair_sync();
    if (leader && threadIdx.x == 0) {
      const uint32_t n0 = ctl->issued[0], n1 = ctl->issued[1];
      const uint32_t hi = n0 > n1 ? n0 : n1;
      // a producer fills stage j only after the MMAs of stage j - kStages finished, so
      // everything below hi - kStages is complete; each j above it is its stage's open phase
      for (uint32_t j = hi > uint32_t(kStages) ? hi - kStages : 0u; j < hi; ++j) {
        const uint32_t fb = smem_u32(&ctl->full[j % kStages]);
        // both CTAs walk the same units, each unit with the same number of K blocks when
        // units have fewer columns (the tail is never split along K)
        int jm, jn, jks, jw = BN;
        if (TS > 1) coords(first_unit + int(j / uint32_t(num_kb)) * unit_stride, jm, jn, jks, jw);
        const uint32_t jb = stage_bytes_for(jw);
        if (j >= n0) mbar_arrive_expect_tx(fb, jb);  // only the follower filled it
        else if (j >= n1) mbar_complete_tx(fb, jb);  // the follower's half never came
        if (!mbar_wait_bounded(fb, (j / kStages) & 1u, nullptr, &g_gemm_error)) atomicOr(&g_gemm_error, kSiteDrain);
      }
    }
  }
  tmem_fence_before();
  __syncthreads();
  if (kTwo) pair_sync();  // the peer's copies, commits and arrivals are done
  tmem_fence_after();
  if (warp == 1) {
    __syncwarp();
    if (kTwo)
      asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" :: "r"(tmem_base), "n"(kTmemCols) : "memory");
    else
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(tmem_base), "n"(kTmemCols) : "memory");
  }
}

constexpr int kMaxSplitParts = 16;  // largest K split (the host planner's limit)

// Split-K epilogue: Y[m, n] = bf16(s_a * s_w[n] * sum_j part[j][m][n] (+ bias[n])), the splits
// summed in order 0, 1, ... (deterministic). One thread per four consecutive columns of a row;
// the partials were written by the GEMM just before (L2-resident), read once.
__global__ void __launch_bounds__(256)
splitk_reduce_kernel(const float* __restrict__ part, int64_t ldp, int splits, int M, int N,
                     const float* __restrict__ s_a, const float* __restrict__ s_w, int per_channel,
                     const uint16_t* __restrict__ bias, uint16_t* __restrict__ y, int64_t ldy, int y_vec) {
  pdl_trigger();
  pdl_wait();  // the partials come from the GEMM just before
  const float sa = s_a ? *s_a : 1.0f;
  const int c4 = (N + 3) >> 2;
  const int64_t items = int64_t(M) * c4;
  const int64_t plane = int64_t(M) * ldp;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < items; i += int64_t(gridDim.x) * blockDim.x) {
    const int m = int(i / c4);
    const int n = int(i - int64_t(m) * c4) * 4;
    const float* src = part + int64_t(m) * ldp + n;
    // every split's load in flight at once (one memory round trip), then the sum in split order
    float4 v[kMaxSplitParts];
#pragma unroll
    for (int j = 0; j < kMaxSplitParts; ++j)
      v[j] = j < splits ? __ldcs(reinterpret_cast<const float4*>(src + j * plane)) : make_float4(0.f, 0.f, 0.f, 0.f);
    float4 acc = v[0];
#pragma unroll
    for (int j = 1; j < kMaxSplitParts; ++j) {
      if (j < splits) {
        acc.x += v[j].x; acc.y += v[j].y; acc.z += v[j].z; acc.w += v[j].w;
      }
    }
    const float a4[4] = {acc.x, acc.y, acc.z, acc.w};
    float o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int nn = min(n + e, N - 1);  // columns past N are computed on a valid index, not stored
      o[e] = fmaf(a4[e], sa * s_w[per_channel ? nn : 0], bias ? bf16_bits_to_float(bias[nn]) : 0.0f);
    }
    uint16_t* yr = y + int64_t(m) * ldy;
    if (y_vec && n + 4 <= N) {
      *reinterpret_cast<uint2*>(yr + n) = make_uint2(pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]));
    } else {
      for (int e = 0; e < 4; ++e)
        if (n + e < N) yr[n + e] = __bfloat16_as_ushort(__float2bfloat16_rn(o[e]));
    }
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

int env_int(const char* name, int dflt) {
  const char* e = std::getenv(name);
  return (e && e[0]) ? std::atoi(e) : dflt;
}

// Run-time switches (read once per process): FP8W8A8_GEMM_PAIR=0 selects one CTA per tile;
// FP8W8A8_GEMM_GROUP_N fixes the raster group; FP8W8A8_GEMM_L2_MB sets the largest W the
// raster keeps hot whole; FP8W8A8_GEMM_L2HINT=0 drops the eviction hints.
struct GemmSwitches {
  bool pair;
  int group_n;
  int64_t l2_budget;
  bool hints;
  int tail;  // largest column split of the last wave's tiles (1: none)
  bool fill;  // also split every tile (up to 4 ways) when the whole grid is one partial wave
  int serpentine;  // -1: planned, 0: never, 1: always
};

const GemmSwitches& switches() {
  static const GemmSwitches s = [] {
    GemmSwitches v;
    v.pair = env_int("FP8W8A8_GEMM_PAIR", 2) != 0;
    v.group_n = env_int("FP8W8A8_GEMM_GROUP_N", 0);
    v.l2_budget = int64_t(std::max(1, env_int("FP8W8A8_GEMM_L2_MB", 72))) << 20;
    v.hints = env_int("FP8W8A8_GEMM_L2HINT", 1) != 0;
    const int t = env_int("FP8W8A8_GEMM_TAIL", 2);
    v.tail = t >= 4 ? 4 : t >= 2 ? 2 : 1;
    v.fill = env_int("FP8W8A8_GEMM_FILL", 1) != 0;
    v.serpentine = env_int("FP8W8A8_GEMM_SERPENTINE", -1);
    return v;
  }();
  return s;
}

// True when p is memory of device `dev` itself. The pair mode's tensor maps may only cover
// this GPU's own memory: pinned or managed host memory, and memory of another GPU, take the
// single-CTA kernel.
bool local_device_memory(const void* p, int dev) {
  cudaPointerAttributes at = {};
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return at.type == cudaMemoryTypeDevice && at.device == dev;
}

PerDeviceCache<const void*, int> g_attr_cache;   // kernel -> attributes set on this device
PerDeviceCache<const void*, int> g_pair_cache;   // kernel -> co-resident clusters of two

// Kernel attributes (dynamic shared memory) are per device: set once on each.
bool ensure_attributes(int dev, const void* kernel) {
  int done = 0;
  return g_attr_cache.get(dev, kernel, &done, [&](int* v) {
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(gemm::kSmemBytes)) !=
        cudaSuccess) {
      cudaGetLastError();
      return false;
    }
    *v = 1;
    return true;
  });
}

// Resident clusters of two for the pair kernel on device `dev`: clusters must fit in one
// GPC, so GPCs with an odd number of free SMs leave one SM out.
int pair_clusters(int dev, const void* kernel) {
  int n = 0;
  g_pair_cache.get(dev, kernel, &n, [&](int* v) {
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(gemm::kThreads);
    cfg.dynamicSmemBytes = gemm::kSmemBytes;
    cfg.gridDim = dim3(2 * 64);  // any multiple of the cluster size
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(v, kernel, &cfg) != cudaSuccess) {
      cudaGetLastError();
      return false;
    }
    if (std::getenv("FP8W8A8_DEBUG")) std::fprintf(stderr, "fp8w8a8: gemm pairs resident on device %d: %d\n", dev, *v);
    return true;
  });
  return n;
}

}  // namespace

namespace {

// Small M, where all tiles fit in half the slots (CTA pairs or CTAs): every tile is split by
// columns into 2 or 4 units over all of K. Measured per layer on a GB300 against the K split
// (Mistral-7B and TinyLlama linears at 33..512 tokens): quarter tiles took TinyLlama qkv at 128
// tokens 15.4 -> 11.8 us and Mistral-7B qkv 22.6 -> 17.9 us, and beat the K split up to 32 K
// blocks (TinyLlama qkv at 33 tokens 13.3 -> 11.8 us); with longer K (the down projections'
// 44-112 blocks) the K split stays far ahead.
constexpr int kFillMaxKb = 32;

bool fill_applies(int units, int slots) { return units > 0 && 2 * units <= slots && switches().fill; }

}  // namespace

// The launch configuration (host logic only; see GemmPlan).
GemmPlan plan_gemm(const void* a, int64_t lda_bytes, const void* w, int64_t ldw_bytes, int M, int N, int dev,
                   int num_sms, int pair_clusters_available) {
  return plan_gemm_model(lda_bytes, ldw_bytes, M, N, local_device_memory(a, dev) && local_device_memory(w, dev),
                         num_sms, pair_clusters_available);
}

GemmPlan plan_gemm_model(int64_t lda_bytes, int64_t ldw_bytes, int M, int N, bool local, int num_sms,
                         int pair_clusters_available) {
  using namespace gemm;
  (void)lda_bytes;
  const GemmSwitches& sw = switches();
  GemmPlan pl;
  pl.m_tiles = (M + BM - 1) / BM;
  pl.n_tiles = (N + BN - 1) / BN;
  pl.two_sm = sw.pair && pl.m_tiles >= 2 && 2 * pair_clusters_available >= (3 * num_sms) / 4 && local;
  const int m_units = pl.two_sm ? (pl.m_tiles + 1) / 2 : pl.m_tiles;
  const int units = m_units * pl.n_tiles;
  pl.splits = 1;
  pl.grid = pl.two_sm ? 2 * std::min(units, pair_clusters_available) : std::min(units, num_sms);
  // raster (GB300 ncu sweeps of the group size, hints on and off): when all of W fits the
  // budget it is kept hot (loaded evict_last, qA evict_first) while the row blocks stream past;
  // otherwise column groups of a ~28 MB W slice with no hints. Keeping qA hot instead (one
  // column at a time, W evict_first) re-read qA ~13 times on the 117 MB gate_up layer.
  // With a single row block (or pair) every W tile is read once: W streams (evict_first) and
  // the few qA rows, read by every column tile, stay (evict_last).
  const int64_t w_bytes = int64_t(N) * ldw_bytes;
  const int64_t w_tile_bytes = int64_t(BN) * ldw_bytes;
  (void)lda_bytes;
  pl.hint_a = pl.hint_b = kHintNormal;
  if (m_units == 1) {
    pl.group_n = pl.n_tiles;
    pl.hint_a = kHintLast;
    pl.hint_b = kHintFirst;
  } else if (w_bytes <= sw.l2_budget) {
    pl.group_n = pl.n_tiles;
    pl.hint_a = kHintFirst;
    pl.hint_b = kHintLast;
  } else {
    pl.group_n = int(std::max<int64_t>(1, std::min<int64_t>(pl.n_tiles, (int64_t(28) << 20) / w_tile_bytes)));
  }
  if (sw.group_n > 0) pl.group_n = std::min(sw.group_n, pl.n_tiles);
  pl.hint_y = kHintFirst;  // Y is written once
  if (!sw.hints) pl.hint_a = pl.hint_b = pl.hint_y = kHintNormal;
  // K direction: a W larger than half of the L2 budget is swept once per wave of row blocks and
  // falls out of L2 before the next wave re-reads it; walking K backwards on every other unit
  // makes a wave start on the blocks the previous one read last (measured on the 59 MB down
  // projection: 12 % fewer DRAM reads, 1.4 % faster; a W that stays in L2 gains nothing)
  pl.serpentine = sw.serpentine >= 0 ? sw.serpentine : (m_units > 1 && w_bytes > sw.l2_budget / 2 ? 1 : 0);
  // the last wave: when fewer tiles than slots are left after the full waves, split each of
  // them by columns into 2 or 4 units (all of K each) so that the wave ends sooner
  const int slots = pl.two_sm ? pair_clusters_available : num_sms;  // co-resident CTA pairs or CTAs
  pl.tail_split = 1;
  pl.tail_start = units;
  const int rem = slots > 0 ? units % slots : 0;
  if (units > slots && rem > 0) {
    for (int f = sw.tail; f >= 2; f /= 2)
      if (f * rem <= slots) {
        pl.tail_split = f;
        pl.tail_start = units - rem;
        break;
      }
  } else if (fill_applies(units, slots)) {
    // one partial wave only (small M): every tile split by columns, as far as the slots allow
    for (int f = 4; f >= 2; f /= 2)
      if (f * units <= slots) {
        pl.tail_split = f;
        pl.tail_start = 0;
        break;
      }
  }
  if (pl.tail_split > 1) {
    const int split_units = pl.tail_start + (units - pl.tail_start) * pl.tail_split;
    pl.grid = pl.two_sm ? 2 * std::min(split_units, pair_clusters_available) : std::min(split_units, num_sms);
  }
  return pl;
}

namespace {

// Split count for `units` work units on `slots` parallel slots with `num_kb` K blocks each, for
// M x N outputs. Time model in us, fitted to GB300 measurements of the Mistral-7B and TinyLlama
// linears at M = 32, 64 and 128 with every split count forced: each of ceil(units * S / slots)
// waves streams ceil(num_kb / S) K blocks at ~0.38 us a block, the first ~4 of them hidden behind
// the pipeline fill; a split adds ~2 us (the reduce kernel) and ~0.5 us per MB of fp32 partials
// (written by the GEMM, read back by the reduce kernel). A split is taken only if it saves 1.5 us.
int choose_splits(int units, int slots, int num_kb, int64_t M, int64_t N, int max_splits) {
  constexpr double kBlockUs = 0.38, kSplitUs = 2.0, kPartialUsPerMB = 0.5, kMinGainUs = 1.5;
  constexpr int kHiddenBlocks = 4;
  auto cost = [&](int S, int kbs) {
    const double waves = double((int64_t(units) * S + slots - 1) / slots);
    double t = waves * std::max(kbs - kHiddenBlocks, 0) * kBlockUs;
    if (S > 1) t += kSplitUs + kPartialUsPerMB * double(splitk_bytes(M, N, S)) / 1e6;
    return t;
  };
  const double base = cost(1, num_kb);
  int best = 1;
  double best_cost = base;
  for (int S = 2; S <= std::min(max_splits, num_kb); ++S) {
    const int kbs = (num_kb + S - 1) / S;
    if ((num_kb + kbs - 1) / kbs != S) continue;  // every split owns blocks
    const double c = cost(S, kbs);
    if (c < best_cost) {
      best = S;
      best_cost = c;
    }
  }
  return best_cost < base - kMinGainUs ? best : 1;
}

constexpr int kMaxSplits = gemm::kMaxSplitParts;

}  // namespace

size_t splitk_bytes(int64_t M, int64_t N, int splits) {
  if (splits <= 1 || M <= 0 || N <= 0) return 0;
  const int64_t ldp = (N + 3) / 4 * 4;
  return size_t(splits) * size_t(M) * size_t(ldp) * 4;
}

int plan_splits(int64_t M, int64_t N, int64_t K, int num_sms, int pair_slots, size_t ws_bytes) {
  using namespace gemm;
  if (M <= 0 || N <= 0 || K <= 0) return 1;
  const int m_tiles = int((M + BM - 1) / BM), n_tiles = int((N + BN - 1) / BN);
  const int num_kb = int((K + BK - 1) / BK);
  const bool two = pair_slots > 0 && m_tiles >= 2 && 2 * pair_slots >= (3 * num_sms) / 4;
  const int units = (two ? (m_tiles + 1) / 2 : m_tiles) * n_tiles;
  const int slots = two ? pair_slots : num_sms;
  // the partials should stay in L2 (written once by the GEMM, read once by the reduce kernel)
  const size_t cap = std::min(ws_bytes, size_t(64) << 20);
  int max_s = kMaxSplits;
  while (max_s > 1 && splitk_bytes(M, N, max_s) > cap) --max_s;
  const int forced = env_int("FP8W8A8_GEMM_SPLITK", 0);  // measurement override
  if (forced > 0) {
    // the largest count not above the request for which every split owns K blocks
    const int S = std::max(1, std::min({forced, max_s, num_kb}));
    const int kbs = (num_kb + S - 1) / S;
    return (num_kb + kbs - 1) / kbs;
  }
  // measured: with CTA pairs (two or more row blocks) a split never paid for itself
  if (two) return 1;
  // short K on few tiles: the column split of every tile (plan_gemm) is faster
  if (num_kb <= kFillMaxKb && fill_applies(units, slots)) return 1;
  return choose_splits(units, slots, num_kb, M, N, max_s);
}

namespace {

template <bool kBf16>
int launch_kind(const void* a, int64_t lda_bytes, const float* s_a, const void* w, int64_t ldw_bytes,
                const float* s_w, int per_channel, const uint16_t* bias, uint16_t* y, int64_t ldy, int M, int N,
                int K, uint32_t idesc, int num_sms, cudaStream_t stream, const SplitK& split) {
  using namespace gemm;
  auto single = gemm_kernel<kBf16, false>;
  auto two_sm = gemm_kernel<kBf16, true>;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (!ensure_attributes(dev, reinterpret_cast<const void*>(single)) ||
      !ensure_attributes(dev, reinterpret_cast<const void*>(two_sm)))
    return 1;
  const int clusters = switches().pair ? pair_clusters(dev, reinterpret_cast<const void*>(two_sm)) : 0;
  GemmPlan pl = plan_gemm(a, lda_bytes, w, ldw_bytes, M, N, dev, num_sms, clusters);
  const int S = std::max(1, split.splits);
  const int num_kb = kBf16 ? (K + BK / 2 - 1) / (BK / 2) : (K + BK - 1) / BK;  // K blocks of 128 bytes
  const int tiles = (pl.two_sm ? (pl.m_tiles + 1) / 2 : pl.m_tiles) * pl.n_tiles;
  const int units = tiles * S;

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
  p.m_tiles = pl.m_tiles;
  p.n_tiles = pl.n_tiles;
  p.group_n = pl.group_n;
  p.y_vec = (ldy % 8 == 0) && (reinterpret_cast<uintptr_t>(y) % 16 == 0);
  p.idesc = idesc;
  p.hint_a = pl.hint_a;
  p.hint_b = pl.hint_b;
  p.hint_y = pl.hint_y;
  p.k_splits = S;
  p.kb_per_split = (num_kb + S - 1) / S;
  p.part = split.part;
  p.ldp = split.ldp;
  if (S > 1 && (split.part == nullptr || (num_kb + p.kb_per_split - 1) / p.kb_per_split != S)) return 4;
  p.tail_split = S > 1 ? 1 : pl.tail_split;  // a K split already fills the GPU
  p.tail_start = p.tail_split > 1 ? pl.tail_start : units;
  const int work = p.tail_split > 1 ? p.tail_start + (tiles - p.tail_start) * p.tail_split : units;
  pl.grid = pl.two_sm ? 2 * std::min(work, clusters) : std::min(work, num_sms);
  p.serpentine = pl.serpentine;

  CUtensorMap ma, mb, mbt;
  const uint32_t b_rows = pl.two_sm ? BN / 2 : BN;
  if (!make_tensor_map(&ma, a, kBf16, M, K, lda_bytes, BM) ||
      !make_tensor_map(&mb, w, kBf16, N, K, ldw_bytes, b_rows))
    return 2;
  mbt = mb;
  if (p.tail_split > 1 && !make_tensor_map(&mbt, w, kBf16, N, K, ldw_bytes, b_rows / p.tail_split)) return 2;

  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cfg.gridDim = dim3(unsigned(pl.grid));
  cudaLaunchAttribute attr[1];
  cfg.attrs = attr;
  if (pl.two_sm) {
    // Launched without programmatic stream serialization: the pair's grid starts only after
    // the kernel before it has finished, so no CTA pair becomes resident while CTAs of an
    // earlier kernel still hold the SMs (its own trigger still lets the next kernel start early).
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, two_sm, ma, mb, mbt, p) != cudaSuccess) return 3;
  } else {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, single, ma, mb, mbt, p) != cudaSuccess) return 3;
  }
  if (S == 1) return 0;
  // the split-K epilogue, launched early (programmatic) so it is resident when the GEMM ends
  const int64_t items = int64_t(M) * ((N + 3) / 4);
  cudaLaunchConfig_t rc = {};
  rc.blockDim = dim3(256);
  rc.gridDim = dim3(unsigned(std::max<int64_t>(1, std::min<int64_t>((items + 255) / 256, int64_t(num_sms) * 8))));
  rc.stream = stream;
  cudaLaunchAttribute rattr[1];
  rattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  rattr[0].val.programmaticStreamSerializationAllowed = 1;
  rc.attrs = rattr;
  rc.numAttrs = 1;
  return cudaLaunchKernelEx(&rc, splitk_reduce_kernel, static_cast<const float*>(split.part), split.ldp, S, M, N,
                            s_a, s_w, per_channel, bias, y, ldy, p.y_vec) == cudaSuccess ? 0 : 3;
}

// Shared launch: operands are FP8 (ld in bytes) or bf16 (ld in bytes as well).
int launch_gemm(bool bf16, const void* a, int64_t lda_bytes, const float* s_a, const void* w, int64_t ldw_bytes,
                const float* s_w, int per_channel, const uint16_t* bias, uint16_t* y, int64_t ldy, int M, int N,
                int K, uint32_t idesc, int num_sms, cudaStream_t stream, const SplitK& split) {
  return bf16 ? launch_kind<true>(a, lda_bytes, s_a, w, ldw_bytes, s_w, per_channel, bias, y, ldy, M, N, K, idesc,
                                  num_sms, stream, split)
              : launch_kind<false>(a, lda_bytes, s_a, w, ldw_bytes, s_w, per_channel, bias, y, ldy, M, N, K, idesc,
                                   num_sms, stream, split);
}

}  // namespace

int gemm_launch(const uint8_t* qa, int64_t ldqa, const float* s_a, const uint8_t* qw, int64_t ldqw,
                const float* s_w, int per_channel, const uint16_t* bias, uint16_t* y, int64_t ldy,
                int M, int N, int K, int fmt_a, int fmt_w, int num_sms, cudaStream_t stream, const SplitK& split) {
  return launch_gemm(false, qa, ldqa, s_a, qw, ldqw, s_w, per_channel, bias, y, ldy, M, N, K,
                     gemm::make_idesc(fmt_a, fmt_w), num_sms, stream, split);
}

int gemm_bf16_launch(const uint16_t* a, int64_t lda, const uint16_t* w, int64_t ldw, const float* s_w,
                     int per_channel, const uint16_t* bias, uint16_t* y, int64_t ldy, int M, int N, int K,
                     int num_sms, cudaStream_t stream) {
  return launch_gemm(true, a, lda * 2, nullptr, w, ldw * 2, s_w, per_channel, bias, y, ldy, M, N, K,
                     gemm::kIdescBf16, num_sms, stream, SplitK());
}

GemmPlan gemm_plan(const void* a, int64_t lda_bytes, const void* w, int64_t ldw_bytes, int M, int N, int num_sms) {
  int dev = 0;
  GemmPlan none{};
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return none;
  }
  const void* k = reinterpret_cast<const void*>(gemm::gemm_kernel<false, true>);
  if (!ensure_attributes(dev, k)) return none;
  const int clusters = switches().pair ? pair_clusters(dev, k) : 0;
  return plan_gemm(a, lda_bytes, w, ldw_bytes, M, N, dev, num_sms, clusters);
}

SplitK gemm_split_plan(const uint8_t* qa, int64_t ldqa, const uint8_t* qw, int64_t ldqw, int M, int N, int K,
                       int num_sms, void* ws, size_t ws_bytes) {
  SplitK sk;
  if (ws == nullptr || ws_bytes == 0) return sk;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return sk;
  }
  const void* k = reinterpret_cast<const void*>(gemm::gemm_kernel<false, true>);
  if (!ensure_attributes(dev, k)) return sk;
  const int clusters = switches().pair ? pair_clusters(dev, k) : 0;
  const GemmPlan pl = plan_gemm(qa, ldqa, qw, ldqw, M, N, dev, num_sms, clusters);
  const int S = plan_splits(M, N, K, num_sms, pl.two_sm ? clusters : 0, ws_bytes);
  if (S <= 1) return sk;
  sk.splits = S;
  sk.part = static_cast<float*>(ws);
  sk.ldp = (int64_t(N) + 3) / 4 * 4;
  return sk;
}

unsigned int gemm_read_and_clear_error() {
  unsigned int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, gemm::g_gemm_error, sizeof(v)) != cudaSuccess) return 0;
  cudaMemcpyToSymbol(gemm::g_gemm_error, &zero, sizeof(zero));
  return v;
}

}  // namespace fp8k
