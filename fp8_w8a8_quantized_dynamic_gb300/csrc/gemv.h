// Host-visible interface of the decode GEMV (kernels in gemv.cuh, instantiated in gemv.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace fp8k {
namespace gemv {

constexpr int kConsumerWarps = 8;
constexpr int kThreads = 32 * (kConsumerWarps + 1);  // + one producer warp
constexpr int kConsumerThreads = 32 * kConsumerWarps;
constexpr int kRows = 16 * kConsumerWarps;            // 128 rows per row block
constexpr int kTileK = 128;                           // bytes of K per tile (one swizzle row)
constexpr int kTileBytes = kRows * kTileK;            // 16 KB
constexpr int kMaxStages = 12;
constexpr int kMinStages = 4;
constexpr int kMaxTokens = 32;                        // largest M (four n8 token tiles)
constexpr int kDefaultMaxM = 32;                      // default decode crossover (M <= this runs the GEMV)
constexpr int kMaxCluster = 8;
constexpr int kMaxRowBlocks = 8;                      // per cluster (partials live in smem)

// Partials a rank receives for one row block: [source rank][its rows][act_rows tokens] fp32,
// at most (kRows + kMaxCluster) rows in total (rows per rank rounded up).
__host__ __device__ inline int part_bytes(int act_rows) { return (kRows + kMaxCluster) * act_rows * 4; }
constexpr int kMaxSlice = 4096;                       // bytes of K per rank
constexpr int kSmemLimit = 227 * 1024;
constexpr int kRegUnits = 8;  // 8-element units of A a consumer thread keeps in registers
constexpr int kQuantUnroll = 4;  // units a consumer thread quantizes per round (independent chains)
constexpr int kMaxSliceBf16 = 4096;  // K elements per rank with bf16 activations (smem permitting)

// Activation modes of the kernel.
constexpr int kModePrequant = 0;  // qA and s_a given (fp8_scaled_mm)
constexpr int kModeQuantize = 1;  // bf16 A quantized in the kernel (dynamic or static scale)
constexpr int kModeBf16 = 2;      // bf16 A used as is: weight-only product, W up-converted to bf16

struct Params {
  const uint8_t* qa;   // pre-quantized: FP8 [M, ldqa], bytes [K, ldqa) zero
  int64_t ldqa;
  const float* s_a;    // pre-quantized: activation scale (device)
  const uint16_t* a;   // quantized here: bf16 [M, lda]
  int64_t lda;
  int vec_a;           // quantized here: A rows allow 16-byte loads
  const float* s_static;  // quantized here: static activation scale (device), or null (dynamic)
  const float* s_w;    // [1] or [N]
  int per_channel;
  const uint16_t* bias;  // bf16 [N] or null
  uint16_t* y;           // bf16 [M, ldy]
  int64_t ldy;
  int M, N, K;
  int kslice;          // bytes of K per rank, multiple of kTileK
  int act_stride;      // smem row stride (bytes) of the activation slice: == 64 mod 128 for FP8
                       // activations, == 16 mod 128 for bf16 (conflict-free fragment loads);
                       // the tcgen05 path stores [K block][token][128 B] instead (stride = kslice)
  int stages;          // ring depth
  int row_blocks;      // ceil(N / kRows)
  int num_clusters;    // C
  int act_rows;        // token rows staged in smem (8 * NT); also the token stride of the partials
  int head_tiles;      // weight tiles issued before the activation loads have landed
  int cluster_amax;    // dynamic scale: 1 = exchange slice maxima over the cluster, 0 = every CTA reads all of A
  int scratch_a;       // quantize mode: 0 = A read with per-thread loads; 1 = all of A, 2 = this rank's
                       // slice, bulk-copied into ring stages [head_tiles, stages) that are idle until
                       // the stream is released
};

// Shared-memory layout (from a 1024-aligned base): ring | act | partials | barriers.
struct Layout {
  uint32_t ring, act, part, bars, total;
};

__host__ __device__ inline Layout layout(int stages, int act_stride, int act_rows, int rb_per_cluster) {
  Layout L;
  L.ring = 0;
  L.act = stages * kTileBytes;
  L.part = L.act + act_rows * act_stride;
  L.bars = L.part + rb_per_cluster * part_bytes(act_rows);
  L.total = L.bars + (2 * kMaxStages + 2) * 8;
  return L;
}

// One instantiation of the kernel: NT n8 token tiles (1: M <= 8, 2: M <= 16, 4: M <= 32), activation
// mode (kMode*), FP8 formats of the activations (fa, unused for kModeBf16) and weights (fw), and
// the main loop on tcgen05 (tc; NT >= 2 with FP8 activations) or on mma.sync.
// The second tensor map covers qA [M, K] in [8 * NT rows x 128 B] boxes (pre-quantized mode on
// tcgen05); the other kernels ignore it.
using KernelFn = void (*)(CUtensorMap, CUtensorMap, Params);
KernelFn kernel_for(int NT, int mode, int fa, int fw, bool tc);

// Enqueues the failure-path self-test kernel (a bounded wait made to run out after limit_ns).
void selftest_timeout(unsigned long long limit_ns, cudaStream_t st);

// Device-side error bits of the GEMV on the current device (read, then cleared).
unsigned int read_and_clear_error();

}  // namespace gemv
}  // namespace fp8k
