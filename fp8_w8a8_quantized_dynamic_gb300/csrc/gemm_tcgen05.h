// Internal interface between the C-ABI layer and the tcgen05 GEMM translation unit.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace fp8k {

struct GemmParams {
  int M, N, K;
  const float* s_a;  // null: 1 (weight-only product)
  const float* s_w;
  int per_channel;
  const uint16_t* bias;
  uint16_t* y;
  int64_t ldy;
  int m_tiles, n_tiles, group_n;
  int y_vec;
  uint32_t idesc;  // tcgen05 instruction descriptor (carries the two operand formats)
  int hint_a, hint_b, hint_y;  // L2 eviction priority of qA / qW loads and Y stores (0 normal, 1 first, 2 last)
  // split-K: each tile's K blocks are divided among k_splits work units (kb_per_split blocks
  // each); every unit writes its unscaled fp32 partial to part [k_splits][M][ldp] and a reduce
  // kernel sums them in split order and runs the epilogue. k_splits == 1: Y written directly.
  int k_splits, kb_per_split;
  float* part;
  int64_t ldp;
  // last wave: work units from tail_start on are tiles split by columns into tail_split units
  // of BN / tail_split columns (all of K); tail_split == 1: no such units
  int tail_start, tail_split;
  int serpentine;  // 1: every other work unit of a CTA walks its K blocks backwards
};

// Workspace of a split-K GEMM: the fp32 partials [splits][M][ldp].
struct SplitK {
  int splits = 1;          // 1: K is not split
  float* part = nullptr;
  int64_t ldp = 0;         // row stride of the partials (elements, multiple of 4)
};

// Bytes of split-K workspace for `splits` (the fp32 partials).
size_t splitk_bytes(int64_t M, int64_t N, int splits);

// Split count for an M x N x K FP8 GEMM on a GPU with `num_sms` SMs and `pair_slots` co-resident
// CTA pairs (0: no pair mode), limited to what `ws_bytes` of split workspace holds. Host logic.
int plan_splits(int64_t M, int64_t N, int64_t K, int num_sms, int pair_slots, size_t ws_bytes);

// Launch configuration of one GEMM call (host logic only).
struct GemmPlan {
  int two_sm;    // 1: CTA pairs on the two-SM MMA; 0: one CTA per tile
  int grid;      // CTAs launched (persistent)
  int m_tiles, n_tiles;
  int group_n;   // raster group (column tiles per group)
  int hint_a, hint_b, hint_y;
  int splits;    // K split count (1: none)
  int tail_split;  // column split of the last wave's tiles (1: none; never with a K split)
  int tail_start;  // first work unit of the split tail
  int serpentine;  // 1: every other work unit of a CTA walks K backwards
};

// The plan for operands a [M, lda_bytes] and w [N, ldw_bytes] on device `dev` with
// `pair_clusters_available` co-resident CTA pairs: the two-SM mode needs at least two row
// blocks, pairs on 3/4 of the SMs, and both operands in this device's own memory.
GemmPlan plan_gemm(const void* a, int64_t lda_bytes, const void* w, int64_t ldw_bytes, int M, int N, int dev,
                   int num_sms, int pair_clusters_available);

// The same rules without a device: `local` says whether both operands are this GPU's own memory,
// `pair_clusters_available` how many CTA pairs are co-resident (host logic only).
GemmPlan plan_gemm_model(int64_t lda_bytes, int64_t ldw_bytes, int M, int N, bool local, int num_sms,
                         int pair_clusters_available);

// The plan gemm_launch would use on the current device (queries pointer attributes and occupancy).
GemmPlan gemm_plan(const void* a, int64_t lda_bytes, const void* w, int64_t ldw_bytes, int M, int N, int num_sms);

// Enqueues the persistent GEMM. Returns 0 on success, non-zero when the tensor maps could
// not be encoded or the launch failed. qa/qw: 16-byte aligned, ld multiples of 16.
// fmt_a / fmt_w: 0 = e4m3, 1 = e5m2. split: K split (the GEMM, then the reduce kernel), or
// the default of no split.
int gemm_launch(const uint8_t* qa, int64_t ldqa, const float* s_a, const uint8_t* qw, int64_t ldqw,
                const float* s_w, int per_channel, const uint16_t* bias, uint16_t* y, int64_t ldy,
                int M, int N, int K, int fmt_a, int fmt_w, int num_sms, cudaStream_t stream,
                const SplitK& split = SplitK());

// The split plan gemm_launch would use for these FP8 operands with `ws_bytes` of split
// workspace at `ws` (256-byte aligned), on the current device.
SplitK gemm_split_plan(const uint8_t* qa, int64_t ldqa, const uint8_t* qw, int64_t ldqw, int M, int N, int K,
                       int num_sms, void* ws, size_t ws_bytes);

// bf16 x bf16 GEMM on the same kernel (tcgen05 kind::f16) for the weight-only product:
//   Y[m, n] = bf16( s_w[n] * sum_k A[m, k] W[n, k]  (+ bias[n]) ).
// a, w: bf16, 16-byte aligned, lda / ldw in elements with lda * 2 and ldw * 2 multiples of 16.
int gemm_bf16_launch(const uint16_t* a, int64_t lda, const uint16_t* w, int64_t ldw, const float* s_w,
                     int per_channel, const uint16_t* bias, uint16_t* y, int64_t ldy, int M, int N, int K,
                     int num_sms, cudaStream_t stream);

// 2-D FP8 (byte) tensor map over [rows, K] (row stride ld bytes), box [box_rows rows x 128 bytes],
// 128-byte swizzle, zero fill outside the matrix. False when the encoder is unavailable or fails.
bool make_fp8_tensor_map(CUtensorMap* map, const uint8_t* base, int64_t rows, int64_t K, int64_t ld,
                         uint32_t box_rows);

// Device-side error bits recorded by the GEMM kernel on the current device (read, then cleared).
unsigned int gemm_read_and_clear_error();

}  // namespace fp8k
