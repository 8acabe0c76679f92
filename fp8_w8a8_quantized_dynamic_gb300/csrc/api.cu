// C ABI of the FP8 W8A8 linear (declared in include/fp8w8a8.h): argument validation,
// M-based dispatch between the decode GEMV and the tcgen05 GEMM, launch configuration.
// Every step of the layer runs in this library's kernels; nothing falls back to the CPU.

#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <map>
#include <mutex>
#include <tuple>
#include <utility>

#include "fp8w8a8.h"
#include "device_common.cuh"
#include "gemm_tcgen05.h"
#include "gemv.h"
#include "quantize.cuh"

#define FP8_API extern "C" __attribute__((visibility("default")))

namespace {

using namespace fp8k;

constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1;
constexpr int kGemvMaxK = gemv::kMaxCluster * gemv::kMaxSlice;  // 32768
// Tokens up to which the GEMV quantizes A itself (two n8 token tiles). With four, the 32-token
// activation area leaves the ring too shallow to hold A, which every cluster would fetch twice
// (for the amax, then for the cast) by per-thread round trips while the weight stream waits
// (measured: 15-25 us on the Mistral-7B gate_up and down layers at 32 tokens); there A is
// quantized once beforehand and the GEMV loads the FP8 slice by TMA.
// FP8W8A8_GEMV_SELFQUANT overrides it (measurement switch; at most 32).
int64_t gemv_self_quant_max_m() {
  static const int64_t v = [] {
    const char* e = std::getenv("FP8W8A8_GEMV_SELFQUANT");
    return e ? std::max<int64_t>(0, std::min<int64_t>(std::atoi(e), gemv::kMaxTokens)) : int64_t(2 * 8);
  }();
  return v;
}

// ---------------------------------------------------------------------------
// device properties (cached per device)
// ---------------------------------------------------------------------------

struct DevInfo {
  int checked = 0;
  int supported = 0;
  int sms = 0;
};

std::mutex g_dev_mu;
DevInfo g_dev[64];

fp8_status current_device(int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FP8_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DevInfo& d = g_dev[dev];
  if (!d.checked) {
    int major = 0, minor = 0, n = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return FP8_ERR_CUDA;
    d.supported = (major == 10 && minor == 3);
    d.sms = n;
    d.checked = 1;
  }
  if (!d.supported) return FP8_ERR_UNSUPPORTED_DEVICE;
  *sms = d.sms;
  return FP8_OK;
}

// Largest M that runs the decode GEMV: FP8W8A8_GEMV_MAX_M at start-up (default
// gemv::kDefaultMaxM), then fp8_set_gemv_max_m; never above gemv::kMaxTokens.
std::atomic<int>& gemv_max_m_value() {
  static std::atomic<int> v{[] {
    const char* e = std::getenv("FP8W8A8_GEMV_MAX_M");
    const int x = e ? std::atoi(e) : gemv::kDefaultMaxM;
    return std::max(0, std::min(x, gemv::kMaxTokens));
  }()};
  return v;
}

int gemv_max_m() { return gemv_max_m_value().load(std::memory_order_relaxed); }

// The GEMV runs every M up to the crossover (default 32, its largest): measured per layer on a
// GB300 (CUDA graph replay), at 17..32 tokens the GEMV on once-quantized activations with its
// tcgen05 main loop beats or ties the split GEMM on every Mistral-7B and TinyLlama linear
// (Mistral-7B down at 32 tokens 19.9 vs 22.6 us, gate_up 29.8 vs 29.1, qkv 13.7 vs 15.6;
// TinyLlama 8.0-13.5 vs 11.1-14.8 us), and below 17 tokens by more.
bool use_gemv(int64_t M, int64_t K, int64_t N) {
  (void)N;
  return K <= kGemvMaxK && M <= gemv_max_m();
}

// Weight tiles the GEMV issues before its activation loads have landed (FP8W8A8_GEMV_HEAD
// overrides the default of 4; 0 holds the whole stream, gemv::kMaxStages lets it run free).
int gemv_head_tiles() {
  static const int v = [] {
    const char* e = std::getenv("FP8W8A8_GEMV_HEAD");
    const int x = e ? std::atoi(e) : 4;
    return std::max(0, std::min(x, 1 << 20));
  }();
  return v;
}

// FP8W8A8_GEMV_SLICE=1: the dynamic-scale GEMV always copies only each rank's slice of A and
// exchanges slice maxima over the cluster (measurement switch).
bool gemv_slice_only() {
  static const bool v = std::getenv("FP8W8A8_GEMV_SLICE") != nullptr && std::atoi(std::getenv("FP8W8A8_GEMV_SLICE")) != 0;
  return v;
}

int64_t round_up16(int64_t k) { return (k + 15) / 16 * 16; }

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Passes `e` through; with FP8W8A8_DEBUG set, a failure is also described on stderr.
cudaError_t report_cuda(cudaError_t e, const char* where) {
  static const bool debug = std::getenv("FP8W8A8_DEBUG") != nullptr;
  if (e != cudaSuccess && debug) std::fprintf(stderr, "fp8w8a8: %s: %s\n", where, cudaGetErrorString(e));
  return e;
}

// ---------------------------------------------------------------------------
// launch helpers
// ---------------------------------------------------------------------------

template <typename... KArgs, typename... Args>
fp8_status launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool pdl,
                  dim3 cluster, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster.x * cluster.y * cluster.z > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster.x;
    attr[n].val.clusterDim.y = cluster.y;
    attr[n].val.clusterDim.z = cluster.z;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return report_cuda(cudaLaunchKernelEx(&cfg, kernel, args...), "kernel launch") == cudaSuccess ? FP8_OK
                                                                                       : FP8_ERR_CUDA;
}

struct BF16Mat {
  const uint16_t* p;
  int64_t rows, cols, ld;
  int contiguous() const { return ld == cols && aligned(p, 16); }
  int vec() const { return aligned(p, 16) && ld % 8 == 0; }
};

// CTAs of the amax pass: at most the partial slots of a workspace, and a whole number per SM
// (6 on a 152-SM GB300) so that no SM carries one more CTA than the others at the end.
int amax_grid(const BF16Mat& a, int sms) {
  const int64_t units = (a.rows * a.cols + 7) / 8;
  const int64_t per_block = int64_t(kQuantThreads) * 4;
  int64_t g = (units + per_block - 1) / per_block;
  const int64_t per_sm = std::max<int64_t>(1, std::min<int64_t>(8, kAmaxMaxBlocks / std::max(sms, 1)));
  g = std::min<int64_t>(g, std::min<int64_t>(kAmaxMaxBlocks, int64_t(sms) * per_sm));
  return int(std::max<int64_t>(g, 1));
}

fp8_status launch_amax(const BF16Mat& a, float* partials, int grid, cudaStream_t st, bool pdl) {
  return launch(amax_partials_kernel, dim3(grid), dim3(kQuantThreads), 0, st, pdl, dim3(1, 1, 1), a.p, a.rows,
                a.cols, a.ld, a.contiguous(), a.vec(), partials, int(pdl));
}

bool valid_fmt(int f) { return f == kFmtE4M3 || f == kFmtE5M2; }

// Cast of A to FP8 of format `fmt`: dynamic scale from `partials` (n_partials of them), or
// the static scale *s_static when partials is null. s_out (may be null) receives the scale.
fp8_status launch_cast(const BF16Mat& a, const float* partials, int n_partials, const float* s_static, float* s_out,
                       uint8_t* q, int64_t ldq, int fmt, int sms, cudaStream_t st, bool pdl) {
  const int64_t units = a.rows * (ldq / 16);
  const int64_t g = std::max<int64_t>(1, std::min<int64_t>((units + kQuantThreads - 1) / kQuantThreads,
                                                           int64_t(sms) * 8));
  const bool narrow = units < (int64_t(1) << 31);
  auto go = [&](auto kernel) {
    return launch(kernel, dim3(unsigned(g)), dim3(kQuantThreads), 0, st, pdl, dim3(1, 1, 1), a.p, a.rows, a.cols,
                  a.ld, a.vec(), partials, n_partials, s_static, s_out, q, ldq, int(pdl));
  };
  if (fmt == kFmtE5M2)
    return narrow ? go(cast_kernel<uint32_t, kFmtE5M2>) : go(cast_kernel<uint64_t, kFmtE5M2>);
  return narrow ? go(cast_kernel<uint32_t, kFmtE4M3>) : go(cast_kernel<uint64_t, kFmtE4M3>);
}

fp8_status launch_fill_bias(const void* bias, void* y, int64_t M, int64_t N, int64_t ldy, int sms, cudaStream_t st) {
  const int64_t total = M * N;
  const int64_t g = std::max<int64_t>(1, std::min<int64_t>((total + 255) / 256, int64_t(sms) * 8));
  return launch(fill_bias_kernel, dim3(unsigned(g)), dim3(256), 0, st, true, dim3(1, 1, 1),
                static_cast<const uint16_t*>(bias), static_cast<uint16_t*>(y), M, N, ldy, 1);
}

gemv::Params gemv_params(const uint8_t* qa, int64_t ldqa, const float* s_a, const float* s_w, int per_channel,
                         const void* bias, void* y, int64_t ldy, int64_t M, int64_t N, int64_t K) {
  gemv::Params p = {};
  p.qa = qa;
  p.ldqa = ldqa;
  p.s_a = s_a;
  p.s_w = s_w;
  p.per_channel = per_channel;
  p.bias = static_cast<const uint16_t*>(bias);
  p.y = static_cast<uint16_t*>(y);
  p.ldy = ldy;
  p.M = int(M);
  p.N = int(N);
  p.K = int(K);
  return p;
}

// Dynamic shared memory the GEMV may use: the device's opt-in per-block limit minus the
// kernel's static shared memory (set as the kernel attribute on first use; cached).
int gemv_smem_limit(gemv::KernelFn kfn) {
  static std::mutex mu;
  static std::map<std::tuple<int, const void*>, int> cache;
  int dev = 0;
  cudaGetDevice(&dev);
  const void* fn = reinterpret_cast<const void*>(kfn);
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(std::make_tuple(dev, fn));
  if (it != cache.end()) return it->second;
  int optin = 0;
  cudaFuncAttributes fa = {};
  int limit = 0;
  if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) == cudaSuccess &&
      cudaFuncGetAttributes(&fa, fn) == cudaSuccess) {
    limit = std::min(optin - int(fa.sharedSizeBytes), gemv::kSmemLimit);
    if (report_cuda(cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, limit),
                    "gemv smem attribute") != cudaSuccess)
      limit = 0;
  }
  cache[std::make_tuple(dev, fn)] = limit;
  return limit;
}

// Largest number of co-resident clusters of `S` CTAs for the GEMV at `smem` bytes (cached).
int gemv_max_clusters(gemv::KernelFn kfn, int S, size_t smem) {
  static std::mutex mu;
  static std::map<std::tuple<int, const void*, int, size_t>, int> cache;
  int dev = 0;
  cudaGetDevice(&dev);
  const void* fn = reinterpret_cast<const void*>(kfn);
  const auto key = std::make_tuple(dev, fn, S, smem);
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(S * 64);
  cfg.blockDim = dim3(gemv::kThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = S;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (report_cuda(cudaOccupancyMaxActiveClusters(&n, fn, &cfg), "gemv cluster occupancy") != cudaSuccess) n = 0;
  cache[key] = n;
  return n;
}

// Persistent split-K GEMV on e4m3 activations. Picks the cluster size S (K split) and the
// number of clusters C so that the CTA with the most work streams as few 16 KB weight tiles
// as possible, every cluster holds at most kMaxRowBlocks row blocks, and the smem fits.
// Shared-memory row stride (bytes) of a K-slice of activations: FP8 rows are padded to 64 mod
// 128, bf16 rows (two bytes an element) to 16 mod 128, so the fragment loads of a warp spread
// over all banks.
// The tcgen05 main loop (tc) keeps the FP8 activations as 128-byte swizzled K blocks of
// [tokens][128 B], kslice bytes a token in all.
int gemv_act_stride(int mode, int kslice, bool tc) {
  if (mode == gemv::kModeBf16) return 2 * kslice + 16;
  if (tc) return kslice;
  return kslice % 128 == 0 ? kslice + 64 : kslice;
}

// 17 to 32 tokens with FP8 activations run the GEMV's main loop on tcgen05: four n8 token tiles
// on mma.sync take about twice the weight stream's time per tile, while at two tiles mma.sync
// keeps up and the tensor-memory round trip only adds latency (measured per layer on a GB300:
// Mistral-7B gate_up at M = 32, 49.6 -> 40.5 us; qkv at M = 12, 12.3 -> 12.9 us).
// FP8W8A8_GEMV_TC: 0 never, 2 from two token tiles on (measurement switches).
bool gemv_tc(int NT, int mode) {
  static const int from = [] {
    const char* e = std::getenv("FP8W8A8_GEMV_TC");
    const int v = e ? std::atoi(e) : 4;
    return v <= 0 ? 1 << 20 : v <= 2 ? 2 : 4;
  }();
  return NT >= from && mode == gemv::kModePrequant;
}

// One GEMV launch configuration: cluster size S (K split), clusters C, ring depth, K slice per
// rank, activation layout and start-up (host logic only).
struct GemvConfig {
  bool ok = false;
  int S = 1, C = 1, stages = gemv::kMinStages, kslice = gemv::kTileK, act_stride = 0, act_rows = 8;
  int head_tiles = 0, cluster_amax = 0, scratch_a = 0;
  size_t smem = 0;
};

// Picks the cluster size S and the number of clusters C so that the CTA with the most work
// streams as few 16 KB weight tiles as possible, every cluster holds at most kMaxRowBlocks row
// blocks and the shared memory fits smem_limit; cmax_of(S) gives the co-resident clusters of S
// CTAs at smem_limit. Then the activation staging (bulk copy of A into idle ring stages when
// A's rows are 16-byte aligned) and where the dynamic maximum comes from.
template <typename ClustersOf>
GemvConfig gemv_configure(int M, int N, int K, int mode, bool tc, bool vec_a, bool static_scale, int smem_limit,
                          ClustersOf&& cmax_of) {
  using namespace gemv;
  GemvConfig g;
  const int R = (N + kRows - 1) / kRows;
  const int KT = (K + kTileK - 1) / kTileK;
  const bool dyn = mode == kModeQuantize;
  const int max_slice = mode == kModeBf16 ? kMaxSliceBf16 : kMaxSlice;
  const int NT = M <= 8 ? 1 : M <= 16 ? 2 : 4;
  g.act_rows = 8 * NT;
  auto smem_for = [&](int stg, int act_stride, int nrb) {
    return size_t(layout(stg, act_stride, g.act_rows, nrb).total) + 1024;
  };
  int best_cost = -1;
  for (int S = 1; S <= kMaxCluster; ++S) {
    if (S > KT) break;
    const int slice_tiles = (KT + S - 1) / S;
    if ((KT + slice_tiles - 1) / slice_tiles != S) continue;  // every rank must own tiles
    const int kslice = slice_tiles * kTileK;
    if (kslice > max_slice) continue;
    const int act_stride = gemv_act_stride(mode, kslice, tc);
    if (smem_for(kMinStages, act_stride, 1) > size_t(smem_limit)) continue;
    // co-resident clusters at the largest shared memory any configuration may take (a lower
    // bound for every configuration, so the grid never runs in waves)
    const int cmax = cmax_of(S);
    if (cmax <= 0) continue;
    int C = std::min(cmax, R);
    const int nrb = (R + C - 1) / C;
    if (nrb > kMaxRowBlocks) continue;
    C = (R + nrb - 1) / nrb;
    if (smem_for(kMinStages, act_stride, nrb) > size_t(smem_limit)) continue;
    // streamed tiles of the busiest CTA, plus (dynamic mode) its activation prologue: each
    // batch of kRegUnits A loads per consumer thread costs about as much as two weight tiles
    const int units = M * (kslice / 8);
    const int batches = dyn ? (units + kRegUnits * kConsumerThreads - 1) / (kRegUnits * kConsumerThreads) : 0;
    const int cost = nrb * slice_tiles + 2 * (batches > 1 ? batches : 0);
    if (best_cost < 0 || cost < best_cost) {
      // with the row blocks known, the deepest ring that fits
      int stg = kMinStages;
      while (stg < kMaxStages && smem_for(stg + 1, act_stride, nrb) <= size_t(smem_limit)) ++stg;
      best_cost = cost;
      g.S = S;
      g.C = C;
      g.stages = stg;
      g.kslice = kslice;
      g.smem = smem_for(stg, act_stride, nrb);
    }
  }
  if (best_cost < 0) return g;
  g.ok = true;
  g.act_stride = gemv_act_stride(mode, g.kslice, tc);
  g.head_tiles = gemv_head_tiles();
  // dynamic scale: every CTA reads all of A when that is at most two load batches per thread
  // (no cluster exchange on the critical path); larger A exchanges the ranks' slice maxima
  const int64_t units_all = int64_t(M) * ((K + 7) / 8);
  g.cluster_amax = (g.S > 1 && units_all > 2 * kRegUnits * kConsumerThreads) ? 1 : 0;
  if (g.S == 1) g.cluster_amax = 1;  // one rank: its slice is all of A
  // quantize mode with row-aligned A: bulk-copy A (all of it for the dynamic maximum when it
  // fits, else this rank's slice) into the ring stages that stay idle until the stream is
  // released, so the prologue reads it from shared memory with no per-thread round trips
  // (the head shrinks, down to one tile, when that makes the copy fit)
  g.scratch_a = 0;
  if (mode == kModeQuantize && vec_a && K % 8 == 0) {
    auto head_for = [&](int64_t bytes) {  // largest head <= the default that leaves `bytes` free
      const int64_t slots = (bytes + kTileBytes - 1) / kTileBytes;
      return int(std::min<int64_t>(g.head_tiles, g.stages - slots));
    };
    const int64_t full_bytes = int64_t(M) * K * 2;
    const int64_t slice_bytes = int64_t(M) * g.kslice * 2;
    if (static_scale) {
      if (head_for(slice_bytes) >= 1) { g.scratch_a = 2; g.head_tiles = head_for(slice_bytes); }
    } else if (!gemv_slice_only() && head_for(full_bytes) >= 1) {
      g.scratch_a = 1;
      g.head_tiles = head_for(full_bytes);
      g.cluster_amax = 0;
    } else if (head_for(slice_bytes) >= 1) {
      g.scratch_a = 2;
      g.head_tiles = head_for(slice_bytes);
      g.cluster_amax = 1;
    }
  }
  return g;
}

fp8_status launch_gemv(gemv::Params p, int mode, int fmt_a, int fmt_w, const uint8_t* qw, int64_t ldqw,
                       cudaStream_t st) {
  using namespace gemv;
  const int NT = p.M <= 8 ? 1 : p.M <= 16 ? 2 : 4;
  const int act_rows = 8 * NT;
  const bool tc = gemv_tc(NT, mode);
  const KernelFn kfn = kernel_for(NT, mode, fmt_a, fmt_w, tc);
  const int smem_limit = gemv_smem_limit(kfn);
  const GemvConfig g = gemv_configure(p.M, p.N, p.K, mode, tc, p.vec_a != 0, p.s_static != nullptr, smem_limit,
                                      [&](int S) { return gemv_max_clusters(kfn, S, size_t(smem_limit)); });
  if (!g.ok) {
    report_cuda(cudaErrorInvalidConfiguration, "no GEMV configuration fits");
    return FP8_ERR_CUDA;
  }
  p.kslice = g.kslice;
  p.act_stride = g.act_stride;
  p.act_rows = g.act_rows;
  p.head_tiles = g.head_tiles;
  p.cluster_amax = g.cluster_amax;
  p.scratch_a = g.scratch_a;
  p.stages = g.stages;
  p.row_blocks = (p.N + kRows - 1) / kRows;
  p.num_clusters = g.C;
  const int bS = g.S, bC = g.C;
  const size_t bsmem = g.smem;
  static const bool debug = std::getenv("FP8W8A8_DEBUG") != nullptr;
  if (debug)
    std::fprintf(stderr, "fp8w8a8: gemv M=%d N=%d K=%d mode=%d cluster=%d clusters=%d stages=%d kslice=%d smem=%zu "
                 "scratch=%d cluster_amax=%d\n", p.M, p.N, p.K, mode, bS, bC, g.stages, g.kslice, bsmem, p.scratch_a,
                 p.cluster_amax);
  CUtensorMap map, amap;
  if (!make_fp8_tensor_map(&map, qw, p.N, p.K, ldqw, kRows)) return FP8_ERR_CUDA;
  amap = map;  // unused unless the pre-quantized tcgen05 kernel loads qA by TMA
  if (tc && mode == kModePrequant && !make_fp8_tensor_map(&amap, p.qa, p.M, p.K, p.ldqa, uint32_t(act_rows)))
    return FP8_ERR_CUDA;
  return launch(kfn, dim3(bC * bS), dim3(kThreads), bsmem, st, true, dim3(bS, 1, 1), map, amap, p);
}

// ---------------------------------------------------------------------------
// validation
// ---------------------------------------------------------------------------

fp8_status check_bf16_mat(const void* p, int64_t rows, int64_t cols, int64_t ld) {
  if (rows < 0 || cols < 0 || rows > kMaxDim || cols > kMaxDim) return FP8_ERR_INVALID_ARG;
  if (ld < std::max<int64_t>(cols, 1)) return FP8_ERR_INVALID_ARG;
  if (rows > 0 && cols > 0 && p == nullptr) return FP8_ERR_INVALID_ARG;
  if (!aligned(p, 2)) return FP8_ERR_MISALIGNED;
  return FP8_OK;
}

fp8_status check_fp8_mat(const void* p, int64_t rows, int64_t cols, int64_t ld) {
  if (rows < 0 || cols < 0 || rows > kMaxDim || cols > kMaxDim) return FP8_ERR_INVALID_ARG;
  if (ld < std::max<int64_t>(round_up16(cols), 16)) return FP8_ERR_INVALID_ARG;
  if (ld % FP8_LD_ALIGN != 0) return FP8_ERR_MISALIGNED;
  if (rows > 0 && p == nullptr) return FP8_ERR_INVALID_ARG;
  if (!aligned(p, 16)) return FP8_ERR_MISALIGNED;
  return FP8_OK;
}

fp8_status check_ws(const void* ws, size_t ws_bytes, size_t need) {
  if (need == 0) return FP8_OK;
  if (ws == nullptr || ws_bytes < need) return FP8_ERR_WORKSPACE;
  if (!aligned(ws, 256)) return FP8_ERR_WORKSPACE;
  return FP8_OK;
}

#define FP8_TRY(expr)                  \
  do {                                 \
    const fp8_status _s = (expr);      \
    if (_s != FP8_OK) return _s;       \
  } while (0)

// Decode shapes need no workspace (the GEMV quantizes A itself); the GEMM path holds the
// partial amax values, s_a and qA [M, round_up(K, 16)]: the least a GEMM-path call accepts.
// Workspace of fp8_linear: the partial amax values, s_a and qA, except for the GEMV at up to
// 16 tokens, which quantizes A itself.
size_t linear_ws_bytes(int64_t M, int64_t K, int64_t N) {
  if (M <= 0 || K <= 0 || (use_gemv(M, K, N) && M <= gemv_self_quant_max_m())) return 0;
  return FP8_QUANT_WORKSPACE_BYTES + size_t(M) * size_t(round_up16(K));
}

size_t round_up_256(size_t b) { return (b + 255) / 256 * 256; }

// What fp8_workspace_bytes reports: the above plus, from the next 256-byte boundary, the
// split-K fp32 partials of the split a 152-SM GB300 (76 CTA pairs) would use.
// A call given less (but at least linear_ws_bytes) splits only as far as its workspace holds.
size_t linear_ws_bytes_full(int64_t M, int64_t K, int64_t N) {
  const size_t base = linear_ws_bytes(M, K, N);
  if (base == 0 || N <= 0 || use_gemv(M, K, N)) return base;
  const int S = fp8k::plan_splits(M, N, K, 152, 76, SIZE_MAX);
  return S > 1 ? round_up_256(base) + fp8k::splitk_bytes(M, N, S) : base;
}

fp8_status linear_impl(const void* a, int64_t M, int64_t K, int64_t lda, int fmt_a, const float* s_static,
                       const uint8_t* qw, int fmt_w, int64_t N, int64_t ldqw, const float* s_w, int per_channel,
                       const void* bias, void* y, int64_t ldy, void* ws, size_t ws_bytes, fp8_stream_t stream) {
  if (!valid_fmt(fmt_a) || !valid_fmt(fmt_w) || (per_channel != 0 && per_channel != 1)) return FP8_ERR_INVALID_ARG;
  FP8_TRY(check_bf16_mat(a, M, K, lda));
  FP8_TRY(check_fp8_mat(qw, N, K, ldqw));
  FP8_TRY(check_bf16_mat(y, M, N, ldy));
  if (N > 0 && s_w == nullptr) return FP8_ERR_INVALID_ARG;
  if (!aligned(bias, 2) || !aligned(s_static, 4)) return FP8_ERR_MISALIGNED;
  if (M == 0 || N == 0) return FP8_OK;
  FP8_TRY(check_ws(ws, ws_bytes, linear_ws_bytes(M, K, N)));
  int sms = 0;
  FP8_TRY(current_device(&sms));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (K == 0) return launch_fill_bias(bias, y, M, N, ldy, sms, st);

  const BF16Mat A{static_cast<const uint16_t*>(a), M, K, lda};
  const bool gemv = use_gemv(M, K, N);
  if (gemv && M <= gemv_self_quant_max_m()) {
    // decode: one persistent GEMV kernel quantizes A (cluster-wide amax, or the static
    // scale) and streams qW
    gemv::Params p = gemv_params(nullptr, 0, nullptr, s_w, per_channel, bias, y, ldy, M, N, K);
    p.a = A.p;
    p.lda = lda;
    p.vec_a = A.vec();
    p.s_static = s_static;
    return launch_gemv(p, gemv::kModeQuantize, fmt_a, fmt_w, qw, ldqw, st);
  }
  // A is quantized once into the workspace (amax pass and cast, or the cast with the static
  // scale), then the GEMM, or for 17..32 tokens the GEMV on the pre-quantized activations
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  float* partials = reinterpret_cast<float*>(wsb);
  uint8_t* qa = wsb + kWsQaOffset;
  const int64_t ldqa = round_up16(K);
  const float* s_a = s_static;
  if (s_static == nullptr) {
    float* s_dyn = reinterpret_cast<float*>(wsb + kWsScaleOffset);
    const int g = amax_grid(A, sms);
    FP8_TRY(launch_amax(A, partials, g, st, true));
    FP8_TRY(launch_cast(A, partials, g, nullptr, s_dyn, qa, ldqa, fmt_a, sms, st, true));
    s_a = s_dyn;
  } else {
    FP8_TRY(launch_cast(A, nullptr, 0, s_static, nullptr, qa, ldqa, fmt_a, sms, st, true));
  }
  if (gemv)
    return launch_gemv(gemv_params(qa, ldqa, s_a, s_w, per_channel, bias, y, ldy, M, N, K), gemv::kModePrequant,
                       fmt_a, fmt_w, qw, ldqw, st);
  // split-K scratch past qA, when the workspace holds it
  const size_t split_off = round_up_256(linear_ws_bytes(M, K, N));
  const fp8k::SplitK sk =
      ws_bytes > split_off
          ? fp8k::gemm_split_plan(qa, ldqa, qw, ldqw, int(M), int(N), int(K), sms, wsb + split_off, ws_bytes - split_off)
          : fp8k::SplitK();
  if (gemm_launch(qa, ldqa, s_a, qw, ldqw, s_w, per_channel, static_cast<const uint16_t*>(bias),
                  static_cast<uint16_t*>(y), ldy, int(M), int(N), int(K), fmt_a, fmt_w, sms, st, sk) != 0)
    return FP8_ERR_CUDA;
  return FP8_OK;
}

fp8_status quantize_weight_impl(const void* w_bf16, int64_t N, int64_t K, int64_t ldw, int per_channel, int fmt,
                                uint8_t* qw, int64_t ldq, float* s_w, void* ws, size_t ws_bytes,
                                fp8_stream_t stream) {
  FP8_TRY(check_bf16_mat(w_bf16, N, K, ldw));
  FP8_TRY(check_fp8_mat(qw, N, K, ldq));
  if ((per_channel != 0 && per_channel != 1) || !valid_fmt(fmt)) return FP8_ERR_INVALID_ARG;
  if (s_w == nullptr) return FP8_ERR_INVALID_ARG;
  if (!per_channel) FP8_TRY(check_ws(ws, ws_bytes, FP8_QUANT_WORKSPACE_BYTES));
  if (per_channel && N == 0) return FP8_OK;
  int sms = 0;
  FP8_TRY(current_device(&sms));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const BF16Mat W{static_cast<const uint16_t*>(w_bf16), N, K, ldw};
  // Weight kernels never trigger programmatic launch early: a following linear call may
  // read qW before its own wait (see the header's launch-ordering note).
  if (per_channel) {
    const int g = int(std::min<int64_t>(N, int64_t(sms) * 8));
    auto go = [&](auto kernel) {
      return launch(kernel, dim3(g), dim3(kQuantThreads), 0, st, false, dim3(1, 1, 1), W.p, N, K, ldw, W.vec(), qw,
                    ldq, s_w);
    };
    return fmt == kFmtE5M2 ? go(quantize_rows_kernel<kFmtE5M2>) : go(quantize_rows_kernel<kFmtE4M3>);
  }
  float* partials = static_cast<float*>(ws);
  const int g = amax_grid(W, sms);
  FP8_TRY(launch_amax(W, partials, g, st, false));
  return launch_cast(W, partials, g, nullptr, s_w, qw, ldq, fmt, sms, st, false);
}

fp8_status quantize_act_impl(const void* a_bf16, int64_t M, int64_t K, int64_t lda, int fmt, const float* s_static,
                             uint8_t* qa, int64_t ldq, float* s_a, void* ws, size_t ws_bytes, fp8_stream_t stream) {
  FP8_TRY(check_bf16_mat(a_bf16, M, K, lda));
  FP8_TRY(check_fp8_mat(qa, M, K, ldq));
  if (s_a == nullptr || !valid_fmt(fmt)) return FP8_ERR_INVALID_ARG;
  if (!aligned(s_static, 4)) return FP8_ERR_MISALIGNED;
  if (s_static == nullptr) FP8_TRY(check_ws(ws, ws_bytes, FP8_QUANT_WORKSPACE_BYTES));
  int sms = 0;
  FP8_TRY(current_device(&sms));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const BF16Mat A{static_cast<const uint16_t*>(a_bf16), M, K, lda};
  if (s_static != nullptr) return launch_cast(A, nullptr, 0, s_static, s_a, qa, ldq, fmt, sms, st, true);
  float* partials = static_cast<float*>(ws);
  const int g = amax_grid(A, sms);
  FP8_TRY(launch_amax(A, partials, g, st, true));
  return launch_cast(A, partials, g, nullptr, s_a, qa, ldq, fmt, sms, st, true);
}

fp8_status scaled_mm_impl(const uint8_t* qa, int fmt_a, int64_t M, int64_t K, int64_t ldqa, const float* s_a,
                          const uint8_t* qw, int fmt_w, int64_t N, int64_t ldqw, const float* s_w, int per_channel,
                          const void* bias_bf16, void* y_bf16, int64_t ldy, fp8_stream_t stream) {
  FP8_TRY(check_fp8_mat(qa, M, K, ldqa));
  FP8_TRY(check_fp8_mat(qw, N, K, ldqw));
  FP8_TRY(check_bf16_mat(y_bf16, M, N, ldy));
  if ((per_channel != 0 && per_channel != 1) || !valid_fmt(fmt_a) || !valid_fmt(fmt_w)) return FP8_ERR_INVALID_ARG;
  if (M > 0 && N > 0 && (s_a == nullptr || s_w == nullptr)) return FP8_ERR_INVALID_ARG;
  if (!aligned(bias_bf16, 2)) return FP8_ERR_MISALIGNED;
  if (M == 0 || N == 0) return FP8_OK;
  int sms = 0;
  FP8_TRY(current_device(&sms));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (K == 0) return launch_fill_bias(bias_bf16, y_bf16, M, N, ldy, sms, st);
  if (use_gemv(M, K, N))
    return launch_gemv(gemv_params(qa, ldqa, s_a, s_w, per_channel, bias_bf16, y_bf16, ldy, M, N, K), gemv::kModePrequant,
                       fmt_a, fmt_w, qw, ldqw, st);
  if (fp8k::gemm_launch(qa, ldqa, s_a, qw, ldqw, s_w, per_channel, static_cast<const uint16_t*>(bias_bf16),
                        static_cast<uint16_t*>(y_bf16), ldy, int(M), int(N), int(K), fmt_a, fmt_w, sms, st) != 0)
    return FP8_ERR_CUDA;
  return FP8_OK;
}

// ---------------------------------------------------------------------------
// weight-only FP8 linear: bf16 activations, FP8 weights up-converted to bf16
// ---------------------------------------------------------------------------

int64_t round_up8(int64_t k) { return (k + 7) / 8 * 8; }
size_t round_up256(size_t b) { return (b + 255) / 256 * 256; }

// Decode shapes stream the FP8 weights through the GEMV, up-converting each tile in registers
// (bf16 activation slices of at most kMaxSliceBf16 per rank); larger shapes up-convert W once
// into the workspace and run the bf16 tcgen05 GEMM.
bool use_gemv_weight_only(int64_t M, int64_t K) {
  return M <= gemv_max_m() && K <= int64_t(gemv::kMaxCluster) * gemv::kMaxSliceBf16;
}

// GEMM path: up-converted W [N, round_up8(K)] bf16, then room for a 16-byte-aligned copy of A
// [M, round_up8(K)] (used only when A's rows are not 16-byte aligned).
size_t weight_only_ws_bytes(int64_t M, int64_t K, int64_t N) {
  if (M <= 0 || K <= 0 || N <= 0 || use_gemv_weight_only(M, K)) return 0;
  return round_up256(size_t(N) * size_t(round_up8(K)) * 2) + size_t(M) * size_t(round_up8(K)) * 2;
}

fp8_status weight_only_impl(const void* a, int64_t M, int64_t K, int64_t lda, const uint8_t* qw, int fmt_w,
                            int64_t N, int64_t ldqw, const float* s_w, int per_channel, const void* bias, void* y,
                            int64_t ldy, void* ws, size_t ws_bytes, fp8_stream_t stream) {
  if (!valid_fmt(fmt_w) || (per_channel != 0 && per_channel != 1)) return FP8_ERR_INVALID_ARG;
  FP8_TRY(check_bf16_mat(a, M, K, lda));
  FP8_TRY(check_fp8_mat(qw, N, K, ldqw));
  FP8_TRY(check_bf16_mat(y, M, N, ldy));
  if (N > 0 && s_w == nullptr) return FP8_ERR_INVALID_ARG;
  if (!aligned(bias, 2)) return FP8_ERR_MISALIGNED;
  if (M == 0 || N == 0) return FP8_OK;
  FP8_TRY(check_ws(ws, ws_bytes, weight_only_ws_bytes(M, K, N)));
  int sms = 0;
  FP8_TRY(current_device(&sms));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (K == 0) return launch_fill_bias(bias, y, M, N, ldy, sms, st);

  const BF16Mat A{static_cast<const uint16_t*>(a), M, K, lda};
  if (use_gemv_weight_only(M, K)) {
    gemv::Params p = gemv_params(nullptr, 0, nullptr, s_w, per_channel, bias, y, ldy, M, N, K);
    p.a = A.p;
    p.lda = lda;
    p.vec_a = A.vec();
    return launch_gemv(p, gemv::kModeBf16, kFmtE4M3, fmt_w, qw, ldqw, st);
  }
  const int64_t ldk = round_up8(K);
  uint16_t* wb = static_cast<uint16_t*>(ws);
  {
    const int64_t units = N * (ldk / 8);
    const int g = int(std::max<int64_t>(1, std::min<int64_t>((units + kQuantThreads - 1) / kQuantThreads,
                                                             int64_t(sms) * 8)));
    auto go = [&](auto kernel) {
      return launch(kernel, dim3(g), dim3(kQuantThreads), 0, st, true, dim3(1, 1, 1), qw, N, K, ldqw, wb, ldk);
    };
    FP8_TRY(fmt_w == kFmtE5M2 ? go(upconvert_kernel<kFmtE5M2>) : go(upconvert_kernel<kFmtE4M3>));
  }
  const uint16_t* a_tma = A.p;
  int64_t lda_tma = lda;
  if ((lda * 2) % 16 != 0 || !aligned(A.p, 16)) {
    uint16_t* acopy = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(ws) + round_up256(size_t(N) * ldk * 2));
    const int64_t units = M * (ldk / 8);
    const int g = int(std::max<int64_t>(1, std::min<int64_t>((units + kQuantThreads - 1) / kQuantThreads,
                                                             int64_t(sms) * 8)));
    FP8_TRY(launch(copy_rows_bf16_kernel, dim3(g), dim3(kQuantThreads), 0, st, true, dim3(1, 1, 1), A.p, M, K, lda,
                   A.vec(), acopy, ldk, 1));
    a_tma = acopy;
    lda_tma = ldk;
  }
  if (gemm_bf16_launch(a_tma, lda_tma, wb, ldk, s_w, per_channel, static_cast<const uint16_t*>(bias),
                       static_cast<uint16_t*>(y), ldy, int(M), int(N), int(K), sms, st) != 0)
    return FP8_ERR_CUDA;
  return FP8_OK;
}

}  // namespace

// ---------------------------------------------------------------------------
// exported C ABI
// ---------------------------------------------------------------------------

FP8_API int64_t fp8_min_ld(int64_t K) { return K <= 0 ? 16 : round_up16(K); }

FP8_API size_t fp8_workspace_bytes(int64_t M, int64_t K, int64_t N) {
  return linear_ws_bytes_full(std::max<int64_t>(M, 0), std::max<int64_t>(K, 0), std::max<int64_t>(N, 0));
}

FP8_API int fp8_set_gemv_max_m(int m) {
  if (m < 0) return gemv_max_m();
  return gemv_max_m_value().exchange(std::min(m, gemv::kMaxTokens));
}

FP8_API int fp8_uses_gemv(int64_t M, int64_t K, int64_t N) {
  return use_gemv(M, K, N) ? 1 : 0;
}

FP8_API fp8_status fp8_quantize_weight(const void* w_bf16, int64_t N, int64_t K, int64_t ldw, int per_channel,
                                       uint8_t* qw, int64_t ldq, float* s_w, void* ws, size_t ws_bytes,
                                       fp8_stream_t stream) {
  return quantize_weight_impl(w_bf16, N, K, ldw, per_channel, kFmtE4M3, qw, ldq, s_w, ws, ws_bytes, stream);
}

FP8_API fp8_status fp8_quantize_weight_ex(const void* w_bf16, int64_t N, int64_t K, int64_t ldw, int per_channel,
                                          fp8_format fmt, uint8_t* qw, int64_t ldq, float* s_w, void* ws,
                                          size_t ws_bytes, fp8_stream_t stream) {
  return quantize_weight_impl(w_bf16, N, K, ldw, per_channel, int(fmt), qw, ldq, s_w, ws, ws_bytes, stream);
}

FP8_API fp8_status fp8_quantize_act(const void* a_bf16, int64_t M, int64_t K, int64_t lda, uint8_t* qa, int64_t ldq,
                                    float* s_a, void* ws, size_t ws_bytes, fp8_stream_t stream) {
  return quantize_act_impl(a_bf16, M, K, lda, kFmtE4M3, nullptr, qa, ldq, s_a, ws, ws_bytes, stream);
}

FP8_API fp8_status fp8_quantize_act_ex(const void* a_bf16, int64_t M, int64_t K, int64_t lda, fp8_format fmt,
                                       const float* s_static, uint8_t* qa, int64_t ldq, float* s_a, void* ws,
                                       size_t ws_bytes, fp8_stream_t stream) {
  return quantize_act_impl(a_bf16, M, K, lda, int(fmt), s_static, qa, ldq, s_a, ws, ws_bytes, stream);
}

FP8_API fp8_status fp8_scaled_mm(const uint8_t* qa, int64_t M, int64_t K, int64_t ldqa, const float* s_a,
                                 const uint8_t* qw, int64_t N, int64_t ldqw, const float* s_w, int per_channel,
                                 const void* bias_bf16, void* y_bf16, int64_t ldy, fp8_stream_t stream) {
  return scaled_mm_impl(qa, kFmtE4M3, M, K, ldqa, s_a, qw, kFmtE4M3, N, ldqw, s_w, per_channel, bias_bf16, y_bf16,
                        ldy, stream);
}

FP8_API fp8_status fp8_scaled_mm_ex(const uint8_t* qa, fp8_format fmt_a, int64_t M, int64_t K, int64_t ldqa,
                                    const float* s_a, const uint8_t* qw, fp8_format fmt_w, int64_t N, int64_t ldqw,
                                    const float* s_w, int per_channel, const void* bias_bf16, void* y_bf16,
                                    int64_t ldy, fp8_stream_t stream) {
  return scaled_mm_impl(qa, int(fmt_a), M, K, ldqa, s_a, qw, int(fmt_w), N, ldqw, s_w, per_channel, bias_bf16,
                        y_bf16, ldy, stream);
}

FP8_API fp8_status fp8_linear(const void* a_bf16, int64_t M, int64_t K, int64_t lda, const uint8_t* qw, int64_t N,
                              int64_t ldqw, const float* s_w, const void* bias_bf16, void* y_bf16, int64_t ldy,
                              void* ws, size_t ws_bytes, fp8_stream_t stream) {
  return linear_impl(a_bf16, M, K, lda, kFmtE4M3, nullptr, qw, kFmtE4M3, N, ldqw, s_w, 0, bias_bf16, y_bf16, ldy,
                     ws, ws_bytes, stream);
}

FP8_API fp8_status fp8_linear_channelwise(const void* a_bf16, int64_t M, int64_t K, int64_t lda, const uint8_t* qw,
                                          int64_t N, int64_t ldqw, const float* s_w, const void* bias_bf16,
                                          void* y_bf16, int64_t ldy, void* ws, size_t ws_bytes,
                                          fp8_stream_t stream) {
  return linear_impl(a_bf16, M, K, lda, kFmtE4M3, nullptr, qw, kFmtE4M3, N, ldqw, s_w, 1, bias_bf16, y_bf16, ldy,
                     ws, ws_bytes, stream);
}

FP8_API fp8_status fp8_linear_static(const void* a_bf16, int64_t M, int64_t K, int64_t lda, const float* s_a,
                                     const uint8_t* qw, int64_t N, int64_t ldqw, const float* s_w, int per_channel,
                                     const void* bias_bf16, void* y_bf16, int64_t ldy, void* ws, size_t ws_bytes,
                                     fp8_stream_t stream) {
  if (M > 0 && N > 0 && s_a == nullptr) return FP8_ERR_INVALID_ARG;
  return linear_impl(a_bf16, M, K, lda, kFmtE4M3, s_a, qw, kFmtE4M3, N, ldqw, s_w, per_channel, bias_bf16, y_bf16,
                     ldy, ws, ws_bytes, stream);
}

FP8_API fp8_status fp8_linear_ex(const void* a_bf16, int64_t M, int64_t K, int64_t lda, fp8_format fmt_a,
                                 const float* s_static, const uint8_t* qw, fp8_format fmt_w, int64_t N, int64_t ldqw,
                                 const float* s_w, int per_channel, const void* bias_bf16, void* y_bf16, int64_t ldy,
                                 void* ws, size_t ws_bytes, fp8_stream_t stream) {
  return linear_impl(a_bf16, M, K, lda, int(fmt_a), s_static, qw, int(fmt_w), N, ldqw, s_w, per_channel, bias_bf16,
                     y_bf16, ldy, ws, ws_bytes, stream);
}

FP8_API size_t fp8_weight_only_workspace_bytes(int64_t M, int64_t K, int64_t N) {
  return weight_only_ws_bytes(M, K, N);
}

FP8_API fp8_status fp8_linear_weight_only(const void* a_bf16, int64_t M, int64_t K, int64_t lda, const uint8_t* qw,
                                          fp8_format fmt_w, int64_t N, int64_t ldqw, const float* s_w,
                                          int per_channel, const void* bias_bf16, void* y_bf16, int64_t ldy,
                                          void* ws, size_t ws_bytes, fp8_stream_t stream) {
  return weight_only_impl(a_bf16, M, K, lda, qw, int(fmt_w), N, ldqw, s_w, per_channel, bias_bf16, y_bf16, ldy, ws,
                          ws_bytes, stream);
}

// The launch a plan and a K split give: CTAs, raster group, split counts (both queries below).
void report_plan(const fp8k::GemmPlan& pl, int S, int sms, int* two_sm, int* grid, int* group_n, int* splits,
                 int* tail_split) {
  const int m_units = pl.two_sm ? (pl.m_tiles + 1) / 2 : pl.m_tiles;
  if (two_sm) *two_sm = pl.two_sm;
  if (grid) *grid = S > 1 ? (pl.two_sm ? std::min(pl.grid, 2 * m_units * pl.n_tiles * S)
                                       : std::min(sms, m_units * pl.n_tiles * S))
                          : pl.grid;
  if (group_n) *group_n = pl.group_n;
  if (splits) *splits = S;
  if (tail_split) *tail_split = S > 1 ? 1 : pl.tail_split;
}

FP8_API fp8_status fp8_gemm_config(const uint8_t* qa, int64_t M, int64_t ldqa, const uint8_t* qw, int64_t N,
                                   int64_t ldqw, int64_t K, size_t ws_bytes, int* two_sm, int* grid, int* group_n,
                                   int* splits, int* tail_split) {
  if (M <= 0 || N <= 0 || K <= 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim || ldqa <= 0 || ldqw <= 0)
    return FP8_ERR_INVALID_ARG;
  int sms = 0;
  FP8_TRY(current_device(&sms));
  const fp8k::GemmPlan pl = fp8k::gemm_plan(qa, ldqa, qw, ldqw, int(M), int(N), sms);
  if (pl.grid <= 0) return FP8_ERR_CUDA;
  // the split fp8_linear would take with a workspace of ws_bytes (the planning needs no memory)
  const size_t split_off = round_up_256(linear_ws_bytes(M, K, N));
  int S = 1;
  if (!use_gemv(M, K, N) && ws_bytes > split_off) {
    alignas(256) static unsigned char probe[256];
    S = fp8k::gemm_split_plan(qa, ldqa, qw, ldqw, int(M), int(N), int(K), sms, probe, ws_bytes - split_off).splits;
  }
  report_plan(pl, S, sms, two_sm, grid, group_n, splits, tail_split);
  return FP8_OK;
}

FP8_API fp8_status fp8_gemv_plan_model(int64_t M, int64_t N, int64_t K, int mode, int static_scale, int smem_limit,
                                       const int* clusters_of_size, int* cluster, int* clusters, int* stages,
                                       int* kslice, int* scratch_a, int* cluster_amax, int* tcgen05) {
  if (M <= 0 || M > gemv::kMaxTokens || N <= 0 || N > kMaxDim || K <= 0 || K > kGemvMaxK || mode < 0 || mode > 2 ||
      smem_limit <= 0 || clusters_of_size == nullptr)
    return FP8_ERR_INVALID_ARG;
  const int NT = M <= 8 ? 1 : M <= 16 ? 2 : 4;
  const bool tc = gemv_tc(NT, mode);
  const GemvConfig g = gemv_configure(int(M), int(N), int(K), mode, tc, true, static_scale != 0, smem_limit,
                                      [&](int S) { return clusters_of_size[S - 1]; });
  if (!g.ok) return FP8_ERR_CUDA;
  if (cluster) *cluster = g.S;
  if (clusters) *clusters = g.C;
  if (stages) *stages = g.stages;
  if (kslice) *kslice = g.kslice;
  if (scratch_a) *scratch_a = g.scratch_a;
  if (cluster_amax) *cluster_amax = g.cluster_amax;
  if (tcgen05) *tcgen05 = tc ? 1 : 0;
  return FP8_OK;
}

FP8_API fp8_status fp8_gemm_plan_model(int64_t M, int64_t N, int64_t K, int num_sms, int pair_slots, size_t ws_bytes,
                                       int* two_sm, int* grid, int* group_n, int* splits, int* tail_split) {
  if (M <= 0 || N <= 0 || K <= 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim || num_sms <= 0 || pair_slots < 0)
    return FP8_ERR_INVALID_ARG;
  const int64_t ld = round_up16(K);
  const fp8k::GemmPlan pl = fp8k::plan_gemm_model(ld, ld, int(M), int(N), true, num_sms, pair_slots);
  const size_t split_off = round_up_256(linear_ws_bytes(M, K, N));
  int S = 1;
  if (!use_gemv(M, K, N) && ws_bytes > split_off)
    S = fp8k::plan_splits(M, N, K, num_sms, pl.two_sm ? pair_slots : 0, ws_bytes - split_off);
  report_plan(pl, S, num_sms, two_sm, grid, group_n, splits, tail_split);
  return FP8_OK;
}

FP8_API fp8_status fp8_last_device_status(fp8_stream_t stream) {
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return FP8_ERR_CUDA;
  const unsigned int e = fp8k::gemm_read_and_clear_error() | gemv::read_and_clear_error();
  if (cudaGetLastError() != cudaSuccess) return FP8_ERR_CUDA;
  return (e & kErrTimeout) ? FP8_ERR_TIMEOUT : FP8_OK;
}

FP8_API fp8_status fp8_selftest_timeout(int64_t limit_ns, fp8_stream_t stream) {
  if (limit_ns < 1000 || limit_ns > 10000000000ll) return FP8_ERR_INVALID_ARG;
  int sms = 0;
  FP8_TRY(current_device(&sms));
  gemv::selftest_timeout(static_cast<unsigned long long>(limit_ns), reinterpret_cast<cudaStream_t>(stream));
  return report_cuda(cudaGetLastError(), "self-test launch") == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

FP8_API const char* fp8_status_string(fp8_status s) {
  switch (s) {
    case FP8_OK: return "FP8_OK";
    case FP8_ERR_INVALID_ARG: return "FP8_ERR_INVALID_ARG";
    case FP8_ERR_MISALIGNED: return "FP8_ERR_MISALIGNED";
    case FP8_ERR_WORKSPACE: return "FP8_ERR_WORKSPACE";
    case FP8_ERR_CUDA: return "FP8_ERR_CUDA";
    case FP8_ERR_TIMEOUT: return "FP8_ERR_TIMEOUT";
    case FP8_ERR_UNSUPPORTED_DEVICE: return "FP8_ERR_UNSUPPORTED_DEVICE";
  }
  return "FP8_ERR_UNKNOWN";
}

// ---------------------------------------------------------------------------
// fp8_linear_noalloc: the linear for callers that cannot allocate device memory
// ---------------------------------------------------------------------------
//
// The scratch the linear needs (partial amax values, the activation scale and, on the GEMM
// path, the quantized activations) lives in this fixed array instead of a caller workspace.
// Every GPU that loads the library holds it until the process exits. Host code must not pass
// the array's name to a kernel: on the host that name is only a stand-in for the symbol, so
// its device address is looked up once per device with cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[FP8_NOALLOC_SCRATCH_BYTES];

namespace {

std::mutex g_noalloc_mu;
struct NoallocAddr {
  void* ptr = nullptr;
  unsigned long long ctx = 0;  // id of the context the address belongs to
};
NoallocAddr g_noalloc_addr[64];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Unique id of the calling thread's current CUDA context (0 when it cannot be read). A device
// reset destroys the primary context and the library's module with it; the next context gets
// a new id, so an address cached for the old one is never reused.
unsigned long long current_context_id() {
  static const std::pair<CtxGetCurrentFn, CtxGetIdFn> fns = [] {
    void* a = nullptr;
    void* b = nullptr;
    cudaDriverEntryPointQueryResult qa, qb;
    const bool ok = cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 12000, cudaEnableDefault, &qa) ==
                        cudaSuccess && qa == cudaDriverEntryPointSuccess &&
                    cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) ==
                        cudaSuccess && qb == cudaDriverEntryPointSuccess;
    return ok ? std::make_pair(reinterpret_cast<CtxGetCurrentFn>(a), reinterpret_cast<CtxGetIdFn>(b))
              : std::make_pair(static_cast<CtxGetCurrentFn>(nullptr), static_cast<CtxGetIdFn>(nullptr));
  }();
  CUcontext c = nullptr;
  unsigned long long id = 0;
  if (fns.first && fns.second && fns.first(&c) == CUDA_SUCCESS && c != nullptr && fns.second(c, &id) == CUDA_SUCCESS)
    return id;
  return 0;
}

// Device address of g_noalloc_scratch on the current device, looked up on first use and again
// whenever the current context is a different one (after a device reset).
fp8_status noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FP8_ERR_CUDA;
  const unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  NoallocAddr& e = g_noalloc_addr[dev];
  if (e.ptr == nullptr || ctx == 0 || e.ctx != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return FP8_ERR_CUDA;
    e.ptr = p;
    e.ctx = current_context_id();  // the lookup above creates the context if there was none
  }
  *out = e.ptr;
  return FP8_OK;
}

}  // namespace

FP8_API fp8_status fp8_linear_noalloc(const void* a_bf16, int64_t M, int64_t K, int64_t lda, const uint8_t* qw,
                                      int64_t N, int64_t ldqw, const float* s_w, int per_channel,
                                      const void* bias_bf16, void* y_bf16, int64_t ldy, fp8_stream_t stream) {
  if (per_channel != 0 && per_channel != 1) return FP8_ERR_INVALID_ARG;
  FP8_TRY(check_bf16_mat(a_bf16, M, K, lda));
  FP8_TRY(check_fp8_mat(qw, N, K, ldqw));
  FP8_TRY(check_bf16_mat(y_bf16, M, N, ldy));
  if (M == 0 || N == 0)
    return linear_impl(a_bf16, M, K, lda, kFmtE4M3, nullptr, qw, kFmtE4M3, N, ldqw, s_w, per_channel, bias_bf16,
                       y_bf16, ldy, nullptr, 0, stream);
  // shapes whose scratch would not fit are refused before anything is enqueued
  if (linear_ws_bytes(M, K, N) > size_t(FP8_NOALLOC_SCRATCH_BYTES)) return FP8_ERR_WORKSPACE;
  void* scratch = nullptr;
  FP8_TRY(noalloc_scratch(&scratch));
  return linear_impl(a_bf16, M, K, lda, kFmtE4M3, nullptr, qw, kFmtE4M3, N, ldqw, s_w, per_channel, bias_bf16,
                     y_bf16, ldy, scratch, size_t(FP8_NOALLOC_SCRATCH_BYTES), stream);
}
