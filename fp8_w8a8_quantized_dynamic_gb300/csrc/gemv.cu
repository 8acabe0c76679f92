// Instantiations of the decode GEMV kernel (gemv.cuh) and its host-side accessors.
// The kernels, their error word and the function that reads it live in this one
// translation unit (one CUDA module), so the host reads the word the kernels write.

#include "gemv.cuh"

namespace fp8k {
namespace gemv {

namespace {

template <int NT, int Mode, bool Tc>
KernelFn pick(int fa, int fw) {
  if constexpr (Mode == kModeBf16) {
    return fw == kFmtE4M3 ? gemv_kernel<NT, Mode, kFmtE4M3, kFmtE4M3, false>
                          : gemv_kernel<NT, Mode, kFmtE4M3, kFmtE5M2, false>;
  } else {
    if (fa == kFmtE4M3)
      return fw == kFmtE4M3 ? gemv_kernel<NT, Mode, kFmtE4M3, kFmtE4M3, Tc> : gemv_kernel<NT, Mode, kFmtE4M3, kFmtE5M2, Tc>;
    return fw == kFmtE4M3 ? gemv_kernel<NT, Mode, kFmtE5M2, kFmtE4M3, Tc> : gemv_kernel<NT, Mode, kFmtE5M2, kFmtE5M2, Tc>;
  }
}

template <int NT, bool Tc>
KernelFn pick_mode(int mode, int fa, int fw) {
  if (mode == kModeQuantize) return pick<NT, kModeQuantize, false>(fa, fw);
  if (mode == kModeBf16) return pick<NT, kModeBf16, false>(fa, fw);
  return pick<NT, kModePrequant, Tc>(fa, fw);
}

}  // namespace

KernelFn kernel_for(int NT, int mode, int fa, int fw, bool tc) {
  if (NT == 1) return pick_mode<1, false>(mode, fa, fw);
  if (NT == 2) return tc ? pick_mode<2, true>(mode, fa, fw) : pick_mode<2, false>(mode, fa, fw);
  return tc ? pick_mode<4, true>(mode, fa, fw) : pick_mode<4, false>(mode, fa, fw);
}

// Failure-path self-test. A two-warp pipeline on a two-stage mbarrier ring, shaped like the
// GEMV's producer / consumer handshake, in which the producer withholds item `withheld`: the
// consumer's bounded wait for it runs out after limit_ns, records kErrTimeout in the GEMV's
// error word and raises the CTA's abort flag, the producer's own bounded waits then give up,
// and the kernel returns normally, leaving the context usable. Nothing faults or hangs.
__global__ void __launch_bounds__(64) selftest_timeout_kernel(unsigned long long limit_ns, int withheld) {
  __shared__ __align__(8) uint64_t full[2], empty[2];
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  volatile int* ab = &abort_flag;
  constexpr int kItems = 4;
  if (lane == 0) {
    for (int it = 0; it < kItems; ++it) {
      const int s = it & 1;
      const uint32_t ph = (it >> 1) & 1u;
      if (warp == 0) {  // producer
        if (!mbar_wait_bounded(smem_u32(&empty[s]), ph ^ 1u, ab, &g_gemv_error, limit_ns)) break;
        if (it != withheld) mbar_arrive(smem_u32(&full[s]));
      } else {          // consumer
        if (!mbar_wait_bounded(smem_u32(&full[s]), ph, ab, &g_gemv_error, limit_ns)) break;
        mbar_arrive(smem_u32(&empty[s]));
      }
    }
  }
  __syncwarp();
  __syncthreads();
}

void selftest_timeout(unsigned long long limit_ns, cudaStream_t st) {
  selftest_timeout_kernel<<<1, 64, 0, st>>>(limit_ns, 2);
}

unsigned int read_and_clear_error() {
  unsigned int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_gemv_error, sizeof(v)) != cudaSuccess) return 0;
  cudaMemcpyToSymbol(g_gemv_error, &zero, sizeof(zero));
  return v;
}

}  // namespace gemv
}  // namespace fp8k
