// Instantiations of the decode GEMV kernel (gemv.cuh) and its host-side accessors.
// The kernels, their error word and the function that reads it live in this one
// translation unit (one CUDA module), so the host reads the word the kernels write.

#include "gemv.cuh"

namespace fp8k {
namespace gemv {

namespace {

template <int NT, int Mode>
KernelFn pick(int fa, int fw) {
  if constexpr (Mode == kModeBf16) {
    return fw == kFmtE4M3 ? gemv_kernel<NT, Mode, kFmtE4M3, kFmtE4M3> : gemv_kernel<NT, Mode, kFmtE4M3, kFmtE5M2>;
  } else {
    if (fa == kFmtE4M3)
      return fw == kFmtE4M3 ? gemv_kernel<NT, Mode, kFmtE4M3, kFmtE4M3> : gemv_kernel<NT, Mode, kFmtE4M3, kFmtE5M2>;
    return fw == kFmtE4M3 ? gemv_kernel<NT, Mode, kFmtE5M2, kFmtE4M3> : gemv_kernel<NT, Mode, kFmtE5M2, kFmtE5M2>;
  }
}

template <int NT>
KernelFn pick_mode(int mode, int fa, int fw) {
  if (mode == kModeQuantize) return pick<NT, kModeQuantize>(fa, fw);
  if (mode == kModeBf16) return pick<NT, kModeBf16>(fa, fw);
  return pick<NT, kModePrequant>(fa, fw);
}

}  // namespace

KernelFn kernel_for(int NT, int mode, int fa, int fw) {
  return NT == 1 ? pick_mode<1>(mode, fa, fw) : pick_mode<2>(mode, fa, fw);
}

unsigned int read_and_clear_error() {
  unsigned int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_gemv_error, sizeof(v)) != cudaSuccess) return 0;
  cudaMemcpyToSymbol(g_gemv_error, &zero, sizeof(zero));
  return v;
}

}  // namespace gemv
}  // namespace fp8k
