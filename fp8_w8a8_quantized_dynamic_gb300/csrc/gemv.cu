// Instantiations of the decode GEMV kernel (gemv.cuh) and its host-side accessors.
// The kernels, their error word and the function that reads it live in this one
// translation unit (one CUDA module), so the host reads the word the kernels write.

#include "gemv.cuh"

namespace fp8k {
namespace gemv {

namespace {

template <int NT, bool D>
KernelFn pick(int fa, int fw) {
  if (fa == kFmtE4M3) return fw == kFmtE4M3 ? gemv_kernel<NT, D, kFmtE4M3, kFmtE4M3> : gemv_kernel<NT, D, kFmtE4M3, kFmtE5M2>;
  return fw == kFmtE4M3 ? gemv_kernel<NT, D, kFmtE5M2, kFmtE4M3> : gemv_kernel<NT, D, kFmtE5M2, kFmtE5M2>;
}

}  // namespace

KernelFn kernel_for(int NT, bool dyn, int fa, int fw) {
  if (NT == 1) return dyn ? pick<1, true>(fa, fw) : pick<1, false>(fa, fw);
  return dyn ? pick<2, true>(fa, fw) : pick<2, false>(fa, fw);
}

unsigned int read_and_clear_error() {
  unsigned int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_gemv_error, sizeof(v)) != cudaSuccess) return 0;
  cudaMemcpyToSymbol(g_gemv_error, &zero, sizeof(zero));
  return v;
}

}  // namespace gemv
}  // namespace fp8k
