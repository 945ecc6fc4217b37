// Pair-kernel instantiations with the tail-slice epilogue: launches whose last,
// partial wave of 256 x 256 tiles is cut into K slices on separate SM pairs,
// the slices' fp32 partials added in slice order before the epilogue (see
// tail_slices and plan_split in gemm_core.cuh).  They live in a translation
// unit of their own, beside the unsliced kernels of gemm_tc.cu and
// gemm_fp8.cu, so that a launch without slices runs code compiled without the
// slice paths (the GeLU and GeLU' epilogues are register-bound).
#include "gemm_core.cuh"

namespace mtl {
namespace tcg {

template <int EPI, bool F32, bool RED, bool F8>
static KernelFn split_ptr() {
  return reinterpret_cast<KernelFn>(gemm_tc2_kernel<EPI, F32, RED, F8, true>);
}

template <bool F8>
static KernelFn select_split(int epi, bool f32, bool red) {
#define SELS(E)                                                                     \
  if (epi == E) {                                                                   \
    if (f32) return red ? split_ptr<E, true, true, F8>() : split_ptr<E, true, false, F8>(); \
    return red ? split_ptr<E, false, true, F8>() : split_ptr<E, false, false, F8>();        \
  }
  SELS(EPI_STORE)
  SELS(EPI_BIAS)
  SELS(EPI_BIAS_RESID)
  SELS(EPI_BIAS_GELU)
  SELS(EPI_DGELU)
#undef SELS
  return nullptr;
}

KernelFn select_kernel2_split(int epi, bool f32, bool red) { return select_split<false>(epi, f32, red); }
KernelFn select_kernel8_split(int epi, bool f32, bool red) { return select_split<true>(epi, f32, red); }

}  // namespace tcg
}  // namespace mtl
