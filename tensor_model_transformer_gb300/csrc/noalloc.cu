// An entry point for callers that cannot allocate device memory: the bias
// gradient (fixed-order column sum) with its partial-sum scratch in a static
// device array instead of a caller workspace.
//
// The scratch holds the per-row-block partial sums the column-sum kernels
// stage between their two passes.  It is a file-scope __device__ array of
// kScratchFloats floats (8 MiB), so every GPU that loads this library keeps it
// until the process exits.  Host code cannot use the array's name as a device
// address (it names a host-side shadow), so the first call on each device looks
// the address up with cudaGetSymbolAddress, with that device current, and
// passes it to the kernels.
#include <mutex>

#include "../../include/mtl.h"
#include "common.cuh"
#include "kernels.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxCols = 16384;
// The column sum stages at most 128 row blocks x cols partial sums.
constexpr size_t kScratchFloats = (size_t)128 * kMaxCols;

__device__ __align__(256) float g_bias_grad_scratch[kScratchFloats];

float* g_scratch_addr[kMaxDevices];
cudaError_t g_setup_status[kMaxDevices];
std::once_flag g_setup_once[kMaxDevices];

}  // namespace

extern "C" mtl_status mtl_bias_grad_noalloc(int32_t dtype, const void* dy, int64_t ld,
                                            int32_t rows, int32_t cols, void* out,
                                            mtl_stream stream) {
  mtl::clear_cuda_error();
  if (dtype != MTL_F32 && dtype != MTL_BF16) return MTL_ERR_INVALID_ARG;
  const int64_t vec = dtype == MTL_BF16 ? 8 : 4;   // elements per 16-byte load
  if (rows < 0 || cols <= 0 || ld < cols || cols % vec || ld % vec) return MTL_ERR_INVALID_ARG;
  if (!dy || !out || (reinterpret_cast<uintptr_t>(dy) & 15) || (reinterpret_cast<uintptr_t>(out) & 3))
    return MTL_ERR_INVALID_ARG;
  if (cols > kMaxCols || mtl::colsum_partial_floats(rows, cols) > kScratchFloats)
    return MTL_ERR_UNSUPPORTED;

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    mtl::record_cuda_error(e, "bias grad: device query");
    return MTL_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return MTL_ERR_UNSUPPORTED;
  std::call_once(g_setup_once[dev], [dev]() {
    g_setup_status[dev] =
        cudaGetSymbolAddress(reinterpret_cast<void**>(&g_scratch_addr[dev]), g_bias_grad_scratch);
  });
  if (g_setup_status[dev] != cudaSuccess) {
    mtl::record_cuda_error(g_setup_status[dev], "bias grad: scratch address");
    return MTL_ERR_CUDA;
  }

  int launches = 0;
  mtl::LaunchCtx c{reinterpret_cast<cudaStream_t>(stream), 0, &launches, nullptr};
  // Every partial the second pass reads is written by the first pass of the
  // same call, so the scratch needs no clearing between calls.
  e = mtl::colsum(dtype, dy, ld, rows, cols, static_cast<float*>(out), g_scratch_addr[dev], c);
  if (e != cudaSuccess) {
    mtl::record_cuda_error(e, "bias grad");
    return MTL_ERR_CUDA;
  }
  return MTL_OK;
}
