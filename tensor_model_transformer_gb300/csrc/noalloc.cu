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
// passes it to the kernels.  Only a successful lookup is kept: a call whose
// lookup failed (for instance one made during stream capture) returns
// MTL_ERR_CUDA and the next call on that device tries again.
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

float* g_scratch_addr[kMaxDevices];   // non-null once the lookup succeeded
std::mutex g_setup_mutex;

// The scratch array's device address on device `dev` (current), looked up on
// the first successful call.
cudaError_t scratch_address(int dev, float** addr) {
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_bias_grad_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = static_cast<float*>(p);
  }
  *addr = g_scratch_addr[dev];
  return cudaSuccess;
}

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
  float* scratch = nullptr;
  e = scratch_address(dev, &scratch);
  if (e != cudaSuccess) {
    cudaGetLastError();   // the failed lookup leaves nothing behind for later calls
    mtl::record_cuda_error(e, "bias grad: scratch address");
    return MTL_ERR_CUDA;
  }

  int launches = 0;
  mtl::LaunchCtx c{reinterpret_cast<cudaStream_t>(stream), 0, &launches, nullptr};
  // Every partial the second pass reads is written by the first pass of the
  // same call, so the scratch needs no clearing between calls.
  e = mtl::colsum(dtype, dy, ld, rows, cols, static_cast<float*>(out), scratch, c);
  if (e != cudaSuccess) {
    mtl::record_cuda_error(e, "bias grad");
    return MTL_ERR_CUDA;
  }
  return MTL_OK;
}
