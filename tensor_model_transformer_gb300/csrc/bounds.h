// Checks of the coordinates and indices the kernels compute, against the
// extents of the tensors they address.  Builds with MTL_DEBUG run them on the
// device before every TMA copy and plain store of the instrumented kernels
// (a failed check records a fault in the workspace status word and skips the
// access, so a wrong coordinate shows up as MTL_ERR_BOUNDS instead of a GPU
// fault); the host unit tests run the same functions on the CPU.
//
// The rules come from the tensor-memory-access requirements of tiled bulk
// tensor copies: the innermost coordinate x times the element size must be a
// multiple of 16 bytes; a load may start at a negative or out-of-range
// coordinate (the box is filled where it lies outside the tensor) but a box
// entirely outside the tensor means the tiling arithmetic is wrong; a store
// must not start at a negative coordinate, nor past the tensor's end.
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define MTL_HD __host__ __device__ __forceinline__
#else
#define MTL_HD inline
#endif

namespace mtl {
namespace bounds {

enum Fault : uint32_t {
  kOk = 0,
  kTmaXMisaligned = 1,     // x * element bytes is not a multiple of 16
  kTmaBoxOutside = 2,      // a load's box lies entirely outside the tensor
  kTmaStoreNegative = 3,   // a store starts at a negative coordinate
  kTmaStoreOutside = 4,    // a store starts past the tensor's end
  kIndexOutside = 5,       // an element index outside [0, n)
};

// A 2D tensor of ext_x (innermost) x ext_y elements of elem_bytes bytes,
// accessed in boxes of box_x x box_y.
struct Box2 {
  int64_t ext_x, ext_y;
  int32_t box_x, box_y, elem_bytes;
};

MTL_HD uint32_t check_tma_x(const Box2& b, int64_t x) {
  const int64_t off = x * b.elem_bytes;
  return (off % 16 != 0) ? kTmaXMisaligned : kOk;
}

MTL_HD uint32_t check_tma_load(const Box2& b, int64_t x, int64_t y) {
  if (check_tma_x(b, x) != kOk) return kTmaXMisaligned;
  if (x >= b.ext_x || y >= b.ext_y || x + b.box_x <= 0 || y + b.box_y <= 0) return kTmaBoxOutside;
  return kOk;
}

MTL_HD uint32_t check_tma_store(const Box2& b, int64_t x, int64_t y) {
  if (check_tma_x(b, x) != kOk) return kTmaXMisaligned;
  if (x < 0 || y < 0) return kTmaStoreNegative;
  if (x >= b.ext_x || y >= b.ext_y) return kTmaStoreOutside;
  return kOk;
}

MTL_HD uint32_t check_index(int64_t i, int64_t n) {
  return (i < 0 || i >= n) ? kIndexOutside : kOk;
}

// Status-word bits of a failed check: the bounds flag (4), the fault in bits
// 8..11 and the call site in bits 16..23 (the first failure's fields may be
// ORed with later ones; the flag is exact).
constexpr uint32_t kStatusBoundsFlag = 4u;

MTL_HD uint32_t status_bits(uint32_t fault, uint32_t site) {
  return fault == kOk ? 0u : (kStatusBoundsFlag | ((fault & 0xFu) << 8) | ((site & 0xFFu) << 16));
}

// Call sites reported in the status word.
enum Site : uint32_t {
  kSiteGemmA = 1, kSiteGemmB = 2, kSiteGemmC = 3, kSiteGemmZ = 4,
  kSiteAttnFwdQ = 5, kSiteAttnFwdKV = 6, kSiteAttnFwdOut = 7,
  kSiteAttnDqLoad = 8, kSiteAttnDqKV = 9, kSiteAttnDqOut = 10,
  kSiteAttnDkvLoad = 11, kSiteAttnDkvQ = 12, kSiteAttnDkvOut = 13,
};

}  // namespace bounds
}  // namespace mtl
