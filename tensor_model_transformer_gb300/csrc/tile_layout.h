// Byte layout of the shared-memory tiles the attention kernels load with TMA
// and hand to tcgen05.mma, and of their epilogue staging buffers.  Plain C++
// (host and device), so the host unit tests check the arithmetic on the CPU.
//
// A swizzled TMA box stores row r of `rowb` bytes at r * rowb, with each
// 16-byte piece p of it moved to p XOR (bits 7.. of the piece's byte offset):
// 128-byte swizzle XORs the piece index (bits 4-6) with offset bits 7-9, that
// is with r % 8 for 128-byte rows; 64-byte swizzle XORs bits 4-5 with bits
// 7-8, that is with (r / 2) % 4 for 64-byte rows.  The boxes start on
// 1024-byte boundaries, so the offset within the box gives the same bits.
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define MTL_LAYOUT_HD __host__ __device__ __forceinline__
#else
#define MTL_LAYOUT_HD inline
#endif

namespace mtl {
namespace layout {

// Byte offset of 16-byte piece p of row r in a box of 64-byte rows, 64-byte swizzle.
MTL_LAYOUT_HD constexpr uint32_t sw64_off(int r, int p) {
  return (uint32_t)(r * 64 + ((p ^ ((r >> 1) & 3)) << 4));
}
// The same for 128-byte rows and 128-byte swizzle.
MTL_LAYOUT_HD constexpr uint32_t sw128_off(int r, int p) {
  return (uint32_t)(r * 128 + ((p ^ (r & 7)) << 4));
}

// A 128-row bf16 operand tile of d = 16 KS columns: atoms of 128 rows x ACOLS
// columns, each the box of one TMA load.  d = 64 and 128: 64-column atoms with
// 128-byte swizzle; d = 96: three 32-column atoms with 64-byte swizzle (24 KB
// a tile, where two 64-column atoms take 32 KB with a quarter unused).
template <int KS>
struct TileFmt {
  static constexpr int D = KS * 16;
  static constexpr bool SW64 = D % 64 != 0;
  static constexpr int ACOLS = SW64 ? 32 : 64;
  static constexpr int ATOMS = D / ACOLS;
  static constexpr uint32_t ROWB = ACOLS * 2;   // bytes of an atom row
  static constexpr uint32_t ATOM = 128 * ROWB;
  static constexpr uint32_t TILE = ATOMS * ATOM;
  static constexpr int KPA = ACOLS / 16;        // 16-column k-steps per atom
  static_assert(D % ACOLS == 0, "a tile is whole atoms");
  // K-major operand: k-step kk (columns 16 kk .. 16 kk + 15) starts at byte
  // 32 (kk % KPA) of the rows of atom kk / KPA
  MTL_LAYOUT_HD static constexpr uint32_t koff(int kk) {
    return (uint32_t)(kk / KPA) * ATOM + (uint32_t)(kk % KPA) * 32;
  }
  // MN-major operand (the tile's rows are the K dimension): k-step kk is rows
  // 16 kk .. 16 kk + 15
  MTL_LAYOUT_HD static constexpr uint32_t mnoff(int kk) { return (uint32_t)kk * 16 * ROWB; }
  // byte offset of 16-byte chunk c (columns 8c .. 8c + 7) of row r
  MTL_LAYOUT_HD static constexpr uint32_t chunk(int r, int c) {
    return (uint32_t)(c / (ACOLS / 8)) * ATOM +
           (SW64 ? sw64_off(r, c % (ACOLS / 8)) : sw128_off(r, c % (ACOLS / 8)));
  }
};

}  // namespace layout
}  // namespace mtl
