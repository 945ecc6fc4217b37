// The tcgen05 GEMM machinery shared by the bf16 kernels (gemm_tc.cu) and the
// FP8 instantiations of the pair kernel (gemm_fp8.cu): tile raster, fused
// epilogue, epilogue warp role, the 2-CTA pair kernel and the tensor-map helper.
#pragma once

#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace mtl {
namespace tcg {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int EPI_WARPS = 8;
constexpr int THREADS = 128 + 32 * EPI_WARPS;
constexpr int LAUNCH_REGS = 168, PRODUCER_REGS = 56, EPILOGUE_REGS = 224;
static_assert(PRODUCER_REGS * 128 + EPILOGUE_REGS * 32 * EPI_WARPS == LAUNCH_REGS * THREADS,
              "register split must add up to the launch total");
constexpr int TMEM_COLS = 2 * BN;
constexpr int BAR_BYTES = 256;
constexpr int STAGE_OUT_BYTES = 4096;                       // epilogue output staging a warp
constexpr int OUT_STAGING_BYTES = EPI_WARPS * STAGE_OUT_BYTES;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + OUT_STAGING_BYTES + BAR_BYTES + 1024;
constexpr int GROUP_M = 16;   // tile raster: groups of 16 M-blocks sweep all N-blocks
constexpr int RASTER_N_MAX = 16;   // at most this many N-blocks: the raster runs N fastest
// Split tiles (pair kernel): a region of a tile's output written by one epilogue
// warp (32 rows x 128 columns, fp32), and the regions of a tile (2 CTAs x 8 warps).
constexpr int SPLIT_REGION_FLOATS = 32 * 128;
constexpr int SPLIT_REGIONS = 2 * EPI_WARPS;

struct Params {
  int M, N, K, parts, kb_per_unit, units_per_tile;
  int a_mn, b_mn;
  int tiles_m, tiles_n, num_tiles;
  const bf16* bias;
  const bf16* R;
  int64_t ldr;
  bf16* Z;
  int64_t ldz;
  void* C;
  int64_t ldc;
  unsigned* status;
  Dropout drop;   // EPI_BIAS_RESID: C = R + dropout(acc + bias), element e = row * N + col
  // FP8 operands (pair kernel with F8): formats (0 E4M3, 1 E5M2) and the
  // device-side per-tensor scales; the accumulator is multiplied by
  // float32(1 / float32(scale_a * scale_b)) before the epilogue.  Null for bf16.
  int fmt_a, fmt_b;
  const float* scale_a;
  const float* scale_b;
  // Raster: raster_n = 1 runs N fastest (every N-block of an M-block together,
  // for narrow outputs whose B operand then stays in L2), else groups of
  // GROUP_M M-blocks sweep the N-blocks.
  int raster_n;
  // Work split (pair kernel).  Tiles [0, dp_tiles) of the raster, whole waves
  // over the pairs, run whole and round-robin.  Each of the remaining tiles
  // (the last, partial wave) is cut into split_s slices of its granules
  // (split_g K-blocks each: a partition when the partials are summed, else one
  // K-block; split_gpt granules a tile), slice j being granules
  // [j * split_gpt / split_s, (j + 1) * split_gpt / split_s); pair q < tail
  // tiles x split_s computes slice q % split_s of tail tile q / split_s.  All
  // slices start together at their own K offset, like the whole waves before
  // them, so pairs that share an operand block still read it at the same time.
  // A slice's epilogue warps write their fp32 partial (a running partition
  // sum, or the slice's K range) to slot j of split_ws and count themselves in
  // split_cnt; the warp that arrives last adds slots 0..split_s-1 in order and
  // runs the epilogue.
  // EPI_DGELU: per-warp column sums of the stored output (32 rows each) go to
  // csum[row / 32][col] (fp32; the bias gradient's partial sums), or nowhere
  // when null.  Whole 32-column chunks only (N % 32 == 0).
  float* csum;
  int dp_tiles;
  int split_s;
  int split_g, split_gpt;
  float* split_ws;       // [tail tile][slot][SPLIT_REGIONS][SPLIT_REGION_FLOATS]
  unsigned* split_cnt;   // [tail tile][SPLIT_REGIONS], zero between launches
};

// One piece of a pair's work: granules [g0, g1) of tile `tile`; split: slice
// `slot` of tail tile `sk` (the tile's other slices run on other pairs).
struct Piece {
  int tile, g0, g1, sk, slot;
  bool split;
};

struct PieceIter {
  int next, step;
  bool tail_done;
};

__device__ __forceinline__ void piece_begin(const Params& p, int pair_id, int npairs,
                                            PieceIter& it) {
  it.next = pair_id;
  it.step = npairs;
  it.tail_done = false;
}

__device__ __forceinline__ bool piece_next(const Params& p, PieceIter& it, Piece& pc) {
  if (it.next < p.dp_tiles) {
    pc.tile = it.next;
    pc.g0 = 0;
    pc.g1 = p.split_gpt;
    pc.sk = -1;
    pc.slot = 0;
    pc.split = false;
    it.next += it.step;
    return true;
  }
  if (it.tail_done || p.split_s <= 1) return false;
  it.tail_done = true;
  // this pair's slice of the tail: pair index = it.next - dp_tiles (whole waves)
  const int q = (it.next - p.dp_tiles);
  if (q < 0 || q >= (p.num_tiles - p.dp_tiles) * p.split_s) return false;
  pc.sk = q / p.split_s;
  pc.slot = q - pc.sk * p.split_s;
  pc.tile = p.dp_tiles + pc.sk;
  pc.g0 = pc.slot * p.split_gpt / p.split_s;
  pc.g1 = (pc.slot + 1) * p.split_gpt / p.split_s;
  pc.split = true;
  return true;
}

__device__ __forceinline__ void tile_coords(const Params& p, int tile, int& mb, int& nb) {
  if (p.raster_n) {
    mb = tile / p.tiles_n;
    nb = tile - mb * p.tiles_n;
    return;
  }
  const int per_group = GROUP_M * p.tiles_n;
  const int g = tile / per_group;
  const int first_m = g * GROUP_M;
  const int gsize = min(GROUP_M, p.tiles_m - first_m);
  const int r = tile - g * per_group;
  mb = first_m + r % gsize;
  nb = r / gsize;
}

// Dropout keep bits of columns [col0, col0+32) of one row (bit e for col0+e),
// all ones without dropout.
template <int EPI>
__device__ __forceinline__ uint32_t chunk_keep(const Params& p, int row, int col0) {
  if (EPI != EPI_BIAS_RESID || !p.drop.on || row >= p.M) return 0xffffffffu;
  const unsigned long long e0 = (unsigned long long)row * p.N + col0;
  if ((p.N & 3) == 0 && col0 + 32 <= p.N) return drop_bits32(e0, p.drop);
  uint32_t bits = 0;
#pragma unroll 1
  for (int e = 0; e < 32 && col0 + e < p.N; ++e) bits |= (drop_keep(e0 + e, p.drop) ? 1u : 0u) << e;
  return bits;
}

// Applies the epilogue to 32 consecutive columns [col0, col0+32) of one row;
// `keep`: dropout bits of EPI_BIAS_RESID (chunk_keep).
template <int EPI, bool OUT_F32>
__device__ __forceinline__ void epi_chunk(const Params& p, int row, int col0, float (&v)[32],
                                          uint32_t keep) {
  if (row >= p.M || col0 >= p.N) return;
  const bool full = col0 + 32 <= p.N;
  if (full) {
    if (EPI == EPI_BIAS || EPI == EPI_BIAS_RESID || EPI == EPI_BIAS_GELU) {
      const uint4* bp = reinterpret_cast<const uint4*>(p.bias + col0);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 u = __ldg(bp + q);
        const bf16* hb = reinterpret_cast<const bf16*>(&u);
#pragma unroll
        for (int e = 0; e < 8; ++e) v[q * 8 + e] += __bfloat162float(hb[e]);
      }
    }
    if (EPI == EPI_BIAS_RESID && p.drop.on) {
#pragma unroll
      for (int e = 0; e < 32; ++e) v[e] = ((keep >> e) & 1u) ? v[e] * p.drop.scale : 0.f;
    }
    if (EPI == EPI_BIAS_RESID) {
      const uint4* rp = reinterpret_cast<const uint4*>(p.R + (size_t)row * p.ldr + col0);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 u = rp[q];
        const bf16* hb = reinterpret_cast<const bf16*>(&u);
#pragma unroll
        for (int e = 0; e < 8; ++e) v[q * 8 + e] += __bfloat162float(hb[e]);
      }
    }
    if (EPI == EPI_DGELU) {
      const uint4* zp = reinterpret_cast<const uint4*>(p.Z + (size_t)row * p.ldz + col0);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 u = zp[q];
        const bf16* hb = reinterpret_cast<const bf16*>(&u);
#pragma unroll
        for (int e = 0; e < 8; ++e) v[q * 8 + e] *= gelu_grad_f(__bfloat162float(hb[e]));
      }
    }
    if (EPI == EPI_BIAS_GELU) {
      uint4* zp = reinterpret_cast<uint4*>(p.Z + (size_t)row * p.ldz + col0);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint4 u;
        bf16* hb = reinterpret_cast<bf16*>(&u);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          hb[e] = __float2bfloat16_rn(v[q * 8 + e]);
          v[q * 8 + e] = gelu_f(v[q * 8 + e]);
        }
        zp[q] = u;
      }
    }
    if (OUT_F32) {
      float4* cp = reinterpret_cast<float4*>(static_cast<float*>(p.C) + (size_t)row * p.ldc + col0);
#pragma unroll
      for (int q = 0; q < 8; ++q)
        cp[q] = make_float4(v[q * 4], v[q * 4 + 1], v[q * 4 + 2], v[q * 4 + 3]);
    } else {
      uint4* cp = reinterpret_cast<uint4*>(static_cast<bf16*>(p.C) + (size_t)row * p.ldc + col0);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint4 u;
        bf16* hb = reinterpret_cast<bf16*>(&u);
#pragma unroll
        for (int e = 0; e < 8; ++e) hb[e] = __float2bfloat16_rn(v[q * 8 + e]);
        cp[q] = u;
      }
    }
  } else {
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      const int col = col0 + e;
      if (col < p.N) {
        float x = v[e];
        if (EPI == EPI_BIAS || EPI == EPI_BIAS_RESID || EPI == EPI_BIAS_GELU)
          x += __bfloat162float(p.bias[col]);
        if (EPI == EPI_BIAS_RESID && p.drop.on) x = ((keep >> e) & 1u) ? x * p.drop.scale : 0.f;
        if (EPI == EPI_BIAS_RESID) x += __bfloat162float(p.R[(size_t)row * p.ldr + col]);
        if (EPI == EPI_DGELU) x *= gelu_grad_f(__bfloat162float(p.Z[(size_t)row * p.ldz + col]));
        if (EPI == EPI_BIAS_GELU) {
          p.Z[(size_t)row * p.ldz + col] = __float2bfloat16_rn(x);
          x = gelu_f(x);
        }
        if (OUT_F32)
          static_cast<float*>(p.C)[(size_t)row * p.ldc + col] = x;
        else
          static_cast<bf16*>(p.C)[(size_t)row * p.ldc + col] = __float2bfloat16_rn(x);
      }
    }
  }
}

// Output staging for the TMA stores of the epilogue: each epilogue warp owns
// STAGE_OUT_BYTES of shared memory (1024-aligned) holding one 32 x 32 chunk of
// C (bf16: 64-byte rows in the 64-byte swizzle; fp32: 128-byte rows in the
// 128-byte swizzle) and, for EPI_BIAS_GELU, the chunk of z (bf16) at +2048.
template <int EPI, bool OUT_F32>
__host__ __device__ constexpr bool tma_out() {   // fp32 C with z would not fit the warp's staging
  return !(EPI == EPI_BIAS_GELU && OUT_F32);
}

// Row r's 16-byte piece q of a 32 x 32 staging chunk with 64-byte rows
// (64-byte swizzle: q ^ bits 7-8 of the offset) and with 128-byte rows
// (128-byte swizzle: q ^ bits 7-9).
__device__ __forceinline__ uint32_t sw64_piece(int r, int q) { return r * 64 + ((q ^ ((r >> 1) & 3)) << 4); }
__device__ __forceinline__ uint32_t sw128_piece(int r, int q) { return r * 128 + ((q ^ (r & 7)) << 4); }

// epi_chunk for a whole chunk (col0 + 32 <= N) of the warp's 32 rows row0 + lane,
// written through the warp's staging buffer by TMA stores (rows >= M are
// computed on zeros and dropped by the tensor map's bounds).  Called by all 32
// lanes; lane 0 issues the stores.
// side: the chunk's 32 bf16 of R (EPI_BIAS_RESID) or Z (EPI_DGELU) of this
// lane's row, read by the caller (side_load).
template <int EPI, bool OUT_F32>
__device__ __forceinline__ void epi_chunk_tma(const Params& p, int row0, int col0,
                                              float (&v)[32], uint32_t keep, int lane,
                                              const uint4 (&side)[4], const CUtensorMap* tmC,
                                              const CUtensorMap* tmZ, uint32_t stage) {
  if (EPI == EPI_BIAS || EPI == EPI_BIAS_RESID || EPI == EPI_BIAS_GELU) {
    const uint4* bp = reinterpret_cast<const uint4*>(p.bias + col0);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 u = __ldg(bp + q);
      const bf16* hb = reinterpret_cast<const bf16*>(&u);
#pragma unroll
      for (int e = 0; e < 8; ++e) v[q * 8 + e] += __bfloat162float(hb[e]);
    }
  }
  if (EPI == EPI_BIAS_RESID && p.drop.on) {
#pragma unroll
    for (int e = 0; e < 32; ++e) v[e] = ((keep >> e) & 1u) ? v[e] * p.drop.scale : 0.f;
  }
  if (EPI == EPI_BIAS_RESID) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const bf16* hb = reinterpret_cast<const bf16*>(&side[q]);
#pragma unroll
      for (int e = 0; e < 8; ++e) v[q * 8 + e] += __bfloat162float(hb[e]);
    }
  }
  if (EPI == EPI_DGELU) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const bf16* hb = reinterpret_cast<const bf16*>(&side[q]);
#pragma unroll
      for (int e = 0; e < 8; ++e) v[q * 8 + e] *= gelu_grad_f(__bfloat162float(hb[e]));
    }
  }
  auto pack2 = [](float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  };
  // the previous chunk's stores have read the staging buffer
  if (lane == 0) bulk_wait_read0();
  __syncwarp();
  if (EPI == EPI_BIAS_GELU) {
#pragma unroll
    for (int q = 0; q < 4; ++q)
      st_shared_v4(stage + 2048 + sw64_piece(lane, q), pack2(v[8 * q], v[8 * q + 1]),
                   pack2(v[8 * q + 2], v[8 * q + 3]), pack2(v[8 * q + 4], v[8 * q + 5]),
                   pack2(v[8 * q + 6], v[8 * q + 7]));
#pragma unroll
    for (int e = 0; e < 32; ++e) v[e] = gelu_f(v[e]);
  }
  if (OUT_F32) {
#pragma unroll
    for (int q = 0; q < 8; ++q)
      st_shared_v4(stage + sw128_piece(lane, q), __float_as_uint(v[4 * q]),
                   __float_as_uint(v[4 * q + 1]), __float_as_uint(v[4 * q + 2]),
                   __float_as_uint(v[4 * q + 3]));
  } else {
#pragma unroll
    for (int q = 0; q < 4; ++q)
      st_shared_v4(stage + sw64_piece(lane, q), pack2(v[8 * q], v[8 * q + 1]),
                   pack2(v[8 * q + 2], v[8 * q + 3]), pack2(v[8 * q + 4], v[8 * q + 5]),
                   pack2(v[8 * q + 6], v[8 * q + 7]));
  }
  fence_proxy_async_shared();
  __syncwarp();
  if (lane == 0) {
    const bounds::Box2 boxc = {p.N, p.M, 32, 32, OUT_F32 ? 4 : 2};
    if (MTL_CHECKED(p.status, bounds::check_tma_store(boxc, col0, row0), bounds::kSiteGemmC))
      tma_store_2d(tmC, stage, col0, row0);
    const bounds::Box2 boxz = {p.N, p.M, 32, 32, 2};
    if (EPI == EPI_BIAS_GELU &&
        MTL_CHECKED(p.status, bounds::check_tma_store(boxz, col0, row0), bounds::kSiteGemmZ))
      tma_store_2d(tmZ, stage + 2048, col0, row0);
    bulk_commit();
  }
  if (EPI == EPI_DGELU && p.csum) {
    // column sums of the chunk as stored, from the staging buffer (rows past M
    // hold zeros: their A rows read as zero)
    if (OUT_F32) {
      // lane l adds column l over the 32 rows, in row order
      float cs = 0.f;
#pragma unroll
      for (int r = 0; r < 32; ++r)
        cs += ld_shared_f32(stage + r * 128 + ((((lane >> 2) ^ (r & 7))) << 4) + (lane & 3) * 4);
      p.csum[(size_t)(row0 >> 5) * p.N + col0 + lane] = cs;
    } else {
      // lane l adds the column pair cp = l % 16 (one 32-bit word of two bf16)
      // over the even rows (l < 16) or the odd rows (l >= 16), in row order --
      // an even and an odd row of the 64-byte-swizzled staging tile lie in
      // opposite halves of the banks -- then the two halves are added
      const int cp = lane & 15, odd = lane >> 4;
      float c0 = 0.f, c1 = 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int r = 2 * i + odd;
        const uint32_t w =
            ld_shared_u32(stage + r * 64 + (((cp >> 2) ^ ((r >> 1) & 3)) << 4) + (cp & 3) * 4);
        c0 += __uint_as_float(w << 16);
        c1 += __uint_as_float(w & 0xffff0000u);
      }
      c0 += __shfl_xor_sync(0xffffffffu, c0, 16);
      c1 += __shfl_xor_sync(0xffffffffu, c1, 16);
      if (!odd)
        *reinterpret_cast<float2*>(p.csum + (size_t)(row0 >> 5) * p.N + col0 + 2 * cp) =
            make_float2(c0, c1);
    }
  }
}

// Epilogue warps 4..11: wait for an accumulator, read it from TMEM (32 columns
// at a time), add partition partials in order, apply the epilogue, store.
// tfull0 / tempty0: addresses of tfull[0] and tempty[0] (tempty as a cluster
// address when PAIR: the epilogue warps of both CTAs of a pair release the
// accumulator to the leader CTA's barrier).  The work is the pieces of pair (or
// CTA) tile0 of tile_step (piece_next); tiles are tile_rows high and this
// CTA's rows start at row_off inside a tile.
// tmC / tmZ: tensor maps of C and z (32 x 32 boxes) for the TMA stores of
// whole chunks; out_stage: the shared staging area (OUT_STAGING_BYTES).
// AHEAD: R / Z of the next chunk are loaded while this one is processed (the
// FP8 kernels, whose shorter main loop leaves the epilogue exposed; measured
// slower for bf16).
template <int EPI, bool OUT_F32, bool REDUCE, bool PAIR, bool AHEAD, bool SPLIT>
__device__ __forceinline__ void epilogue_role(const Params& p, uint32_t tmem_base, uint32_t tfull0,
                                              uint32_t tempty0, volatile int* abort_flag,
                                              int warp, int lane, int tile0, int tile_step,
                                              int tile_rows, int row_off, const CUtensorMap* tmC,
                                              const CUtensorMap* tmZ, uint32_t out_stage) {
  auto tfull_bar = [&](int b) { return tfull0 + 8u * b; };
  auto tempty_bar = [&](int b) { return tempty0 + 8u * b; };
  const int ew = warp - 4;
  const int quarter = warp & 3;
  const int chalf = ew >> 2;
  // FP8 descale (exactly 1 for bf16 operands)
  const float ds = p.scale_a ? __fdiv_rn(1.0f, __fmul_rn(*p.scale_a, *p.scale_b)) : 1.0f;
  const uint32_t stage = out_stage + ew * STAGE_OUT_BYTES;
  // one 32 x 32 chunk of the epilogue: whole chunks through TMA stores, ragged
  // ones (col0 + 32 > N) element by element
  // R (EPI_BIAS_RESID) or Z (EPI_DGELU) of a whole chunk is read into
  // registers; with AHEAD one chunk ahead (the first chunk of a tile before its
  // accumulator is waited for), so the global-load latency overlaps the
  // previous chunk's work
  constexpr bool SIDE = tma_out<EPI, OUT_F32>() && (EPI == EPI_BIAS_RESID || EPI == EPI_DGELU);
  auto side_load = [&](int row, int col0, uint4(&dst)[4]) {
    if constexpr (SIDE) {
      if (row < p.M && col0 + 32 <= p.N) {
        const bf16* src = EPI == EPI_DGELU ? p.Z + (size_t)row * p.ldz + col0
                                           : p.R + (size_t)row * p.ldr + col0;
#pragma unroll
        for (int q = 0; q < 4; ++q) dst[q] = reinterpret_cast<const uint4*>(src)[q];
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) dst[q] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
  };
  auto chunk = [&](int row, int col0, float(&v)[32], uint32_t keep, const uint4(&side)[4]) {
    if (col0 >= p.N) return;
    const int row0 = row - lane;
    if constexpr (tma_out<EPI, OUT_F32>()) {
      if (col0 + 32 <= p.N) {
        if (row0 < p.M) epi_chunk_tma<EPI, OUT_F32>(p, row0, col0, v, keep, lane, side, tmC, tmZ, stage);
        return;
      }
    }
    epi_chunk<EPI, OUT_F32>(p, row, col0, v, keep);
  };
  // A split piece's partial: this warp's 32 rows x 128 columns in slot `slot`
  // of split tile `sk`, as [column group of 4][row][4] (a warp's float4 stores
  // cover 512 contiguous bytes).
  auto split_region = [&](int sk, int slot) -> float* {
    return p.split_ws + ((size_t)(sk * p.split_s + slot) * SPLIT_REGIONS +
                         (size_t)row_off / 128 * EPI_WARPS + ew) *
                            SPLIT_REGION_FLOATS;
  };
  auto split_store4 = [&](float* reg, int q, float a, float b, float c, float d) {
    reinterpret_cast<float4*>(reg)[q * 32 + lane] = make_float4(a, b, c, d);
  };
  int unit = 0;
  bool ok = true;
  PieceIter pit;
  piece_begin(p, tile0, tile_step, pit);
  Piece pc;
  while (ok && piece_next(p, pit, pc)) {
    int mb, nb;
    tile_coords(p, pc.tile, mb, nb);
    const int row = mb * tile_rows + row_off + quarter * 32 + lane;
    const int colbase = nb * BN + chalf * 128;
    const bool split = SPLIT && pc.split;
    float* sreg = split ? split_region(pc.sk, pc.slot) : nullptr;
    // R or Z of this lane's row of the piece (two 128-byte lines) into L2 now,
    // so the epilogue's loads of it, after the piece's products, hit L2
    if constexpr (SIDE) {
      if (!split && row < p.M && colbase + 128 <= p.N) {
        const bf16* src = EPI == EPI_DGELU ? p.Z + (size_t)row * p.ldz + colbase
                                           : p.R + (size_t)row * p.ldr + colbase;
        prefetch_l2(src);
        prefetch_l2(src + 64);
      }
    }
    uint4 side[4];
    if (!REDUCE && AHEAD && !split) side_load(row, colbase, side);
    // the running partition sum starts at +0 in every piece, so no value of it
    // lives from one piece into the next (x + 0 = x: the same sums)
    float sum[REDUCE ? 128 : 1];
    if constexpr (REDUCE) {
#pragma unroll
      for (int i = 0; i < 128; ++i) sum[i] = 0.f;
    }
    // (a run-time unit count in both cases: units_per_tile is 1 without partial
    // sums; the loop keeps the same shape either way)
    const int nunits = REDUCE ? pc.g1 - pc.g0 : p.units_per_tile;
    for (int u = 0; u < nunits; ++u, ++unit) {
      const int buf = unit & 1;
      const uint32_t uphase = (unit >> 1) & 1;
      if (!mbar_wait_bounded(tfull_bar(buf), uphase, p.status, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t tb = tmem_base + buf * BN + chalf * 128 + ((uint32_t)(quarter * 32) << 16);
      if constexpr (REDUCE) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t r[32];
          tmem_ld32(tb + c * 32, r);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) sum[c * 32 + i] += __uint_as_float(r[i]);
        }
      } else if (split) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t r[32];
          tmem_ld32(tb + c * 32, r);
          tmem_ld_wait();
#pragma unroll
          for (int q = 0; q < 8; ++q)
            split_store4(sreg, c * 8 + q, __uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                         __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3]));
        }
      } else {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint32_t keep = chunk_keep<EPI>(p, row, colbase + c * 32);
          uint32_t r[32];
          tmem_ld32(tb + c * 32, r);
          tmem_ld_wait();
          uint4 next[4];
          if (AHEAD && c < 3) side_load(row, colbase + (c + 1) * 32, next);
          if (!AHEAD) side_load(row, colbase + c * 32, side);
          float v[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]) * ds;
          chunk(row, colbase + c * 32, v, keep, side);
          if (AHEAD && c < 3) {
#pragma unroll
            for (int q = 0; q < 4; ++q) side[q] = next[q];
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if constexpr (PAIR)
          mbar_arrive_cluster(tempty_bar(buf));
        else
          mbar_arrive(tempty_bar(buf));
      }
    }
    if (!ok) break;
    if constexpr (REDUCE) {
      if (split) {
#pragma unroll
        for (int q = 0; q < 32; ++q)
          split_store4(sreg, q, sum[4 * q], sum[4 * q + 1], sum[4 * q + 2], sum[4 * q + 3]);
      } else {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint32_t keep = chunk_keep<EPI>(p, row, colbase + c * 32);
          side_load(row, colbase + c * 32, side);   // (128 partition sums leave no room ahead)
          float v[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = sum[c * 32 + i] * ds;
          chunk(row, colbase + c * 32, v, keep, side);
        }
      }
    }
    if (SPLIT && split) {
      // publish this slice's partial; the warp of the tile's last slice to
      // arrive adds the slices in slice order and runs the epilogue
      __threadfence();
      __syncwarp();
      unsigned* cnt = p.split_cnt + (size_t)pc.sk * SPLIT_REGIONS + row_off / 128 * EPI_WARPS + ew;
      unsigned old = 0;
      if (lane == 0) old = atomicAdd(cnt, 1u);
      old = __shfl_sync(0xffffffffu, old, 0);
      if (old == (unsigned)(p.split_s - 1)) {
        __threadfence();
        // this lane's row of the tile region, chunk by chunk, summed over the
        // slices in slot order (slot j is SPLIT_REGIONS regions after slot
        // j - 1), two slots' loads in flight at a time; one copy of the chunk
        // epilogue (a rarely taken path: kept small, not unrolled)
        constexpr int SLOT4 = SPLIT_REGIONS * SPLIT_REGION_FLOATS / 4;
        const float4* s0 = reinterpret_cast<const float4*>(split_region(pc.sk, 0)) + lane;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          const uint32_t keep = chunk_keep<EPI>(p, row, colbase + c * 32);
          side_load(row, colbase + c * 32, side);
          float v[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0.f;
          const float4* sc = s0 + c * 8 * 32;
#pragma unroll 1
          for (int jj = 0; jj < p.split_s; jj += 2) {
            const bool two = jj + 1 < p.split_s;
            float4 a[8], b[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              a[q] = __ldcg(sc + jj * SLOT4 + q * 32);
              b[q] = two ? __ldcg(sc + (jj + 1) * SLOT4 + q * 32) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              v[4 * q] += a[q].x;
              v[4 * q + 1] += a[q].y;
              v[4 * q + 2] += a[q].z;
              v[4 * q + 3] += a[q].w;
            }
            if (two) {
#pragma unroll
              for (int q = 0; q < 8; ++q) {
                v[4 * q] += b[q].x;
                v[4 * q + 1] += b[q].y;
                v[4 * q + 2] += b[q].z;
                v[4 * q + 3] += b[q].w;
              }
            }
          }
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] *= ds;
          chunk(row, colbase + c * 32, v, keep, side);
        }
        if (lane == 0) *cnt = 0u;   // ready for the next launch
      }
    }
  }
  __syncwarp();
  if (lane == 0) bulk_wait0();   // the last stores are written before the kernel ends
  __syncwarp();
}

// ============================================================================
// Pair kernel: a cluster of two CTAs computes 256x256 tiles with cta_group::2
// MMAs (M = 256 across the pair, N = 256).  Each CTA loads its 128-row half of
// A and its 128-row half of B; the leader CTA (rank 0) issues every MMA, which
// reads both CTAs' shared memory and writes each CTA's 128 rows into its own
// TMEM.  One tcgen05.mma does twice the work of the single-CTA kernel's, so the
// one issuing thread keeps the tensor pipes busy.  K stages are 128 deep (two
// 64-wide swizzle boxes), three stages of 64 KB per CTA.  With F8 the operands
// are FP8 (tcgen05 kind::f8f6f4, K-major only): a 128-deep stage is one
// 128-byte box per row (32 KB per CTA), six stages, four MMAs of K = 32; the
// byte layout and descriptor steps are the bf16 ones.
//   full[s]   leader only: both CTAs' TMA loads complete on it
//   empty[s]  both CTAs: multicast commit after the stage's MMAs
//   tfull[b]  both CTAs: multicast commit after a work unit's MMAs
//   tempty[b] leader only: 16 arrivals, the epilogue warps of both CTAs
constexpr int P_BK = 128, P_HALF = 128;              // K elements per stage, rows per CTA
constexpr int P_ATOM = P_HALF * 128;                 // one [128 rows][128 bytes] box
constexpr int P_SMEM_BYTES = 3 * 2 * 2 * P_ATOM + OUT_STAGING_BYTES + BAR_BYTES + 1024;   // 192 KB of stages

template <int EPI, bool OUT_F32, bool REDUCE, bool F8, bool SPLIT = false>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
    gemm_tc2_kernel(const __grid_constant__ CUtensorMap tmA,
                    const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmC,
                    const __grid_constant__ CUtensorMap tmZ, const Params p) {
  constexpr int P_NBOX = F8 ? 1 : 2;                 // 128-byte boxes per row and stage
  constexpr int P_STAGES = F8 ? 6 : 3;
  constexpr int P_A_BYTES = P_NBOX * P_ATOM;
  constexpr int P_B_BYTES = P_NBOX * P_ATOM;
  constexpr int P_STAGE_BYTES = P_A_BYTES + P_B_BYTES;
  constexpr int P_KSTEPS = F8 ? P_BK / 32 : P_BK / 16;   // MMAs per stage
  static_assert(P_STAGES * P_STAGE_BYTES + OUT_STAGING_BYTES + BAR_BYTES + 1024 <= P_SMEM_BYTES,
                "stage ring");
  static_assert(P_SMEM_BYTES <= 232448, "shared memory of one CTA");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sA0 = smem_u32(smem);
  const uint32_t sB0 = sA0 + P_STAGES * P_A_BYTES;
  const uint32_t out_stage = sA0 + P_STAGES * P_STAGE_BYTES;   // 1024-aligned
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + P_STAGES * P_STAGE_BYTES + OUT_STAGING_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * P_STAGES + 4);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (P_STAGES + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * P_STAGES + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * P_STAGES + 2 + b); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_cta_rank();
  const int pair_id = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  if (threadIdx.x == 0) {
    for (int s = 0; s < P_STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), 2 * EPI_WARPS);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc_pair(smem_u32(tmem_slot), TMEM_COLS);
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmC);
    if (EPI == EPI_BIAS_GELU) tma_prefetch_desc(&tmZ);
  }
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(PRODUCER_REGS));
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(EPILOGUE_REGS));
  }

  if (warp >= 4) {
    epilogue_role<EPI, OUT_F32, REDUCE, true, F8, SPLIT>(p, tmem_base, tfull_bar(0),
                                              cluster_map(tempty_bar(0), 0), abort_flag, warp,
                                              lane, pair_id, npairs, 2 * P_HALF, P_HALF * rank,
                                              &tmC, &tmZ, out_stage);
  } else if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      PieceIter pit;
      piece_begin(p, pair_id, npairs, pit);
      Piece pc;
      while (ok && piece_next(p, pit, pc)) {
        int mb, nb;
        tile_coords(p, pc.tile, mb, nb);
        const int m0 = mb * 2 * P_HALF + P_HALF * rank, n0 = nb * 2 * P_HALF + P_HALF * rank;
        for (int kb = pc.g0 * p.split_g; kb < pc.g1 * p.split_g; ++kb) {
          if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, p.status, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t fb = cluster_map(full_bar(stage), 0);
          if (rank == 0) mbar_arrive_expect_tx(full_bar(stage), 2 * P_STAGE_BYTES);
          const int k0 = kb * P_BK;
          const uint32_t sa = sA0 + stage * P_A_BYTES, sb = sB0 + stage * P_B_BYTES;
#pragma unroll
          for (int j = 0; j < P_NBOX; ++j) {
            // K-major boxes: 64 K (128 bytes of FP8) x 128 rows; MN-major: 64 M
            // or N x 128 K
            const bool ak = F8 || !p.a_mn, bk = F8 || !p.b_mn;
            const int ax = ak ? k0 + 64 * j : m0 + 64 * j, ay = ak ? m0 : k0;
            const int bx = bk ? k0 + 64 * j : n0 + 64 * j, by = bk ? n0 : k0;
            const bounds::Box2 boxa = {ak ? p.K : p.M, ak ? p.M : p.K, F8 ? 128 : 64, 128,
                                       F8 ? 1 : 2};
            const bounds::Box2 boxb = {bk ? p.K : p.N, bk ? p.N : p.K, F8 ? 128 : 64, 128,
                                       F8 ? 1 : 2};
            if (MTL_CHECKED(p.status, bounds::check_tma_load(boxa, ax, ay), bounds::kSiteGemmA))
              tma_load_2d_pair(sa + j * P_ATOM, &tmA, fb, ax, ay);
            if (MTL_CHECKED(p.status, bounds::check_tma_load(boxb, bx, by), bounds::kSiteGemmB))
              tma_load_2d_pair(sb + j * P_ATOM, &tmB, fb, bx, by);
          }
          if (++stage == P_STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (leader)
    if (lane == 0 && rank == 0) {
      const uint32_t idesc = F8 ? idesc_f8_f32(2 * P_HALF, BN, p.fmt_a, p.fmt_b)
                                : idesc_bf16_f32(2 * P_HALF, BN, p.a_mn != 0, p.b_mn != 0);
      const bool a_mn = !F8 && p.a_mn, b_mn = !F8 && p.b_mn;
      const uint64_t a_desc0 = a_mn ? desc_mnbase(sA0, P_ATOM) : desc_kbase(sA0);
      const uint64_t b_desc0 = b_mn ? desc_mnbase(sB0, P_ATOM) : desc_kbase(sB0);
      int stage = 0;
      uint32_t phase = 0;
      int unit = 0;
      bool ok = true;
      PieceIter pit;
      piece_begin(p, pair_id, npairs, pit);
      Piece pc;
      while (ok && piece_next(p, pit, pc)) {
        // a unit is one partition (partials summed) or the piece's whole K range
        const int nunits = REDUCE ? pc.g1 - pc.g0 : 1;
        const int kb_unit = REDUCE ? p.kb_per_unit : (pc.g1 - pc.g0) * p.split_g;
        for (int u = 0; u < nunits && ok; ++u, ++unit) {
          const int buf = unit & 1;
          const uint32_t uphase = (unit >> 1) & 1;
          if (!mbar_wait_bounded_cluster(tempty_bar(buf), uphase ^ 1u, p.status, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + buf * BN;
          for (int kb = 0; kb < kb_unit; ++kb) {
            if (!mbar_wait_bounded(full_bar(stage), phase, p.status, abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t ad0 = a_desc0 + (uint64_t)(stage * (P_A_BYTES / 16));
            const uint64_t bd0 = b_desc0 + (uint64_t)(stage * (P_B_BYTES / 16));
#pragma unroll
            for (int kk = 0; kk < P_KSTEPS; ++kk) {
              const uint32_t ao = a_mn ? mnmajor_off(kk) : kmajor_off(kk, P_ATOM);
              const uint32_t bo = b_mn ? mnmajor_off(kk) : kmajor_off(kk, P_ATOM);
              if (F8)
                tc_mma_f8_pair(d_tmem, desc_add(ad0, ao), desc_add(bd0, bo), idesc,
                               (kb > 0 || kk > 0) ? 1u : 0u);
              else
                tc_mma_bf16_pair(d_tmem, desc_add(ad0, ao), desc_add(bd0, bo), idesc,
                                 (kb > 0 || kk > 0) ? 1u : 0u);
            }
            tc_commit_pair_mc(empty_bar(stage), 3);
            if (++stage == P_STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (ok) tc_commit_pair_mc(tfull_bar(buf), 3);
        }
      }
    }
    __syncwarp();
  }

  tc_fence_before();
  cluster_sync();
  if (warp == 1) {
    if (*abort_flag) {
      const long long t0 = clock64();
      while (clock64() - t0 < 2000000LL) {
      }
    }
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

// ---------------------------------------------------------------- host side

typedef void (*KernelFn)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, Params);

// The pair kernels with the tail-slice epilogue (gemm_split.cu): bf16 and FP8.
KernelFn select_kernel2_split(int epi, bool f32, bool red);
KernelFn select_kernel8_split(int epi, bool f32, bool red);

// Slices per tile of the last, partial wave of num_tiles tiles over npairs
// pairs (1: no split): as many as give every tail slice its own pair, at most
// one per granule and at most MAX_SLICES, for tiles of at least
// SPLIT_MIN_KBLOCKS 128-deep K-blocks (a shorter tile's saved time, ~0.5 us a
// K-block, does not pay for the slices' write-out and the ordered re-read).
constexpr int MAX_SLICES = 16;
constexpr int SPLIT_MIN_KBLOCKS = 48;
inline int tail_slices(int num_tiles, int npairs, int gpt, int kb_per_tile) {
  if (npairs < 2 || num_tiles < npairs || kb_per_tile < SPLIT_MIN_KBLOCKS) return 1;
  const int rem = num_tiles % npairs;
  if (rem == 0) return 1;
  int s = npairs / rem;
  if (s > gpt) s = gpt;
  if (s > MAX_SLICES) s = MAX_SLICES;
  return s < 2 ? 1 : s;
}

// Scratch bound for M x N outputs over npairs pairs (any K): slots for the
// tail tiles' slices, and counters.
inline void split_scratch_for(int num_tiles, int npairs, size_t* bytes, size_t* counters) {
  const int s = tail_slices(num_tiles, npairs, MAX_SLICES, SPLIT_MIN_KBLOCKS);
  const int rem = s > 1 ? num_tiles % npairs : 0;
  *bytes = (size_t)rem * s * SPLIT_REGIONS * SPLIT_REGION_FLOATS * sizeof(float);
  *counters = (size_t)rem * SPLIT_REGIONS;
}

// Fills the work-split fields of p (granules, raster, tail slices) for a
// launch over npairs pairs; the tail is split only with enough scratch in a
// (else every tile runs whole).
inline void plan_split(Params& p, bool reduce, int npairs, bool pair_kernel, const GemmArgs& a) {
  p.csum = a.epi == EPI_DGELU && a.N % 32 == 0 ? a.colsum_part : nullptr;
  p.raster_n = p.tiles_n <= RASTER_N_MAX;
  p.split_g = reduce ? p.kb_per_unit : 1;
  p.split_gpt = reduce ? p.units_per_tile : p.kb_per_unit;
  p.dp_tiles = p.num_tiles;
  p.split_s = 1;
  p.split_ws = nullptr;
  p.split_cnt = nullptr;
  if (!pair_kernel) return;
  const int s = tail_slices(p.num_tiles, npairs, p.split_gpt, p.split_gpt * p.split_g);
  if (s <= 1) return;
  const int rem = p.num_tiles % npairs;
  const size_t bytes = (size_t)rem * s * SPLIT_REGIONS * SPLIT_REGION_FLOATS * sizeof(float);
  if (!a.split_ws || !a.split_cnt || a.split_ws_bytes < bytes ||
      a.split_cnt_count < (size_t)rem * SPLIT_REGIONS)
    return;
  p.dp_tiles = p.num_tiles - rem;
  p.split_s = s;
  p.split_ws = a.split_ws;
  p.split_cnt = a.split_cnt;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, []() {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// 2D map over a row-major matrix with `rows` rows of `cols` elements (row pitch
// ld elements; bf16, or bytes when fp8), box of box_cols x box_rows, 128-byte
// swizzle, out-of-range elements read as zero.
inline bool make_map(CUtensorMap* m, const void* ptr, uint64_t cols, uint64_t rows, int64_t ld,
                     uint32_t box_cols, uint32_t box_rows, bool fp8 = false) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld * (fp8 ? 1 : 2)};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
             const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor map of a GEMM output for the epilogue's TMA stores: [rows][cols] of
// bf16 or fp32 with row pitch ld elements, 32 x 32 boxes in the swizzle the
// staging chunk uses (64-byte rows: 64-byte swizzle; 128-byte rows: 128-byte).
inline bool make_out_map(CUtensorMap* m, const void* ptr, uint64_t cols, uint64_t rows,
                         int64_t ld, bool f32) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld * (f32 ? 4 : 2)};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
             const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             f32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
             CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The C and z maps of a GEMM (z: EPI_BIAS_GELU with a bf16 C; otherwise a copy
// of the C map, never used).
inline bool make_epilogue_maps(CUtensorMap* mc, CUtensorMap* mz, const GemmArgs& a) {
  if (!make_out_map(mc, a.C, (uint64_t)a.N, (uint64_t)a.M, a.ldc, a.c_f32)) return false;
  if (a.epi == EPI_BIAS_GELU && !a.c_f32)
    return make_out_map(mz, a.Z, (uint64_t)a.N, (uint64_t)a.M, a.ldz, false);
  *mz = *mc;
  return true;
}

}  // namespace tcg
}  // namespace mtl
