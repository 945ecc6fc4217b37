// FP8 GEMMs and per-tensor FP8 quantization for sm_103a.
//
// The pages list FP8 training ("--fp8-hybrid") among the framework's features
// without a recipe; read here as: forward GEMM operands (activations and
// weights) in E4M3, gradient operands in E5M2, each tensor scaled by
// fmt_max / amax over the whole tensor (all t partitions together), the
// accumulator multiplied back by 1 / (scale_a * scale_b) in fp32 before the
// fused epilogue.  The GEMM is the 2-CTA pair kernel of gemm_core.cuh
// instantiated with FP8 operands (tcgen05.mma kind::f8f6f4); both operands are
// K-major, so a transposed use of a tensor (a weight or data gradient) gets a
// transposed FP8 copy from the quantizer rather than a transposed descriptor.
#include <cuda_fp8.h>

#include <cstring>

#include "gemm_core.cuh"

namespace mtl {
namespace f8 {

constexpr int QTHREADS = 256;

// A thread takes the same column vectors of QROWS rows at once (rows
// blockIdx.x + k * gridDim.x), so that up to QROWS * ceil(cols / (QTHREADS * E))
// 16-byte loads are in flight.
constexpr int QROWS = 4;

// Block-wide max of non-negative floats, then one atomicMax on the bits (for
// non-negative IEEE floats the unsigned order is the float order).
template <typename T>
__global__ void __launch_bounds__(QTHREADS) amax_kernel(const T* __restrict__ x, int64_t rows,
                                                        int64_t cols, int64_t ld,
                                                        unsigned* __restrict__ amax_bits) {
  constexpr int E = Vec<T>::N;
  __shared__ float red[QTHREADS / 32];
  float m = 0.f;
  const int64_t G = gridDim.x;
  for (int64_t r0 = blockIdx.x; r0 < rows; r0 += QROWS * G) {
    for (int64_t c = (int64_t)threadIdx.x * E; c < cols; c += (int64_t)QTHREADS * E) {
      Vec<T> v[QROWS];
#pragma unroll
      for (int k = 0; k < QROWS; ++k)
        if (r0 + k * G < rows) v[k].load(x + (r0 + k * G) * ld + c);
#pragma unroll
      for (int k = 0; k < QROWS; ++k) {
        if (r0 + k * G >= rows) continue;
        float f[E];
        v[k].unpack(f);
#pragma unroll
        for (int e = 0; e < E; ++e) m = fmaxf(m, fabsf(f[e]));
      }
    }
  }
  m = warp_max(m);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < QTHREADS / 32; ++w) m = fmaxf(m, red[w]);
    atomicMax(amax_bits, __float_as_uint(m));
  }
}

// 16 fp32 values -> 16 fp8 bytes (saturating, round to nearest even).
template <int FMT>
__device__ __forceinline__ uint4 to_fp8x16(const float (&f)[16]) {
  const __nv_fp8_interpretation_t kind = FMT == 0 ? __NV_E4M3 : __NV_E5M2;
  uint32_t w[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t lo =
        __nv_cvt_float2_to_fp8x2(make_float2(f[4 * k], f[4 * k + 1]), __NV_SATFINITE, kind);
    const uint32_t hi =
        __nv_cvt_float2_to_fp8x2(make_float2(f[4 * k + 2], f[4 * k + 3]), __NV_SATFINITE, kind);
    w[k] = (lo & 0xFFFFu) | (hi << 16);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// q = fp8(x * scale), 16 elements (16 bytes out) per thread, row and step.
template <typename T, int FMT>
__global__ void __launch_bounds__(QTHREADS) cast_kernel(const T* __restrict__ x, int64_t rows,
                                                        int64_t cols, int64_t ld,
                                                        const unsigned* __restrict__ amax_bits,
                                                        float* __restrict__ scale_out,
                                                        uint8_t* __restrict__ q, int64_t ldq) {
  constexpr int E = Vec<T>::N;
  const float amax = __uint_as_float(*amax_bits);
  const float maxv = FMT == 0 ? 448.0f : 57344.0f;
  const float scale = amax > 0.f ? __fdiv_rn(maxv, amax) : 1.0f;
  if (blockIdx.x == 0 && threadIdx.x == 0) *scale_out = scale;
  const int64_t G = gridDim.x;
  for (int64_t r0 = blockIdx.x; r0 < rows; r0 += QROWS * G) {
    for (int64_t c = (int64_t)threadIdx.x * 16; c < cols; c += (int64_t)QTHREADS * 16) {
      Vec<T> v[QROWS][16 / E];
#pragma unroll
      for (int k = 0; k < QROWS; ++k)
        if (r0 + k * G < rows) {
#pragma unroll
          for (int j = 0; j < 16 / E; ++j) v[k][j].load(x + (r0 + k * G) * ld + c + j * E);
        }
#pragma unroll
      for (int k = 0; k < QROWS; ++k) {
        if (r0 + k * G >= rows) continue;
        float f[16];
#pragma unroll
        for (int j = 0; j < 16 / E; ++j) {
          float g[E];
          v[k][j].unpack(g);
#pragma unroll
          for (int e = 0; e < E; ++e) f[j * E + e] = __fmul_rn(g[e], scale);
        }
        *reinterpret_cast<uint4*>(q + (r0 + k * G) * ldq + c) = to_fp8x16<FMT>(f);
      }
    }
  }
}

// qT = fp8(x * scale) transposed: qT[c][r] for x [rows][cols], and optionally
// the row-major q from the same read.  A CTA takes CTX tiles of 64 x 64 side by
// side along the columns (all their loads issued first) and converts them
// row-wise into byte tiles in shared memory, 16 elements per thread and tile
// (those 16 bytes also go to q).  Then each thread reads a 16 x 4 block (16
// rows, one 32-bit word each) of one tile, transposes it with byte permutes and
// stores four 16-byte pieces of output rows.  A tile row is 16 words; rows
// 16j..16j+15 start 8j words further on, so that the four 16-row groups a warp
// reads fall on disjoint banks.  rows % 16 == 0.
constexpr int CT = 64, CTX = 4;
constexpr int TILE_WORDS = CT * 16 + 32;
__device__ __forceinline__ int tile_word(int row, int wcol) { return row * 16 + (row >> 4) * 8 + wcol; }

template <typename T, int FMT>
__global__ void __launch_bounds__(QTHREADS) cast_transpose_kernel(
    const T* __restrict__ x, int64_t rows, int64_t cols, int64_t ld,
    const unsigned* __restrict__ amax_bits, float* __restrict__ scale_out,
    uint8_t* __restrict__ qT, int64_t ldqT, uint8_t* __restrict__ q, int64_t ldq) {
  static_assert(QTHREADS == CTX * 64, "one thread per 16 x 4 block of each tile");
  constexpr int E = Vec<T>::N;
  __shared__ __align__(16) uint32_t tile[CTX * TILE_WORDS];
  const float amax = __uint_as_float(*amax_bits);
  const float maxv = FMT == 0 ? 448.0f : 57344.0f;
  const float scale = amax > 0.f ? __fdiv_rn(maxv, amax) : 1.0f;
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *scale_out = scale;
  const int64_t r0 = (int64_t)blockIdx.y * CT, cb = (int64_t)blockIdx.x * CT * CTX;
  // convert: thread -> (row tr, 16 columns from tc) of every tile
  {
    const int tr = threadIdx.x >> 2, tc = (threadIdx.x & 3) * 16;
    const int64_t r = r0 + tr;
    Vec<T> v[CTX][16 / E];
#pragma unroll
    for (int t = 0; t < CTX; ++t) {
      const int64_t c = cb + t * CT + tc;
      if (r < rows && c < cols) {   // cols % 16 == 0: the 16 columns are all in range
#pragma unroll
        for (int j = 0; j < 16 / E; ++j) v[t][j].load(x + r * ld + c + j * E);
      }
    }
#pragma unroll
    for (int t = 0; t < CTX; ++t) {
      const int64_t c = cb + t * CT + tc;
      const bool live = r < rows && c < cols;
      float f[16];
#pragma unroll
      for (int j = 0; j < 16 / E; ++j) {
        float g[E];
        if (live) v[t][j].unpack(g);
#pragma unroll
        for (int e = 0; e < E; ++e) f[j * E + e] = live ? __fmul_rn(g[e], scale) : 0.f;
      }
      const uint4 w = to_fp8x16<FMT>(f);
      *reinterpret_cast<uint4*>(&tile[t * TILE_WORDS + tile_word(tr, tc / 4)]) = w;
      if (q && live) *reinterpret_cast<uint4*>(q + r * ldq + c) = w;
    }
  }
  __syncthreads();
  // transpose: thread -> tile t, 16-row group rg, word column wc (columns 4wc..4wc+3)
  {
    const int t = threadIdx.x >> 6, l = threadIdx.x & 63;
    const int rg = l & 3, wc = l >> 2;
    const int64_t r = r0 + rg * 16, c = cb + t * CT + wc * 4;
    if (r < rows && c < cols) {   // cols % 16 == 0: the 4 columns are all in range
      const uint32_t* src = &tile[t * TILE_WORDS];
      uint32_t w[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) w[i] = src[tile_word(rg * 16 + i, wc)];
      uint32_t o[4][4];   // o[j][k]: column 4wc+j, rows 4k..4k+3 of the group
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t t0 = __byte_perm(w[4 * k], w[4 * k + 1], 0x5140);
        const uint32_t t1 = __byte_perm(w[4 * k], w[4 * k + 1], 0x7362);
        const uint32_t t2 = __byte_perm(w[4 * k + 2], w[4 * k + 3], 0x5140);
        const uint32_t t3 = __byte_perm(w[4 * k + 2], w[4 * k + 3], 0x7362);
        o[0][k] = __byte_perm(t0, t2, 0x5410);
        o[1][k] = __byte_perm(t0, t2, 0x7632);
        o[2][k] = __byte_perm(t1, t3, 0x5410);
        o[3][k] = __byte_perm(t1, t3, 0x7632);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j)
        *reinterpret_cast<uint4*>(qT + (c + j) * ldqT + r) = make_uint4(o[j][0], o[j][1], o[j][2], o[j][3]);
    }
  }
}

}  // namespace f8

namespace tcg {

template <int EPI, bool F32, bool RED>
static KernelFn kernel8_ptr() {
  return reinterpret_cast<KernelFn>(gemm_tc2_kernel<EPI, F32, RED, true>);
}

static KernelFn select_kernel8(int epi, bool f32, bool red) {
#define SEL8(E)                                                                          \
  if (epi == E) {                                                                        \
    if (f32) return red ? kernel8_ptr<E, true, true>() : kernel8_ptr<E, true, false>();  \
    return red ? kernel8_ptr<E, false, true>() : kernel8_ptr<E, false, false>();         \
  }
  SEL8(EPI_STORE)
  SEL8(EPI_BIAS)
  SEL8(EPI_BIAS_RESID)
  SEL8(EPI_BIAS_GELU)
  SEL8(EPI_DGELU)
#undef SEL8
  return nullptr;
}

}  // namespace tcg

bool gemm_fp8_supported(const GemmArgs& a, int num_sms) {
  if (num_sms < 2) return false;
  if (a.parts < 1 || a.K <= 0 || a.K % a.parts || (a.K / a.parts) % tcg::P_BK) return false;
  if (!a.A.k_major || !a.B.k_major) return false;
  if ((a.fmt_a != 0 && a.fmt_a != 1) || (a.fmt_b != 0 && a.fmt_b != 1)) return false;
  if (!a.scale_a || !a.scale_b) return false;
  auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  if (!al16(a.A.ptr) || !al16(a.B.ptr) || !al16(a.C)) return false;
  if ((a.A.ld % 16) || (a.B.ld % 16) || (a.ldc % 8)) return false;
  if (a.epi == EPI_BIAS_RESID && ((a.ldr % 8) || !al16(a.R))) return false;
  if ((a.epi == EPI_BIAS_GELU || a.epi == EPI_DGELU) && ((a.ldz % 8) || !al16(a.Z))) return false;
  if ((a.epi == EPI_BIAS || a.epi == EPI_BIAS_RESID || a.epi == EPI_BIAS_GELU) && !al16(a.bias))
    return false;
  return true;
}

cudaError_t gemm_fp8(const GemmArgs& a, const LaunchCtx& c) {
  using namespace tcg;
  if (a.M == 0 || a.N == 0) return cudaSuccess;
  if (!gemm_fp8_supported(a, c.num_sms)) return cudaErrorInvalidValue;
  CUtensorMap ma, mb;
  // K-major boxes: 128 rows of 128 fp8 (one 128-byte swizzle span)
  if (!make_map(&ma, a.A.ptr, (uint64_t)a.K, (uint64_t)a.M, a.A.ld, 128, 128, true) ||
      !make_map(&mb, a.B.ptr, (uint64_t)a.K, (uint64_t)a.N, a.B.ld, 128, 128, true))
    return cudaErrorInvalidValue;
  CUtensorMap mc, mz;
  if (!make_epilogue_maps(&mc, &mz, a)) return cudaErrorInvalidValue;
  Params p;
  memset(&p, 0, sizeof(p));
  p.M = a.M;
  p.N = a.N;
  p.K = a.K;
  p.parts = a.parts;
  const bool reduce = a.parts > 1;
  p.units_per_tile = reduce ? a.parts : 1;
  p.kb_per_unit = (a.K / a.parts) / P_BK;
  p.tiles_m = (a.M + 2 * P_HALF - 1) / (2 * P_HALF);
  p.tiles_n = (a.N + BN - 1) / BN;
  p.num_tiles = p.tiles_m * p.tiles_n;
  p.bias = static_cast<const bf16*>(a.bias);
  p.R = static_cast<const bf16*>(a.R);
  p.ldr = a.ldr;
  p.Z = static_cast<bf16*>(a.Z);
  p.ldz = a.ldz;
  p.C = a.C;
  p.ldc = a.ldc;
  p.status = a.status;
  p.drop = a.drop;
  p.fmt_a = a.fmt_a;
  p.fmt_b = a.fmt_b;
  p.scale_a = a.scale_a;
  p.scale_b = a.scale_b;
  plan_split(p, reduce, c.num_sms / 2, true, a);
  KernelFn fn = p.split_s > 1 ? select_kernel8_split(a.epi, a.c_f32, reduce)
                              : select_kernel8(a.epi, a.c_f32, reduce);
  if (!fn) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void*>(fn),
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, P_SMEM_BYTES);
  if (e != cudaSuccess) return e;
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, reinterpret_cast<const void*>(fn));
  if (e != cudaSuccess) return e;
  if (fa.numRegs != LAUNCH_REGS) return cudaErrorInvalidConfiguration;
  const int pairs = c.num_sms / 2;
  const int grid = 2 * (p.num_tiles < pairs ? p.num_tiles : pairs);
  c.before(KK_GEMM_FP8, 2.0 * a.M * a.N * a.K);
  fn<<<grid, THREADS, P_SMEM_BYTES, c.stream>>>(ma, mb, mc, mz, p);
  c.after();
  return cudaGetLastError();
}

cudaError_t fp8_amax(int src_dtype, const void* x, int64_t rows, int64_t cols, int64_t ld,
                     unsigned* amax_bits, const LaunchCtx& c) {
  using namespace f8;
  if (rows == 0 || cols == 0) return cudaSuccess;
  if (cols % 16) return cudaErrorInvalidValue;
  const int64_t want = 4LL * c.num_sms;
  const int grid = (int)(rows < want ? rows : want);
  c.before(KK_QUANT, (double)rows * cols * (src_dtype == kBF16 ? 2 : 4));
  if (src_dtype == kBF16)
    amax_kernel<bf16><<<grid, QTHREADS, 0, c.stream>>>(static_cast<const bf16*>(x), rows, cols, ld,
                                                       amax_bits);
  else
    amax_kernel<float><<<grid, QTHREADS, 0, c.stream>>>(static_cast<const float*>(x), rows, cols,
                                                        ld, amax_bits);
  c.after();
  return cudaGetLastError();
}

cudaError_t fp8_cast(int src_dtype, const void* x, int64_t rows, int64_t cols, int64_t ld,
                     int fmt, const unsigned* amax_bits, float* scale, void* q, int64_t ldq,
                     void* qT, int64_t ldqT, const LaunchCtx& c) {
  using namespace f8;
  if (rows == 0 || cols == 0) return cudaSuccess;
  if (cols % 16 || (qT && rows % 16) || (fmt != 0 && fmt != 1)) return cudaErrorInvalidValue;
  const int esz = src_dtype == kBF16 ? 2 : 4;
  uint8_t* qr = static_cast<uint8_t*>(q);
  if (qT) {
    dim3 grid((unsigned)((cols + CT * CTX - 1) / (CT * CTX)), (unsigned)((rows + CT - 1) / CT));
    c.before(KK_QUANT, (double)rows * cols * (esz + (q ? 2 : 1)));
    uint8_t* qb = static_cast<uint8_t*>(qT);
#define CASTT(T, F)                                                                      \
  cast_transpose_kernel<T, F><<<grid, QTHREADS, 0, c.stream>>>(                          \
      static_cast<const T*>(x), rows, cols, ld, amax_bits, scale, qb, ldqT, qr, ldq)
    if (src_dtype == kBF16) {
      if (fmt == 0) CASTT(bf16, 0); else CASTT(bf16, 1);
    } else {
      if (fmt == 0) CASTT(float, 0); else CASTT(float, 1);
    }
#undef CASTT
  } else {
    const int64_t want = 4LL * c.num_sms;
    const int grid = (int)(rows < want ? rows : want);
    c.before(KK_QUANT, (double)rows * cols * (esz + 1));
#define CAST(T, F)                                                                              \
  cast_kernel<T, F><<<grid, QTHREADS, 0, c.stream>>>(static_cast<const T*>(x), rows, cols, ld, \
                                                     amax_bits, scale, qr, ldq)
    if (src_dtype == kBF16) {
      if (fmt == 0) CAST(bf16, 0); else CAST(bf16, 1);
    } else {
      if (fmt == 0) CAST(float, 0); else CAST(float, 1);
    }
#undef CAST
  }
  c.after();
  return cudaGetLastError();
}

cudaError_t fp8_quantize2(int src_dtype, const void* x, int64_t rows, int64_t cols, int64_t ld,
                          int fmt, unsigned* amax_bits, float* scale, void* q, int64_t ldq,
                          void* qT, int64_t ldqT, const LaunchCtx& c) {
  if (rows == 0 || cols == 0) return cudaSuccess;
  if (cols % 16 || (qT && rows % 16) || (fmt != 0 && fmt != 1)) return cudaErrorInvalidValue;
  const cudaError_t e = fp8_amax(src_dtype, x, rows, cols, ld, amax_bits, c);
  if (e != cudaSuccess) return e;
  return fp8_cast(src_dtype, x, rows, cols, ld, fmt, amax_bits, scale, q, ldq, qT, ldqT, c);
}

cudaError_t fp8_quantize(int src_dtype, const void* x, int64_t rows, int64_t cols, int64_t ld,
                         int fmt, unsigned* amax_bits, float* scale, void* q, int64_t ldq,
                         const LaunchCtx& c) {
  return fp8_quantize2(src_dtype, x, rows, cols, ld, fmt, amax_bits, scale, q, ldq, nullptr, 0, c);
}

}  // namespace mtl
