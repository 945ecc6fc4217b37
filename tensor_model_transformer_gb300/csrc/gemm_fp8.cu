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

// Block-wide max of non-negative floats, then one atomicMax on the bits (for
// non-negative IEEE floats the unsigned order is the float order).
template <typename T>
__global__ void __launch_bounds__(QTHREADS) amax_kernel(const T* __restrict__ x, int64_t rows,
                                                        int64_t cols, int64_t ld,
                                                        unsigned* __restrict__ amax_bits) {
  constexpr int E = Vec<T>::N;
  __shared__ float red[QTHREADS / 32];
  float m = 0.f;
  for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
    const T* row = x + r * ld;
    for (int64_t c = (int64_t)threadIdx.x * E; c < cols; c += (int64_t)QTHREADS * E) {
      Vec<T> v;
      v.load(row + c);
#pragma unroll
      for (int e = 0; e < E; ++e) m = fmaxf(m, fabsf(v.get(e)));
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

// q = fp8(x * scale), 16 elements (16 bytes out) per thread and step.
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
  const __nv_fp8_interpretation_t kind = FMT == 0 ? __NV_E4M3 : __NV_E5M2;
  for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
    const T* row = x + r * ld;
    uint8_t* qrow = q + r * ldq;
    for (int64_t c = (int64_t)threadIdx.x * 16; c < cols; c += (int64_t)QTHREADS * 16) {
      float f[16];
#pragma unroll
      for (int j = 0; j < 16 / E; ++j) {
        Vec<T> v;
        v.load(row + c + j * E);
#pragma unroll
        for (int e = 0; e < E; ++e) f[j * E + e] = __fmul_rn(v.get(e), scale);
      }
      uint4 out;
      uint32_t* w = reinterpret_cast<uint32_t*>(&out);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(f[4 * k], f[4 * k + 1]),
                                                     __NV_SATFINITE, kind);
        const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(f[4 * k + 2], f[4 * k + 3]),
                                                     __NV_SATFINITE, kind);
        w[k] = (lo & 0xFFFFu) | (hi << 16);
      }
      *reinterpret_cast<uint4*>(qrow + c) = out;
    }
  }
}

// qT = fp8(x * scale) transposed: qT[c][r] for x [rows][cols], and optionally
// the row-major q from the same read.  A CTA converts a 64 x 64 tile row-wise
// into a byte tile in shared memory (16 elements per thread; those 16 bytes
// also go to q), then writes it column-wise: 16 consecutive rows of one column
// make one 16-byte store of an output row.  rows % 16 == 0.
constexpr int CT = 64;
template <typename T, int FMT>
__global__ void __launch_bounds__(QTHREADS) cast_transpose_kernel(
    const T* __restrict__ x, int64_t rows, int64_t cols, int64_t ld,
    const unsigned* __restrict__ amax_bits, float* __restrict__ scale_out,
    uint8_t* __restrict__ qT, int64_t ldqT, uint8_t* __restrict__ q, int64_t ldq) {
  constexpr int E = Vec<T>::N;
  __shared__ __align__(16) uint8_t tile[CT][CT + 16];   // rows of 80 bytes: 16-byte aligned
  const float amax = __uint_as_float(*amax_bits);
  const float maxv = FMT == 0 ? 448.0f : 57344.0f;
  const float scale = amax > 0.f ? __fdiv_rn(maxv, amax) : 1.0f;
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *scale_out = scale;
  const __nv_fp8_interpretation_t kind = FMT == 0 ? __NV_E4M3 : __NV_E5M2;
  const int64_t r0 = (int64_t)blockIdx.y * CT, c0 = (int64_t)blockIdx.x * CT;
  // load: thread -> (row tr, 16 columns from tc)
  {
    const int tr = threadIdx.x >> 2, tc = (threadIdx.x & 3) * 16;
    const int64_t r = r0 + tr, c = c0 + tc;
    float f[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) f[i] = 0.f;
    if (r < rows && c < cols) {   // cols % 16 == 0: the 16 columns are all in range
#pragma unroll
      for (int j = 0; j < 16 / E; ++j) {
        Vec<T> v;
        v.load(x + r * ld + c + j * E);
#pragma unroll
        for (int e = 0; e < E; ++e) f[j * E + e] = __fmul_rn(v.get(e), scale);
      }
    }
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(f[4 * k], f[4 * k + 1]),
                                                   __NV_SATFINITE, kind);
      const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(f[4 * k + 2], f[4 * k + 3]),
                                                   __NV_SATFINITE, kind);
      w[k] = (lo & 0xFFFFu) | (hi << 16);
    }
    *reinterpret_cast<uint4*>(&tile[tr][tc]) = make_uint4(w[0], w[1], w[2], w[3]);
    if (q && r < rows && c < cols)
      *reinterpret_cast<uint4*>(q + r * ldq + c) = make_uint4(w[0], w[1], w[2], w[3]);
  }
  __syncthreads();
  // store: thread -> (output row oc = tile column, 16 rows from orr)
  {
    const int oc = threadIdx.x >> 2, orr = (threadIdx.x & 3) * 16;
    const int64_t c = c0 + oc, r = r0 + orr;
    if (c < cols && r < rows) {
      uint32_t w[4];
#pragma unroll
      for (int k = 0; k < 4; ++k)
        w[k] = (uint32_t)tile[orr + 4 * k][oc] | ((uint32_t)tile[orr + 4 * k + 1][oc] << 8) |
               ((uint32_t)tile[orr + 4 * k + 2][oc] << 16) |
               ((uint32_t)tile[orr + 4 * k + 3][oc] << 24);
      *reinterpret_cast<uint4*>(qT + c * ldqT + r) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

}  // namespace f8

namespace tcg {

typedef void (*KernelFn)(CUtensorMap, CUtensorMap, Params);

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
  KernelFn fn = select_kernel8(a.epi, a.c_f32, reduce);
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
  fn<<<grid, THREADS, P_SMEM_BYTES, c.stream>>>(ma, mb, p);
  c.after();
  return cudaGetLastError();
}

cudaError_t fp8_quantize2(int src_dtype, const void* x, int64_t rows, int64_t cols, int64_t ld,
                          int fmt, unsigned* amax_bits, float* scale, void* q, int64_t ldq,
                          void* qT, int64_t ldqT, const LaunchCtx& c) {
  using namespace f8;
  if (rows == 0 || cols == 0) return cudaSuccess;
  if (cols % 16 || rows % 16 || (fmt != 0 && fmt != 1)) return cudaErrorInvalidValue;
  cudaError_t e;
  if (!qT) {
    // amax, then the row-major cast (which also writes the scale)
    return fp8_quantize(src_dtype, x, rows, cols, ld, fmt, amax_bits, scale, q, ldq, c);
  }
  {
    const int64_t want = 4LL * c.num_sms;
    const int grid = (int)(rows < want ? rows : want);
    c.before(KK_QUANT, (double)rows * cols * (src_dtype == kBF16 ? 2 : 4));
    if (src_dtype == kBF16)
      amax_kernel<bf16><<<grid, QTHREADS, 0, c.stream>>>(static_cast<const bf16*>(x), rows, cols,
                                                         ld, amax_bits);
    else
      amax_kernel<float><<<grid, QTHREADS, 0, c.stream>>>(static_cast<const float*>(x), rows,
                                                          cols, ld, amax_bits);
    c.after();
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  dim3 grid((unsigned)((cols + CT - 1) / CT), (unsigned)((rows + CT - 1) / CT));
  c.before(KK_QUANT, (double)rows * cols * ((src_dtype == kBF16 ? 2 : 4) + (q ? 2 : 1)));
  uint8_t* qb = static_cast<uint8_t*>(qT);
  uint8_t* qr = static_cast<uint8_t*>(q);
#define CASTT(T, F)                                                                      \
  cast_transpose_kernel<T, F><<<grid, QTHREADS, 0, c.stream>>>(                          \
      static_cast<const T*>(x), rows, cols, ld, amax_bits, scale, qb, ldqT, qr, ldq)
  if (src_dtype == kBF16) {
    if (fmt == 0) CASTT(bf16, 0); else CASTT(bf16, 1);
  } else {
    if (fmt == 0) CASTT(float, 0); else CASTT(float, 1);
  }
#undef CASTT
  c.after();
  return cudaGetLastError();
}

cudaError_t fp8_quantize(int src_dtype, const void* x, int64_t rows, int64_t cols, int64_t ld,
                         int fmt, unsigned* amax_bits, float* scale, void* q, int64_t ldq,
                         const LaunchCtx& c) {
  using namespace f8;
  if (rows == 0 || cols == 0) return cudaSuccess;
  if (cols % 16 || (fmt != 0 && fmt != 1)) return cudaErrorInvalidValue;
  const int64_t want = 4LL * c.num_sms;
  const int grid = (int)(rows < want ? rows : want);
  const double bytes = (double)rows * cols * (src_dtype == kBF16 ? 2 : 4);
  c.before(KK_QUANT, bytes);
  if (src_dtype == kBF16)
    amax_kernel<bf16><<<grid, QTHREADS, 0, c.stream>>>(static_cast<const bf16*>(x), rows, cols, ld,
                                                       amax_bits);
  else
    amax_kernel<float><<<grid, QTHREADS, 0, c.stream>>>(static_cast<const float*>(x), rows, cols,
                                                        ld, amax_bits);
  c.after();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  c.before(KK_QUANT, bytes + (double)rows * cols);
  uint8_t* qb = static_cast<uint8_t*>(q);
#define CAST(T, F)                                                                              \
  cast_kernel<T, F><<<grid, QTHREADS, 0, c.stream>>>(static_cast<const T*>(x), rows, cols, ld, \
                                                     amax_bits, scale, qb, ldq)
  if (src_dtype == kBF16) {
    if (fmt == 0) CAST(bf16, 0); else CAST(bf16, 1);
  } else {
    if (fmt == 0) CAST(float, 0); else CAST(float, 1);
  }
#undef CAST
  c.after();
  return cudaGetLastError();
}

}  // namespace mtl
