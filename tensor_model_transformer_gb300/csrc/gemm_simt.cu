// CUDA-core GEMM with exact fp32 arithmetic: the path of fp32 layers, whose
// tolerance (1e-5 of the largest output) rules out tensor-core tf32.
//
// C = epi( sum_{p = 0..parts-1} P_p ),  P_p = sum_{k in part p} A(m,k) B(n,k)
// Each part is accumulated on its own and the parts are added in order -- the
// row-parallel GEMM's partial outputs and their g / f sum ("Megatron-LM:
// GPU-Cluster Training Parallelism", section "Paper 1: The f/g Conjugate
// Operators").  64x64 output tile per 256-thread block, 4x4 per thread.
#include "common.cuh"
#include "kernels.h"

namespace mtl {
namespace {

constexpr int TM = 64, TN = 64, TK = 16;

template <typename T, int EPI, bool OUT_F32>
__global__ void __launch_bounds__(256) gemm_simt_kernel(GemmArgs a) {
  __shared__ float As[TK][TM + 4];
  __shared__ float Bs[TK][TN + 4];
  const T* Ap = static_cast<const T*>(a.A.ptr);
  const T* Bp = static_cast<const T*>(a.B.ptr);
  const int m0 = blockIdx.y * TM, n0 = blockIdx.x * TN;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float sum[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) sum[i][j] = 0.f;
  const int kpart = a.K / a.parts;
  for (int p = 0; p < a.parts; ++p) {
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
    const int kbeg = p * kpart, kend = kbeg + kpart;
    for (int k0 = kbeg; k0 < kend; k0 += TK) {
      for (int i = threadIdx.x; i < TM * TK; i += 256) {
        int mm, kk;
        if (a.A.k_major) { kk = i % TK; mm = i / TK; } else { mm = i % TM; kk = i / TM; }
        const int gm = m0 + mm, gk = k0 + kk;
        float v = 0.f;
        if (gm < a.M && gk < kend)
          v = to_f<T>(a.A.k_major ? Ap[(size_t)gm * a.A.ld + gk] : Ap[(size_t)gk * a.A.ld + gm]);
        As[kk][mm] = v;
      }
      for (int i = threadIdx.x; i < TN * TK; i += 256) {
        int nn, kk;
        if (a.B.k_major) { kk = i % TK; nn = i / TK; } else { nn = i % TN; kk = i / TN; }
        const int gn = n0 + nn, gk = k0 + kk;
        float v = 0.f;
        if (gn < a.N && gk < kend)
          v = to_f<T>(a.B.k_major ? Bp[(size_t)gn * a.B.ld + gk] : Bp[(size_t)gk * a.B.ld + gn]);
        Bs[kk][nn] = v;
      }
      __syncthreads();
#pragma unroll
      for (int kk = 0; kk < TK; ++kk) {
        float av[4], bv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) av[i] = As[kk][ty * 4 + i];
#pragma unroll
        for (int j = 0; j < 4; ++j) bv[j] = Bs[kk][tx * 4 + j];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
      }
      __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) sum[i][j] += acc[i][j];
  }
  const T* bias = static_cast<const T*>(a.bias);
  const T* R = static_cast<const T*>(a.R);
  T* Z = static_cast<T*>(a.Z);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty * 4 + i;
    if (m >= a.M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n >= a.N) continue;
      float v = sum[i][j];
      if (EPI == EPI_BIAS || EPI == EPI_BIAS_RESID || EPI == EPI_BIAS_GELU) v += to_f<T>(bias[n]);
      if (EPI == EPI_BIAS_RESID && a.drop.on)
        v = drop_keep((unsigned long long)m * a.N + n, a.drop) ? v * a.drop.scale : 0.f;
      if (EPI == EPI_BIAS_RESID) v += to_f<T>(R[(size_t)m * a.ldr + n]);
      if (EPI == EPI_DGELU) v *= gelu_grad_f(to_f<T>(Z[(size_t)m * a.ldz + n]));
      if (EPI == EPI_BIAS_GELU) {
        Z[(size_t)m * a.ldz + n] = from_f<T>(v);
        v = gelu_f(v);
      }
      if (OUT_F32)
        static_cast<float*>(a.C)[(size_t)m * a.ldc + n] = v;
      else
        static_cast<T*>(a.C)[(size_t)m * a.ldc + n] = from_f<T>(v);
    }
  }
}

template <typename T, int EPI>
cudaError_t launch_epi(const GemmArgs& a, const LaunchCtx& c) {
  dim3 grid((a.N + TN - 1) / TN, (a.M + TM - 1) / TM);
  c.before(KK_GEMM_SIMT, 2.0 * a.M * a.N * a.K);
  if (a.c_f32)
    gemm_simt_kernel<T, EPI, true><<<grid, 256, 0, c.stream>>>(a);
  else
    gemm_simt_kernel<T, EPI, false><<<grid, 256, 0, c.stream>>>(a);
  c.after();
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_t(const GemmArgs& a, const LaunchCtx& c) {
  switch (a.epi) {
    case EPI_STORE: return launch_epi<T, EPI_STORE>(a, c);
    case EPI_BIAS: return launch_epi<T, EPI_BIAS>(a, c);
    case EPI_BIAS_RESID: return launch_epi<T, EPI_BIAS_RESID>(a, c);
    case EPI_BIAS_GELU: return launch_epi<T, EPI_BIAS_GELU>(a, c);
    case EPI_DGELU: return launch_epi<T, EPI_DGELU>(a, c);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t gemm_simt(int dtype, const GemmArgs& a, const LaunchCtx& c) {
  if (a.M == 0 || a.N == 0) return cudaSuccess;
  return dtype == kBF16 ? launch_t<bf16>(a, c) : launch_t<float>(a, c);
}

}  // namespace mtl
