// Causal multi-head attention on CUDA cores, exact fp32 arithmetic: the path of
// fp32 layers.  One warp per query row (forward, dQ) or key row (dK, dV).
//
// Each head is local to its partition: the head-interleaved QKV layout puts a
// head's Q, K and V in one contiguous column block ("Megatron-LM: GPU-Cluster
// Training Parallelism", section "Paper 1: QKV Column-Parallel Splitting in
// Detail"), so no partition reads another's columns.  Scale 1/sqrt(d); keys
// after the query get probability 0 (causal scale-mask-softmax, section "Fused
// Transformer Kernels").
#include "common.cuh"
#include "kernels.h"

namespace mtl {
namespace {

constexpr int kWarps = 4;
constexpr int kMaxDPerLane = 4;   // d <= 128

template <typename T>
__device__ __forceinline__ float dot_row(const float* __restrict__ a_smem,
                                         const T* __restrict__ b, int d) {
  float s = 0.f;
  for (int c = 0; c < d; ++c) s = fmaf(a_smem[c], to_f<T>(b[c]), s);
  return s;
}

// grid (ceil(seq / rows_per_block), heads, batch); dynamic smem: kWarps*seq
// floats of scores + kWarps*d floats of query.
// Attention dropout numbering: element (query i, key j) of head hd, batch b is
// e = ((b * heads + hd) * seq + i) * seq + j.
__device__ __forceinline__ unsigned long long drop_index(int b, int hd, int heads, int seq, int i,
                                                         int j) {
  return (((unsigned long long)b * heads + hd) * seq + i) * (unsigned long long)seq + j;
}

template <typename T>
__global__ void attn_fwd_simt_kernel(const T* __restrict__ qkv, T* __restrict__ ctx,
                                     float* __restrict__ lse, int seq, int heads, int d,
                                     int rows_per_block, Dropout drop) {
  extern __shared__ float sm[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* sc = sm + warp * seq;
  float* qs = sm + kWarps * seq + warp * d;
  const int head = blockIdx.y, b = blockIdx.z;
  const int h = heads * d;
  const size_t ld = 3 * (size_t)h;
  const T* base = qkv + (size_t)b * seq * ld + (size_t)head * 3 * d;
  const float scale = 1.0f / sqrtf((float)d);
  const int i0 = blockIdx.x * rows_per_block;
  const int i1 = min(seq, i0 + rows_per_block);
  for (int i = i0 + warp; i < i1; i += kWarps) {
    for (int c = lane; c < d; c += 32) qs[c] = to_f<T>(base[(size_t)i * ld + c]);
    __syncwarp();
    float mx = -INFINITY;
    for (int j = lane; j <= i; j += 32) {
      const float s = dot_row<T>(qs, base + (size_t)j * ld + d, d) * scale;
      sc[j] = s;
      mx = fmaxf(mx, s);
    }
    mx = warp_max(mx);
    float sum = 0.f;
    for (int j = lane; j <= i; j += 32) {
      const float e = expf(sc[j] - mx);
      sc[j] = e;
      sum += e;
    }
    sum = warp_sum(sum);
    if (drop.on) {
      // O = (P * keep / (1 - p)) V; the row sum stays that of the undropped P
      for (int j = lane; j <= i; j += 32)
        sc[j] = drop_keep(drop_index(b, head, heads, seq, i, j), drop) ? sc[j] * drop.scale : 0.f;
    }
    __syncwarp();
    float o[kMaxDPerLane];
#pragma unroll
    for (int k = 0; k < kMaxDPerLane; ++k) o[k] = 0.f;
    for (int j = 0; j <= i; ++j) {
      const float pj = sc[j];
      const T* vr = base + (size_t)j * ld + 2 * d;
#pragma unroll
      for (int k = 0; k < kMaxDPerLane; ++k) {
        const int c = lane + 32 * k;
        if (c < d) o[k] = fmaf(pj, to_f<T>(vr[c]), o[k]);
      }
    }
    const float inv = 1.0f / sum;
    T* orow = ctx + ((size_t)b * seq + i) * h + (size_t)head * d;
#pragma unroll
    for (int k = 0; k < kMaxDPerLane; ++k) {
      const int c = lane + 32 * k;
      if (c < d) orow[c] = from_f<T>(o[k] * inv);
    }
    if (lane == 0) lse[((size_t)b * heads + head) * seq + i] = mx + logf(sum);
    __syncwarp();
  }
}

// dQ and D_i = sum_c dO_ic O_ic, one warp per query row.
template <typename T>
__global__ void attn_bwd_dq_simt_kernel(const T* __restrict__ qkv, const T* __restrict__ ctx,
                                        const float* __restrict__ lse, const T* __restrict__ dctx,
                                        T* __restrict__ dqkv, float* __restrict__ dsum, int seq,
                                        int heads, int d, int rows_per_block, Dropout drop) {
  extern __shared__ float sm[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* sc = sm + warp * seq;
  float* qs = sm + kWarps * seq + warp * 2 * d;
  float* dos = qs + d;
  const int head = blockIdx.y, b = blockIdx.z;
  const int h = heads * d;
  const size_t ld = 3 * (size_t)h;
  const T* base = qkv + (size_t)b * seq * ld + (size_t)head * 3 * d;
  const float scale = 1.0f / sqrtf((float)d);
  const int i0 = blockIdx.x * rows_per_block;
  const int i1 = min(seq, i0 + rows_per_block);
  for (int i = i0 + warp; i < i1; i += kWarps) {
    const size_t orow = ((size_t)b * seq + i) * h + (size_t)head * d;
    float dpart = 0.f;
    for (int c = lane; c < d; c += 32) {
      qs[c] = to_f<T>(base[(size_t)i * ld + c]);
      const float g = to_f<T>(dctx[orow + c]);
      dos[c] = g;
      dpart = fmaf(g, to_f<T>(ctx[orow + c]), dpart);
    }
    const float Di = warp_sum(dpart);
    __syncwarp();
    const float li = lse[((size_t)b * heads + head) * seq + i];
    for (int j = lane; j <= i; j += 32) {
      const float s = dot_row<T>(qs, base + (size_t)j * ld + d, d) * scale;
      const float p = expf(s - li);
      float dp = dot_row<T>(dos, base + (size_t)j * ld + 2 * d, d);
      if (drop.on) dp = drop_keep(drop_index(b, head, heads, seq, i, j), drop) ? dp * drop.scale : 0.f;
      sc[j] = p * (dp - Di);
    }
    __syncwarp();
    float acc[kMaxDPerLane];
#pragma unroll
    for (int k = 0; k < kMaxDPerLane; ++k) acc[k] = 0.f;
    for (int j = 0; j <= i; ++j) {
      const float ds = sc[j];
      const T* kr = base + (size_t)j * ld + d;
#pragma unroll
      for (int k = 0; k < kMaxDPerLane; ++k) {
        const int c = lane + 32 * k;
        if (c < d) acc[k] = fmaf(ds, to_f<T>(kr[c]), acc[k]);
      }
    }
    T* dq = dqkv + ((size_t)b * seq + i) * ld + (size_t)head * 3 * d;
#pragma unroll
    for (int k = 0; k < kMaxDPerLane; ++k) {
      const int c = lane + 32 * k;
      if (c < d) dq[c] = from_f<T>(acc[k] * scale);
    }
    if (lane == 0) dsum[((size_t)b * heads + head) * seq + i] = Di;
    __syncwarp();
  }
}

// dK and dV, one warp per key row j, over queries i >= j.
template <typename T>
__global__ void attn_bwd_dkv_simt_kernel(const T* __restrict__ qkv, const float* __restrict__ lse,
                                         const T* __restrict__ dctx, const float* __restrict__ dsum,
                                         T* __restrict__ dqkv, int seq, int heads, int d,
                                         int rows_per_block, Dropout drop) {
  extern __shared__ float sm[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* sp = sm + warp * 2 * seq;
  float* sds = sp + seq;
  float* ks = sm + kWarps * 2 * seq + warp * 2 * d;
  float* vs = ks + d;
  const int head = blockIdx.y, b = blockIdx.z;
  const int h = heads * d;
  const size_t ld = 3 * (size_t)h;
  const T* base = qkv + (size_t)b * seq * ld + (size_t)head * 3 * d;
  const T* dob = dctx + (size_t)b * seq * h + (size_t)head * d;
  const float* lrow = lse + ((size_t)b * heads + head) * seq;
  const float* drow = dsum + ((size_t)b * heads + head) * seq;
  const float scale = 1.0f / sqrtf((float)d);
  const int j0 = blockIdx.x * rows_per_block;
  const int j1 = min(seq, j0 + rows_per_block);
  for (int j = j0 + warp; j < j1; j += kWarps) {
    for (int c = lane; c < d; c += 32) {
      ks[c] = to_f<T>(base[(size_t)j * ld + d + c]);
      vs[c] = to_f<T>(base[(size_t)j * ld + 2 * d + c]);
    }
    __syncwarp();
    for (int i = j + lane; i < seq; i += 32) {
      const float s = dot_row<T>(ks, base + (size_t)i * ld, d) * scale;
      const float p = expf(s - lrow[i]);
      float dp = dot_row<T>(vs, dob + (size_t)i * h, d);
      float pd = p;
      if (drop.on) {
        const bool kept = drop_keep(drop_index(b, head, heads, seq, i, j), drop);
        pd = kept ? p * drop.scale : 0.f;
        dp = kept ? dp * drop.scale : 0.f;
      }
      sp[i] = pd;
      sds[i] = p * (dp - drow[i]);
    }
    __syncwarp();
    float dk[kMaxDPerLane], dv[kMaxDPerLane];
#pragma unroll
    for (int k = 0; k < kMaxDPerLane; ++k) dk[k] = dv[k] = 0.f;
    for (int i = j; i < seq; ++i) {
      const float p = sp[i], ds = sds[i];
      const T* qr = base + (size_t)i * ld;
      const T* dor = dob + (size_t)i * h;
#pragma unroll
      for (int k = 0; k < kMaxDPerLane; ++k) {
        const int c = lane + 32 * k;
        if (c < d) {
          dv[k] = fmaf(p, to_f<T>(dor[c]), dv[k]);
          dk[k] = fmaf(ds, to_f<T>(qr[c]), dk[k]);
        }
      }
    }
    T* out = dqkv + ((size_t)b * seq + j) * ld + (size_t)head * 3 * d;
#pragma unroll
    for (int k = 0; k < kMaxDPerLane; ++k) {
      const int c = lane + 32 * k;
      if (c < d) {
        out[d + c] = from_f<T>(dk[k] * scale);
        out[2 * d + c] = from_f<T>(dv[k]);
      }
    }
    __syncwarp();
  }
}

constexpr int kRowsPerBlock = 16;

template <typename T>
cudaError_t fwd_t(const void* qkv, void* ctx, float* lse, int batch, int seq, int heads, int d,
                  const Dropout& drop, const LaunchCtx& c) {
  dim3 grid((seq + kRowsPerBlock - 1) / kRowsPerBlock, heads, batch);
  const size_t smem = (size_t)kWarps * (seq + d) * sizeof(float);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(attn_fwd_simt_kernel<T>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  c.before(KK_ATTN_FWD, 2.0 * batch * (double)seq * (seq + 1) * heads * d);
  attn_fwd_simt_kernel<T><<<grid, kWarps * 32, smem, c.stream>>>((const T*)qkv, (T*)ctx, lse, seq,
                                                                 heads, d, kRowsPerBlock, drop);
  c.after();
  return cudaGetLastError();
}

template <typename T>
cudaError_t bwd_t(const void* qkv, const void* ctx, const float* lse, const void* dctx,
                  void* dqkv, float* dsum, int batch, int seq, int heads, int d,
                  const Dropout& drop, const LaunchCtx& c) {
  dim3 grid((seq + kRowsPerBlock - 1) / kRowsPerBlock, heads, batch);
  const size_t smem1 = (size_t)kWarps * (seq + 2 * d) * sizeof(float);
  const size_t smem2 = (size_t)kWarps * (2 * seq + 2 * d) * sizeof(float);
  cudaError_t e;
  if (smem1 > 48 * 1024) {
    e = cudaFuncSetAttribute(attn_bwd_dq_simt_kernel<T>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem1);
    if (e != cudaSuccess) return e;
  }
  if (smem2 > 48 * 1024) {
    e = cudaFuncSetAttribute(attn_bwd_dkv_simt_kernel<T>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem2);
    if (e != cudaSuccess) return e;
  }
  const double tri = (double)batch * seq * (seq + 1) / 2.0 * heads * d;
  c.before(KK_ATTN_BWD, 2.0 * 2.0 * tri);
  attn_bwd_dq_simt_kernel<T><<<grid, kWarps * 32, smem1, c.stream>>>(
      (const T*)qkv, (const T*)ctx, lse, (const T*)dctx, (T*)dqkv, dsum, seq, heads, d,
      kRowsPerBlock, drop);
  c.after();
  c.before(KK_ATTN_BWD, 2.0 * 4.0 * tri);
  attn_bwd_dkv_simt_kernel<T><<<grid, kWarps * 32, smem2, c.stream>>>(
      (const T*)qkv, lse, (const T*)dctx, dsum, (T*)dqkv, seq, heads, d, kRowsPerBlock,
      drop);
  c.after();
  return cudaGetLastError();
}

}  // namespace

cudaError_t attn_fwd_simt(int dtype, const void* qkv, void* ctx, float* lse, int batch, int seq,
                          int heads, int d, const Dropout& drop, const LaunchCtx& c) {
  if (batch == 0 || seq == 0) return cudaSuccess;
  return dtype == kBF16 ? fwd_t<bf16>(qkv, ctx, lse, batch, seq, heads, d, drop, c)
                        : fwd_t<float>(qkv, ctx, lse, batch, seq, heads, d, drop, c);
}

cudaError_t attn_bwd_simt(int dtype, const void* qkv, const void* ctx, const float* lse,
                          const void* dctx, void* dqkv, float* dsum, int batch, int seq,
                          int heads, int d, const Dropout& drop, const LaunchCtx& c) {
  if (batch == 0 || seq == 0) return cudaSuccess;
  return dtype == kBF16
             ? bwd_t<bf16>(qkv, ctx, lse, dctx, dqkv, dsum, batch, seq, heads, d, drop, c)
             : bwd_t<float>(qkv, ctx, lse, dctx, dqkv, dsum, batch, seq, heads, d, drop, c);
}

}  // namespace mtl
