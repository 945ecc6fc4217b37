// LayerNorm forward / backward (+ residual gradient) and fixed-order column sums.
//
// Pre-LN ("Megatron-LM: GPU-Cluster Training Parallelism", section "Paper 1: BERT
// LayerNorm Rearrangement"): every sublayer reads LayerNorm(x).  These kernels are
// HBM-bound: each row is read once into registers as 16-byte vectors, reduced
// with warp shuffles, and written once.  Parameter gradients (dgamma, dbeta) and
// bias gradients are reduced deterministically: fixed row blocks write partial
// column sums, then one pass adds the partials in block order.
#include <cstring>

#include "common.cuh"
#include "kernels.h"

namespace mtl {
namespace {

constexpr int kLnThreadsMax = 512;
constexpr int kLnBwdBlocks = 512;     // most row blocks of the dgamma/dbeta reduction
constexpr int kLnBwdPerSM = 2;        // LN backward blocks per SM (one wave)
constexpr int kLnBwdThreadsMax = 512; // threads per row of the LN backward
// With the folded column sums, rows of one vector a thread and at most this
// many threads, so that two blocks of it fit an SM's registers.
constexpr int kLnSumsThreadsMax = 384;
constexpr int kColsumThreads = 256;   // threads per block of the bias-gradient column sums
constexpr int kColsumDropBlocks = 512;  // the same with dropout (Philox work per element)

// Sums NV values over the block in place; `red` holds NV*32 floats.  Every
// thread adds the per-warp sums in the same order.
template <int NV>
__device__ __forceinline__ void block_sum_n(float (&v)[NV], float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nw = (blockDim.x + 31) >> 5;
#pragma unroll
  for (int i = 0; i < NV; ++i) v[i] = warp_sum(v[i]);
  __syncthreads();  // earlier readers of `red` are done
  if (lane == 0) {
#pragma unroll
    for (int i = 0; i < NV; ++i) red[i * 32 + warp] = v[i];
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    float s = 0.f;
    for (int w = 0; w < nw; ++w) s += red[i * 32 + w];
    v[i] = s;
  }
}

// R rows per iteration: the loads of all R rows are issued before the block
// reductions, so each thread keeps R*V 16-byte loads in flight.  Each element
// is converted to fp32 once; gamma and beta are held as fp32 for all rows.
// AMAX: also fold max |u| into *amax_bits.
template <typename T, int V, int R, bool AMAX>
__global__ void __launch_bounds__(kLnThreadsMax, V == 1 ? 4 : 1)   // short rows: 32 registers
    ln_fwd_kernel(const T* __restrict__ x, const T* __restrict__ gamma, const T* __restrict__ beta,
                  T* __restrict__ u, float* __restrict__ mean_out, float* __restrict__ rstd_out,
                  int n, int h, float eps, int rows_per_block, unsigned* __restrict__ amax_bits) {
  constexpr int E = Vec<T>::N;
  __shared__ float red[R * 32];
  float umax = 0.f;   // max |u| of this thread's outputs before rounding (AMAX)
  griddep_wait();   // no-op unless launched as a programmatic dependent
  if (threadIdx.x == 0) griddep_launch_dependents();
  const int nvec = h / E;
  const int r_begin = blockIdx.x * rows_per_block;
  const int r_end = min(n, r_begin + rows_per_block);
  const float inv_h = 1.0f / (float)h;
  // gamma and beta are reloaded (from L1) for every row: holding them in
  // registers would cost occupancy, which this latency-bound kernel needs more
  constexpr bool GB_REG = false;
  constexpr int VG = GB_REG ? V : 1;
  float gf[VG][E], bf[VG][E];
  if (GB_REG) {
#pragma unroll
    for (int i = 0; i < VG; ++i) {
      const int vi = threadIdx.x + i * blockDim.x;
      if (vi < nvec) {
        Vec<T> tg, tb;
        tg.load(gamma + vi * E);
        tb.load(beta + vi * E);
        tg.unpack(gf[i]);
        tb.unpack(bf[i]);
      }
    }
  }
  for (int r0 = r_begin; r0 < r_end; r0 += R) {
    float xf[R][V][E];
    float s[R];
#pragma unroll
    for (int rr = 0; rr < R; ++rr) {
      s[rr] = 0.f;
#pragma unroll
      for (int i = 0; i < V; ++i) {
        const int vi = threadIdx.x + i * blockDim.x;
        if (r0 + rr < r_end && vi < nvec) {
          Vec<T> xv;
          xv.load(x + (size_t)(r0 + rr) * h + vi * E);
          xv.unpack(xf[rr][i]);
#pragma unroll
          for (int e = 0; e < E; ++e) s[rr] += xf[rr][i][e];
        }
      }
    }
    block_sum_n<R>(s, red);
    float mean[R], ss[R];
#pragma unroll
    for (int rr = 0; rr < R; ++rr) {
      mean[rr] = s[rr] * inv_h;
      ss[rr] = 0.f;
#pragma unroll
      for (int i = 0; i < V; ++i) {
        const int vi = threadIdx.x + i * blockDim.x;
        if (r0 + rr < r_end && vi < nvec) {
#pragma unroll
          for (int e = 0; e < E; ++e) {
            const float dlt = xf[rr][i][e] - mean[rr];
            ss[rr] += dlt * dlt;
          }
        }
      }
    }
    block_sum_n<R>(ss, red);
#pragma unroll
    for (int rr = 0; rr < R; ++rr) {
      if (r0 + rr >= r_end) continue;
      const float rs = 1.0f / sqrtf(ss[rr] * inv_h + eps);
#pragma unroll
      for (int i = 0; i < V; ++i) {
        const int vi = threadIdx.x + i * blockDim.x;
        if (vi >= nvec) continue;
        float gv[E], bv[E];
        if (GB_REG) {
#pragma unroll
          for (int e = 0; e < E; ++e) {
            gv[e] = gf[GB_REG ? i : 0][e];
            bv[e] = bf[GB_REG ? i : 0][e];
          }
        } else {
          Vec<T> tg, tb;
          tg.load(gamma + vi * E);
          tb.load(beta + vi * E);
          tg.unpack(gv);
          tb.unpack(bv);
        }
        float of[E];
#pragma unroll
        for (int e = 0; e < E; ++e) {
          of[e] = (xf[rr][i][e] - mean[rr]) * rs * gv[e] + bv[e];
          if (AMAX) umax = fmaxf(umax, fabsf(of[e]));
        }
        Vec<T> o;
        o.pack(of);
        o.store(u + (size_t)(r0 + rr) * h + vi * E);
      }
    }
    if (threadIdx.x == 0) {
#pragma unroll
      for (int rr = 0; rr < R; ++rr) {
        if (r0 + rr < r_end) {
          mean_out[r0 + rr] = mean[rr];
          rstd_out[r0 + rr] = 1.0f / sqrtf(ss[rr] * inv_h + eps);
        }
      }
    }
  }
  if (AMAX) {
    // max |u| of the stored values: rounding to T is monotone and symmetric, so
    // the rounded maximum is the maximum of the rounded values
    umax = warp_max(umax);
    __syncthreads();   // the last block_sum_n's readers of `red` are done
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = umax;
    __syncthreads();
    if (threadIdx.x == 0) {
      for (int w = 1; w < (int)(blockDim.x + 31) / 32; ++w) umax = fmaxf(umax, red[w]);
      atomicMax(amax_bits, __float_as_uint(Vec<T>::round(umax)));
    }
  }
}

// One warp per row, for rows of at most kLnWarpMaxVec 16-byte vectors a lane:
// lane l holds vectors l, l + 32, ... of the row (each load instruction of the
// warp covers 512 contiguous bytes), so a whole row's loads are in flight at
// once and both reductions are warp shuffles, with no block barrier.  The
// arithmetic per element is ln_fwd_kernel's: the mean, then the centred second
// moment, and the output expression ln_apply_kernel uses to rebuild u bit for
// bit from the saved statistics.
constexpr int kLnWarpMaxVec = 16;
constexpr int kLnWarpThreads = 256;
template <typename T, int VL, bool AMAX>
__global__ void __launch_bounds__(kLnWarpThreads)
    ln_fwd_warp_kernel(const T* __restrict__ x, const T* __restrict__ gamma,
                       const T* __restrict__ beta, T* __restrict__ u, float* __restrict__ mean_out,
                       float* __restrict__ rstd_out, int n, int h, float eps,
                       unsigned* __restrict__ amax_bits) {
  constexpr int E = Vec<T>::N;
  griddep_wait();   // no-op unless launched as a programmatic dependent
  if (threadIdx.x == 0) griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int wpb = blockDim.x >> 5;
  const int nvec = h / E;
  const float inv_h = 1.0f / (float)h;
  float umax = 0.f;
  for (int r = blockIdx.x * wpb + (threadIdx.x >> 5); r < n; r += gridDim.x * wpb) {
    Vec<T> xv[VL];
#pragma unroll
    for (int i = 0; i < VL; ++i)
      if (lane + 32 * i < nvec) xv[i].load(x + (size_t)r * h + (lane + 32 * i) * E);
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < VL; ++i) {
      if (lane + 32 * i < nvec) {
        float f[E];
        xv[i].unpack(f);
#pragma unroll
        for (int e = 0; e < E; ++e) s += f[e];
      }
    }
    const float mean = warp_sum(s) * inv_h;
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < VL; ++i) {
      if (lane + 32 * i < nvec) {
        float f[E];
        xv[i].unpack(f);
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const float dlt = f[e] - mean;
          ss += dlt * dlt;
        }
      }
    }
    ss = warp_sum(ss);
    const float rs = 1.0f / sqrtf(ss * inv_h + eps);
#pragma unroll
    for (int i = 0; i < VL; ++i) {
      const int vi = lane + 32 * i;
      if (vi >= nvec) continue;
      float f[E], gv[E], bv[E], of[E];
      xv[i].unpack(f);
      Vec<T> tg, tb;
      tg.load(gamma + vi * E);
      tb.load(beta + vi * E);
      tg.unpack(gv);
      tb.unpack(bv);
#pragma unroll
      for (int e = 0; e < E; ++e) {
        of[e] = (f[e] - mean) * rs * gv[e] + bv[e];
        if (AMAX) umax = fmaxf(umax, fabsf(of[e]));
      }
      Vec<T> o;
      o.pack(of);
      o.store(u + (size_t)r * h + vi * E);
    }
    if (lane == 0) {
      mean_out[r] = mean;
      rstd_out[r] = rs;
    }
  }
  if (AMAX) {
    // max |u| of the stored values: rounding to T is monotone and symmetric,
    // so the rounded maximum is the maximum of the rounded values
    umax = warp_max(umax);
    if (lane == 0) atomicMax(amax_bits, __float_as_uint(Vec<T>::round(umax)));
  }
}

// Each block sums du * xhat and du over its rows for the dgamma / dbeta
// partials; a thread owns the same columns in every row, so the sums need no
// atomics and keep row order.  Short rows (V <= 2) keep those sums and gamma in
// registers; longer rows keep the sums in dynamic shared memory (2 * h floats).
// R rows per iteration, their loads issued before the reduction.
// MODE 0: du fp32, dx = resid + LN_bwd(du) (Pre-LN);  MODE 1: du = du2 (of type
// T), dx = LN_bwd(du);  MODE 2: du = du (fp32) + du2 (T), dx = LN_bwd(du) (the
// Post-LN layer's two LayerNorms).
// SUMS (MODE 0, rows of at most two vectors a thread): the block also sums the
// residual input and the stored output dx column by column into part_r and
// part_o (the Pre-LN layer's db_fc2 = sum dy and db_o = sum dx1, read here
// anyway).
template <typename T, int V, int R, int MODE, bool SUMS>
__device__ __forceinline__ void ln_bwd_body(
    const float* __restrict__ du, const T* __restrict__ du2, const T* __restrict__ x,
    const float* __restrict__ mean_in, const float* __restrict__ rstd_in,
    const T* __restrict__ gamma, const T* __restrict__ resid, T* __restrict__ dx,
    float* __restrict__ part_g, float* __restrict__ part_b, int n, int h, int rows_per_block,
    float* __restrict__ part_r, float* __restrict__ part_o) {
  constexpr int E = Vec<T>::N;
  constexpr bool ACC_REG = V <= 2;
  constexpr int VA = ACC_REG ? V : 1;
  static_assert(!SUMS || (MODE == 0 && V == 1), "column sums need MODE 0 and one vector a thread");
  constexpr int VS = SUMS ? VA : 1;
  float ar[VS][E], ao[VS][E];
  if (SUMS) {
#pragma unroll
    for (int i = 0; i < VS; ++i)
#pragma unroll
      for (int e = 0; e < E; ++e) ar[i][e] = ao[i][e] = 0.f;
  }
  extern __shared__ float lsm[];
  float* acc_g = lsm;
  float* acc_b = lsm + h;
  __shared__ float red[2 * R * 32];
  const int nvec = h / E;
  float ag[VA][E], ab[VA][E], gf[VA][E];
  if (ACC_REG) {
#pragma unroll
    for (int i = 0; i < VA; ++i) {
      const int vi = threadIdx.x + i * blockDim.x;
#pragma unroll
      for (int e = 0; e < E; ++e) ag[i][e] = ab[i][e] = gf[i][e] = 0.f;
      if (vi < nvec) {
        Vec<T> tg;
        tg.load(gamma + vi * E);
        tg.unpack(gf[i]);
      }
    }
  } else {
    // accumulator layout [e][vi]: consecutive threads touch consecutive words;
    // each thread reads back only the columns it wrote: no barrier needed
    for (int vi = threadIdx.x; vi < nvec; vi += blockDim.x) {
#pragma unroll
      for (int e = 0; e < E; ++e) {
        acc_g[e * nvec + vi] = 0.f;
        acc_b[e * nvec + vi] = 0.f;
      }
    }
  }
  const int r_begin = blockIdx.x * rows_per_block;
  const int r_end = min(n, r_begin + rows_per_block);
  const float inv_h = 1.0f / (float)h;
  for (int r0 = r_begin; r0 < r_end; r0 += R) {
    Vec<T> rv[R][V];
    float xh[R][V][E], dd[R][V][E];
    float mu[R], rs[R], s[2 * R];
#pragma unroll
    for (int rr = 0; rr < R; ++rr) {
      const bool live = r0 + rr < r_end;
      mu[rr] = live ? mean_in[r0 + rr] : 0.f;
      rs[rr] = live ? rstd_in[r0 + rr] : 0.f;
      s[2 * rr] = 0.f;
      s[2 * rr + 1] = 0.f;
#pragma unroll
      for (int i = 0; i < V; ++i) {
        const int vi = threadIdx.x + i * blockDim.x;
        if (live && vi < nvec) {
          const size_t off = (size_t)(r0 + rr) * h + vi * E;
          Vec<T> xv;
          xv.load(x + off);
          xv.unpack(xh[rr][i]);
          if (MODE == 0) rv[rr][i].load(resid + off);
          if (MODE != 1) {
#pragma unroll
            for (int e = 0; e < E; e += 4) {
              const float4 q = *reinterpret_cast<const float4*>(du + off + e);
              dd[rr][i][e] = q.x;
              dd[rr][i][e + 1] = q.y;
              dd[rr][i][e + 2] = q.z;
              dd[rr][i][e + 3] = q.w;
            }
          }
          if (MODE != 0) {
            Vec<T> d2;
            d2.load(du2 + off);
            float f2[E];
            d2.unpack(f2);
#pragma unroll
            for (int e = 0; e < E; ++e) dd[rr][i][e] = (MODE == 2 ? dd[rr][i][e] : 0.f) + f2[e];
          }
        }
      }
    }
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const int vi = threadIdx.x + i * blockDim.x;
      if (vi >= nvec) continue;
      float gv[E];
      if (ACC_REG) {
#pragma unroll
        for (int e = 0; e < E; ++e) gv[e] = gf[ACC_REG ? i : 0][e];
      } else {
        Vec<T> tg;
        tg.load(gamma + vi * E);
        tg.unpack(gv);
      }
#pragma unroll
      for (int rr = 0; rr < R; ++rr) {
        if (r0 + rr >= r_end) continue;
#pragma unroll
        for (int e = 0; e < E; ++e) {
          xh[rr][i][e] = (xh[rr][i][e] - mu[rr]) * rs[rr];
          const float gd = dd[rr][i][e] * gv[e];
          s[2 * rr] += gd;
          s[2 * rr + 1] += gd * xh[rr][i][e];
        }
      }
    }
    block_sum_n<2 * R>(s, red);
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const int vi = threadIdx.x + i * blockDim.x;
      if (vi >= nvec) continue;
      float gv[E];
      if (ACC_REG) {
#pragma unroll
        for (int e = 0; e < E; ++e) gv[e] = gf[ACC_REG ? i : 0][e];
      } else {
        Vec<T> tg;
        tg.load(gamma + vi * E);
        tg.unpack(gv);
      }
      float sg[E], sb[E];
#pragma unroll
      for (int e = 0; e < E; ++e) sg[e] = sb[e] = 0.f;
#pragma unroll
      for (int rr = 0; rr < R; ++rr) {
        if (r0 + rr >= r_end) continue;
        const float m1 = s[2 * rr] * inv_h, m2 = s[2 * rr + 1] * inv_h;
        float rf[E], of[E];
        if (MODE == 0) rv[rr][i].unpack(rf);
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const float gd = dd[rr][i][e] * gv[e];
          of[e] = (MODE == 0 ? rf[e] : 0.f) + rs[rr] * (gd - m1 - xh[rr][i][e] * m2);
          sg[e] += dd[rr][i][e] * xh[rr][i][e];
          sb[e] += dd[rr][i][e];
        }
        Vec<T> o;
        o.pack(of);
        o.store(dx + (size_t)(r0 + rr) * h + vi * E);
        if (SUMS) {
          // the residual as read and the output as stored, row by row
          float ofr[E];
          o.unpack(ofr);
#pragma unroll
          for (int e = 0; e < E; ++e) {
            ar[SUMS ? i : 0][e] += rf[e];
            ao[SUMS ? i : 0][e] += ofr[e];
          }
        }
      }
      if (ACC_REG) {
#pragma unroll
        for (int e = 0; e < E; ++e) {
          ag[ACC_REG ? i : 0][e] += sg[e];
          ab[ACC_REG ? i : 0][e] += sb[e];
        }
      } else {
#pragma unroll
        for (int e = 0; e < E; ++e) {
          acc_g[e * nvec + vi] += sg[e];
          acc_b[e * nvec + vi] += sb[e];
        }
      }
    }
  }
  if (ACC_REG) {
#pragma unroll
    for (int i = 0; i < VA; ++i) {
      const int vi = threadIdx.x + i * blockDim.x;
      if (vi >= nvec) continue;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        part_g[(size_t)blockIdx.x * h + vi * E + e] = ag[i][e];
        part_b[(size_t)blockIdx.x * h + vi * E + e] = ab[i][e];
        if (SUMS) {
          part_r[(size_t)blockIdx.x * h + vi * E + e] = ar[SUMS ? i : 0][e];
          part_o[(size_t)blockIdx.x * h + vi * E + e] = ao[SUMS ? i : 0][e];
        }
      }
    }
  } else {
    for (int vi = threadIdx.x; vi < nvec; vi += blockDim.x) {
#pragma unroll
      for (int e = 0; e < E; ++e) {
        part_g[(size_t)blockIdx.x * h + vi * E + e] = acc_g[e * nvec + vi];
        part_b[(size_t)blockIdx.x * h + vi * E + e] = acc_b[e * nvec + vi];
      }
    }
  }
}

template <typename T, int V, int R, int MODE>
__global__ void __launch_bounds__(kLnThreadsMax)
    ln_bwd_kernel(const float* __restrict__ du, const T* __restrict__ du2, const T* __restrict__ x,
                  const float* __restrict__ mean_in, const float* __restrict__ rstd_in,
                  const T* __restrict__ gamma, const T* __restrict__ resid, T* __restrict__ dx,
                  float* __restrict__ part_g, float* __restrict__ part_b, int n, int h,
                  int rows_per_block) {
  ln_bwd_body<T, V, R, MODE, false>(du, du2, x, mean_in, rstd_in, gamma, resid, dx, part_g,
                                    part_b, n, h, rows_per_block, nullptr, nullptr);
}

// The Pre-LN form (MODE 0, one vector a thread) with the column sums of the
// residual and of the output; bounded to two blocks an SM.
template <typename T>
__global__ void __launch_bounds__(kLnSumsThreadsMax, kLnBwdPerSM)
    ln_bwd_sums_kernel(const float* __restrict__ du, const T* __restrict__ x,
                       const float* __restrict__ mean_in, const float* __restrict__ rstd_in,
                       const T* __restrict__ gamma, const T* __restrict__ resid,
                       T* __restrict__ dx, float* __restrict__ part_g, float* __restrict__ part_b,
                       int n, int h, int rows_per_block, float* __restrict__ part_r,
                       float* __restrict__ part_o) {
  ln_bwd_body<T, 1, 1, 0, true>(du, nullptr, x, mean_in, rstd_in, gamma, resid, dx, part_g,
                                part_b, n, h, rows_per_block, part_r, part_o);
}

// Row blocks of a column sum over n rows of N columns with E elements a
// thread: about 1024 blocks in all (several waves on any SM count), between
// 128 and 512 row blocks; rows_blocks * N stays within 1024 * 2048 floats for
// N up to 16384.
int colsum_row_blocks(int n, int N, int E) {
  const int cb = (N / E + kColsumThreads - 1) / kColsumThreads;
  int b = 1024 / (cb > 0 ? cb : 1);
  b = b < 128 ? 128 : (b > 512 ? 512 : b);
  return n < b ? (n > 0 ? n : 1) : b;
}

// out[c] = sum over row blocks b = 0..nblk-1 of part[b*N + c].  One CTA per
// 32 columns: warp w sums the row blocks w, w+32, w+64, ... (coalesced 128-byte
// rows, several loads in flight), then the 32 warp sums are added in warp
// order: a fixed order for any launch.
constexpr int kFinWarps = 32;
__device__ __forceinline__ void finalize_cols(const float* __restrict__ part, int nblk, int N,
                                              float* __restrict__ out, int cblock) {
  __shared__ float red[kFinWarps][33];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c = cblock * 32 + lane;
  float s = 0.f;
  if (c < N) {
#pragma unroll 4
    for (int b = warp; b < nblk; b += kFinWarps) s += part[(size_t)b * N + c];
  }
  red[warp][lane] = s;
  __syncthreads();
  if (warp == 0 && c < N) {
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < kFinWarps; ++w) t += red[w][lane];
    out[c] = t;
  }
}

__global__ void __launch_bounds__(kFinWarps * 32)
    finalize_cols_kernel(const float* __restrict__ part, int nblk, int N,
                         float* __restrict__ out) {
  finalize_cols(part, nblk, N, out, blockIdx.x);
}

// Several finalizes in one launch: job k owns the column blocks
// [first[k], first[k + 1]) of the grid.  Each column is summed exactly as
// finalize_cols_kernel sums it.
struct FinalizeArgs {
  const float* part[FinalizeJobs::kMax];
  float* out[FinalizeJobs::kMax];
  int nblk[FinalizeJobs::kMax], N[FinalizeJobs::kMax], first[FinalizeJobs::kMax + 1];
  int n;
};

__global__ void __launch_bounds__(kFinWarps * 32) finalize_multi_kernel(const FinalizeArgs a) {
  int k = 0;
  while (k + 1 < a.n && (int)blockIdx.x >= a.first[k + 1]) ++k;
  finalize_cols(a.part[k], a.nblk[k], a.N[k], a.out[k], blockIdx.x - a.first[k]);
}

// With AMAX, max |Y| of the block's elements also goes to *amax_bits (one
// atomicMax a block).
template <typename T, bool AMAX>
__global__ void __launch_bounds__(kColsumThreads)
    colsum_partial_kernel(const T* __restrict__ Y, int64_t ld, int n, int N, int rows_per_block,
                          float* __restrict__ part, unsigned* __restrict__ amax_bits) {
  constexpr int E = Vec<T>::N;
  const int c0 = (blockIdx.x * blockDim.x + threadIdx.x) * E;
  float m = 0.f;
  if (c0 < N) {
    float acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
    const int r0 = blockIdx.y * rows_per_block;
    const int r1 = min(n, r0 + rows_per_block);
    // unrolled so that 8 row loads are in flight; the adds keep row order
#pragma unroll 8
    for (int r = r0; r < r1; ++r) {
      Vec<T> v;
      v.load(Y + (size_t)r * ld + c0);
      float f[E];
      v.unpack(f);
#pragma unroll
      for (int e = 0; e < E; ++e) {
        acc[e] += f[e];
        if (AMAX) m = fmaxf(m, fabsf(f[e]));
      }
    }
#pragma unroll
    for (int e = 0; e < E; ++e) part[(size_t)blockIdx.y * N + c0 + e] = acc[e];
  }
  if (AMAX) {
    __shared__ float red[kColsumThreads / 32];
    m = warp_max(m);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
      for (int w = 1; w < kColsumThreads / 32; ++w) m = fmaxf(m, red[w]);
      atomicMax(amax_bits, __float_as_uint(m));
    }
  }
}

// colsum_partial_kernel on Y * keep / (1 - p), also writing that product to Ym.
template <typename T>
__global__ void colsum_dropout_partial_kernel(const T* __restrict__ Y, T* __restrict__ Ym,
                                              int64_t ld, int n, int N, int rows_per_block,
                                              Dropout drop, float* __restrict__ part) {
  constexpr int E = Vec<T>::N;   // 8 or 4: whole Philox blocks, N % 4 == 0
  const int c0 = (blockIdx.x * blockDim.x + threadIdx.x) * E;
  if (c0 >= N) return;
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  const int r0 = blockIdx.y * rows_per_block;
  const int r1 = min(n, r0 + rows_per_block);
  for (int r = r0; r < r1; ++r) {
    Vec<T> v;
    v.load(Y + (size_t)r * ld + c0);
    const unsigned long long blk = ((unsigned long long)r * N + c0) >> 2;
    uint32_t bits = drop_bits4(blk, drop);
    if (E == 8) bits |= drop_bits4(blk + 1, drop) << 4;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const float x = ((bits >> e) & 1u) ? v.get(e) * drop.scale : 0.f;
      acc[e] += x;
      v.set(e, x);
    }
    v.store(Ym + (size_t)r * ld + c0);
  }
#pragma unroll
  for (int e = 0; e < E; ++e) part[(size_t)blockIdx.y * N + c0 + e] = acc[e];
}

// Vectors per thread and threads per block for a row of h elements.
template <typename T>
void row_plan(int h, int* vpt, int* threads, int max_threads = kLnThreadsMax) {
  const int nvec = h / Vec<T>::N;
  int v = 1;
  while ((nvec + v - 1) / v > max_threads) v *= 2;
  *vpt = v;
  *threads = (((nvec + v - 1) / v) + 31) / 32 * 32;
}

template <typename T>
cudaError_t ln_fwd_t(const void* x, const void* g, const void* b, void* u, float* mean,
                     float* rstd, int n, int h, float eps, const LaunchCtx& c,
                     unsigned* amax_bits) {
  if (n == 0) return cudaSuccess;
  const int vl = (h / Vec<T>::N + 31) / 32;   // vectors a lane with one warp a row
  if (vl <= kLnWarpMaxVec) {
    const int wpb = kLnWarpThreads / 32;
    const int wgrid = (n + wpb - 1) / wpb;
    c.before(KK_LN_FWD, (double)n * h * (2.0 * sizeof(T)) + 8.0 * n);
    cudaError_t we = cudaSuccess;
#define LN_FWD_WARP(VV)                                                                       \
  if (vl <= VV) {                                                                           \
    we = amax_bits ? launch_ex(c, ln_fwd_warp_kernel<T, VV, true>, dim3(wgrid),               \
                               dim3(kLnWarpThreads), 0, 1, (const T*)x, (const T*)g,          \
                               (const T*)b, (T*)u, mean, rstd, n, h, eps, amax_bits)          \
                   : launch_ex(c, ln_fwd_warp_kernel<T, VV, false>, dim3(wgrid),              \
                               dim3(kLnWarpThreads), 0, 1, (const T*)x, (const T*)g,          \
                               (const T*)b, (T*)u, mean, rstd, n, h, eps, amax_bits);         \
  } else
    LN_FWD_WARP(1)
    LN_FWD_WARP(2)
    LN_FWD_WARP(4)
    LN_FWD_WARP(8)
    LN_FWD_WARP(12)
    LN_FWD_WARP(16)
    {}
#undef LN_FWD_WARP
    c.after();
    if (we != cudaSuccess) return we;
    return cudaGetLastError();
  }
  int vpt, threads;
  row_plan<T>(h, &vpt, &threads);
  const int rows = n >= 4 * c.num_sms * 4 ? 4 : 1;
  const int grid = (n + rows - 1) / rows;
  c.before(KK_LN_FWD, (double)n * h * (2.0 * sizeof(T)) + 8.0 * n);
#define LN_FWD_CASE(VV, RR)                                                                  \
  case VV:                                                                                   \
    e = amax_bits                                                                            \
            ? launch_ex(c, ln_fwd_kernel<T, VV, RR, true>, dim3(grid), dim3(threads), 0, 1,  \
                        (const T*)x, (const T*)g, (const T*)b, (T*)u, mean, rstd, n, h, eps, \
                        rows, amax_bits)                                                     \
            : launch_ex(c, ln_fwd_kernel<T, VV, RR, false>, dim3(grid), dim3(threads), 0, 1, \
                        (const T*)x, (const T*)g, (const T*)b, (T*)u, mean, rstd, n, h, eps, \
                        rows, amax_bits);                                                    \
    break;
  cudaError_t e = cudaSuccess;
  switch (vpt) {
    LN_FWD_CASE(1, 1)
    LN_FWD_CASE(2, 1)
    LN_FWD_CASE(4, 1)
    LN_FWD_CASE(8, 1)
    default:
      return cudaErrorInvalidValue;
  }
#undef LN_FWD_CASE
  c.after();
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// One finalize of nblk rows of partial column sums: deferred into *defer when
// given, else launched now.
cudaError_t finalize_or_defer(const float* part, int nblk, int N, float* out, const LaunchCtx& c,
                              FinalizeJobs* defer) {
  if (defer) return defer->add(part, nblk, N, out) ? cudaSuccess : cudaErrorInvalidValue;
  c.before(KK_FINALIZE, 4.0 * nblk * N);
  finalize_cols_kernel<<<(N + 31) / 32, kFinWarps * 32, 0, c.stream>>>(part, nblk, N, out);
  c.after();
  return cudaGetLastError();
}

template <typename T, int MODE>
cudaError_t ln_bwd_t(const float* du, const void* du2, const void* x, const float* mean,
                     const float* rstd, const void* g, const void* resid, void* dx, float* dgamma,
                     float* dbeta, float* partial, int n, int h, const LaunchCtx& c,
                     FinalizeJobs* defer = nullptr, float* dresid = nullptr,
                     float* ddx = nullptr) {
  int vpt, threads;
  row_plan<T>(h, &vpt, &threads, kLnBwdThreadsMax);
  // one wave of kLnBwdPerSM blocks per SM, at most kLnBwdBlocks (the partial
  // buffer's rows)
  const int want = kLnBwdPerSM * c.num_sms < kLnBwdBlocks ? kLnBwdPerSM * c.num_sms : kLnBwdBlocks;
  const int nblk = n < want ? (n > 0 ? n : 1) : want;
  const int rows = (n + nblk - 1) / nblk;
  float* pg = partial;
  float* pb = partial + (size_t)nblk * h;
  float* pr = partial + 2 * (size_t)nblk * h;
  float* po = partial + 3 * (size_t)nblk * h;
  const bool sums = dresid && ddx;
  if (sums && MODE != 0) return cudaErrorInvalidValue;
  const size_t smem = vpt <= 2 ? 0 : 2 * (size_t)h * sizeof(float);
  c.before(KK_LN_BWD, (double)n * h * (3.0 * sizeof(T) + 4.0) + 8.0 * n);
#define LN_BWD_CASE(VV, RR)                                                                 \
  case VV:                                                                                  \
    if (smem > 48 * 1024) {                                                                 \
      cudaError_t fe = cudaFuncSetAttribute(ln_bwd_kernel<T, VV, RR, MODE>,                 \
                                            cudaFuncAttributeMaxDynamicSharedMemorySize,    \
                                            (int)smem);                                     \
      if (fe != cudaSuccess) return fe;                                                     \
    }                                                                                       \
    ln_bwd_kernel<T, VV, RR, MODE><<<nblk, threads, smem, c.stream>>>(                      \
        du, (const T*)du2, (const T*)x, mean, rstd, (const T*)g, (const T*)resid, (T*)dx,   \
        pg, pb, n, h, rows);                                                                \
    break;
  if (sums) {
    if constexpr (MODE == 0) {
      if (vpt != 1 || threads > kLnSumsThreadsMax) return cudaErrorInvalidValue;
      ln_bwd_sums_kernel<T><<<nblk, threads, 0, c.stream>>>(
          du, (const T*)x, mean, rstd, (const T*)g, (const T*)resid, (T*)dx, pg, pb, n, h, rows,
          pr, po);
    }
  } else {
    switch (vpt) {
      LN_BWD_CASE(1, 1)
      LN_BWD_CASE(2, 1)
      LN_BWD_CASE(4, 1)
      LN_BWD_CASE(8, 1)
      default:
        return cudaErrorInvalidValue;
    }
  }
#undef LN_BWD_CASE
  c.after();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if ((e = finalize_or_defer(pg, nblk, h, dgamma, c, defer)) != cudaSuccess) return e;
  if ((e = finalize_or_defer(pb, nblk, h, dbeta, c, defer)) != cudaSuccess) return e;
  if (sums) {
    if ((e = finalize_or_defer(pr, nblk, h, dresid, c, defer)) != cudaSuccess) return e;
    if ((e = finalize_or_defer(po, nblk, h, ddx, c, defer)) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

template <typename T>
cudaError_t colsum_t(const void* Y, int64_t ld, int n, int N, float* out, float* partial,
                     const LaunchCtx& c, unsigned* amax_bits, FinalizeJobs* defer) {
  constexpr int E = Vec<T>::N;
  const int nblk = colsum_row_blocks(n, N, E);
  const int rows = (n + nblk - 1) / nblk;
  const int threads = kColsumThreads;
  dim3 grid((N / E + threads - 1) / threads, nblk);
  c.before(KK_COLSUM, (double)n * N * sizeof(T));
  if (amax_bits)
    colsum_partial_kernel<T, true><<<grid, threads, 0, c.stream>>>((const T*)Y, ld, n, N, rows,
                                                                   partial, amax_bits);
  else
    colsum_partial_kernel<T, false><<<grid, threads, 0, c.stream>>>((const T*)Y, ld, n, N, rows,
                                                                    partial, nullptr);
  c.after();
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return finalize_or_defer(partial, nblk, N, out, c, defer);
}

template <typename T>
cudaError_t colsum_dropout_t(const void* Y, void* Ym, int64_t ld, int n, int N,
                             const Dropout& drop, float* out, float* partial,
                             const LaunchCtx& c) {
  constexpr int E = Vec<T>::N;
  const int nblk = n < kColsumDropBlocks ? (n > 0 ? n : 1) : kColsumDropBlocks;
  const int rows = (n + nblk - 1) / nblk;
  const int threads = 256;
  dim3 grid((N / E + threads - 1) / threads, nblk);
  c.before(KK_COLSUM, 2.0 * n * N * sizeof(T));
  colsum_dropout_partial_kernel<T><<<grid, threads, 0, c.stream>>>((const T*)Y, (T*)Ym, ld, n, N,
                                                                   rows, drop, partial);
  c.after();
  c.before(KK_FINALIZE, 4.0 * nblk * N);
  finalize_cols_kernel<<<(N + 31) / 32, kFinWarps * 32, 0, c.stream>>>(partial, nblk, N, out);
  c.after();
  return cudaGetLastError();
}

}  // namespace

size_t ln_bwd_partial_floats(int n, int h, bool sums) {
  const size_t nblk = n < kLnBwdBlocks ? (n > 0 ? n : 1) : kLnBwdBlocks;
  return (sums ? 4 : 2) * nblk * (size_t)h;
}

bool ln_bwd_can_sum(int dtype, int h) {
  // one vector a thread (the sums stay in registers) and a block small enough
  // for two a SM
  return h / (dtype == kBF16 ? 8 : 4) <= kLnSumsThreadsMax;
}

bool FinalizeJobs::add(const float* p, int nb, int cols, float* o) {
  if (n >= kMax) return false;
  part[n] = p;
  nblk[n] = nb;
  N[n] = cols;
  out[n] = o;
  ++n;
  return true;
}

cudaError_t finalize_jobs(FinalizeJobs& j, const LaunchCtx& c) {
  if (j.n == 0) return cudaSuccess;
  FinalizeArgs a;
  memset(&a, 0, sizeof(a));
  a.n = j.n;
  int blocks = 0;
  double bytes = 0;
  for (int k = 0; k < j.n; ++k) {
    a.part[k] = j.part[k];
    a.out[k] = j.out[k];
    a.nblk[k] = j.nblk[k];
    a.N[k] = j.N[k];
    a.first[k] = blocks;
    blocks += (j.N[k] + 31) / 32;
    bytes += 4.0 * j.nblk[k] * j.N[k];
  }
  a.first[j.n] = blocks;
  j.n = 0;
  if (blocks == 0) return cudaSuccess;
  c.before(KK_FINALIZE, bytes);
  finalize_multi_kernel<<<blocks, kFinWarps * 32, 0, c.stream>>>(a);
  c.after();
  return cudaGetLastError();
}
size_t colsum_dropout_partial_floats(int n, int N) {
  const size_t nblk = n < kColsumDropBlocks ? (n > 0 ? n : 1) : kColsumDropBlocks;
  return nblk * (size_t)N;
}
size_t colsum_partial_floats(int n, int N) {
  // the bf16 plan (8 elements a thread) has the most row blocks for a width
  return (size_t)colsum_row_blocks(n, N, 8) * N;
}

cudaError_t ln_fwd(int dtype, const void* x, const void* g, const void* b, void* u, float* mean,
                   float* rstd, int n, int h, float eps, const LaunchCtx& c, unsigned* amax_bits) {
  return dtype == kBF16 ? ln_fwd_t<bf16>(x, g, b, u, mean, rstd, n, h, eps, c, amax_bits)
                        : ln_fwd_t<float>(x, g, b, u, mean, rstd, n, h, eps, c, amax_bits);
}

cudaError_t ln_bwd(int dtype, const float* du, const void* x, const float* mean,
                   const float* rstd, const void* g, const void* resid, void* dx,
                   float* dgamma, float* dbeta, float* partial, int n, int h,
                   const LaunchCtx& c, FinalizeJobs* defer, float* dresid, float* ddx) {
  return dtype == kBF16 ? ln_bwd_t<bf16, 0>(du, nullptr, x, mean, rstd, g, resid, dx, dgamma,
                                            dbeta, partial, n, h, c, defer, dresid, ddx)
                        : ln_bwd_t<float, 0>(du, nullptr, x, mean, rstd, g, resid, dx, dgamma,
                                             dbeta, partial, n, h, c, defer, dresid, ddx);
}

cudaError_t ln_bwd_sum(int dtype, const float* du, const void* du2, const void* x,
                       const float* mean, const float* rstd, const void* g, void* dx,
                       float* dgamma, float* dbeta, float* partial, int n, int h,
                       const LaunchCtx& c) {
  if (!du2) return cudaErrorInvalidValue;
  if (dtype == kBF16)
    return du ? ln_bwd_t<bf16, 2>(du, du2, x, mean, rstd, g, nullptr, dx, dgamma, dbeta, partial,
                                  n, h, c)
              : ln_bwd_t<bf16, 1>(nullptr, du2, x, mean, rstd, g, nullptr, dx, dgamma, dbeta,
                                  partial, n, h, c);
  return du ? ln_bwd_t<float, 2>(du, du2, x, mean, rstd, g, nullptr, dx, dgamma, dbeta, partial,
                                 n, h, c)
            : ln_bwd_t<float, 1>(nullptr, du2, x, mean, rstd, g, nullptr, dx, dgamma, dbeta,
                                 partial, n, h, c);
}

// ---------------------------------------------------------------- recomputation
// u = (x - mean) * rstd * gamma + beta from saved statistics: the same
// arithmetic as ln_fwd_kernel's output, so the values match it bit for bit.
template <typename T>
__global__ void ln_apply_kernel(const T* __restrict__ x, const float* __restrict__ mean,
                                const float* __restrict__ rstd, const T* __restrict__ gamma,
                                const T* __restrict__ beta, T* __restrict__ u, int n, int h) {
  constexpr int E = Vec<T>::N;
  const int nvec = h / E;
  for (int r = blockIdx.x; r < n; r += gridDim.x) {
    const float mu = mean[r], rs = rstd[r];
    for (int vi = threadIdx.x; vi < nvec; vi += blockDim.x) {
      Vec<T> xv, tg, tb, o;
      xv.load(x + (size_t)r * h + vi * E);
      tg.load(gamma + vi * E);
      tb.load(beta + vi * E);
#pragma unroll
      for (int e = 0; e < E; ++e) o.set(e, (xv.get(e) - mu) * rs * tg.get(e) + tb.get(e));
      o.store(u + (size_t)r * h + vi * E);
    }
  }
}

template <typename T>
__global__ void gelu_apply_kernel(const T* __restrict__ z, T* __restrict__ a, int64_t nvec) {
  constexpr int E = Vec<T>::N;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nvec;
       i += (int64_t)gridDim.x * blockDim.x) {
    Vec<T> v;
    v.load(z + i * E);
#pragma unroll
    for (int e = 0; e < E; ++e) v.set(e, gelu_f(v.get(e)));
    v.store(a + i * E);
  }
}

cudaError_t ln_apply(int dtype, const void* x, const float* mean, const float* rstd,
                     const void* g, const void* b, void* u, int n, int h, const LaunchCtx& c) {
  if (n == 0) return cudaSuccess;
  const int grid = n < 8 * c.num_sms ? n : 8 * c.num_sms;
  c.before(KK_LN_FWD, (double)n * h * 2.0 * (dtype == kBF16 ? 2 : 4));
  if (dtype == kBF16)
    ln_apply_kernel<bf16><<<grid, 256, 0, c.stream>>>((const bf16*)x, mean, rstd, (const bf16*)g,
                                                      (const bf16*)b, (bf16*)u, n, h);
  else
    ln_apply_kernel<float><<<grid, 256, 0, c.stream>>>((const float*)x, mean, rstd,
                                                       (const float*)g, (const float*)b,
                                                       (float*)u, n, h);
  c.after();
  return cudaGetLastError();
}

cudaError_t gelu_apply(int dtype, const void* z, void* a, int64_t count, const LaunchCtx& c) {
  if (count == 0) return cudaSuccess;
  const int64_t nvec = count / (dtype == kBF16 ? 8 : 4);
  const int grid = 8 * c.num_sms;
  c.before(KK_LN_FWD, (double)count * 2.0 * (dtype == kBF16 ? 2 : 4));
  if (dtype == kBF16)
    gelu_apply_kernel<bf16><<<grid, 256, 0, c.stream>>>((const bf16*)z, (bf16*)a, nvec);
  else
    gelu_apply_kernel<float><<<grid, 256, 0, c.stream>>>((const float*)z, (float*)a, nvec);
  c.after();
  return cudaGetLastError();
}

cudaError_t colsum(int dtype, const void* Y, int64_t ld, int n, int N, float* out,
                   float* partial, const LaunchCtx& c, unsigned* amax_bits, FinalizeJobs* defer) {
  return dtype == kBF16 ? colsum_t<bf16>(Y, ld, n, N, out, partial, c, amax_bits, defer)
                        : colsum_t<float>(Y, ld, n, N, out, partial, c, amax_bits, defer);
}

cudaError_t colsum_dropout(int dtype, const void* Y, void* Ym, int64_t ld, int n, int N,
                           const Dropout& drop, float* out, float* partial, const LaunchCtx& c) {
  if (N % 4) return cudaErrorInvalidValue;
  return dtype == kBF16 ? colsum_dropout_t<bf16>(Y, Ym, ld, n, N, drop, out, partial, c)
                        : colsum_dropout_t<float>(Y, Ym, ld, n, N, drop, out, partial, c);
}

}  // namespace mtl
