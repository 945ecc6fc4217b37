// Inference kernels: prefill's KV-cache write and the one-token decode step.
//
// Page "Megatron-LM: GPU-Cluster Training Parallelism", section "Paper 1: QKV
// Column-Parallel Splitting in Detail" (inference-time behaviour): the column
// split is the training one; during decode each partition appends the new
// token's K and V of its own heads to its local cache shard, so the cache
// divides evenly by t.  Here the shards are the head blocks of one cache
// [batch][heads][max_seq][d] (K, then V): partition p's shard is heads
// [p*H/t, (p+1)*H/t) of every batch row.
//
// A decode step reads every weight once and the cache up to each sequence's
// length: it is HBM-bound.  Its GEMMs have M = batch (a few tokens), so they
// run "swapped": the weight rows are the tcgen05 M dimension (128 output
// features per CTA) and the tokens the N dimension (batch rounded up to 16).
// K is split over the CTAs of a thread-block cluster (up to 8) so the grid
// covers the SMs about twice; each CTA leaves its fp32 partial tile in its own
// shared memory and the cluster adds the slices in slice order through
// distributed shared memory (deterministic, no global round trip).  The
// row-parallel GEMMs' partition sum (g) is that ordered sum over K slices.
// The decode kernels are chained with programmatic dependent launch: a GEMM
// starts streaming its weights (which no earlier kernel writes) while the
// previous kernel finishes, and waits only before touching activations.
#include "common.cuh"
#include "kernels.h"

namespace mtl {
namespace dec {

constexpr int TILE = 128;        // output features per CTA (MMA M)
constexpr int BK = 64;           // K per stage (one 128-byte swizzled box)
constexpr int THREADS = 192;     // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
constexpr int MAX_STAGES = 8;
constexpr int A_BYTES = TILE * BK * 2;   // 16 KB of weights per stage
constexpr int MAX_SPLITS = 8;            // K slices = CTAs of a (portable) cluster

struct GemvParams {
  int N, K, batch, nb;             // nb = batch rounded up to 16 (MMA N)
  int splits, kb_per_split, stages;
  const bf16* bias;
  const bf16* R;                   // residual [batch][N] (EPI_BIAS_RESID)
  bf16* out;                       // [batch][N]
  unsigned* status;
};

template <int EPI>
__device__ __forceinline__ float gemv_epi(const GemvParams& p, int f, int b, float acc) {
  float v = acc + __bfloat162float(p.bias[f]);
  if (EPI == EPI_BIAS_RESID) v += __bfloat162float(p.R[(size_t)b * p.N + f]);
  if (EPI == EPI_BIAS_GELU) v = gelu_f(v);
  return v;
}

// One CTA: output features [128*blockIdx.x, +128) over K slice blockIdx.y; the
// p.splits slices of a tile are one cluster.
template <int EPI>
__global__ void __launch_bounds__(THREADS) gemv_tc_kernel(const __grid_constant__ CUtensorMap tw,
                                                          const __grid_constant__ CUtensorMap tx,
                                                          const GemvParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(base);
  const uint32_t b_bytes = (uint32_t)p.nb * BK * 2;
  const uint32_t stage_bytes = A_BYTES + b_bytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + p.stages * stage_bytes);
  const uint32_t bar0 = smem_u32(bars);
  auto FULL = [&](int s) { return bar0 + 8u * s; };
  auto EMPTY = [&](int s) { return bar0 + 8u * (MAX_STAGES + s); };
  const uint32_t DONE = bar0 + 8u * (2 * MAX_STAGES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * MAX_STAGES + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // partial tile [batch][128] fp32, over the stage buffers once the MMAs are done
  float* red = reinterpret_cast<float*>(base);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = blockIdx.x, split = blockIdx.y;
  const int kb0 = split * p.kb_per_split;
  const uint32_t ncols = p.nb <= 32 ? 32u : p.nb <= 64 ? 64u : p.nb <= 128 ? 128u : 256u;

  if (threadIdx.x == 0) {
    for (int i = 0; i < p.stages; ++i) {
      mbar_init(FULL(i), 1);
      mbar_init(EMPTY(i), 1);
    }
    mbar_init(DONE, 1);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_shared();
  }
  __syncthreads();
  if (threadIdx.x == 0) griddep_launch_dependents();

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&tw);
      tma_prefetch_desc(&tx);
      // The weights are never written by an earlier kernel: fill the first
      // stages with them before waiting for the activations.
      const int pre = p.kb_per_split < p.stages ? p.kb_per_split : p.stages;
      for (int kb = 0; kb < pre; ++kb) {
        mbar_arrive_expect_tx(FULL(kb), stage_bytes);
        tma_load_2d(sbase + kb * stage_bytes, &tw, FULL(kb), (kb0 + kb) * BK, tile * TILE);
      }
      griddep_wait();
      for (int kb = 0; kb < pre; ++kb)
        tma_load_2d(sbase + kb * stage_bytes + A_BYTES, &tx, FULL(kb), (kb0 + kb) * BK, 0);
      for (int kb = pre; kb < p.kb_per_split; ++kb) {
        const int s = kb % p.stages;
        const uint32_t ph = (kb / p.stages) & 1;
        if (!mbar_wait_bounded(EMPTY(s), ph ^ 1u, p.status, abort_flag)) break;
        mbar_arrive_expect_tx(FULL(s), stage_bytes);
        const uint32_t sa = sbase + s * stage_bytes;
        tma_load_2d(sa, &tw, FULL(s), (kb0 + kb) * BK, tile * TILE);
        tma_load_2d(sa + A_BYTES, &tx, FULL(s), (kb0 + kb) * BK, 0);
      }
    } else {
      griddep_wait();
    }
    __syncwarp();
  } else {
    griddep_wait();
    if (warp == 1) {
      tmem_alloc(smem_u32(tmem_slot), ncols);
      tc_fence_before();
    }
    named_bar_sync(2, THREADS - 32);   // warps 1..5: the TMEM address is in place
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    if (warp == 1) {
      if (lane == 0) {
        const uint32_t idesc = idesc_bf16_f32(TILE, p.nb, false, false);
        bool ok = true;
        for (int kb = 0; kb < p.kb_per_split && ok; ++kb) {
          const int s = kb % p.stages;
          const uint32_t ph = (kb / p.stages) & 1;
          if (!mbar_wait_bounded(FULL(s), ph, p.status, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = sbase + s * stage_bytes;
          const uint64_t da = desc_kbase(sa), db = desc_kbase(sa + A_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            tc_mma_bf16(tmem, desc_add(da, kk * 32), desc_add(db, kk * 32), idesc,
                        (kb > 0 || kk > 0) ? 1u : 0u);
          tc_commit(EMPTY(s));
        }
        if (ok) tc_commit(DONE);
      }
      __syncwarp();
    } else {
      // epilogue: warp w reads TMEM lanes 32*(w%4) .. +31 = output features
      const int q4 = warp & 3;
      const int fl = q4 * 32 + lane;
      const int f = tile * TILE + fl;
      if (mbar_wait_bounded(DONE, 0, p.status, abort_flag)) {
        tc_fence_after();
        for (int c0 = 0; c0 < p.nb; c0 += 32) {
          uint32_t r[32];
          tmem_ld32(tmem + ((uint32_t)(q4 * 32) << 16) + c0, r);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int b = c0 + i;
            if (b < p.batch) {
              const float acc = __uint_as_float(r[i]);
              if (p.splits == 1) {
                if (f < p.N)
                  p.out[(size_t)b * p.N + f] = __float2bfloat16_rn(gemv_epi<EPI>(p, f, b, acc));
              } else {
                red[b * TILE + fl] = acc;
              }
            }
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (p.splits > 1) {
    // the cluster's slices, added in slice order; CTA `rank` finishes outputs
    // [rank*per, (rank+1)*per) of the tile's batch x 128
    cluster_sync();
    const int rank = (int)cluster_cta_rank();
    const int total = p.batch * TILE;
    const int per = (total + p.splits - 1) / p.splits;
    const int o1 = min(total, (rank + 1) * per);
    const uint32_t red_u32 = smem_u32(red);
    for (int o = rank * per + (int)threadIdx.x; o < o1; o += THREADS) {
      float v[MAX_SPLITS];
#pragma unroll
      for (int s = 0; s < MAX_SPLITS; ++s)
        if (s < p.splits) v[s] = ld_dsmem_f32(cluster_map(red_u32 + 4u * o, s));
      float acc = v[0];
#pragma unroll
      for (int s = 1; s < MAX_SPLITS; ++s)
        if (s < p.splits) acc += v[s];
      const int b = o / TILE, f = tile * TILE + o % TILE;
      if (f < p.N) p.out[(size_t)b * p.N + f] = __float2bfloat16_rn(gemv_epi<EPI>(p, f, b, acc));
    }
    cluster_sync();   // no CTA leaves while another may still read its partial
  }
  if (warp == 1) {
    if (*abort_flag) {
      const long long t0 = clock64();
      while (clock64() - t0 < 2000000LL) {
      }
    }
    tc_fence_after();
    tmem_dealloc(*tmem_slot, ncols);
  }
}

// ---------------------------------------------------------------- decode attention
constexpr int ATT_CHUNK = 128;   // keys per CTA
constexpr int ATT_THREADS = 128;

template <typename T>
struct AttnDecParams {
  int batch, heads, d, max_seq, splits_max;
  float scale_log2;
  const T* qkv;          // [batch][3h] head-interleaved
  T* kc;                 // K cache [batch][heads][max_seq][d]
  T* vc;                 // V cache
  const int* cache_len;  // [batch]
  T* ctx;                // [batch][h]
  float* part;           // [batch*heads][splits_max][d + 2] (o, m, l)
  int* counters;         // [batch*heads], zero on entry, left zero
  unsigned* status;
};

template <typename T>
__device__ __forceinline__ void unpack16(const uint4& u, float (&v)[16 / sizeof(T)]) {
  Vec<T> x;
  x.raw = *reinterpret_cast<const decltype(x.raw)*>(&u);
#pragma unroll
  for (int i = 0; i < Vec<T>::N; ++i) v[i] = x.get(i);
}

// One CTA per (chunk of 128 keys, head, batch row).  The chunk's cached K and
// V rows are contiguous in the head-major cache, so one thread starts two bulk
// copies into shared memory before anything else (the cache rows below the
// current length were written by earlier steps, so this runs ahead of the
// programmatic wait on the QKV GEMM).  Scores: four lanes per key, each
// summing a quarter of the 16-byte chunks of the row (chunk order chosen so
// the 8 lanes of a shared-memory phase hit 8 different bank groups); the new
// token's own key and value come from the QKV output.  P V: thread = (16-byte
// channel chunk, key group).  Chunks of a (batch, head) combine in chunk order
// in the last CTA to finish; the chunk holding position L writes the new K, V.
template <typename T>
__global__ void __launch_bounds__(ATT_THREADS) attn_decode_kernel(const AttnDecParams<T> p) {
  constexpr int VEC = 16 / sizeof(T);
  extern __shared__ __align__(128) uint8_t att_smem[];   // K [CHUNK][d], V [CHUNK][d]
  __shared__ __align__(8) uint64_t bar;
  __shared__ float s_q[128];
  __shared__ float s_p[ATT_CHUNK];
  __shared__ float s_red[ATT_THREADS / 32];
  __shared__ float s_o[ATT_THREADS * (VEC + 1)];   // padded: conflict-free stores
  __shared__ int s_last;
  __shared__ int s_abort;
  const int sp = blockIdx.x, hd = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int d = p.d, h = p.heads * d;
  const int row_bytes = d * (int)sizeof(T);
  const int nch = row_bytes / 16;                 // 16-byte chunks per row
  T* sK = reinterpret_cast<T*>(att_smem);
  T* sV = reinterpret_cast<T*>(att_smem + ATT_CHUNK * row_bytes);
  // cache lengths are advanced only at the end of a step
  const int L = p.cache_len[b];
  if (L < 0 || L >= p.max_seq) {
    griddep_wait();
    if (tid == 0 && sp == 0 && hd == 0) atomicOr(p.status, kDevErrBadArg);
    return;
  }
  const int nk = L + 1;
  const int nsplit = (nk + ATT_CHUNK - 1) / ATT_CHUNK;
  if (sp >= nsplit) {
    griddep_wait();
    return;
  }
  const int j0 = sp * ATT_CHUNK, j1 = min(nk, j0 + ATT_CHUNK);
  const int ncached = min(j1, L) - j0;            // rows already in the cache
  const size_t head_off = ((size_t)b * p.heads + hd) * p.max_seq;
  if (tid == 0) {
    mbar_init(smem_u32(&bar), 1);
    s_abort = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (tid == 0 && ncached > 0) {
    const uint32_t bytes = (uint32_t)ncached * row_bytes;
    mbar_arrive_expect_tx(smem_u32(&bar), 2 * bytes);
    bulk_load(smem_u32(sK), p.kc + (head_off + j0) * d, bytes, smem_u32(&bar));
    bulk_load(smem_u32(sV), p.vc + (head_off + j0) * d, bytes, smem_u32(&bar));
  }
  griddep_wait();
  if (tid == 0) griddep_launch_dependents();
  const T* qrow = p.qkv + (size_t)b * 3 * h + (size_t)hd * 3 * d;
  for (int c = tid; c < d; c += ATT_THREADS) s_q[c] = to_f<T>(qrow[c]) * p.scale_log2;
  if (sp == nsplit - 1) {
    // position L: the new key and value, into the cache and into this chunk
    for (int c = tid; c < d; c += ATT_THREADS) {
      const T kv = qrow[d + c], vv = qrow[2 * d + c];
      p.kc[(head_off + L) * d + c] = kv;
      p.vc[(head_off + L) * d + c] = vv;
      sK[(L - j0) * d + c] = kv;
      sV[(L - j0) * d + c] = vv;
    }
  }
  if (ncached > 0 && !mbar_wait_bounded(smem_u32(&bar), 0, p.status, &s_abort)) {
    // bulk copy never completed: the status word has the timeout; finish
    // without trusting the rows
  }
  __syncthreads();
  // scores (log2 domain): lanes 4k..4k+3 of a warp take key 8*pass + k of the warp
  const int nrows = j1 - j0;
  const int pp = lane & 3, kk = (lane >> 2) & 1;
  const int sh = (nch % 8 == 0) ? 4 : 0;
  float mx = -INFINITY;
  for (int r0 = warp * 8; r0 < nrows; r0 += 32) {
    const int r = r0 + (lane >> 2);
    float s = 0.f;
    if (r < nrows) {
      const uint8_t* krow = reinterpret_cast<const uint8_t*>(sK) + (size_t)r * row_bytes;
      for (int t = pp; t < nch; t += 4) {
        int c = t + kk * sh;
        if (c >= nch) c -= nch;
        const uint4 u = *reinterpret_cast<const uint4*>(krow + c * 16);
        float kv[VEC];
        unpack16<T>(u, kv);
#pragma unroll
        for (int i = 0; i < VEC; ++i) s = fmaf(s_q[c * VEC + i], kv[i], s);
      }
    }
    s += __shfl_xor_sync(0xffffffffu, s, 1);
    s += __shfl_xor_sync(0xffffffffu, s, 2);
    if (r < nrows) {
      if (pp == 0) s_p[r] = s;
      mx = fmaxf(mx, s);
    }
  }
  mx = warp_max(mx);
  if (lane == 0) s_red[warp] = mx;
  __syncthreads();
  mx = s_red[0];
  for (int w = 1; w < ATT_THREADS / 32; ++w) mx = fmaxf(mx, s_red[w]);
  __syncthreads();
  float l = 0.f;
  for (int r = tid; r < nrows; r += ATT_THREADS) {
    const float e = exp2f(s_p[r] - mx);
    s_p[r] = e;
    l += e;
  }
  l = warp_sum(l);
  if (lane == 0) s_red[warp] = l;
  __syncthreads();
  l = 0.f;
  for (int w = 0; w < ATT_THREADS / 32; ++w) l += s_red[w];
  // o = sum_r p_r v_r: thread = (channel chunk cg, key group kg)
  const int kg_n = ATT_THREADS / nch;
  const int cg = tid % nch, kg = tid / nch;
  float acc[VEC];
#pragma unroll
  for (int i = 0; i < VEC; ++i) acc[i] = 0.f;
  if (kg < kg_n) {
    const uint8_t* vbase = reinterpret_cast<const uint8_t*>(sV) + cg * 16;
    for (int r = kg; r < nrows; r += kg_n) {
      const float pr = s_p[r];
      float vv[VEC];
      unpack16<T>(*reinterpret_cast<const uint4*>(vbase + (size_t)r * row_bytes), vv);
#pragma unroll
      for (int i = 0; i < VEC; ++i) acc[i] = fmaf(pr, vv[i], acc[i]);
    }
  }
#pragma unroll
  for (int i = 0; i < VEC; ++i) s_o[tid * (VEC + 1) + i] = acc[i];
  __syncthreads();
  const int bh = b * p.heads + hd;
  float* mypart = p.part + ((size_t)bh * p.splits_max + sp) * (d + 2);
  for (int c = tid; c < d; c += ATT_THREADS) {
    const int g = c / VEC, i = c % VEC;
    float o = 0.f;
    for (int k = 0; k < kg_n; ++k) o += s_o[(k * nch + g) * (VEC + 1) + i];
    if (nsplit == 1)
      p.ctx[(size_t)b * h + (size_t)hd * d + c] = from_f<T>(o / l);
    else
      mypart[c] = o;
  }
  if (nsplit == 1) return;
  if (tid == 0) {
    mypart[d] = mx;
    mypart[d + 1] = l;
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(&p.counters[bh], 1) == nsplit - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const float* pp_ = p.part + (size_t)bh * p.splits_max * (d + 2);
  float M = -INFINITY;
  for (int s = 0; s < nsplit; ++s) M = fmaxf(M, __ldcg(pp_ + (size_t)s * (d + 2) + d));
  float Lsum = 0.f;
  for (int s = 0; s < nsplit; ++s)
    Lsum += __ldcg(pp_ + (size_t)s * (d + 2) + d + 1) * exp2f(__ldcg(pp_ + (size_t)s * (d + 2) + d) - M);
  for (int c = tid; c < d; c += ATT_THREADS) {
    float o = 0.f;
    for (int s = 0; s < nsplit; ++s)
      o += __ldcg(pp_ + (size_t)s * (d + 2) + c) * exp2f(__ldcg(pp_ + (size_t)s * (d + 2) + d) - M);
    p.ctx[(size_t)b * h + (size_t)hd * d + c] = from_f<T>(o / Lsum);
  }
  if (tid == 0) p.counters[bh] = 0;
}

// ---------------------------------------------------------------- cache bookkeeping
// Prefill: K and V of tokens (b, i < seq) from qkv [batch*seq][3h] to the cache
// at positions i; lengths set to seq.  One block per token.
template <typename T>
__global__ void kv_write_kernel(const T* __restrict__ qkv, T* __restrict__ kc, T* __restrict__ vc,
                                int* __restrict__ cache_len, int seq, int heads, int d,
                                int max_seq) {
  constexpr int VEC = 16 / sizeof(T);
  const int row = blockIdx.x;
  const int b = row / seq, i = row % seq;
  const int h = heads * d;
  const T* src = qkv + (size_t)row * 3 * h;
  const int per_head = d / VEC;
  for (int v = threadIdx.x; v < 2 * heads * per_head; v += blockDim.x) {
    const int which = v / (heads * per_head);          // 0: K, 1: V
    const int r = v % (heads * per_head);
    const int hd = r / per_head, c = (r % per_head) * VEC;
    Vec<T> x;
    x.load(src + (size_t)hd * 3 * d + (which + 1) * d + c);
    T* dst = (which == 0 ? kc : vc) + (((size_t)b * heads + hd) * max_seq + i) * d + c;
    x.store(dst);
  }
  if (i == 0 && threadIdx.x == 0) cache_len[b] = seq;
}

__global__ void kv_advance_kernel(int* cache_len, int batch, int max_seq) {
  griddep_wait();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < batch && cache_len[b] >= 0 && cache_len[b] < max_seq) cache_len[b] += 1;
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

bool make_map(CUtensorMap* m, const void* ptr, uint64_t cols, uint64_t rows, uint32_t box_rows) {
  static EncodeTiledFn enc = nullptr;
  if (!enc) {
    void* fp = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fp, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return false;
    enc = reinterpret_cast<EncodeTiledFn>(fp);
  }
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {BK, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int round16(int v) { return (v + 15) / 16 * 16; }

}  // namespace dec

using namespace dec;

// Split of K for a decode GEMM: the largest divisor of the 64-wide K block
// count, at most one cluster (8), that keeps the grid near two CTAs per SM.
static int gemv_splits(int N, int K, int num_sms) {
  if (num_sms > kDecodeSmCap) num_sms = kDecodeSmCap;
  const int tiles = (N + TILE - 1) / TILE;
  const int nkb = K / BK;
  int target = (2 * num_sms + tiles - 1) / tiles;
  if (target > MAX_SPLITS) target = MAX_SPLITS;
  if (target > nkb) target = nkb;
  int s = 1;
  for (int c = 1; c <= target; ++c)
    if (nkb % c == 0) s = c;
  return s;
}

bool gemv_tc_supported(int N, int K, int batch) {
  return batch >= 1 && batch <= kDecodeMaxBatch && K % BK == 0 && K > 0 && N > 0;
}

cudaError_t gemv_tc(int epi, int N, int K, int batch, const void* W, const void* X,
                    const void* bias, const void* R, void* out, unsigned* status,
                    const LaunchCtx& c) {
  if (batch == 0) return cudaSuccess;
  if (!gemv_tc_supported(N, K, batch)) return cudaErrorInvalidValue;
  GemvParams p;
  p.N = N;
  p.K = K;
  p.batch = batch;
  p.nb = round16(batch);
  p.splits = gemv_splits(N, K, c.num_sms);
  p.kb_per_split = K / BK / p.splits;
  const int stage_bytes = A_BYTES + p.nb * BK * 2;
  int stages = (96 * 1024) / stage_bytes;
  p.stages = stages < 2 ? 2 : stages > MAX_STAGES ? MAX_STAGES : stages;
  p.bias = static_cast<const bf16*>(bias);
  p.R = static_cast<const bf16*>(R);
  p.out = static_cast<bf16*>(out);
  p.status = status;
  CUtensorMap tw, tx;
  if (!make_map(&tw, W, (uint64_t)K, (uint64_t)N, TILE) ||
      !make_map(&tx, X, (uint64_t)K, (uint64_t)batch, (uint32_t)p.nb))
    return cudaErrorInvalidValue;
  // the partial tile [batch][128] fp32 reuses the stage buffers
  size_t smem = (size_t)p.stages * stage_bytes;
  if (smem < (size_t)batch * TILE * 4) return cudaErrorInvalidValue;
  smem += 1024 + 256;
  dim3 grid((N + TILE - 1) / TILE, p.splits);
  cudaError_t e;
  void (*fn)(const CUtensorMap, const CUtensorMap, const GemvParams) = nullptr;
  switch (epi) {
    case EPI_BIAS: fn = gemv_tc_kernel<EPI_BIAS>; break;
    case EPI_BIAS_RESID: fn = gemv_tc_kernel<EPI_BIAS_RESID>; break;
    case EPI_BIAS_GELU: fn = gemv_tc_kernel<EPI_BIAS_GELU>; break;
    default: return cudaErrorInvalidValue;
  }
  if ((e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) !=
      cudaSuccess)
    return e;
  c.before(KK_GEMV_TC, (double)N * K * 2 + (double)batch * (K + N) * 2);
  e = launch_ex(c, fn, grid, dim3(THREADS), smem, p.splits, tw, tx, p);
  c.after();
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

int attn_decode_splits(int max_seq) { return (max_seq + ATT_CHUNK - 1) / ATT_CHUNK; }

template <typename T>
static cudaError_t attn_decode_t(const void* qkv, void* kcache, void* vcache, const int* cache_len,
                                 void* ctx, float* part, int* counters, int batch, int heads,
                                 int d, int max_seq, double kv_bytes, unsigned* status,
                                 const LaunchCtx& c) {
  AttnDecParams<T> p;
  p.batch = batch;
  p.heads = heads;
  p.d = d;
  p.max_seq = max_seq;
  p.splits_max = attn_decode_splits(max_seq);
  p.scale_log2 = 1.4426950408889634f / sqrtf((float)d);
  p.qkv = static_cast<const T*>(qkv);
  p.kc = static_cast<T*>(kcache);
  p.vc = static_cast<T*>(vcache);
  p.cache_len = cache_len;
  p.ctx = static_cast<T*>(ctx);
  p.part = part;
  p.counters = counters;
  p.status = status;
  dim3 grid(p.splits_max, heads, batch);
  const size_t smem = 2 * (size_t)ATT_CHUNK * d * sizeof(T);
  cudaError_t e = cudaFuncSetAttribute(attn_decode_kernel<T>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  c.before(KK_ATTN_DECODE, kv_bytes);
  e = launch_ex(c, attn_decode_kernel<T>, grid, dim3(ATT_THREADS), smem, 1, p);
  c.after();
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t attn_decode(int dtype, const void* qkv, void* kcache, void* vcache,
                        const int* cache_len, void* ctx, float* part, int* counters, int batch,
                        int heads, int d, int max_seq, double kv_bytes, unsigned* status,
                        const LaunchCtx& c) {
  if (batch == 0) return cudaSuccess;
  return dtype == kBF16 ? attn_decode_t<bf16>(qkv, kcache, vcache, cache_len, ctx, part, counters,
                                              batch, heads, d, max_seq, kv_bytes, status, c)
                        : attn_decode_t<float>(qkv, kcache, vcache, cache_len, ctx, part,
                                               counters, batch, heads, d, max_seq, kv_bytes,
                                               status, c);
}

cudaError_t kv_write(int dtype, const void* qkv, void* kcache, void* vcache, int* cache_len,
                     int batch, int seq, int heads, int d, int max_seq, const LaunchCtx& c) {
  if (batch == 0) return cudaSuccess;
  const double bytes = 4.0 * batch * seq * heads * d * (dtype == kBF16 ? 2 : 4);
  c.before(KK_KV_WRITE, bytes);
  if (dtype == kBF16)
    kv_write_kernel<bf16><<<batch * seq, 256, 0, c.stream>>>(
        static_cast<const bf16*>(qkv), static_cast<bf16*>(kcache), static_cast<bf16*>(vcache),
        cache_len, seq, heads, d, max_seq);
  else
    kv_write_kernel<float><<<batch * seq, 256, 0, c.stream>>>(
        static_cast<const float*>(qkv), static_cast<float*>(kcache), static_cast<float*>(vcache),
        cache_len, seq, heads, d, max_seq);
  c.after();
  return cudaGetLastError();
}

cudaError_t kv_advance(int* cache_len, int batch, int max_seq, const LaunchCtx& c) {
  if (batch == 0) return cudaSuccess;
  c.before(KK_KV_WRITE, 8.0 * batch);
  cudaError_t e = launch_ex(c, kv_advance_kernel, dim3((batch + 127) / 128), dim3(128), 0, 1,
                            cache_len, batch, max_seq);
  c.after();
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace mtl
