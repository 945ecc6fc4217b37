// Shared device helpers: bf16 conversion, vector IO, GeLU, mbarrier / TMA /
// tcgen05 inline PTX wrappers and the bounded device-side wait.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "bounds.h"
#include "kernels.h"

namespace mtl {

// ---------------------------------------------------------------- status word
// The first bytes of every workspace hold a device status word; kernels OR these
// codes into it, the host reads it in mtl_layer_check.
constexpr unsigned kDevErrTimeout = 1u;
constexpr unsigned kDevErrBadArg = 2u;
constexpr unsigned kDevErrBounds = bounds::kStatusBoundsFlag;   // MTL_DEBUG builds

// Coordinate checks of builds with MTL_DEBUG: MTL_CHECKED(status, fault, site)
// records a failed check (fault != 0) in the status word and is false, so the
// caller skips the access; without MTL_DEBUG it is `true` and the check is not
// compiled.
__device__ __forceinline__ bool dcheck(unsigned* status, uint32_t fault, uint32_t site) {
  if (fault != bounds::kOk) {
    atomicOr(status, bounds::status_bits(fault, site));
    return false;
  }
  return true;
}
#ifdef MTL_DEBUG
#define MTL_CHECKED(status, fault, site) ::mtl::dcheck((status), (fault), (site))
#else
#define MTL_CHECKED(status, fault, site) true
#endif
// Words of the same 256-byte status block (zeroed by every API call) that the
// persistent attention kernels use as work counters {next item, CTAs done};
// the last CTA of a launch sets its pair back to zero.
constexpr int kSchedFwd = 32, kSchedDq = 34, kSchedDkv = 36;

// A device-side wait gives up after this many SM clock cycles (about 2 s at
// 2 GHz), records kDevErrTimeout and lets the kernel wind down.
constexpr long long kWaitLimitCycles = 4000000000LL;

using bf16 = __nv_bfloat16;

// ---------------------------------------------------------------- elementwise
// The standard normal Phi(z) and phi(z) from one exponential.  With
// x = |z| / sqrt 2: erfc(x) ~ t (a1 + a2 t + ... + a5 t^4) exp(-x^2),
// t = 1 / (1 + p x), the rational approximation 7.1.26 of Abramowitz and
// Stegun, Handbook of Mathematical Functions (|error| <= 1.5e-7 on erf, with
// its published p and a1..a5); Phi(-|z|) = erfc(x) / 2 and
// phi(z) = exp(-x^2) / sqrt(2 pi).  A GeLU epilogue thus costs one reciprocal
// and one exp2 per element.
__device__ __forceinline__ void normal_cdf_pdf(float z, float& cdf, float& pdf) {
  const float x = fabsf(z) * 0.70710678118654752f;
  const float t = __fdividef(1.0f, fmaf(0.3275911f, x, 1.0f));
  float q = fmaf(t, 1.061405429f, -1.453152027f);
  q = fmaf(t, q, 1.421413741f);
  q = fmaf(t, q, -0.284496736f);
  q = fmaf(t, q, 0.254829592f);
  const float g = exp2f(-0.72134752044448170f * z * z);  // exp(-x^2) = exp(-z^2 / 2)
  const float tail = 0.5f * t * q * g;                  // Phi(-|z|)
  cdf = z >= 0.f ? 1.0f - tail : tail;
  pdf = 0.39894228040143268f * g;
}
__device__ __forceinline__ float gelu_f(float z) {
  // GeLU(z) = z * Phi(z)
  float cdf, pdf;
  normal_cdf_pdf(z, cdf, pdf);
  return z * cdf;
}
__device__ __forceinline__ float gelu_grad_f(float z) {
  // d/dz GeLU = Phi(z) + z * phi(z)
  float cdf, pdf;
  normal_cdf_pdf(z, cdf, pdf);
  return fmaf(z, pdf, cdf);
}

template <typename T> __device__ __forceinline__ float to_f(T v);
template <> __device__ __forceinline__ float to_f<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f<bf16>(bf16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f(float v);
template <> __device__ __forceinline__ float from_f<float>(float v) { return v; }
template <> __device__ __forceinline__ bf16 from_f<bf16>(float v) { return __float2bfloat16_rn(v); }

// 16-byte vector of T: 8 bf16 or 4 float.
template <typename T> struct Vec;
template <> struct Vec<bf16> {
  static constexpr int N = 8;
  uint4 raw;
  __device__ __forceinline__ void load(const bf16* p) { raw = *reinterpret_cast<const uint4*>(p); }
  __device__ __forceinline__ void store(bf16* p) const { *reinterpret_cast<uint4*>(p) = raw; }
  __device__ __forceinline__ float get(int i) const {
    const bf16* h = reinterpret_cast<const bf16*>(&raw);
    return __bfloat162float(h[i]);
  }
  __device__ __forceinline__ void set(int i, float v) {
    bf16* h = reinterpret_cast<bf16*>(&raw);
    h[i] = __float2bfloat16_rn(v);
  }
  // v rounded to bf16 (round to nearest even), as fp32
  static __device__ __forceinline__ float round(float v) {
    return __bfloat162float(__float2bfloat16_rn(v));
  }
  // all N elements to / from fp32 (a bf16 is the high half of an fp32 word)
  __device__ __forceinline__ void unpack(float (&f)[N]) const {
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  __device__ __forceinline__ void pack(const float (&f)[N]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 v = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
      w[i] = *reinterpret_cast<uint32_t*>(&v);
    }
    raw = make_uint4(w[0], w[1], w[2], w[3]);
  }
};
template <> struct Vec<float> {
  static constexpr int N = 4;
  float4 raw;
  __device__ __forceinline__ void load(const float* p) { raw = *reinterpret_cast<const float4*>(p); }
  __device__ __forceinline__ void store(float* p) const { *reinterpret_cast<float4*>(p) = raw; }
  __device__ __forceinline__ float get(int i) const { return (&raw.x)[i]; }
  __device__ __forceinline__ void set(int i, float v) { (&raw.x)[i] = v; }
  static __device__ __forceinline__ float round(float v) { return v; }
  __device__ __forceinline__ void unpack(float (&f)[N]) const {
    f[0] = raw.x;
    f[1] = raw.y;
    f[2] = raw.z;
    f[3] = raw.w;
  }
  __device__ __forceinline__ void pack(const float (&f)[N]) { raw = make_float4(f[0], f[1], f[2], f[3]); }
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// ---------------------------------------------------------------- shared memory
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking probe of the same phase (cheaper than try_wait when the phase has
// already completed, the common case on a pipeline's fast path).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase with parity `parity` of barrier `bar` to complete.  Gives
// up after `limit` SM cycles (kWaitLimitCycles by default, or at once if *abort
// is set by another role of the CTA), records the timeout in the status word
// and sets *abort.  Returns false when it gave up.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  unsigned* status, volatile int* abort,
                                                  long long limit = kWaitLimitCycles) {
  if (mbar_test_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (clock64() - t0 > limit) {
      atomicOr(status, kDevErrTimeout);
      *abort = 1;
      return false;
    }
  }
}

// Arrive on a barrier given by a cluster shared-memory address (possibly in
// another CTA of the cluster), with release semantics at cluster scope.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// mbar_wait_bounded for a barrier whose arrivals come from other CTAs of the
// cluster (acquire at cluster scope).
__device__ __forceinline__ bool mbar_wait_bounded_cluster(uint32_t bar, uint32_t parity,
                                                          unsigned* status, volatile int* abort) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if (*abort) return false;
    if (clock64() - t0 > kWaitLimitCycles) {
      atomicOr(status, kDevErrTimeout);
      *abort = 1;
      return false;
    }
  }
}

// ---------------------------------------------------------------- clusters
__device__ __forceinline__ uint32_t cluster_cta_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// The cluster shared-memory address of the same location in CTA `rank`.
__device__ __forceinline__ uint32_t cluster_map(uint32_t addr, uint32_t rank) {
  uint32_t o;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(o) : "r"(addr), "r"(rank));
  return o;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::
          : "memory");
}

// Load a float from another CTA's shared memory (address from cluster_map).
__device__ __forceinline__ float ld_dsmem_f32(uint32_t cluster_addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(cluster_addr) : "memory");
  return v;
}

// ---------------------------------------------------------------- programmatic dependent launch
// Wait until the kernel this one programmatically depends on has completed and
// its memory is visible (returns at once when launched without that
// dependency).  Every kernel that may be launched this way calls it before its
// first read of a predecessor's output and before its first global write.
__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
// Let the next kernel of the stream begin launching once every CTA of this
// grid has called this or exited (its own griddep_wait still waits for this
// grid to finish).
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" :::);
}

// ---------------------------------------------------------------- TMA
// Brings the 128-byte line holding `p` into L2 (no register or shared-memory
// cost; the load that later reads it hits L2).
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<uint64_t>(p)));
}
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* m, uint32_t bar,
                                            int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(x), "r"(y)
      : "memory");
}
// Load into this CTA's shared memory; completion is signalled on `bar`, which
// may be the barrier of the pair's leader CTA (cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* m, uint32_t bar,
                                                 int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(x), "r"(y)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* m, uint32_t bar,
                                            int32_t x, int32_t y, int32_t z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// Plain bulk copy global -> shared (16-byte aligned addresses, size a multiple
// of 16), completing on the mbarrier's transaction count.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

// ---------------------------------------------------------------- tcgen05
// Shared-memory matrix descriptor (tcgen05 form): start address, leading and
// stride byte offsets (all >> 4), the fixed version bits 46..47 = 1, base
// offset 0 (tiles are 1024-byte aligned), swizzle mode in bits 61..63
// (2 = 128-byte swizzle, 4 = 64-byte swizzle).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo, uint32_t mode) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;
  d |= static_cast<uint64_t>(mode & 7u) << 61;
  return d;
}
// swizzle modes of the descriptor
constexpr uint32_t kDescSw128 = 2, kDescSw64 = 4;
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return smem_desc(addr, lbo, sbo, kDescSw128);
}

// Instruction descriptor of tcgen05.mma kind::f16 with bf16 A/B and fp32
// accumulate.  a_mn / b_mn select MN-major (transposed) operands.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4)                       // D format: f32
         | (1u << 7)                     // A format: bf16
         | (1u << 10)                    // B format: bf16
         | ((a_mn ? 1u : 0u) << 15)      // A major
         | ((b_mn ? 1u : 0u) << 16)      // B major
         | ((uint32_t)(N >> 3) << 17)    // N / 8
         | ((uint32_t)(M >> 4) << 24);   // M / 16
}

// Instruction descriptor of tcgen05.mma kind::f8f6f4 with fp32 accumulate and
// K-major operands; fa / fb: operand formats, 0 = E4M3, 1 = E5M2.
__host__ __device__ constexpr uint32_t idesc_f8_f32(int M, int N, int fa, int fb) {
  return (1u << 4)                       // D format: f32
         | ((uint32_t)fa << 7)           // A format
         | ((uint32_t)fb << 10)          // B format
         | ((uint32_t)(N >> 3) << 17)    // N / 8
         | ((uint32_t)(M >> 4) << 24);   // M / 16
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Whole warp: allocate `ncols` TMEM columns, base address written to smem.
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, issued by one thread.
__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]^T: the A operand (M rows = TMEM lanes, K
// along the columns, two 16-bit elements per 32-bit column, the lower K index
// in the low half) is read from tensor memory.
__device__ __forceinline__ void tc_mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                               uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// The mbarrier gets one arrival once all earlier tcgen05.mma of this thread are done.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}
// 32 lanes x 32 consecutive 32-bit columns: thread i of the warp gets lane
// (base lane + i), columns col .. col+31.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
// Pair (cta_group::2) forms: one warp of each CTA of the pair allocates /
// frees the same columns in both CTAs; the leader CTA issues MMAs that span
// both CTAs' shared memory and TMEM; a commit can signal both CTAs' barriers.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_mma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                                 uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// The FP8 form (kind::f8f6f4, K = 32 per instruction), issued by the leader.
__device__ __forceinline__ void tc_mma_f8_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                               uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void tc_commit_pair_mc(uint32_t bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 "
      "[%0], %1;" ::"r"(bar),
      "h"(cta_mask)
      : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
// 32 lanes x 32 consecutive 32-bit columns from registers into TMEM.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
// 32 lanes x 16 consecutive 32-bit columns from registers into TMEM.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 2^x with the hardware approximation (ex2.approx), for softmax exponentials.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Shared-memory operand tiles loaded by TMA as 128-byte-swizzled boxes of
// [rows][64 bf16]: a tile is `atoms` such boxes, `atom_bytes` apart, each box
// covering 64 consecutive elements of the contiguous (channel) dimension.
// K-major use (rows = M or N, channels = K): K step kk of 16 elements.
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t base, uint32_t atom_bytes, int kk) {
  return smem_desc_sw128(base + (kk >> 2) * atom_bytes + (kk & 3) * 32, 16, 1024);
}
// MN-major use (rows = K, channels = M or N): K step kk of 16 rows; the
// leading byte offset steps between 64-wide channel boxes.
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t base, uint32_t atom_bytes, int kk) {
  return smem_desc_sw128(base + kk * 2048, atom_bytes, 1024);
}

// The same descriptors built from a precomputed base: the start address is the
// low field, so a tile offset is added directly (off >> 4, no carry out of the
// 14-bit field for shared-memory addresses).  With kk a compile-time constant
// the offsets fold, so the single MMA-issuing thread spends a couple of integer
// instructions per MMA instead of rebuilding the descriptor.
__host__ __device__ constexpr uint32_t kmajor_off(int kk, uint32_t atom_bytes) {
  return (uint32_t)(kk >> 2) * atom_bytes + (uint32_t)(kk & 3) * 32;
}
__host__ __device__ constexpr uint32_t mnmajor_off(int kk) { return (uint32_t)kk * 2048; }
__device__ __forceinline__ uint64_t desc_kbase(uint32_t base) {
  return smem_desc_sw128(base, 16, 1024);
}
__device__ __forceinline__ uint64_t desc_mnbase(uint32_t base, uint32_t atom_bytes) {
  return smem_desc_sw128(base, atom_bytes, 1024);
}
__device__ __forceinline__ uint64_t desc_add(uint64_t desc, uint32_t byte_off) {
  return desc + (uint64_t)(byte_off >> 4);
}

// Byte offset of 16-byte chunk `c` of row `r` inside a [rows][64 bf16] box
// with 128-byte swizzle (the layout TMA writes and the MMA reads).
__device__ __forceinline__ uint32_t sw128_offset(int r, int c) {
  return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
}

// Barrier over `count` threads (a multiple of 32) on hardware barrier `id`.
__device__ __forceinline__ void named_bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
// TMA tensor store of a shared-memory box to global coordinates (x, y), as a
// bulk group of the issuing thread; bulk_commit closes the group,
// bulk_wait_read0 waits until every group of this thread has finished
// reading shared memory, bulk_wait0 until their writes are done.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* m, uint32_t src, int32_t x,
                                             int32_t y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(m)),
               "r"(src), "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
// One fp32 / one bf16 (as fp32) from a shared-memory address.
__device__ __forceinline__ float ld_shared_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t ld_shared_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ float ld_shared_bf16(uint32_t addr) {
  unsigned short b;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(b) : "r"(addr));
  return __uint_as_float((uint32_t)b << 16);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

// ---------------------------------------------------------------- Philox dropout
// Philox4x32 with 10 rounds (Salmon, Moraes, Dror, Shaw, "Parallel random
// numbers: as easy as 1, 2, 3", SC'11): per round, counter words 0 and 2 are
// multiplied by the two Philox multipliers; the high halves of the products are
// XORed with words 1 / 3 and the round key, the low halves move to words 1 / 3;
// the key advances by the two Weyl increments between rounds (Dropout::rk holds
// the ten round keys, precomputed on the host).
__device__ __forceinline__ uint4 philox4x32_10_rk(uint4 c, const uint32_t (&rk)[20]) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const unsigned long long p0 = (unsigned long long)c.x * 0xD2511F53u;
    const unsigned long long p1 = (unsigned long long)c.z * 0xCD9E8D57u;
    c = make_uint4((uint32_t)(p1 >> 32) ^ c.y ^ rk[2 * r], (uint32_t)p1,
                   (uint32_t)(p0 >> 32) ^ c.w ^ rk[2 * r + 1], (uint32_t)p0);
  }
  return c;
}

// Keep bits of elements 4*blk .. 4*blk+3 of a dropout site: bit k for 4*blk+k.
__device__ __forceinline__ uint32_t drop_bits4(unsigned long long blk, const Dropout& d) {
  const uint4 w =
      philox4x32_10_rk(make_uint4((uint32_t)blk, (uint32_t)(blk >> 32), d.site, 0u), d.rk);
  return (w.x >= d.thresh ? 1u : 0u) | (w.y >= d.thresh ? 2u : 0u) |
         (w.z >= d.thresh ? 4u : 0u) | (w.w >= d.thresh ? 8u : 0u);
}

// Keep bits of 32 consecutive elements e0 .. e0+31 (e0 % 4 == 0): bit k for e0+k.
__device__ __forceinline__ uint32_t drop_bits32(unsigned long long e0, const Dropout& d) {
  uint32_t bits = 0;
#pragma unroll
  for (int q = 0; q < 8; ++q) bits |= drop_bits4((e0 >> 2) + q, d) << (4 * q);
  return bits;
}

// Whether element e is kept (any alignment; one Philox block per call).
__device__ __forceinline__ bool drop_keep(unsigned long long e, const Dropout& d) {
  return (drop_bits4(e >> 2, d) >> (e & 3)) & 1u;
}

}  // namespace mtl
