// Tensor-core GEMM for sm_103a: TMA -> shared memory -> tcgen05.mma -> TMEM ->
// fused epilogue.  bf16 operands, fp32 accumulation.
//
//   C = epi( sum_{p = 0..parts-1} P_p ),  P_p = sum_{k in part p} A(m,k) B(n,k)
//
// Row-parallel GEMMs (out-proj and fc2 forward; the fc1 and QKV input-gradient
// GEMMs backward) split K into t partitions.  Each partition's partial product
// is accumulated on its own in TMEM and the epilogue adds the partials in
// partition order in fp32: the g (forward) and f (backward) all-reduces of
// "Megatron-LM: GPU-Cluster Training Parallelism", section "Paper 1: The f/g
// Conjugate Operators", done as a fixed-order in-GPU sum.  Column-parallel
// GEMMs (QKV, fc1) have no reduction; their bias / GeLU ride the epilogue
// (section "Fused Transformer Kernels").
//
// Kernel shape: persistent, one 384-thread CTA per SM, 128x256 output tile,
// K blocks of 64 in a 4-stage TMA ring (48 KB per stage, 128-byte swizzle).
//   warp 0       TMA producer (one thread)
//   warp 1       TMEM allocator and MMA issuer (one thread)
//   warps 2..3   idle
//   warps 4..11  epilogue: warp w reads TMEM lanes 32*(w%4).., columns
//                128*((w-4)/4).. of the tile
// Registers: the launch gives 168 per thread; the producer warpgroup (warps
// 0..3) drops to 40 and the two epilogue warpgroups rise to 232, which holds
// the 128 fp32 running partition sums per thread (40*128 + 232*256 = 168*384).
// The host launches the kernel only if it was compiled to exactly 168.
// TMEM holds two 128x256 fp32 accumulators (all 512 columns) so the epilogue
// of one work unit overlaps the MMAs of the next.  A work unit is one
// partition of one tile.  Operands may be K-major or MN-major (the backward's
// data and weight gradients read activations and weights transposed); MN-major
// tiles are loaded as 64-wide column boxes and described to the MMA with the
// leading byte offset stepping between them.
#include <cstring>

#include "gemm_core.cuh"

namespace mtl {
namespace tcg {

template <int EPI, bool OUT_F32, bool REDUCE>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmZ,
                   const Params p) {
  static_assert(SMEM_BYTES <= 232448, "shared memory of one CTA");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sA0 = smem_u32(smem);
  const uint32_t sB0 = sA0 + STAGES * A_BYTES;
  const uint32_t out_stage = sA0 + STAGES * STAGE_BYTES;   // 1024-aligned
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES + OUT_STAGING_BYTES);
  // bars[0..S): full, [S..2S): empty, [2S..2S+2): tmem full, [2S+2..2S+4): tmem empty
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 4);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + 2 + b); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), EPI_WARPS);
    }
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_shared();
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmC);
    if (EPI == EPI_BIAS_GELU) tma_prefetch_desc(&tmZ);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(PRODUCER_REGS));
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(EPILOGUE_REGS));
  }

  if (warp >= 4) {
    epilogue_role<EPI, OUT_F32, REDUCE, false, false, false>(p, tmem_base, tfull_bar(0), tempty_bar(0),
                                               abort_flag, warp, lane, blockIdx.x, gridDim.x, BM,
                                               0, &tmC, &tmZ, out_stage);
  } else if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      const int kb_per_tile = p.kb_per_unit * p.units_per_tile;
      bool ok = true;
      for (int tile = blockIdx.x; tile < p.num_tiles && ok; tile += gridDim.x) {
        int mb, nb;
        tile_coords(p, tile, mb, nb);
        for (int kb = 0; kb < kb_per_tile; ++kb) {
          if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, p.status, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t fb = full_bar(stage);
          mbar_arrive_expect_tx(fb, STAGE_BYTES);
          const int k0 = kb * BK;
          const uint32_t sa = sA0 + stage * A_BYTES, sb = sB0 + stage * B_BYTES;
          // K-major: one 64 (K) x BM / BN box; MN-major: 64 x 64 (K) boxes
          if (!p.a_mn) {
            const bounds::Box2 b = {p.K, p.M, BK, BM, 2};
            if (MTL_CHECKED(p.status, bounds::check_tma_load(b, k0, mb * BM), bounds::kSiteGemmA))
              tma_load_2d(sa, &tmA, fb, k0, mb * BM);
          } else {
#pragma unroll
            for (int j = 0; j < BM / 64; ++j) {
              const bounds::Box2 b = {p.M, p.K, 64, BK, 2};
              if (MTL_CHECKED(p.status, bounds::check_tma_load(b, mb * BM + 64 * j, k0),
                              bounds::kSiteGemmA))
                tma_load_2d(sa + j * (BK * 128), &tmA, fb, mb * BM + 64 * j, k0);
            }
          }
          if (!p.b_mn) {
            const bounds::Box2 b = {p.K, p.N, BK, BN, 2};
            if (MTL_CHECKED(p.status, bounds::check_tma_load(b, k0, nb * BN), bounds::kSiteGemmB))
              tma_load_2d(sb, &tmB, fb, k0, nb * BN);
          } else {
#pragma unroll
            for (int j = 0; j < BN / 64; ++j) {
              const bounds::Box2 b = {p.N, p.K, 64, BK, 2};
              if (MTL_CHECKED(p.status, bounds::check_tma_load(b, nb * BN + 64 * j, k0),
                              bounds::kSiteGemmB))
                tma_load_2d(sb + j * (BK * 128), &tmB, fb, nb * BN + 64 * j, k0);
            }
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(BM, BN, p.a_mn != 0, p.b_mn != 0);
      // K-major tiles: rows of 128 bytes, 8-row groups 1024 bytes apart; a
      // 16-deep K step moves 32 bytes along the row.  MN-major tiles: 64-wide
      // column boxes of BK rows (8 KB apart, the leading byte offset), 8-row
      // K groups 1024 bytes apart; a K step moves 16 rows = 2048 bytes.
      const uint32_t a_lbo = p.a_mn ? BK * 128 : 16, b_lbo = p.b_mn ? BK * 128 : 16;
      // base descriptors of stage 0; a stage or K step only moves the start
      // address field (in 16-byte units)
      const uint64_t a_desc0 = smem_desc_sw128(sA0, a_lbo, 1024);
      const uint64_t b_desc0 = smem_desc_sw128(sB0, b_lbo, 1024);
      const uint32_t a_kstep16 = p.a_mn ? 2048 / 16 : 32 / 16, b_kstep16 = p.b_mn ? 2048 / 16 : 32 / 16;
      int stage = 0;
      uint32_t phase = 0;
      int unit = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < p.num_tiles && ok; tile += gridDim.x) {
        for (int u = 0; u < p.units_per_tile && ok; ++u, ++unit) {
          const int buf = unit & 1;
          const uint32_t uphase = (unit >> 1) & 1;
          if (!mbar_wait_bounded(tempty_bar(buf), uphase ^ 1u, p.status, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + buf * BN;
          for (int kb = 0; kb < p.kb_per_unit; ++kb) {
            if (!mbar_wait_bounded(full_bar(stage), phase, p.status, abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t ad0 = a_desc0 + (uint64_t)(stage * (A_BYTES / 16));
            const uint64_t bd0 = b_desc0 + (uint64_t)(stage * (B_BYTES / 16));
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk)
              tc_mma_bf16(d_tmem, ad0 + kk * a_kstep16, bd0 + kk * b_kstep16, idesc,
                          (kb > 0 || kk > 0) ? 1u : 0u);
            tc_commit(empty_bar(stage));
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (ok) tc_commit(tfull_bar(buf));
        }
      }
    }
    __syncwarp();
  }

  __syncthreads();
  if (warp == 1) {
    if (*abort_flag) {
      // A role gave up on a wait (after ~2 s).  Copies and MMAs issued before
      // that finish in microseconds; pause ~1 ms so none is still writing
      // shared memory or TMEM when they are released.
      const long long t0 = clock64();
      while (clock64() - t0 < 2000000LL) {
      }
    }
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}


// K-major operand (rows x K): box 64 (K) x rows_box.  MN-major operand stored
// [K][MN]: box 64 (MN) x BK (K).
bool make_operand_map(CUtensorMap* m, const GemmOperand& op, int mn, int K, int box_rows) {
  if (op.k_major) return make_map(m, op.ptr, (uint64_t)K, (uint64_t)mn, op.ld, BK, box_rows);
  return make_map(m, op.ptr, (uint64_t)mn, (uint64_t)K, op.ld, 64, BK);
}

template <int EPI, bool F32, bool RED>
KernelFn kernel_ptr() {
  return reinterpret_cast<KernelFn>(gemm_tc_kernel<EPI, F32, RED>);
}

template <int EPI, bool F32, bool RED>
KernelFn kernel2_ptr() {
  return reinterpret_cast<KernelFn>(gemm_tc2_kernel<EPI, F32, RED, false>);
}

KernelFn select_kernel2(int epi, bool f32, bool red) {
#define SEL2(E)                                                                          \
  if (epi == E) {                                                                        \
    if (f32) return red ? kernel2_ptr<E, true, true>() : kernel2_ptr<E, true, false>();  \
    return red ? kernel2_ptr<E, false, true>() : kernel2_ptr<E, false, false>();         \
  }
  SEL2(EPI_STORE)
  SEL2(EPI_BIAS)
  SEL2(EPI_BIAS_RESID)
  SEL2(EPI_BIAS_GELU)
  SEL2(EPI_DGELU)
#undef SEL2
  return nullptr;
}

KernelFn select_kernel(int epi, bool f32, bool red) {
#define SEL(E)                                                                         \
  if (epi == E) {                                                                      \
    if (f32) return red ? kernel_ptr<E, true, true>() : kernel_ptr<E, true, false>();  \
    return red ? kernel_ptr<E, false, true>() : kernel_ptr<E, false, false>();         \
  }
  SEL(EPI_STORE)
  SEL(EPI_BIAS)
  SEL(EPI_BIAS_RESID)
  SEL(EPI_BIAS_GELU)
  SEL(EPI_DGELU)
#undef SEL
  return nullptr;
}

}  // namespace tcg

size_t gemm_split_bytes(int M, int N, int num_sms) {
  using namespace tcg;
  const int tiles = ((M + 2 * P_HALF - 1) / (2 * P_HALF)) * ((N + BN - 1) / BN);
  size_t bytes, counters;
  split_scratch_for(tiles, num_sms / 2, &bytes, &counters);
  return bytes;
}

size_t gemm_split_counters(int M, int N, int num_sms) {
  using namespace tcg;
  const int tiles = ((M + 2 * P_HALF - 1) / (2 * P_HALF)) * ((N + BN - 1) / BN);
  size_t bytes, counters;
  split_scratch_for(tiles, num_sms / 2, &bytes, &counters);
  return counters;
}

bool gemm_tc_supported(const GemmArgs& a) {
  if (a.parts < 1 || a.K % a.parts) return false;
  const int kpart = a.K / a.parts;
  if (a.parts > 1 && kpart % tcg::BK) return false;
  auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  if (!al16(a.A.ptr) || !al16(a.B.ptr) || !al16(a.C)) return false;
  if ((a.A.ld % 8) || (a.B.ld % 8) || (a.ldc % 8)) return false;
  if (a.epi == EPI_BIAS_RESID && ((a.ldr % 8) || !al16(a.R))) return false;
  if ((a.epi == EPI_BIAS_GELU || a.epi == EPI_DGELU) && ((a.ldz % 8) || !al16(a.Z))) return false;
  if ((a.epi == EPI_BIAS || a.epi == EPI_BIAS_RESID || a.epi == EPI_BIAS_GELU) && !al16(a.bias))
    return false;
  return true;
}

cudaError_t gemm_tc(const GemmArgs& a, const LaunchCtx& c) {
  using namespace tcg;
  if (a.M == 0 || a.N == 0) return cudaSuccess;
  if (!gemm_tc_supported(a)) return cudaErrorInvalidValue;
  // The pair kernel needs K partitions that are whole 128-deep stages.
  const bool use_pair = c.num_sms >= 2 && (a.parts == 1 || (a.K / a.parts) % P_BK == 0);
  CUtensorMap ma, mb;
  if (use_pair) {
    // every box is 64 wide and 128 deep (K-major: 128 rows of 64 K; MN-major:
    // 128 K rows of 64 M or N)
    auto pmap = [](CUtensorMap* m, const GemmOperand& op, int mn, int K) {
      return op.k_major ? make_map(m, op.ptr, (uint64_t)K, (uint64_t)mn, op.ld, 64, 128)
                        : make_map(m, op.ptr, (uint64_t)mn, (uint64_t)K, op.ld, 64, 128);
    };
    if (!pmap(&ma, a.A, a.M, a.K) || !pmap(&mb, a.B, a.N, a.K)) return cudaErrorInvalidValue;
  } else if (!make_operand_map(&ma, a.A, a.M, a.K, BM) ||
             !make_operand_map(&mb, a.B, a.N, a.K, BN)) {
    return cudaErrorInvalidValue;
  }
  CUtensorMap mc, mz;
  if (!make_epilogue_maps(&mc, &mz, a)) return cudaErrorInvalidValue;
  Params p;
  memset(&p, 0, sizeof(p));   // no FP8 scales: the epilogue's descale is 1
  p.M = a.M;
  p.N = a.N;
  p.K = a.K;
  p.parts = a.parts;
  const bool reduce = a.parts > 1;
  const int bk = use_pair ? P_BK : BK;
  const int tile_m = use_pair ? 2 * P_HALF : BM;
  const int nkb = (a.K + bk - 1) / bk;
  p.units_per_tile = reduce ? a.parts : 1;
  p.kb_per_unit = reduce ? (a.K / a.parts) / bk : nkb;
  p.a_mn = a.A.k_major ? 0 : 1;
  p.b_mn = a.B.k_major ? 0 : 1;
  p.tiles_m = (a.M + tile_m - 1) / tile_m;
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
  plan_split(p, reduce, use_pair ? c.num_sms / 2 : c.num_sms, use_pair, a);
  KernelFn fn = !use_pair          ? select_kernel(a.epi, a.c_f32, reduce)
                : p.split_s > 1    ? select_kernel2_split(a.epi, a.c_f32, reduce)
                                   : select_kernel2(a.epi, a.c_f32, reduce);
  if (!fn) return cudaErrorInvalidValue;
  const int smem_bytes = use_pair ? P_SMEM_BYTES : SMEM_BYTES;
  cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void*>(fn),
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
  if (e != cudaSuccess) return e;
  // The warpgroup register split assumes exactly LAUNCH_REGS registers per
  // thread at launch; with fewer, setmaxnreg.inc could never be satisfied.
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, reinterpret_cast<const void*>(fn));
  if (e != cudaSuccess) return e;
  if (fa.numRegs != LAUNCH_REGS) return cudaErrorInvalidConfiguration;
  if (p.kb_per_unit == 0) {
    // K == 0: nothing to accumulate; the kernel is not launched
    return cudaErrorInvalidValue;
  }
  int grid;
  if (use_pair) {
    const int pairs = c.num_sms / 2;
    grid = 2 * (p.num_tiles < pairs ? p.num_tiles : pairs);
  } else {
    grid = p.num_tiles < c.num_sms ? p.num_tiles : c.num_sms;
  }
  c.before(KK_GEMM_TC, 2.0 * a.M * a.N * a.K);
  fn<<<grid, THREADS, smem_bytes, c.stream>>>(ma, mb, mc, mz, p);
  c.after();
  return cudaGetLastError();
}

}  // namespace mtl
