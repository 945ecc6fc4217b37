// Causal flash attention on tcgen05 tensor cores (bf16 in, fp32 accumulate),
// forward and a deterministic two-kernel backward.
//
// Each head is local to its partition: Q, K and V of head `hd` are the three
// d-wide column blocks at hd*3d of the head-interleaved qkv activation ("Megatron-
// LM: GPU-Cluster Training Parallelism", section "Paper 1: QKV Column-Parallel
// Splitting in Detail"), so the kernels read them straight from qkv with TMA
// boxes -- no transpose kernel (section "Fused Transformer Kernels": layout
// change instead of transposes, fused scale-mask-softmax).
//
//   S = Q K^T / sqrt(d), keys after the query excluded, P = softmax(S), O = P V,
//   lse = log sum exp(S) per query row.
//   Backward: D_i = sum_c dO_ic O_ic;  dS = P * (dO V^T - D);  dQ = dS K / sqrt d;
//   dK = dS^T Q / sqrt d;  dV = P^T dO.
// With attention dropout (keep mask M from the Philox stream, scale 1/(1-p)):
//   O = (P * M / (1-p)) V, lse still that of the undropped P;
//   dV = (P * M / (1-p))^T dO;  dS = P * ((dO V^T) * M / (1-p) - D).
// The forward draws M and stores it as bits (one bit per causal element, an
// eighth of a bf16 P); the two backward kernels read the bits instead of
// drawing again, which trades 2 of 3 Philox passes for a few MB of traffic.
//
// All three kernels are persistent (one CTA per SM) with warp roles:
//   warp 0      TMA producer
//   warp 1      TMEM allocator, MMA issuer
//   the rest    row threads: thread (warp%4)*32+lane owns TMEM lane = one row of
//               a 128-row block.
// Operand tiles are [atoms][rows][64] 128-byte-swizzled boxes straight from TMA;
// the same box serves as a K-major operand (rows = M/N) or an MN-major one
// (rows = K), e.g. dO is the K-major B of dO V^T and the MN-major B of P^T dO.
// P and dS go from registers to shared memory in the same swizzled layout.
// Every wait is bounded; a timeout is recorded in the status word.
#include "common.cuh"
#include "kernels.h"

namespace mtl {
namespace attn {

constexpr int FWD_THREADS = 384;   // forward kernel: 4 control warps, two warpgroups of row threads
constexpr int BWD_THREADS = 384;   // backward kernels: two warpgroups of row threads
constexpr int ATOM128 = 128 * 128;   // [128 rows][64 bf16]
constexpr int ATOM64 = 64 * 128;     // [64 rows][64 bf16]
constexpr int BWD_STAGES = 3;      // TMA ring depth of the backward kernels
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;

struct Params {
  int batch, seq, heads, d, h, nqb;
  float scale_log2;   // log2(e) / sqrt(d)
  float scale;        // 1 / sqrt(d)
  bf16* ctx;          // fwd out / bwd in (O)
  float* lse;
  const bf16* dctx;   // dO
  bf16* dqkv;
  float* dsum;
  unsigned* status;
  Dropout drop;       // attention dropout: element (query i, key j) of head hd, batch b
                      // is e = ((b * heads + hd) * seq + i) * seq + j
  uint32_t* mask;     // keep bits written by the forward, read by the backward
  unsigned* sched;    // work counter pair {next item, CTAs done}: zero before the launch,
                      // reset to zero by the last CTA
  int chunk;          // (batch, head) pairs per scheduling chunk of the forward
};

// Keep bits of the forward, one 2 KB tile per (batch, head, query block qb, key
// block kb <= qb) of 128 x 128: tiles of a (batch, head) pair in the order
// qb (qb + 1) / 2 + kb; inside a tile, word w (keys 32w .. 32w+31 of the block,
// bit = key % 32) of row r sits at w * 128 + r, so a warp's 32 rows are 128
// contiguous bytes.
__device__ __forceinline__ uint32_t* mask_tile(const Params& p, int b, int hd, int qb, int kb) {
  const size_t ntile = (size_t)p.nqb * (p.nqb + 1) / 2;
  return p.mask + (((size_t)b * p.heads + hd) * ntile + (size_t)qb * (qb + 1) / 2 + kb) * 512;
}

// 32 x 32 bit transpose across a warp: on entry lane l holds row l (bit k =
// element (l, k)); on exit lane k holds column k (bit l = element (l, k)).
// Five exchange stages swap the off-diagonal halves of ever smaller blocks.
__device__ __forceinline__ uint32_t warp_transpose32(uint32_t w, int lane) {
#pragma unroll
  for (int j = 16, i = 0; j >= 1; j >>= 1, ++i) {
    const uint32_t m = i == 0 ? 0x0000FFFFu : i == 1 ? 0x00FF00FFu : i == 2 ? 0x0F0F0F0Fu
                     : i == 3 ? 0x33333333u : 0x55555555u;
    const uint32_t o = __shfl_xor_sync(0xffffffffu, w, j);
    w = (lane & j) ? ((w & ~m) | ((o >> j) & m)) : ((w & m) | ((o << j) & ~m));
  }
  return w;
}

// First element index of query row i, head hd, batch b in the attention
// dropout numbering.
__device__ __forceinline__ unsigned long long drop_row(const Params& p, int b, int hd, int i) {
  return (((unsigned long long)b * p.heads + hd) * p.seq + i) * (unsigned long long)p.seq;
}

struct Smem {
  uint8_t* base;
  uint32_t u32;
};

__device__ __forceinline__ Smem smem_aligned(uint8_t* raw) {
  uint8_t* p = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) &
                                          ~static_cast<uintptr_t>(1023));
  return {p, smem_u32(p)};
}

// Work item -> (row block, head, batch) for the persistent kernels.  Items go
// (batch, head)-major, so the items running at once on all SMs cover few pairs
// and reuse each other's K/V from L2; within a pair the row block index is
// rotated by the pair index, so a CTA that takes every gridDim-th item meets
// every row block (and so every amount of causal work) in turn.
__device__ __forceinline__ void item_coords(const Params& p, int item, bool desc, int& blk,
                                            int& hd, int& b) {
  const int pair = item / p.nqb;
  const int i = (item % p.nqb + pair) % p.nqb;
  blk = desc ? (p.nqb - 1 - i) : i;
  hd = pair % p.heads;
  b = pair / p.heads;
}

// ============================================================================ forward
// Persistent: one CTA per SM takes (query pair, head, batch) work items from a
// global counter.  An item is 256 queries as two tiles of 128 rows, A (rows
// 0..127) and B (rows 128..255).  Each tile has a warpgroup of row threads
// (a thread owns one query row and all 128 keys of a block, so row maxima and
// sums stay in registers) and its own P and O in TMEM.  K and V blocks of 128
// keys stream through one TMA ring that both tiles read.  The S buffer in
// TMEM serves the tiles in turn, S uses A(0) B(0) A(1) B(1) ...: the next
// turn's Q K^T runs on the tensor cores while the previous owner computes its
// exponentials.  A warpgroup writes its bf16 P block into TMEM,
// where the PV MMA reads it as the A operand; nothing in TMEM is written by
// an MMA while another MMA may still read it.
// Causal: tile A of query pair q reads key blocks 0..2q, tile B 0..2q+1 (the
// last one is the diagonal block of each); with seq % 256 == 128 the last
// pair has no tile B.
// Items go longest first within chunks of (batch, head) pairs whose K/V fit
// in L2 together, so K/V come from HBM about once and the launch ends on
// short items.
// Warps: 0 scheduler and TMA producer, 1 TMEM allocator and Q K^T issuer, 2 P V
// issuer, 3 register donor, 4..7 row threads of tile A, 8..11 of tile B.  The
// two MMA streams touch disjoint TMEM columns and each commit tracks only its
// own thread's MMAs, so neither issuer waits on the other's dependencies.
// smem: Q_A, Q_B, ring[FWD_RING] (NA atoms of 16 KB each), item ids.
// TMEM: S cols 0..127, P_A 128..191, P_B 192..255, O_A 256.., O_B 384..
constexpr int FWD_RING = 4;
static_assert(FWD_RING % 2 == 0, "K and V must keep to their own ring slots");
constexpr uint32_t TM_S = 0, TM_P = 128, TM_O = 256;
// Register split: warps 0..3 (producer, MMA issuer, two idle) give registers
// to the row warps 4..11, which hold a 128-key score row each.  The split is
// balanced on every SM sub-partition (warp w runs on sub-partition w % 4: one
// giving warp and two taking warps on each), since setmaxnreg.inc waits, with
// no bound, for registers released on its own sub-partition.
constexpr int FWD_LAUNCH_REGS = 168, FWD_LOW_REGS = 56, FWD_ROW_REGS = 224;
static_assert(FWD_THREADS == 384, "one giving and two taking warps per sub-partition");
static_assert(FWD_LOW_REGS + 2 * FWD_ROW_REGS <= 3 * FWD_LAUNCH_REGS,
              "register split exceeds a sub-partition's launch allocation");

struct FwdItem {
  int qp, hd, b;
  int n0, n1;   // key blocks of tile A / tile B (0: tile absent)
  __device__ __forceinline__ int n(int x) const { return x ? n1 : n0; }
};

__device__ __forceinline__ FwdItem fwd_item(const Params& p, int k) {
  const int nq2 = (p.nqb + 1) >> 1;
  const int pairs = p.batch * p.heads;
  const int per_chunk = p.chunk * nq2;
  const int c = k / per_chunk;
  const int cp = min(p.chunk, pairs - c * p.chunk);   // pairs in this chunk
  const int r = k - c * per_chunk;
  const int pair = c * p.chunk + r % cp;
  FwdItem it;
  it.qp = nq2 - 1 - r / cp;
  it.hd = pair % p.heads;
  it.b = pair / p.heads;
  it.n0 = 2 * it.qp + 1;
  it.n1 = 2 * it.qp + 1 < p.nqb ? 2 * it.qp + 2 : 0;
  return it;
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// Two fp32 lanes in one instruction: (a0, a1) * (b0, b1) + (c0, c1), and a sum.
__device__ __forceinline__ void ffma2(float& d0, float& d1, float a0, float a1, float b0, float b1,
                                      float c0, float c1) {
  unsigned long long ra, rb, rc, rd;
  asm("mov.b64 %0, {%1, %2};" : "=l"(ra) : "f"(a0), "f"(a1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(rb) : "f"(b0), "f"(b1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(rc) : "f"(c0), "f"(c1));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(rd) : "l"(ra), "l"(rb), "l"(rc));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(d0), "=f"(d1) : "l"(rd));
}
__device__ __forceinline__ void fadd2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
  unsigned long long ra, rb, rd;
  asm("mov.b64 %0, {%1, %2};" : "=l"(ra) : "f"(a0), "f"(a1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(rb) : "f"(b0), "f"(b1));
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(rd) : "l"(ra), "l"(rb));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(d0), "=f"(d1) : "l"(rd));
}

template <int NA, int KS, bool DROP>
__global__ void __launch_bounds__(FWD_THREADS, 1)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  const Smem sm = smem_aligned(smem_raw);
  constexpr uint32_t TILE = NA * ATOM128;
  constexpr int D = KS * 16;
  const uint32_t sQ0 = sm.u32, sR0 = sQ0 + 2 * TILE;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm.base + (2 + FWD_RING) * TILE);
  const uint32_t bar0 = smem_u32(bars);
  auto B = [&](int i) { return bar0 + 8u * i; };
  // barriers; per-tile ones come in pairs (A, B), item ones in pairs (slot 0, 1)
  // (a barrier waited on by several threads at different progress must never
  // get two completions ahead of any of them: hence S-full per tile)
  constexpr int QF = 0, QE = 2, RF = 4, RE = RF + FWD_RING, SF = RE + FWD_RING, SE = SF + 2,
                PF = SE + 1, PE = PF + 2, IF = PE + 2, IE = IF + 2, NBAR = IE + 2;
  constexpr int ROW_WARPS = FWD_THREADS / 32 - 4;
  int* s_item = reinterpret_cast<int*>(bars + NBAR);   // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(s_item + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_items = ((p.nqb + 1) >> 1) * p.heads * p.batch;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NBAR; ++i) {
      uint32_t cnt = 1;
      if (i == SE || i == PF || i == PF + 1) cnt = 128;
      if (i == IE || i == IE + 1) cnt = 2 + ROW_WARPS;   // 2 MMA issuers + a lane per row warp
      mbar_init(B(i), cnt);
    }
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_shared();
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------ scheduler, TMA producer
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(FWD_LOW_REGS));
    if (lane == 0) {
      tma_prefetch_desc(&tm);
      int g = 0, ni = 0, nit0 = 0, nit1 = 0;
      bool ok = true;
      while (ok) {
        const int slot = ni & 1;
        if (ni >= 2 &&
            !mbar_wait_bounded(B(IE + slot), ((ni >> 1) - 1) & 1, p.status, abort_flag))
          break;
        const int k = (int)atomicAdd(p.sched, 1u);
        s_item[slot] = k;
        mbar_arrive(B(IF + slot));
        ++ni;
        if (k >= n_items) break;
        const FwdItem it = fwd_item(p, k);
        const int colq = it.hd * 3 * p.d, row0 = it.b * p.seq;
        for (int x = 0; x < 2 && ok; ++x) {
          if (!it.n(x)) continue;
          const int nq = x ? nit1++ : nit0++;
          if (nq > 0 && !mbar_wait_bounded(B(QE + x), (nq - 1) & 1, p.status, abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(B(QF + x), TILE);
          for (int a = 0; a < NA; ++a)
            tma_load_2d(sQ0 + x * TILE + a * ATOM128, &tm, B(QF + x), colq + 64 * a,
                        row0 + it.qp * 256 + x * 128);
        }
        const int nkv = it.n0 > it.n1 ? it.n0 : it.n1;
        for (int j = 0; j < nkv && ok; ++j) {
          for (int kv = 0; kv < 2; ++kv, ++g) {
            const int s = g % FWD_RING, use = g / FWD_RING;
            if (use > 0 && !mbar_wait_bounded(B(RE + s), (use - 1) & 1, p.status, abort_flag)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(B(RF + s), TILE);
            for (int a = 0; a < NA; ++a)
              tma_load_2d(sR0 + s * TILE + a * ATOM128, &tm, B(RF + s),
                          colq + (1 + kv) * p.d + 64 * a, row0 + j * 128);
          }
        }
      }
      // the last CTA out leaves the counters at zero for the next launch
      __threadfence();
      if (atomicAdd(p.sched + 1, 1u) == gridDim.x - 1) {
        atomicExch(p.sched, 0u);
        atomicExch(p.sched + 1, 0u);
      }
    }
    __syncwarp();
  } else if (warp == 1 || warp == 2) {
    // ------------------------------------------ MMA issuers: warp 1 Q K^T, warp 2 P V
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(FWD_LOW_REGS));
    if (lane == 0) {
      const bool is_qk = warp == 1;
      const uint32_t id_qk = idesc_bf16_f32(128, 128, false, false);
      const uint32_t id_pv = idesc_bf16_f32(128, D, false, true);
      const uint64_t dQ0 = desc_kbase(sQ0), dR0 = desc_kbase(sR0);
      const uint64_t dRmn0 = desc_mnbase(sR0, ATOM128);
      int g = 0, su = 0, ni = 0;        // ring loads, S uses and items before this item
      int npv0 = 0, npv1 = 0, nit0 = 0, nit1 = 0;
      int ring_seen = -1;               // last ring load this thread waited for
      bool ok = true;
      auto wait = [&](int bar, int k) -> bool {   // completion k (0-based) of barrier `bar`
        if (!mbar_wait_bounded(B(bar), k & 1, p.status, abort_flag)) ok = false;
        return ok;
      };
      // ring load gi (K(j) = g + 2j, V(j) = g + 2j + 1) is in shared memory; with an
      // even ring each slot only ever holds K or only V, so it has a single waiter
      auto wait_ring = [&](int gi) -> bool {
        if (gi <= ring_seen) return true;
        ring_seen = gi;
        return wait(RF + gi % FWD_RING, gi / FWD_RING);
      };
      while (ok) {
        const int slot = ni & 1;
        if (!wait(IF + slot, ni >> 1)) break;
        const int k = *reinterpret_cast<volatile int*>(&s_item[slot]);
        mbar_arrive(B(IE + slot));
        ++ni;
        if (k >= n_items) break;
        const FwdItem it = fwd_item(p, k);
        const int nuse = it.n0 + it.n1;
        const bool last_b = it.n1 > 0;           // tile B is the last reader of K and V
        for (int v = 0; v < nuse && ok; ++v) {
          // S use v -> tile x, key block j: A(0) B(0) A(1) B(1) ... [B(n0)]
          int x, j;
          if (!last_b) {
            x = 0;
            j = v;
          } else if (v < 2 * it.n0) {
            x = v & 1;
            j = v >> 1;
          } else {
            x = 1;
            j = v - it.n0;
          }
          if (is_qk) {
            // S = Q_X K(j)^T once the previous S use has been read
            const int gk = g + 2 * j, s = gk % FWD_RING;
            if (j == 0 && !wait(QF + x, x ? nit1 : nit0)) break;
            if (!wait_ring(gk)) break;
            if (su + v > 0 && !wait(SE, su + v - 1)) break;
            tc_fence_after();
            const uint64_t dQ = desc_add(dQ0, x * TILE), dK = desc_add(dR0, s * TILE);
#pragma unroll
            for (int kk = 0; kk < KS; ++kk)
              tc_mma_bf16(tmem + TM_S, desc_add(dQ, kmajor_off(kk, ATOM128)),
                          desc_add(dK, kmajor_off(kk, ATOM128)), id_qk, kk > 0);
            tc_commit(B(SF + x));
            if (j == it.n(x) - 1) tc_commit(B(QE + x));
            if (x == 1 || !last_b) tc_commit(B(RE + s));
          } else {
            // O_X (+)= P_X V(j), P_X read from TMEM
            // (PF_X of a tile's first block also means its last epilogue read O_X)
            const int gv = g + 2 * j + 1, s = gv % FWD_RING;
            if (!wait(PF + x, x ? npv1 : npv0)) break;
            if (!wait_ring(gv)) break;
            tc_fence_after();
            const uint64_t dV = desc_add(dRmn0, s * TILE);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              tc_mma_bf16_ts(tmem + TM_O + 128 * x, tmem + TM_P + 64 * x + 8 * kk,
                             desc_add(dV, mnmajor_off(kk)), id_pv, (j > 0 || kk > 0) ? 1u : 0u);
            tc_commit(B(PE + x));
            if (x) ++npv1; else ++npv0;
            if (x == 1 || !last_b) tc_commit(B(RE + s));
          }
        }
        if (!ok) break;
        g += 2 * (it.n0 > it.n1 ? it.n0 : it.n1);
        su += nuse;
        if (it.n0) ++nit0;
        if (it.n1) ++nit1;
      }
    }
    __syncwarp();
  } else if (warp == 3) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(FWD_LOW_REGS));
  } else {
    // ---------------------------------------------------------------- row threads
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(FWD_ROW_REGS));
    const int x = (warp - 4) >> 2;                 // tile
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;                  // row = TMEM lane
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    const uint32_t tS = tmem + TM_S + lane_off, tP = tmem + TM_P + 64 * x + lane_off;
    const uint32_t tO = tmem + TM_O + 128 * x + lane_off;
    int cnt = 0, ni = 0;           // blocks of this tile so far, items read
    // A tile's epilogue (O / l to ctx, lse) runs when the tile's next item has
    // its first P block computed: the last PV of the item is done by then, and
    // PV_X(0) of the next item waits for that P block, so O_X is read first.
    bool pend = false;
    float pm = 0.f, pl = 1.f;
    size_t po = 0, plse = 0;       // ctx offset of the row's head slice, lse index
    auto epilogue = [&]() {
      const float inv = (DROP ? p.drop.scale : 1.0f) / pl;
      bf16* orow = p.ctx + po;
#pragma unroll 1
      for (int c = 0; c < D; c += 32) {   // one 32-column chunk live at a time
        uint32_t v[32];
        tmem_ld32(tO + c, v);
        tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint4 w;
          w.x = pack_bf16x2(__uint_as_float(v[q * 8 + 0]) * inv, __uint_as_float(v[q * 8 + 1]) * inv);
          w.y = pack_bf16x2(__uint_as_float(v[q * 8 + 2]) * inv, __uint_as_float(v[q * 8 + 3]) * inv);
          w.z = pack_bf16x2(__uint_as_float(v[q * 8 + 4]) * inv, __uint_as_float(v[q * 8 + 5]) * inv);
          w.w = pack_bf16x2(__uint_as_float(v[q * 8 + 6]) * inv, __uint_as_float(v[q * 8 + 7]) * inv);
          *reinterpret_cast<uint4*>(orow + c + q * 8) = w;
        }
      }
      p.lse[plse] = (pm + __log2f(pl)) * LN2;
    };
    bool ok = true;
    while (ok) {
      const int slot = ni & 1;
      if (!mbar_wait_bounded(B(IF + slot), (ni >> 1) & 1, p.status, abort_flag)) {
        ok = false;
        break;
      }
      const int k = *reinterpret_cast<volatile int*>(&s_item[slot]);
      __syncwarp();
      if (lane == 0) mbar_arrive(B(IE + slot));
      ++ni;
      if (k >= n_items) break;
      const FwdItem it = fwd_item(p, k);
      const int nx = it.n(x);
      const int qb = 2 * it.qp + x;                // 128-row query block of this tile
      float m_used = -INFINITY, l = 0.f;
      for (int j = 0; j < nx; ++j) {
        uint32_t keep[4] = {0xffffffffu, 0xffffffffu, 0xffffffffu, 0xffffffffu};
        if (DROP) {
          // keep bits of this row's 128 keys, drawn before S arrives
          const unsigned long long e0 = drop_row(p, it.b, it.hd, qb * 128 + r) + j * 128;
          uint32_t* mt = mask_tile(p, it.b, it.hd, qb, j);
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            keep[w] = drop_bits32(e0 + 32 * w, p.drop);
            mt[w * 128 + r] = keep[w];
          }
        }
        if (!mbar_wait_bounded(B(SF + x), cnt & 1, p.status, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        float s[128];
        {
          uint32_t v0[32], v1[32], v2[32], v3[32];
          tmem_ld32(tS, v0);
          tmem_ld32(tS + 32, v1);
          tmem_ld32(tS + 64, v2);
          tmem_ld32(tS + 96, v3);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            s[i] = __uint_as_float(v0[i]);
            s[32 + i] = __uint_as_float(v1[i]);
            s[64 + i] = __uint_as_float(v2[i]);
            s[96 + i] = __uint_as_float(v3[i]);
          }
        }
        tc_fence_before();
        mbar_arrive(B(SE));                        // the S buffer may take the next turn
        if (j == nx - 1) {                         // diagonal block: keys after the query
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c > r) s[c] = -INFINITY;
        }
        float mxa[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          float a = fmax3(s[q], s[q + 8], s[q + 16]);
#pragma unroll
          for (int t = 3; t < 15; t += 2) a = fmax3(a, s[q + 8 * t], s[q + 8 * t + 8]);
          mxa[q] = fmaxf(a, s[q + 120]);
        }
        const float mx = fmax3(fmax3(mxa[0], mxa[1], mxa[2]), fmax3(mxa[3], mxa[4], mxa[5]),
                               fmaxf(mxa[6], mxa[7]));
        const float m_new = fmaxf(m_used, mx * p.scale_log2);
        // Rescale only when the running maximum grew by more than 2^8: the
        // exponentials stay below 256 and the final O / l is exact either way.
        const bool resc = m_new > m_used + 8.0f;
        const float alpha = resc ? fast_exp2(m_used - m_new) : 1.0f;
        if (resc) m_used = m_new;
        const float neg = -m_used;
        // P_X and O_X are free once the previous PV of this tile is done
        if (cnt > 0 && !mbar_wait_bounded(B(PE + x), (cnt - 1) & 1, p.status, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (j == 0 && pend) {
          epilogue();
          pend = false;
        }
        // exponentials and row sum a 32-key chunk at a time, each chunk's bf16
        // P stored into TMEM while the next one is computed
        float rs[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) rs[q] = 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
#pragma unroll
          for (int c = 32 * q; c < 32 * q + 32; c += 2) {
            ffma2(s[c], s[c + 1], s[c], s[c + 1], p.scale_log2, p.scale_log2, neg, neg);
            s[c] = fast_exp2(s[c]);
            s[c + 1] = fast_exp2(s[c + 1]);
            const int e = (c >> 1) & 3;
            fadd2(rs[2 * e], rs[2 * e + 1], rs[2 * e], rs[2 * e + 1], s[c], s[c + 1]);
          }
          if (DROP) {
            // dropped probabilities leave the row sum but not P V
#pragma unroll
            for (int c = 0; c < 32; ++c)
              if (!((keep[q] >> c) & 1u)) s[32 * q + c] = 0.f;
          }
          uint32_t pk[16];
#pragma unroll
          for (int c = 0; c < 16; ++c) pk[c] = pack_bf16x2(s[32 * q + 2 * c], s[32 * q + 2 * c + 1]);
          tmem_st16(tP + 16 * q, pk);
        }
        l = l * alpha + (((rs[0] + rs[1]) + (rs[2] + rs[3])) + ((rs[4] + rs[5]) + (rs[6] + rs[7])));
        if (j > 0 && __any_sync(0xffffffffu, resc)) {
          // O_X *= alpha before PV_X(j) (rare)
#pragma unroll
          for (int c = 0; c < D; c += 32) {
            uint32_t v[32];
            tmem_ld32(tO + c, v);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
            tmem_st32(tO + c, v);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(B(PF + x));
        ++cnt;
      }
      if (!ok) break;
      if (nx) {
        pend = true;
        pm = m_used;
        pl = l;
        po = (size_t)(it.b * p.seq + qb * 128 + r) * p.h + (size_t)it.hd * D;
        plse = ((size_t)it.b * p.heads + it.hd) * p.seq + qb * 128 + r;
      }
    }
    if (ok && pend) {
      if (mbar_wait_bounded(B(PE + x), (cnt - 1) & 1, p.status, abort_flag)) {
        tc_fence_after();
        epilogue();
      }
    }
    __syncwarp();
  }
  __syncthreads();
  if (warp == 1) {
    if (*abort_flag) {
      const long long t0 = clock64();
      while (clock64() - t0 < 2000000LL) {
      }
    }
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ============================================================================ dQ
// Persistent: one CTA per SM walks the query-block work items.  Per item: 128
// queries; K/V blocks of 64 keys in a BWD_STAGES-deep ring that runs on across
// items.  S and dP are double-buffered in TMEM (the MMAs of block j+2 run while
// the row threads work on block j), and so is the dQ accumulator (an item's
// epilogue overlaps the next item's MMAs).  Two warpgroups of row threads each
// take 32 of the 64 key columns.  Also writes D_i = sum_c dO_ic O_ic for the
// dK/dV kernel.
// smem: Q, dO (NA atoms of 16 KB), K[ST], V[ST] (NA atoms of 8 KB), dS (1 atom
// of 16 KB), D exchange.  TMEM: S[b] cols 64b, dP[b] cols 128+64b, dQ[b] cols
// 256+128b.
template <int NA, int KS, bool DROP>
__global__ void __launch_bounds__(BWD_THREADS, 1)
    attn_bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap tm128,
                          const __grid_constant__ CUtensorMap tm64,
                          const __grid_constant__ CUtensorMap tmdo128, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  const Smem sm = smem_aligned(smem_raw);
  constexpr uint32_t T128 = NA * ATOM128, T64 = NA * ATOM64;
  constexpr int ST = BWD_STAGES;
  const uint32_t sQ = sm.u32, sDO = sQ + T128, sK0 = sQ + 2 * T128, sV0 = sK0 + ST * T64,
                 sDS = sV0 + ST * T64;
  float* s_dpart = reinterpret_cast<float*>(sm.base + 2 * T128 + 2 * ST * T64 + ATOM128);
  uint64_t* bars =
      reinterpret_cast<uint64_t*>(sm.base + 2 * T128 + 2 * ST * T64 + ATOM128 + 2048);
  const uint32_t bar0 = smem_u32(bars);
  auto B = [&](int i) { return bar0 + 8u * i; };
  // 0 q/do full, 1 q/do empty, 2..ST+1 kv_full, ST+2..2ST+1 kv_empty,
  // then s_full[2], ds_full, dq_done, dq_free[2], d_exchange
  const int QF = 0, QE = 1, KVF = 2, KVE = 2 + ST, SF = 2 + 2 * ST, DSF = 4 + 2 * ST,
            DQD = 5 + 2 * ST, DQFREE = 6 + 2 * ST, DXB = 8 + 2 * ST, NBAR = 9 + 2 * ST;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NBAR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_items = p.nqb * p.heads * p.batch;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NBAR; ++i) {
      const bool rows = i == DSF || i == DQFREE || i == DQFREE + 1 || i == DXB;
      mbar_init(B(i), rows ? 256 : 1);
    }
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_shared();
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS = tmem, tDP = tmem + 128;

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&tm128);
      tma_prefetch_desc(&tm64);
      tma_prefetch_desc(&tmdo128);
      int g = 0, n = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x, ++n) {
        int qb, hd, b;
        item_coords(p, item, true, qb, hd, b);
        const int colq = hd * 3 * p.d;
        const int row0 = b * p.seq + qb * 128;
        if (!mbar_wait_bounded(B(QE), (n & 1) ^ 1u, p.status, abort_flag)) break;
        mbar_arrive_expect_tx(B(QF), 2 * T128);
        for (int a = 0; a < NA; ++a) {
          tma_load_2d(sQ + a * ATOM128, &tm128, B(QF), colq + 64 * a, row0);
          tma_load_2d(sDO + a * ATOM128, &tmdo128, B(QF), hd * p.d + 64 * a, row0);
        }
        const int nkv = 2 * qb + 2;
        for (int j = 0; j < nkv; ++j, ++g) {
          const int s = g % ST;
          const int krow = b * p.seq + j * 64;
          if (!mbar_wait_bounded(B(KVE + s), ((g / ST) & 1) ^ 1u, p.status, abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(B(KVF + s), 2 * T64);
          for (int a = 0; a < NA; ++a) {
            tma_load_2d(sK0 + s * T64 + a * ATOM64, &tm64, B(KVF + s), colq + p.d + 64 * a, krow);
            tma_load_2d(sV0 + s * T64 + a * ATOM64, &tm64, B(KVF + s), colq + 2 * p.d + 64 * a,
                        krow);
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t id_s = idesc_bf16_f32(128, 64, false, false);
      const uint32_t id_dq = idesc_bf16_f32(128, p.d, false, true);
      const uint64_t dQd = desc_kbase(sQ), dDO = desc_kbase(sDO), dK0 = desc_kbase(sK0),
                     dV0 = desc_kbase(sV0), dDS = desc_kbase(sDS);
      const uint64_t dKmn0 = desc_mnbase(sK0, ATOM64);
      int gb = 0, n = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x, ++n) {
        int qb, hd, b;
        item_coords(p, item, true, qb, hd, b);
        const int nkv = 2 * qb + 2;
        if (!mbar_wait_bounded(B(QF), n & 1, p.status, abort_flag)) break;
        tc_fence_after();
        // S(block gg), dP(block gg) into TMEM buffer gg % 2
        auto issue_s = [&](int j) -> bool {
          const int gg = gb + j, s = gg % ST;
          if (!mbar_wait_bounded(B(KVF + s), (gg / ST) & 1, p.status, abort_flag)) return false;
          tc_fence_after();
          const uint32_t bo = (gg & 1) * 64;
          const uint64_t dK = desc_add(dK0, s * T64), dV = desc_add(dV0, s * T64);
#pragma unroll
          for (int kk = 0; kk < KS; ++kk)
            tc_mma_bf16(tS + bo, desc_add(dQd, kmajor_off(kk, ATOM128)),
                        desc_add(dK, kmajor_off(kk, ATOM64)), id_s, kk > 0);
#pragma unroll
          for (int kk = 0; kk < KS; ++kk)
            tc_mma_bf16(tDP + bo, desc_add(dDO, kmajor_off(kk, ATOM128)),
                        desc_add(dV, kmajor_off(kk, ATOM64)), id_s, kk > 0);
          tc_commit(B(SF + (gg & 1)));
          if (j == nkv - 1) tc_commit(B(QE));
          return true;
        };
        ok = issue_s(0) && issue_s(1);   // nkv >= 2
        const uint32_t tDQ = tmem + 256 + 128 * (n & 1);
        for (int j = 0; j < nkv && ok; ++j) {
          const int gg = gb + j, s = gg % ST;
          // row threads wrote dS(gg) and are done reading buffer gg % 2
          if (!mbar_wait_bounded(B(DSF), gg & 1, p.status, abort_flag)) {
            ok = false;
            break;
          }
          if (j == 0 &&
              !mbar_wait_bounded(B(DQFREE + (n & 1)), ((n >> 1) & 1) ^ 1u, p.status, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t dKmn = desc_add(dKmn0, s * T64);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc_mma_bf16(tDQ, desc_add(dDS, kmajor_off(kk, ATOM128)), desc_add(dKmn, mnmajor_off(kk)),
                        id_dq, (j > 0 || kk > 0) ? 1u : 0u);
          tc_commit(B(KVE + s));
          tc_commit(B(DQD));
          if (j + 2 < nkv && !issue_s(j + 2)) ok = false;
        }
        gb += nkv;
      }
    }
    __syncwarp();
  } else if (warp >= 4) {
    const int wg = (warp - 4) >> 2;                 // column half of the 64 keys
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    int gb = 0, n = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x, ++n) {
      int qb, hd, b;
      item_coords(p, item, true, qb, hd, b);
      const int nkv = 2 * qb + 2;
      const int row0 = b * p.seq + qb * 128;
      const int colq = hd * 3 * p.d;
      // D_r = dO_r . O_r: each warpgroup sums half of the channels
      const size_t orow = (size_t)(row0 + r) * p.h + (size_t)hd * p.d;
      const int half = p.d / 2;
      float Dp = 0.f;
      for (int c = wg * half; c < (wg + 1) * half; c += 8) {
        const uint4 go = *reinterpret_cast<const uint4*>(p.dctx + orow + c);
        const uint4 oo = *reinterpret_cast<const uint4*>(p.ctx + orow + c);
        const bf16* gv = reinterpret_cast<const bf16*>(&go);
        const bf16* ov = reinterpret_cast<const bf16*>(&oo);
#pragma unroll
        for (int e = 0; e < 8; ++e) Dp = fmaf(__bfloat162float(gv[e]), __bfloat162float(ov[e]), Dp);
      }
      float* dpart = s_dpart + (n & 1) * 256;
      dpart[wg * 128 + r] = Dp;
      mbar_arrive(B(DXB));
      if (!mbar_wait_bounded(B(DXB), n & 1, p.status, abort_flag)) {
        ok = false;
        break;
      }
      const float Dr = dpart[r] + dpart[128 + r];
      const size_t lrow = ((size_t)b * p.heads + hd) * p.seq + qb * 128 + r;
      if (wg == 0) p.dsum[lrow] = Dr;
      const float lse2 = p.lse[lrow] * LOG2E;
      const uint32_t tDQ = tmem + 256 + 128 * (n & 1);
      for (int j = 0; j < nkv; ++j) {
        const int gg = gb + j;
        // keep bits of this row over the block's 32 keys, loaded before the wait
        const uint32_t keep =
            DROP ? mask_tile(p, b, hd, qb, j >> 1)[((j & 1) * 2 + wg) * 128 + r] : 0xffffffffu;
        if (!mbar_wait_bounded(B(SF + (gg & 1)), (gg >> 1) & 1, p.status, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t col = (gg & 1) * 64 + wg * 32;
        float ds[32];
        {
          uint32_t sv[32], dv[32];
          tmem_ld32(tS + lane_off + col, sv);
          tmem_ld32(tDP + lane_off + col, dv);
          tmem_ld_wait();
          const float dsc = DROP ? p.drop.scale : 1.0f;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int key = j * 64 + wg * 32 + i;
            float pr = fast_exp2(__uint_as_float(sv[i]) * p.scale_log2 - lse2);
            if (key > qb * 128 + r) pr = 0.f;
            const float dp = ((keep >> i) & 1u) ? __uint_as_float(dv[i]) * dsc : 0.f;
            ds[i] = pr * (dp - Dr);
          }
        }
        if (gg > 0) {
          // the dQ MMA of the previous block has read the dS buffer
          if (!mbar_wait_bounded(B(DQD), (gg - 1) & 1, p.status, abort_flag)) {
            ok = false;
            break;
          }
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int k = c * 8;
          st_shared_v4(sDS + sw128_offset(r, wg * 4 + c), pack_bf16x2(ds[k], ds[k + 1]),
                       pack_bf16x2(ds[k + 2], ds[k + 3]), pack_bf16x2(ds[k + 4], ds[k + 5]),
                       pack_bf16x2(ds[k + 6], ds[k + 7]));
        }
        fence_proxy_async_shared();
        tc_fence_before();
        mbar_arrive(B(DSF));
      }
      if (!ok) break;
      if (!mbar_wait_bounded(B(DQD), (gb + nkv - 1) & 1, p.status, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // the two warpgroups store alternate 32-column chunks of dQ
      bf16* dq = p.dqkv + (size_t)(row0 + r) * 3 * p.h + colq;
      for (int c = wg * 32; c < p.d; c += 64) {
        uint32_t v[32];
        tmem_ld32(tDQ + lane_off + c, v);
        tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint4 u;
          u.x = pack_bf16x2(__uint_as_float(v[q * 8 + 0]) * p.scale, __uint_as_float(v[q * 8 + 1]) * p.scale);
          u.y = pack_bf16x2(__uint_as_float(v[q * 8 + 2]) * p.scale, __uint_as_float(v[q * 8 + 3]) * p.scale);
          u.z = pack_bf16x2(__uint_as_float(v[q * 8 + 4]) * p.scale, __uint_as_float(v[q * 8 + 5]) * p.scale);
          u.w = pack_bf16x2(__uint_as_float(v[q * 8 + 6]) * p.scale, __uint_as_float(v[q * 8 + 7]) * p.scale);
          *reinterpret_cast<uint4*>(dq + c + q * 8) = u;
        }
      }
      tc_fence_before();
      mbar_arrive(B(DQFREE + (n & 1)));
      gb += nkv;
    }
    __syncwarp();
  }
  __syncthreads();
  if (warp == 1) {
    if (*abort_flag) {
      const long long t0 = clock64();
      while (clock64() - t0 < 2000000LL) {
      }
    }
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ============================================================================ dK, dV
// Persistent: one CTA per SM walks the key-block work items.  Per item: 128
// keys; query blocks of 64 from the diagonal on, in a BWD_STAGES-deep ring that
// runs on across items.  S^T and dP^T are double-buffered in TMEM; two
// warpgroups of row threads each take 32 of the 64 query columns.  The next
// item's K/V load and first S^T / dP^T MMAs overlap this item's epilogue.
// smem: K, V (NA atoms of 16 KB), Q[ST], dO[ST] (NA atoms of 8 KB), P^T and dS^T
// (1 atom of 16 KB each), lse / D per stage.  TMEM: S^T[b] cols 64b, dP^T[b]
// cols 128+64b, dV 256.., dK 384..
template <int NA, int KS, bool DROP>
__global__ void __launch_bounds__(BWD_THREADS, 1)
    attn_bwd_dkv_tc_kernel(const __grid_constant__ CUtensorMap tm128,
                           const __grid_constant__ CUtensorMap tm64,
                           const __grid_constant__ CUtensorMap tmdo64, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  const Smem sm = smem_aligned(smem_raw);
  constexpr uint32_t T128 = NA * ATOM128, T64 = NA * ATOM64;
  constexpr int ST = BWD_STAGES;
  const uint32_t sK = sm.u32, sV = sK + T128, sQ0 = sK + 2 * T128, sDO0 = sQ0 + ST * T64,
                 sPT = sDO0 + ST * T64, sDST = sPT + ATOM128;
  // lse and D of the 64-query block of each stage, copied in with its Q / dO
  float* s_lse0 = reinterpret_cast<float*>(sm.base + 2 * T128 + 2 * ST * T64 + 2 * ATOM128);
  float* s_d0 = s_lse0 + 64 * ST;
  const uint32_t s_lse_u32 = smem_u32(s_lse0), s_d_u32 = smem_u32(s_d0);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm.base + 2 * T128 + 2 * ST * T64 + 2 * ATOM128 +
                                               512 * ST);
  const uint32_t bar0 = smem_u32(bars);
  auto B = [&](int i) { return bar0 + 8u * i; };
  // 0 kv_full, 1 kv_empty, 2..ST+1 qdo_full, ST+2..2ST+1 qdo_empty, then
  // st_full[2], pt_full, mm_done, acc_free
  const int KVF = 0, KVE = 1, QF = 2, QE = 2 + ST, STF = 2 + 2 * ST, PTF = 4 + 2 * ST,
            MMD = 5 + 2 * ST, ACCFREE = 6 + 2 * ST, NBAR = 7 + 2 * ST;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NBAR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_items = p.nqb * p.heads * p.batch;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NBAR; ++i) mbar_init(B(i), (i == PTF || i == ACCFREE) ? 256 : 1);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_shared();
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tST = tmem, tDPT = tmem + 128, tDV = tmem + 256, tDK = tmem + 384;

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&tm128);
      tma_prefetch_desc(&tm64);
      tma_prefetch_desc(&tmdo64);
      int g = 0, n = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x, ++n) {
        int kb, hd, b;
        item_coords(p, item, false, kb, hd, b);
        const int colq = hd * 3 * p.d;
        const int first = 2 * kb, nq = 2 * p.nqb - first;
        if (!mbar_wait_bounded(B(KVE), (n & 1) ^ 1u, p.status, abort_flag)) break;
        mbar_arrive_expect_tx(B(KVF), 2 * T128);
        for (int a = 0; a < NA; ++a) {
          tma_load_2d(sK + a * ATOM128, &tm128, B(KVF), colq + p.d + 64 * a, b * p.seq + kb * 128);
          tma_load_2d(sV + a * ATOM128, &tm128, B(KVF), colq + 2 * p.d + 64 * a,
                      b * p.seq + kb * 128);
        }
        for (int i = 0; i < nq; ++i, ++g) {
          const int s = g % ST;
          const int qrow = b * p.seq + (first + i) * 64;
          if (!mbar_wait_bounded(B(QE + s), ((g / ST) & 1) ^ 1u, p.status, abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(B(QF + s), 2 * T64 + 512);
          for (int a = 0; a < NA; ++a) {
            tma_load_2d(sQ0 + s * T64 + a * ATOM64, &tm64, B(QF + s), colq + 64 * a, qrow);
            tma_load_2d(sDO0 + s * T64 + a * ATOM64, &tmdo64, B(QF + s), hd * p.d + 64 * a, qrow);
          }
          const size_t lo = ((size_t)b * p.heads + hd) * p.seq + (first + i) * 64;
          bulk_load(s_lse_u32 + s * 256, p.lse + lo, 256, B(QF + s));
          bulk_load(s_d_u32 + s * 256, p.dsum + lo, 256, B(QF + s));
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t id_st = idesc_bf16_f32(128, 64, false, false);
      const uint32_t id_acc = idesc_bf16_f32(128, p.d, false, true);
      const uint64_t dKd = desc_kbase(sK), dVd = desc_kbase(sV), dQ0 = desc_kbase(sQ0),
                     dDO0 = desc_kbase(sDO0), dPT = desc_kbase(sPT), dDST = desc_kbase(sDST);
      const uint64_t dQmn0 = desc_mnbase(sQ0, ATOM64), dDOmn0 = desc_mnbase(sDO0, ATOM64);
      int gb = 0, n = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x, ++n) {
        int kb, hd, b;
        item_coords(p, item, false, kb, hd, b);
        const int nq = 2 * p.nqb - 2 * kb;
        if (!mbar_wait_bounded(B(KVF), n & 1, p.status, abort_flag)) break;
        tc_fence_after();
        // S^T(block gg), dP^T(block gg) into TMEM buffer gg % 2
        auto issue_st = [&](int i) -> bool {
          const int gg = gb + i, s = gg % ST;
          if (!mbar_wait_bounded(B(QF + s), (gg / ST) & 1, p.status, abort_flag)) return false;
          tc_fence_after();
          const uint32_t bo = (gg & 1) * 64;
          const uint64_t dQ = desc_add(dQ0, s * T64), dDO = desc_add(dDO0, s * T64);
#pragma unroll
          for (int kk = 0; kk < KS; ++kk)
            tc_mma_bf16(tST + bo, desc_add(dKd, kmajor_off(kk, ATOM128)),
                        desc_add(dQ, kmajor_off(kk, ATOM64)), id_st, kk > 0);
#pragma unroll
          for (int kk = 0; kk < KS; ++kk)
            tc_mma_bf16(tDPT + bo, desc_add(dVd, kmajor_off(kk, ATOM128)),
                        desc_add(dDO, kmajor_off(kk, ATOM64)), id_st, kk > 0);
          tc_commit(B(STF + (gg & 1)));
          if (i == nq - 1) tc_commit(B(KVE));
          return true;
        };
        ok = issue_st(0) && issue_st(1);   // nq >= 2
        for (int i = 0; i < nq && ok; ++i) {
          const int gg = gb + i, s = gg % ST;
          // row threads wrote P^T(gg), dS^T(gg) and are done reading buffer gg % 2
          if (!mbar_wait_bounded(B(PTF), gg & 1, p.status, abort_flag)) {
            ok = false;
            break;
          }
          if (i == 0 &&
              !mbar_wait_bounded(B(ACCFREE), (n & 1) ^ 1u, p.status, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t dDOmn = desc_add(dDOmn0, s * T64), dQmn = desc_add(dQmn0, s * T64);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc_mma_bf16(tDV, desc_add(dPT, kmajor_off(kk, ATOM128)), desc_add(dDOmn, mnmajor_off(kk)),
                        id_acc, (i > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc_mma_bf16(tDK, desc_add(dDST, kmajor_off(kk, ATOM128)), desc_add(dQmn, mnmajor_off(kk)),
                        id_acc, (i > 0 || kk > 0) ? 1u : 0u);
          tc_commit(B(QE + s));
          tc_commit(B(MMD));
          if (i + 2 < nq && !issue_st(i + 2)) ok = false;
        }
        gb += nq;
      }
    }
    __syncwarp();
  } else if (warp >= 4) {
    const int wg = (warp - 4) >> 2;   // column half of the 64 queries
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;     // key row
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    int gb = 0, n = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x, ++n) {
      int kb, hd, b;
      item_coords(p, item, false, kb, hd, b);
      const int first = 2 * kb, nq = 2 * p.nqb - first;
      const int key = kb * 128 + r;
      for (int i = 0; i < nq; ++i) {
        const int gg = gb + i;
        const int q0 = (first + i) * 64 + wg * 32;
        // the forward's keep word of query q0+lane over this warp's keys, loaded
        // before the waits so its latency hides behind them
        const uint32_t kword =
            DROP ? mask_tile(p, b, hd, q0 >> 7, kb)[q4 * 128 + (q0 & 127) + lane] : 0u;
        if (!mbar_wait_bounded(B(STF + (gg & 1)), (gg >> 1) & 1, p.status, abort_flag)) {
          ok = false;
          break;
        }
        // lse / D of this block arrive with its Q / dO tiles: observe that
        // barrier's phase too (stage gg % ST is not refilled before this
        // iteration ends: its release follows our arrival below)
        if (!mbar_wait_bounded(B(QF + gg % ST), (gg / ST) & 1, p.status, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float* s_lse = s_lse0 + (gg % ST) * 64 + wg * 32;
        const float* s_d = s_d0 + (gg % ST) * 64 + wg * 32;
        const uint32_t col = (gg & 1) * 64 + wg * 32;
        float pt[32], dst[32];
        {
          uint32_t sv[32], dv[32];
          tmem_ld32(tST + lane_off + col, sv);
          tmem_ld32(tDPT + lane_off + col, dv);
          tmem_ld_wait();
          // Keep bits of queries q0 .. q0+31 for this thread's key: lane l reads
          // the forward's word of query q0+l over this warp's 32 keys, and a
          // warp transpose hands lane k the word over queries for key k.
          const uint32_t keep = DROP ? warp_transpose32(kword, lane) : 0xffffffffu;
          const float dsc = DROP ? p.drop.scale : 1.0f;
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            float pr = fast_exp2(__uint_as_float(sv[e]) * p.scale_log2 - s_lse[e] * LOG2E);
            if (q0 + e < key) pr = 0.f;
            const bool kept = (keep >> e) & 1u;
            pt[e] = kept ? pr * dsc : 0.f;
            dst[e] = pr * ((kept ? __uint_as_float(dv[e]) * dsc : 0.f) - s_d[e]);
          }
        }
        if (gg > 0) {
          // the dV / dK MMAs of the previous block have read P^T / dS^T
          if (!mbar_wait_bounded(B(MMD), (gg - 1) & 1, p.status, abort_flag)) {
            ok = false;
            break;
          }
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int k = c * 8;
          st_shared_v4(sPT + sw128_offset(r, wg * 4 + c), pack_bf16x2(pt[k], pt[k + 1]),
                       pack_bf16x2(pt[k + 2], pt[k + 3]), pack_bf16x2(pt[k + 4], pt[k + 5]),
                       pack_bf16x2(pt[k + 6], pt[k + 7]));
          st_shared_v4(sDST + sw128_offset(r, wg * 4 + c), pack_bf16x2(dst[k], dst[k + 1]),
                       pack_bf16x2(dst[k + 2], dst[k + 3]), pack_bf16x2(dst[k + 4], dst[k + 5]),
                       pack_bf16x2(dst[k + 6], dst[k + 7]));
        }
        fence_proxy_async_shared();
        tc_fence_before();
        mbar_arrive(B(PTF));
      }
      if (!ok) break;
      if (!mbar_wait_bounded(B(MMD), (gb + nq - 1) & 1, p.status, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // warpgroup 0 writes dK (scaled), warpgroup 1 writes dV
      bf16* out = p.dqkv + (size_t)(b * p.seq + kb * 128 + r) * 3 * p.h + hd * 3 * p.d;
      const uint32_t tsrc = wg == 0 ? tDK : tDV;
      const float sc = wg == 0 ? p.scale : 1.0f;
      bf16* dst_row = out + (wg == 0 ? p.d : 2 * p.d);
      for (int c = 0; c < p.d; c += 32) {
        uint32_t v[32];
        tmem_ld32(tsrc + lane_off + c, v);
        tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint4 u;
          u.x = pack_bf16x2(__uint_as_float(v[q * 8 + 0]) * sc, __uint_as_float(v[q * 8 + 1]) * sc);
          u.y = pack_bf16x2(__uint_as_float(v[q * 8 + 2]) * sc, __uint_as_float(v[q * 8 + 3]) * sc);
          u.z = pack_bf16x2(__uint_as_float(v[q * 8 + 4]) * sc, __uint_as_float(v[q * 8 + 5]) * sc);
          u.w = pack_bf16x2(__uint_as_float(v[q * 8 + 6]) * sc, __uint_as_float(v[q * 8 + 7]) * sc);
          *reinterpret_cast<uint4*>(dst_row + c + q * 8) = u;
        }
      }
      tc_fence_before();
      mbar_arrive(B(ACCFREE));
      gb += nq;
    }
    __syncwarp();
  }
  __syncthreads();
  if (warp == 1) {
    if (*abort_flag) {
      const long long t0 = clock64();
      while (clock64() - t0 < 2000000LL) {
      }
    }
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
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
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t fwd_smem(int na) {
  const size_t need = (size_t)(2 + FWD_RING) * na * ATOM128 + 256 + 1024;
  return need < 120 * 1024 ? 120 * 1024 : need;   // one CTA per SM (512 TMEM columns)
}
// The backward kernels hold all 512 TMEM columns: their shared memory requests
// keep them at one CTA per SM so a second CTA never waits in tcgen05.alloc.
size_t dq_smem(int na) {
  const size_t need =
      (size_t)2 * na * ATOM128 + 2 * BWD_STAGES * na * ATOM64 + ATOM128 + 2048 + 256 + 1024;
  return need < 120 * 1024 ? 120 * 1024 : need;
}
size_t dkv_smem(int na) {
  const size_t need = (size_t)2 * na * ATOM128 + 2 * BWD_STAGES * na * ATOM64 + 2 * ATOM128 +
                      512 * BWD_STAGES + 256 + 1024;
  return need < 120 * 1024 ? 120 * 1024 : need;
}

Params make_params(int batch, int seq, int heads, int d, unsigned* status, const Dropout& drop) {
  Params p;
  p.drop = drop;
  p.batch = batch;
  p.seq = seq;
  p.heads = heads;
  p.d = d;
  p.h = heads * d;
  p.nqb = seq / 128;
  p.scale = 1.0f / sqrtf((float)d);
  p.scale_log2 = LOG2E * p.scale;
  p.ctx = nullptr;
  p.lse = nullptr;
  p.dctx = nullptr;
  p.dqkv = nullptr;
  p.dsum = nullptr;
  p.status = status;
  p.mask = nullptr;
  p.sched = nullptr;
  p.chunk = 1;
  return p;
}

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}
// A kernel with a setmaxnreg split must start with exactly the registers the
// split was sized for, or setmaxnreg.inc could never be satisfied.
template <typename K>
cudaError_t check_regs(K kernel, int regs) {
  cudaFuncAttributes fa;
  const cudaError_t e = cudaFuncGetAttributes(&fa, kernel);
  if (e != cudaSuccess) return e;
  return fa.numRegs == regs ? cudaSuccess : cudaErrorInvalidConfiguration;
}

}  // namespace attn

bool attn_tc_supported(int seq, int d) { return seq % 128 == 0 && (d == 64 || d == 96 || d == 128); }

size_t attn_mask_bytes(int batch, int seq, int heads) {
  const size_t nqb = (size_t)seq / 128;
  return (size_t)batch * heads * (nqb * (nqb + 1) / 2) * 2048;
}

cudaError_t attn_fwd_tc(const void* qkv, void* ctx, float* lse, int batch, int seq, int heads,
                        int d, const Dropout& drop, uint32_t* mask, unsigned* status,
                        const LaunchCtx& c) {
  using namespace attn;
  if (batch == 0) return cudaSuccess;
  if (!attn_tc_supported(seq, d)) return cudaErrorInvalidValue;
  CUtensorMap tm;
  if (!make_map(&tm, qkv, 3ull * heads * d, (uint64_t)batch * seq, 128)) return cudaErrorInvalidValue;
  if (drop.on && !mask) return cudaErrorInvalidValue;
  Params p = make_params(batch, seq, heads, d, status, drop);
  p.mask = mask;
  p.ctx = static_cast<bf16*>(ctx);
  p.lse = lse;
  p.sched = status + kSchedFwd;
  // pairs whose K/V (NA 128-byte boxes per row) fit in about 48 MB of L2
  {
    const size_t kv = 2ull * seq * (d > 64 ? 2 : 1) * 128;
    const size_t c = ((size_t)48 << 20) / kv;
    p.chunk = c < 1 ? 1 : (c > (size_t)batch * heads ? batch * heads : (int)c);
  }
  const int items = ((p.nqb + 1) / 2) * heads * batch;
  const int grid = items < c.num_sms ? items : c.num_sms;
  const double flops = 2.0 * 2.0 * batch * heads * d * ((double)seq * (seq + 1) / 2.0);
  cudaError_t e;
#define FWD_CASE(NA_, KS_, DR_)                                                          \
  {                                                                                      \
    const size_t sm = fwd_smem(NA_);                                                     \
    if ((e = set_smem(attn_fwd_tc_kernel<NA_, KS_, DR_>, sm)) != cudaSuccess) return e;  \
    if ((e = check_regs(attn_fwd_tc_kernel<NA_, KS_, DR_>, FWD_LAUNCH_REGS)) != cudaSuccess) \
      return e;                                                                          \
    c.before(KK_ATTN_FWD, flops);                                                        \
    attn_fwd_tc_kernel<NA_, KS_, DR_><<<grid, FWD_THREADS, sm, c.stream>>>(tm, p);       \
  }
  if (drop.on) {
    if (d == 64) FWD_CASE(1, 4, true)
    else if (d == 96) FWD_CASE(2, 6, true)
    else FWD_CASE(2, 8, true)
  } else {
    if (d == 64) FWD_CASE(1, 4, false)
    else if (d == 96) FWD_CASE(2, 6, false)
    else FWD_CASE(2, 8, false)
  }
#undef FWD_CASE
  c.after();
  return cudaGetLastError();
}

cudaError_t attn_bwd_tc(const void* qkv, const void* ctx, const float* lse, const void* dctx,
                        void* dqkv, float* dsum, int batch, int seq, int heads, int d,
                        const Dropout& drop, const uint32_t* mask, unsigned* status,
                        const LaunchCtx& c) {
  using namespace attn;
  if (batch == 0) return cudaSuccess;
  if (!attn_tc_supported(seq, d)) return cudaErrorInvalidValue;
  const uint64_t n = (uint64_t)batch * seq;
  CUtensorMap tm128, tm64, tmdo128, tmdo64;
  if (!make_map(&tm128, qkv, 3ull * heads * d, n, 128) || !make_map(&tm64, qkv, 3ull * heads * d, n, 64) ||
      !make_map(&tmdo128, dctx, (uint64_t)heads * d, n, 128) ||
      !make_map(&tmdo64, dctx, (uint64_t)heads * d, n, 64))
    return cudaErrorInvalidValue;
  if (drop.on && !mask) return cudaErrorInvalidValue;
  Params p = make_params(batch, seq, heads, d, status, drop);
  p.mask = const_cast<uint32_t*>(mask);
  p.ctx = static_cast<bf16*>(const_cast<void*>(ctx));
  p.lse = const_cast<float*>(lse);
  p.dctx = static_cast<const bf16*>(dctx);
  p.dqkv = static_cast<bf16*>(dqkv);
  p.dsum = dsum;
  const int items = p.nqb * heads * batch;
  const int grid = items < c.num_sms ? items : c.num_sms;
  const double tri = (double)batch * heads * d * ((double)seq * (seq + 1) / 2.0);
  cudaError_t e;
#define BWD_CASE(NA_, KS_, DR_)                                                                \
  {                                                                                            \
    if ((e = set_smem(attn_bwd_dq_tc_kernel<NA_, KS_, DR_>, dq_smem(NA_))) != cudaSuccess)       \
      return e;                                                                                \
    if ((e = set_smem(attn_bwd_dkv_tc_kernel<NA_, KS_, DR_>, dkv_smem(NA_))) != cudaSuccess)     \
      return e;                                                                                \
    c.before(KK_ATTN_BWD, 2.0 * 3.0 * tri);                                                    \
    attn_bwd_dq_tc_kernel<NA_, KS_, DR_><<<grid, BWD_THREADS, dq_smem(NA_), c.stream>>>(        \
        tm128, tm64, tmdo128, p);                                                              \
    c.after();                                                                                 \
    if ((e = cudaGetLastError()) != cudaSuccess) return e;                                     \
    c.before(KK_ATTN_BWD, 2.0 * 4.0 * tri);                                                    \
    attn_bwd_dkv_tc_kernel<NA_, KS_, DR_><<<grid, BWD_THREADS, dkv_smem(NA_), c.stream>>>(      \
        tm128, tm64, tmdo64, p);                                                               \
    c.after();                                                                                 \
  }
  if (drop.on) {
    if (d == 64) BWD_CASE(1, 4, true)
    else if (d == 96) BWD_CASE(2, 6, true)
    else BWD_CASE(2, 8, true)
  } else {
    if (d == 64) BWD_CASE(1, 4, false)
    else if (d == 96) BWD_CASE(2, 6, false)
    else BWD_CASE(2, 8, false)
  }
#undef BWD_CASE
  return cudaGetLastError();
}

}  // namespace mtl
