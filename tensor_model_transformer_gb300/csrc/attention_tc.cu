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
// All three kernels are persistent (one CTA per SM, work items from a global
// counter) with warp roles:
//   warp 0      scheduler and TMA producer
//   warp 1      TMEM allocator and the MMA issuer of the score-sized products
//   warp 2      the MMA issuer of the products that read P / dS
//   warp 3      gives its registers to the row threads
//   warps 4-11  row threads: thread (warp%4)*32+lane owns TMEM lane = one row of
//               a 128-row block.
// Operand tiles are [atoms][rows][64] 128-byte-swizzled boxes straight from TMA;
// the same box serves as a K-major operand (rows = M/N) or an MN-major one
// (rows = K), e.g. dO is the K-major B of dO V^T and the MN-major B of P^T dO.
// P, dS, P^T and dS^T go from registers to TMEM as bf16 and are read there as
// the A operand of the next product.
// Every wait is bounded; a timeout is recorded in the status word.
#include "common.cuh"
#include "kernels.h"
#include "tile_layout.h"

namespace mtl {
namespace attn {

constexpr int FWD_THREADS = 384;   // forward kernel: 4 control warps, two warpgroups of row threads
constexpr int BWD_THREADS = 384;   // backward kernels: 4 control warps, two warpgroups of row threads
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

// A TMA load of one 64 x 128 box of a bf16 activation with `cols` x `rows`
// elements (qkv: 3h x n; ctx and dctx: h x n), its coordinates checked in
// MTL_DEBUG builds.
__device__ __forceinline__ void load_box(uint32_t dst, const CUtensorMap* m, uint32_t bar, int x,
                                         int y, int64_t cols, int64_t rows, unsigned* status,
                                         uint32_t site, int box_cols = 64) {
  const bounds::Box2 b = {cols, rows, box_cols, 128, 2};
  (void)b;
  if (MTL_CHECKED(status, bounds::check_tma_load(b, x, y), site)) tma_load_2d(dst, m, bar, x, y);
}

// The operand tile layout (tile_layout.h) with its tcgen05 descriptors: K-major
// with 8-row groups ROWB * 8 bytes apart; MN-major with the N atoms ATOM bytes
// apart.
template <int KS>
struct Fmt : layout::TileFmt<KS> {
  using L = layout::TileFmt<KS>;
  static constexpr uint32_t MODE = L::SW64 ? kDescSw64 : kDescSw128;
  __device__ static uint64_t kdesc(uint32_t a) { return smem_desc(a, 16, 8 * L::ROWB, MODE); }
  __device__ static uint64_t mndesc(uint32_t a) { return smem_desc(a, L::ATOM, 8 * L::ROWB, MODE); }
};

struct Smem {
  uint8_t* base;
  uint32_t u32;
};

__device__ __forceinline__ Smem smem_aligned(uint8_t* raw) {
  uint8_t* p = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) &
                                          ~static_cast<uintptr_t>(1023));
  return {p, smem_u32(p)};
}

// Epilogue stores.  A warp's 32 rows (lane = row) of an output tile leave 32
// columns at a time as TMA tensor stores of a 32 x 32 box: each lane writes
// its row's 64 bytes into the warp's 2 KB staging buffer, in the 64-byte
// swizzle the tensor map names (16-byte piece p of row r at r * 64 + ((p ^
// ((r / 2) % 4)) * 16), which also keeps the row-wise writes at four
// shared-memory wavefronts), and one lane issues the store.  The copy engine
// writes global memory while the rows go on; a lane-per-row store of 16 bytes
// from registers touched 32 cache lines per instruction and held the rows for
// thousands of cycles an item.  Before a buffer is rewritten its previous
// store must have read it (cp.async.bulk.wait_group.read).
constexpr uint32_t STAGE_WARP_BYTES = 32 * 64;
constexpr uint32_t STAGE_BYTES = 8 * STAGE_WARP_BYTES;   // the eight row warps

__device__ __forceinline__ uint32_t stage_off(int row, int piece) { return layout::sw64_off(row, piece); }

// 32 fp32 TMEM columns at taddr (this lane's row), times sc, as bf16 to the
// box of 32 columns x 32 rows at (x, y) of the tensor map m (y: the warp's
// first row).  `stage` is the warp's buffer (1024-byte aligned pattern base).
__device__ __forceinline__ void store_acc32_tma(uint32_t taddr, float sc, const CUtensorMap* m, int x,
                                                int y, uint32_t stage, int lane) {
  uint32_t v[32];
  tmem_ld32(taddr, v);
  tmem_ld_wait();
  if (lane == 0) bulk_wait_read0();   // the buffer's previous store has read it
  __syncwarp();
#pragma unroll
  for (int q = 0; q < 4; ++q)
    st_shared_v4(stage + stage_off(lane, q),
                 pack_bf16x2(__uint_as_float(v[q * 8 + 0]) * sc, __uint_as_float(v[q * 8 + 1]) * sc),
                 pack_bf16x2(__uint_as_float(v[q * 8 + 2]) * sc, __uint_as_float(v[q * 8 + 3]) * sc),
                 pack_bf16x2(__uint_as_float(v[q * 8 + 4]) * sc, __uint_as_float(v[q * 8 + 5]) * sc),
                 pack_bf16x2(__uint_as_float(v[q * 8 + 6]) * sc, __uint_as_float(v[q * 8 + 7]) * sc));
  fence_proxy_async_shared();         // the generic writes, before the copy engine reads them
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(m, stage, x, y);
    bulk_commit();
  }
}

// In MTL_DEBUG builds: the 32 x 32 store box at (x, y) of a cols x rows bf16
// tensor starts inside it on a 16-byte boundary.
__device__ __forceinline__ bool store_box_ok(unsigned* status, int x, int y, int64_t cols, int64_t rows,
                                             uint32_t site) {
  const bounds::Box2 b = {cols, rows, 32, 32, 2};
  (void)b;
  (void)status;
  (void)site;
  return MTL_CHECKED(status, bounds::check_tma_store(b, x, y), site);
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
// smem: Q_A, Q_B, ring[FWD_RING] (tiles in the Fmt layout), the epilogue
// staging buffers, item ids.
// TMEM: S cols 0..127, P_A 128..191, P_B 192..255, O_A 256.., O_B 384..
constexpr int FWD_RING = 4;
static_assert(FWD_RING % 2 == 0, "K and V must keep to their own ring slots");
constexpr uint32_t TM_S = 0, TM_P = 128, TM_O = 256;
// Register split: warps 0..3 (producer, two MMA issuers, one idle) give
// registers to the row warps 4..11, which hold a 128-key score row each.  The split is
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

template <int KS, bool DROP>
__global__ void __launch_bounds__(FWD_THREADS, 1)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm, const __grid_constant__ CUtensorMap tmc,
                       const Params p) {
  extern __shared__ uint8_t smem_raw[];
  const Smem sm = smem_aligned(smem_raw);
  using F = Fmt<KS>;
  constexpr uint32_t TILE = F::TILE;
  constexpr int D = KS * 16;
  const uint32_t sQ0 = sm.u32, sR0 = sQ0 + 2 * TILE;
  const uint32_t sStage = sQ0 + (2 + FWD_RING) * TILE;   // epilogue staging, 2 KB a row warp
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm.base + (2 + FWD_RING) * TILE + STAGE_BYTES);
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
        const int64_t cols = 3 * (int64_t)p.h, rows = (int64_t)p.batch * p.seq;
        auto load_q = [&](int x) -> bool {
          const int nq = x ? nit1++ : nit0++;
          if (nq > 0 && !mbar_wait_bounded(B(QE + x), (nq - 1) & 1, p.status, abort_flag))
            return false;
          mbar_arrive_expect_tx(B(QF + x), TILE);
          for (int a = 0; a < F::ATOMS; ++a)
            load_box(sQ0 + x * TILE + a * F::ATOM, &tm, B(QF + x), colq + F::ACOLS * a,
                     row0 + it.qp * 256 + x * 128, cols, rows, p.status, bounds::kSiteAttnFwdQ, F::ACOLS);
          return true;
        };
        auto load_kv = [&](int j) -> bool {   // K(j) and V(j) into the next two ring slots
          for (int kv = 0; kv < 2; ++kv, ++g) {
            const int s = g % FWD_RING, use = g / FWD_RING;
            if (use > 0 && !mbar_wait_bounded(B(RE + s), (use - 1) & 1, p.status, abort_flag))
              return false;
            mbar_arrive_expect_tx(B(RF + s), TILE);
            for (int a = 0; a < F::ATOMS; ++a)
              load_box(sR0 + s * TILE + a * F::ATOM, &tm, B(RF + s),
                       colq + (1 + kv) * p.d + F::ACOLS * a, row0 + j * 128, cols, rows, p.status,
                       bounds::kSiteAttnFwdKV, F::ACOLS);
          }
          return true;
        };
        // Tile A's Q, the first K / V block, then tile B's Q: the previous
        // item's last Q K^T (tile B's) frees B's Q buffer only at the end of
        // that item, and this item's first product (tile A's) needs just Q_A
        // and K(0), which thus load while the previous item finishes.
        const int nkv = it.n0 > it.n1 ? it.n0 : it.n1;
        ok = load_q(0) && load_kv(0) && (!it.n1 || load_q(1));
        for (int j = 1; j < nkv && ok; ++j) ok = load_kv(j);
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
      const uint64_t dQ0 = F::kdesc(sQ0), dR0 = F::kdesc(sR0);
      const uint64_t dRmn0 = F::mndesc(sR0);
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
              tc_mma_bf16(tmem + TM_S, desc_add(dQ, F::koff(kk)), desc_add(dK, F::koff(kk)), id_qk,
                          kk > 0);
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
                             desc_add(dV, F::mnoff(kk)), id_pv, (j > 0 || kk > 0) ? 1u : 0u);
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
    // A tile's epilogue (O / l to ctx, lse) runs when the tile has taken its
    // next item, once the item's last PV is done; PV_X(0) of the next item
    // waits for that item's first P block, so O_X is read first.
    bool pend = false;
    float pm = 0.f, pl = 1.f;
    size_t plse = 0;               // lse index of the row
    int px = 0, py = 0;            // ctx column of the head slice, the warp's first row
    const uint32_t stage = sStage + (warp - 4) * STAGE_WARP_BYTES;
    auto epilogue = [&]() {
      const float inv = (DROP ? p.drop.scale : 1.0f) / pl;
      // the warp's rows of the head slice lie inside ctx [n][h], the row's lse
      // inside [batch][heads][seq] (the warp stores its rows together: it
      // skips them all if one check fails)
      if (!__all_sync(0xffffffffu,
                      MTL_CHECKED(p.status,
                                  bounds::check_index((int64_t)plse, (int64_t)p.batch * p.heads * p.seq),
                                  bounds::kSiteAttnFwdOut)) ||
          !store_box_ok(p.status, px, py, p.h, (int64_t)p.batch * p.seq, bounds::kSiteAttnFwdOut))
        return;
#pragma unroll 1
      for (int c = 0; c < D; c += 32) store_acc32_tma(tO + c, inv, &tmc, px + c, py, stage, lane);
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
      // The previous item's O / l leave while this item's first S is on its
      // way (tile A's first block waits for tile B's extra diagonal block of
      // the previous item); PV_X(0) of this item waits for its first P block.
      if (pend) {
        if (!mbar_wait_bounded(B(PE + x), (cnt - 1) & 1, p.status, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        epilogue();
        pend = false;
      }
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
        plse = ((size_t)it.b * p.heads + it.hd) * p.seq + qb * 128 + r;
        px = it.hd * D;
        py = it.b * p.seq + qb * 128 + q4 * 32;
      }
    }
    if (ok && pend) {
      if (mbar_wait_bounded(B(PE + x), (cnt - 1) & 1, p.status, abort_flag)) {
        tc_fence_after();
        epilogue();
      }
    }
    if (lane == 0) bulk_wait0();   // this warp's stores are done before shared memory goes
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

// ============================================================================ backward
// Two persistent kernels, each with the forward's warp roles: warp 0 takes
// work items from a global counter (longest first within L2-sized chunks of
// (batch, head) pairs) and drives TMA; warp 1 allocates TMEM and issues the
// products that make the score-sized blocks; warp 2 issues the accumulating
// products; warp 3 only gives its registers up; warps 4..11 are two
// warpgroups of row threads, warpgroup w owning columns 64w..64w+63 of every
// 128 x 128 block (P comes from the saved lse, not a row maximum, so the two
// halves never need each other).  A slot of the TMA ring that both issuers
// read is released by two commits.
constexpr int BWD_RING = 4;
constexpr size_t kSmemMax = 227 * 1024;   // dynamic shared memory a CTA may request
static_assert(BWD_RING % 2 == 0, "each ring slot keeps to one operand");

struct BwdItem {
  int blk, hd, b;
};

// Work item k -> (128-row block, head, batch); within a chunk of pairs the
// blocks go by decreasing work: the dQ kernel's query blocks from the last,
// the dK/dV kernel's key blocks from the first.
__device__ __forceinline__ BwdItem bwd_item(const Params& p, int k, bool last_first) {
  const int pairs = p.batch * p.heads;
  const int per_chunk = p.chunk * p.nqb;
  const int c = k / per_chunk;
  const int cp = min(p.chunk, pairs - c * p.chunk);
  const int r = k - c * per_chunk;
  const int pair = c * p.chunk + r % cp;
  const int lvl = r / cp;
  BwdItem it;
  it.blk = last_first ? p.nqb - 1 - lvl : lvl;
  it.hd = pair % p.heads;
  it.b = pair / p.heads;
  return it;
}

// Work-item hand-off through two shared-memory slots: the producer publishes,
// the MMA issuers and one lane of each row warp acknowledge.
struct ItemRing {
  int* slot;
  uint32_t full, empty;   // barrier addresses of slot 0 (slot 1 follows at +8)
};

__device__ __forceinline__ bool item_publish(const ItemRing& q, int ni, int k, unsigned* status,
                                             volatile int* abort_flag) {
  const int s = ni & 1;
  if (ni >= 2 && !mbar_wait_bounded(q.empty + 8u * s, ((ni >> 1) - 1) & 1, status, abort_flag))
    return false;
  q.slot[s] = k;
  mbar_arrive(q.full + 8u * s);
  return true;
}

// Returns false on abort; k >= n_items means no work is left.
__device__ __forceinline__ bool item_take(const ItemRing& q, int ni, bool ack, int& k,
                                          unsigned* status, volatile int* abort_flag) {
  const int s = ni & 1;
  if (!mbar_wait_bounded(q.full + 8u * s, (ni >> 1) & 1, status, abort_flag)) return false;
  k = *reinterpret_cast<volatile int*>(&q.slot[s]);
  __syncwarp(__activemask());
  if (ack) mbar_arrive(q.empty + 8u * s);
  return true;
}

__device__ __forceinline__ void sched_done(unsigned* sched) {
  __threadfence();
  if (atomicAdd(sched + 1, 1u) == gridDim.x - 1) {
    atomicExch(sched, 0u);
    atomicExch(sched + 1, 0u);
  }
}

constexpr int BWD_LAUNCH_REGS = 168, BWD_LOW_REGS = 72, BWD_ROW_REGS = 216;
static_assert(BWD_THREADS == 384, "one giving and two taking warps per sub-partition");
static_assert(BWD_LOW_REGS + 2 * BWD_ROW_REGS <= 3 * BWD_LAUNCH_REGS,
              "register split exceeds a sub-partition's launch allocation");

// Shared memory of the dQ kernel with `qb` Q/dO buffer pairs of `tile` bytes.
__host__ __device__ constexpr size_t dq_need(uint32_t tile, int qb) {
  return (size_t)(2 * qb + 1 + BWD_RING) * tile + 256 + 1024 + 1024;
}
// Q and dO are double-buffered when the tiles leave room (d = 64, 96), so the
// next item's Q and dO load while the current item runs.
__host__ __device__ constexpr int dq_q_bufs(uint32_t tile) { return dq_need(tile, 2) <= kSmemMax ? 2 : 1; }

// ============================================================================ dQ
// Item: 128 queries (Q, dO resident) against key blocks j = 0..qb of 128 keys
// (K(j), V(j) through the ring).  Per block: S = Q K^T and dP = dO V^T (warp
// 1); the row threads' dS = P * (dP - D) with P = exp2(S log2(e) / sqrt(d) -
// lse log2(e)) (zero after the query), written to TMEM as bf16; dQ += dS K
// (warp 2, dS as the A operand).  The row threads also form D_i = sum_c dO_ic
// O_ic from the dO and O tiles in shared memory and store it for the dK/dV
// kernel.  An item's dQ is written out when the rows have formed the next
// item's D (its last dQ product done), while that item's first S and dP are
// on their way; the first dQ product of the next item waits for its dS.
// smem: Q and dO (two pairs where they fit: dq_q_bufs), O, ring[BWD_RING]
// (tiles in the Fmt layout), the halves of D, item ids.  Of the
// ring, DQ_KSLOTS slots hold K blocks and one holds V: K(j) stays until dQ +=
// dS K(j) has read it, about a block after S, so K is loaded up to two blocks
// ahead; V(j) is free once dP(j) is done, and V(j + 1) loads while the rows
// work on block j.  (With K and V alternating in the four slots, K(j + 2)
// waited for dQ(j) and the next S = Q K^T for the load.)
// TMEM: S 0..127, dP 128..255, dS 256..319, dQ 384..
constexpr uint32_t TQ_S = 0, TQ_DP = 128, TQ_DS = 256, TQ_ACC = 384;
constexpr int DQ_KSLOTS = BWD_RING - 1, DQ_VSLOT = BWD_RING - 1;

template <int KS, bool DROP>
__global__ void __launch_bounds__(BWD_THREADS, 1)
    attn_bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap tm,
                          const __grid_constant__ CUtensorMap tmdo,
                          const __grid_constant__ CUtensorMap tmo,
                          const __grid_constant__ CUtensorMap tmdq, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  const Smem sm = smem_aligned(smem_raw);
  using F = Fmt<KS>;
  constexpr uint32_t TILE = F::TILE;
  constexpr int D = KS * 16;
  constexpr int NQB = dq_q_bufs(TILE);   // Q/dO buffers: item m uses buffer m % NQB
  // Q(u) at sQ + 2u TILE with dO(u) after it; then O, then the ring
  const uint32_t sQ = sm.u32, sO = sQ + 2 * NQB * TILE, sR0 = sO + TILE;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm.base + (2 * NQB + 1 + BWD_RING) * TILE);
  const uint32_t bar0 = smem_u32(bars);
  auto B = [&](int i) { return bar0 + 8u * i; };
  // QF / QE (one per Q/dO buffer): Q and dO loaded / the item's last S and dP
  // products done with them; OF: O loaded; DE: the row threads are done with
  // dO and O for D and with the O tile as staging (for a one-block item the
  // products can finish before the rows get to D, so the rows gate dO too)
  constexpr int QF = 0, QE = 2, OF = 4, RF = 5, RE = RF + BWD_RING, SF = RE + BWD_RING, SE = SF + 1,
                DSF = SE + 1, DQD = DSF + 1, DE = DQD + 1, IF = DE + 1, IE = IF + 2, NBAR = IE + 2;
  // the two warpgroups' halves of D for the item's 128 rows
  volatile float* s_dhalf =
      reinterpret_cast<volatile float*>(sm.base + (2 * NQB + 1 + BWD_RING) * TILE + 256);
  int* s_item = reinterpret_cast<int*>(bars + NBAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(s_item + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const ItemRing iq{s_item, B(IF), B(IE)};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_items = p.nqb * p.heads * p.batch;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NBAR; ++i) {
      uint32_t cnt = 1;
      if (i == SE || i == DSF || i == DE) cnt = 256;
      if (i == IE || i == IE + 1) cnt = 2 + 8;            // two issuers + a lane per row warp
      if (i >= RE && i < RE + DQ_KSLOTS) cnt = 2;   // K slots: read by both issuers
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
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(BWD_LOW_REGS));
    if (lane == 0) {
      tma_prefetch_desc(&tm);
      tma_prefetch_desc(&tmdo);
      tma_prefetch_desc(&tmo);
      int g = 0, ni = 0, nit = 0, ksl = 0, kuse = 0;   // K slot and its use count
      bool ok = true;
      while (ok) {
        const int k = (int)atomicAdd(p.sched, 1u);
        if (!item_publish(iq, ni++, k, p.status, abort_flag) || k >= n_items) break;
        const BwdItem it = bwd_item(p, k, true);
        const int colq = it.hd * 3 * p.d, row0 = it.b * p.seq;
        // Q and dO of item nit into buffer u once item nit - NQB is done with
        // them (its products, and its rows' D: waited on below for the
        // previous item, before its O load); then O once the rows are done
        // with the previous item's O
        const int u = nit % NQB, use = nit / NQB;
        if (use > 0 && !mbar_wait_bounded(B(QE + u), (use - 1) & 1, p.status, abort_flag)) break;
        if (NQB == 1 && nit > 0 && !mbar_wait_bounded(B(DE), (nit - 1) & 1, p.status, abort_flag)) break;
        const uint32_t sQu = sQ + 2 * u * TILE, sDOu = sQu + TILE;
        mbar_arrive_expect_tx(B(QF + u), 2 * TILE);
        for (int a = 0; a < F::ATOMS; ++a) {
          load_box(sQu + a * F::ATOM, &tm, B(QF + u), colq + F::ACOLS * a, row0 + it.blk * 128,
                   3 * (int64_t)p.h, (int64_t)p.batch * p.seq, p.status, bounds::kSiteAttnDqLoad, F::ACOLS);
          load_box(sDOu + a * F::ATOM, &tmdo, B(QF + u), it.hd * p.d + F::ACOLS * a, row0 + it.blk * 128,
                   (int64_t)p.h, (int64_t)p.batch * p.seq, p.status, bounds::kSiteAttnDqLoad, F::ACOLS);
        }
        if (NQB == 2 && nit > 0 && !mbar_wait_bounded(B(DE), (nit - 1) & 1, p.status, abort_flag)) break;
        ++nit;
        mbar_arrive_expect_tx(B(OF), TILE);
        for (int a = 0; a < F::ATOMS; ++a)
          load_box(sO + a * F::ATOM, &tmo, B(OF), it.hd * p.d + F::ACOLS * a, row0 + it.blk * 128,
                   (int64_t)p.h, (int64_t)p.batch * p.seq, p.status, bounds::kSiteAttnDqLoad, F::ACOLS);
        for (int j = 0; j <= it.blk && ok; ++j, ++g) {   // g: blocks so far
          for (int kv = 0; kv < 2; ++kv) {
            const int s = kv ? DQ_VSLOT : ksl, use = kv ? g : kuse;
            if (use > 0 && !mbar_wait_bounded(B(RE + s), (use - 1) & 1, p.status, abort_flag)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(B(RF + s), TILE);
            for (int a = 0; a < F::ATOMS; ++a)
              load_box(sR0 + s * TILE + a * F::ATOM, &tm, B(RF + s), colq + (1 + kv) * p.d + F::ACOLS * a,
                       row0 + j * 128, 3 * (int64_t)p.h, (int64_t)p.batch * p.seq, p.status,
                       bounds::kSiteAttnDqKV, F::ACOLS);
          }
          if (++ksl == DQ_KSLOTS) {
            ksl = 0;
            ++kuse;
          }
        }
      }
      sched_done(p.sched);
    }
    __syncwarp();
  } else if (warp == 1 || warp == 2) {
    // ------------------------------------------ MMA issuers: warp 1 S, dP; warp 2 dQ
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(BWD_LOW_REGS));
    if (lane == 0) {
      const bool first = warp == 1;
      const uint32_t id_s = idesc_bf16_f32(128, 128, false, false);
      const uint32_t id_acc = idesc_bf16_f32(128, D, false, true);
      const uint64_t dQ0 = F::kdesc(sQ), dR0 = F::kdesc(sR0);
      const uint64_t dRmn0 = F::mndesc(sR0);
      int ni = 0, nit = 0, nb = 0;      // nb: blocks so far
      int sk = 0, kuse = 0;             // K slot of this block and its use count
      bool ok = true;
      auto wait = [&](int bar, int k) -> bool {
        if (!mbar_wait_bounded(B(bar), k & 1, p.status, abort_flag)) ok = false;
        return ok;
      };
      while (ok) {
        int k;
        if (!item_take(iq, ni++, true, k, p.status, abort_flag)) break;
        if (k >= n_items) break;
        const BwdItem it = bwd_item(p, k, true);
        const int nkv = it.blk + 1;
        const int u = nit % NQB;
        const uint64_t dQd = desc_add(dQ0, 2 * u * TILE), dDO = desc_add(dQd, TILE);
        for (int j = 0; j < nkv && ok; ++j, ++nb) {
          if (first) {
            if (j == 0 && !wait(QF + u, nit / NQB)) break;
            if (!wait(RF + sk, kuse)) break;
            if (nb > 0 && !wait(SE, nb - 1)) break;   // the row threads hold S, dP of the last block
            tc_fence_after();
            const uint64_t dK = desc_add(dR0, sk * TILE), dV = desc_add(dR0, DQ_VSLOT * TILE);
#pragma unroll
            for (int kk = 0; kk < KS; ++kk)
              tc_mma_bf16(tmem + TQ_S, desc_add(dQd, F::koff(kk)), desc_add(dK, F::koff(kk)), id_s,
                          kk > 0);
            // V(j) may land after S is under way
            if (!wait(RF + DQ_VSLOT, nb)) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < KS; ++kk)
              tc_mma_bf16(tmem + TQ_DP, desc_add(dDO, F::koff(kk)), desc_add(dV, F::koff(kk)), id_s,
                          kk > 0);
            tc_commit(B(SF));
            tc_commit(B(RE + sk));
            tc_commit(B(RE + DQ_VSLOT));
            if (j == nkv - 1) tc_commit(B(QE + u));
          } else {
            if (!wait(DSF, nb)) break;                // dS of this block is in TMEM
            if (!wait(RF + sk, kuse)) break;
            tc_fence_after();
            const uint64_t dKmn = desc_add(dRmn0, sk * TILE);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              tc_mma_bf16_ts(tmem + TQ_ACC, tmem + TQ_DS + 8 * kk, desc_add(dKmn, F::mnoff(kk)),
                             id_acc, (j > 0 || kk > 0) ? 1u : 0u);
            tc_commit(B(DQD));
            tc_commit(B(RE + sk));
          }
          if (++sk == DQ_KSLOTS) {
            sk = 0;
            ++kuse;
          }
        }
        if (!ok) break;
        ++nit;
      }
    }
    __syncwarp();
  } else if (warp == 3) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(BWD_LOW_REGS));
  } else {
    // ---------------------------------------------------------------- row threads
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(BWD_ROW_REGS));
    const int wg = (warp - 4) >> 2;            // key columns 64 wg .. 64 wg + 63
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;              // query row = TMEM lane
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    const float dsc = DROP ? p.drop.scale : 1.0f;
    int ni = 0, nb = 0, nit = 0;
    bool pend = false;
    int px = 0, py = 0;                        // dqkv column of the pending dQ, the warp's first row
    // the epilogue stages its stores in the O tile, which is free from the
    // moment every row thread has formed D until the rows arrive on DE
    const uint32_t stage = sO + (warp - 4) * STAGE_WARP_BYTES;
    auto epilogue = [&]() {
      // warpgroup wg writes 32-column chunks wg, wg + 2, ... of the rows' dQ,
      // inside dqkv [n][3h]
      if (!store_box_ok(p.status, px, py, 3 * (int64_t)p.h, (int64_t)p.batch * p.seq, bounds::kSiteAttnDqOut))
        return;
#pragma unroll 1
      for (int c = 32 * wg; c < D; c += 64)
        store_acc32_tma(tmem + TQ_ACC + lane_off + c, p.scale, &tmdq, px + c, py, stage, lane);
    };
    bool ok = true;
    while (ok) {
      int k;
      if (!item_take(iq, ni++, lane == 0, k, p.status, abort_flag)) {
        ok = false;
        break;
      }
      if (k >= n_items) break;
      const BwdItem it = bwd_item(p, k, true);
      const int qb = it.blk;
      // D_r = dO_r . O_r from the tiles in shared memory (they are not reloaded
      // before every row thread has arrived on DE, after the previous item's
      // epilogue below)
      const int u = nit % NQB;
      const uint32_t sDO = sQ + (2 * u + 1) * TILE;
      if (!mbar_wait_bounded(B(QF + u), (nit / NQB) & 1, p.status, abort_flag) ||
          !mbar_wait_bounded(B(OF), nit & 1, p.status, abort_flag)) {
        ok = false;
        break;
      }
      ++nit;
      // warpgroup wg sums columns wg D/2 .. (wg + 1) D/2 - 1; both then add
      // the two halves in the same order
      float Dp = 0.f;
#pragma unroll
      for (int i = 0; i < D / 16; ++i) {
        const int c = wg * (D / 16) + i;
        const uint32_t off = F::chunk(r, c);
        Vec<bf16> go, oo;
        go.raw = ld_shared_v4(sDO + off);
        oo.raw = ld_shared_v4(sO + off);
        float gf[8], of[8];
        go.unpack(gf);
        oo.unpack(of);
#pragma unroll
        for (int e = 0; e < 8; ++e) Dp = fmaf(gf[e], of[e], Dp);
      }
      s_dhalf[wg * 128 + r] = Dp;
      named_bar_sync(1, 256);                  // every row is done with the O tile
      const float Dr = s_dhalf[r] + s_dhalf[128 + r];
      // the previous item's dQ leaves now, staged in the O tile, while this
      // item's first S and dP are on their way (its last dQ product is done)
      if (pend) {
        if (!mbar_wait_bounded(B(DQD), (nb - 1) & 1, p.status, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        epilogue();
        pend = false;
      }
      // the next item's Q, dO and O may load once the stores have read their
      // staging buffers
      if (lane == 0) bulk_wait_read0();
      __syncwarp();
      mbar_arrive(B(DE));
      const size_t lrow = ((size_t)it.b * p.heads + it.hd) * p.seq + qb * 128 + r;
      if (wg == 0) p.dsum[lrow] = Dr;
      const float lse2 = p.lse[lrow] * LOG2E;
      for (int j = 0; j <= qb; ++j, ++nb) {
        uint32_t keep[2] = {0xffffffffu, 0xffffffffu};
        if (DROP) {
          const uint32_t* mt = mask_tile(p, it.b, it.hd, qb, j);
          keep[0] = mt[(2 * wg) * 128 + r];
          keep[1] = mt[(2 * wg + 1) * 128 + r];
        }
        if (!mbar_wait_bounded(B(SF), nb & 1, p.status, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        float ds[64];
        {
          uint32_t s0[32], s1[32], d0[32], d1[32];
          tmem_ld32(tmem + TQ_S + lane_off + 64 * wg, s0);
          tmem_ld32(tmem + TQ_S + lane_off + 64 * wg + 32, s1);
          tmem_ld32(tmem + TQ_DP + lane_off + 64 * wg, d0);
          tmem_ld32(tmem + TQ_DP + lane_off + 64 * wg + 32, d1);
          tmem_ld_wait();
          tc_fence_before();
          mbar_arrive(B(SE));                    // S, dP may take the next block
          // the previous dQ product has read dS (and, at an item's first block,
          // finished the previous item's dQ)
          if (nb > 0 && !mbar_wait_bounded(B(DQD), (nb - 1) & 1, p.status, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const bool diag = j == qb;
          const float nl = -lse2;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            // 32 columns: exponentials, dS, and their bf16 store while the next
            // half is computed
#pragma unroll
            for (int c = 32 * h; c < 32 * h + 32; c += 2) {
              float x0, x1;
              ffma2(x0, x1, __uint_as_float(h ? s1[c - 32] : s0[c]),
                    __uint_as_float(h ? s1[c - 31] : s0[c + 1]), p.scale_log2, p.scale_log2, nl, nl);
              float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
              if (diag && 64 * wg + c > r) p0 = 0.f;
              if (diag && 64 * wg + c + 1 > r) p1 = 0.f;
              const float dv0 = __uint_as_float(h ? d1[c - 32] : d0[c]);
              const float dv1 = __uint_as_float(h ? d1[c - 31] : d0[c + 1]);
              const float dp0 = ((keep[h] >> (c & 31)) & 1u) ? dv0 * dsc : 0.f;
              const float dp1 = ((keep[h] >> ((c + 1) & 31)) & 1u) ? dv1 * dsc : 0.f;
              ds[c] = p0 * (dp0 - Dr);
              ds[c + 1] = p1 * (dp1 - Dr);
            }
            uint32_t pk[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) pk[c] = pack_bf16x2(ds[32 * h + 2 * c], ds[32 * h + 2 * c + 1]);
            tmem_st16(tmem + TQ_DS + lane_off + 32 * wg + 16 * h, pk);
          }
        }
        if (!ok) break;
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(B(DSF));
      }
      if (!ok) break;
      pend = true;
      px = it.hd * 3 * D;
      py = it.b * p.seq + qb * 128 + q4 * 32;
    }
    if (ok && pend && mbar_wait_bounded(B(DQD), (nb - 1) & 1, p.status, abort_flag)) {
      tc_fence_after();
      epilogue();
    }
    if (lane == 0) bulk_wait0();   // this warp's stores are done before shared memory goes
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

// Shared memory of the dK/dV kernel with `kvb` K/V buffers of `tile` bytes.
__host__ __device__ constexpr size_t dkv_need(uint32_t tile, int kvb) {
  return (size_t)(2 * kvb + BWD_RING) * tile + STAGE_BYTES + 2048 + 256 + 1024;
}
// K and V are double-buffered when the tiles leave room (d = 64, 96), so the
// next item's K and V load while the current item runs.
__host__ __device__ constexpr int dkv_kv_bufs(uint32_t tile) { return dkv_need(tile, 2) <= kSmemMax ? 2 : 1; }

// ============================================================================ dK, dV
// Item: 128 keys (K, V resident) against query blocks i = kb..nqb-1 (Q(i) with
// the lse and D of its queries, dO(i): through the ring).  Per block: S^T =
// K Q^T, then dP^T = V dO^T into the same TMEM columns once the row threads
// have read S^T (warp 1); the row threads' P^T (with the forward's keep mask
// and scale) and dS^T = P^T * (dP^T - D), written to TMEM as bf16; dV += P^T
// dO and dK += dS^T Q (warp 2, A operands from TMEM).  An item's dK and dV are
// written out when the rows take the next item (its last dV and dK products
// done), while that item's K, V and first S^T are on their way.
// smem: K and V (two pairs where they fit: dkv_kv_bufs), ring[BWD_RING] (tiles
// in the Fmt layout), the epilogue staging buffers, lse and D of the two Q
// slots, item ids.  TMEM: S^T / dP^T 0..127, P^T 128..191, dS^T 192..255,
// dV 256.., dK 384..
constexpr uint32_t TK_S = 0, TK_P = 128, TK_DS = 192, TK_DV = 256, TK_DK = 384;

template <int KS, bool DROP>
__global__ void __launch_bounds__(BWD_THREADS, 1)
    attn_bwd_dkv_tc_kernel(const __grid_constant__ CUtensorMap tm,
                           const __grid_constant__ CUtensorMap tmdo,
                           const __grid_constant__ CUtensorMap tmdq, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  const Smem sm = smem_aligned(smem_raw);
  using F = Fmt<KS>;
  constexpr uint32_t TILE = F::TILE;
  constexpr int D = KS * 16;
  constexpr int NKV = dkv_kv_bufs(TILE);   // K/V buffers: item m uses buffer m % NKV
  const uint32_t sK = sm.u32, sR0 = sK + 2 * NKV * TILE;   // K(u) at sK + 2u TILE, V(u) after it
  const uint32_t sStage = sR0 + BWD_RING * TILE;           // epilogue staging, 2 KB a row warp
  // lse, D of the queries in Q slot 2m: 128 + 128 floats at s_ld + 256 m
  float* s_ld = reinterpret_cast<float*>(sm.base + (2 * NKV + BWD_RING) * TILE + STAGE_BYTES);
  const uint32_t s_ld_u32 = smem_u32(s_ld);
  uint64_t* bars = reinterpret_cast<uint64_t*>(s_ld + 128 * BWD_RING);
  const uint32_t bar0 = smem_u32(bars);
  auto B = [&](int i) { return bar0 + 8u * i; };
  // KVF / KVE: one barrier per K/V buffer
  constexpr int KVF = 0, KVE = 2, RF = 4, RE = RF + BWD_RING, SF = RE + BWD_RING, SE = SF + 1,
                DPF = SE + 1, DPE = DPF + 1, PF = DPE + 1, PE = PF + 1, DSF = PE + 1,
                DSE = DSF + 1, IF = DSE + 1, IE = IF + 2, NBAR = IE + 2;
  int* s_item = reinterpret_cast<int*>(bars + NBAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(s_item + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const ItemRing iq{s_item, B(IF), B(IE)};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_items = p.nqb * p.heads * p.batch;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NBAR; ++i) {
      uint32_t cnt = 1;
      if (i == SE || i == DPE || i == PF || i == DSF) cnt = 256;
      if (i == IE || i == IE + 1) cnt = 2 + 8;
      if (i >= RE && i < RE + BWD_RING) cnt = 2;           // Q and dO: both issuers
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
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(BWD_LOW_REGS));
    if (lane == 0) {
      tma_prefetch_desc(&tm);
      tma_prefetch_desc(&tmdo);
      int g = 0, ni = 0, nit = 0;
      bool ok = true;
      while (ok) {
        const int k = (int)atomicAdd(p.sched, 1u);
        if (!item_publish(iq, ni++, k, p.status, abort_flag) || k >= n_items) break;
        const BwdItem it = bwd_item(p, k, false);
        const int colq = it.hd * 3 * p.d, row0 = it.b * p.seq;
        // K and V of item nit into buffer u once item nit - NKV is done with it
        const int u = nit % NKV, use = nit / NKV;
        if (use > 0 && !mbar_wait_bounded(B(KVE + u), (use - 1) & 1, p.status, abort_flag)) break;
        ++nit;
        const uint32_t sKu = sK + 2 * u * TILE, sVu = sKu + TILE;
        mbar_arrive_expect_tx(B(KVF + u), 2 * TILE);
        for (int a = 0; a < F::ATOMS; ++a) {
          load_box(sKu + a * F::ATOM, &tm, B(KVF + u), colq + p.d + F::ACOLS * a, row0 + it.blk * 128,
                   3 * (int64_t)p.h, (int64_t)p.batch * p.seq, p.status, bounds::kSiteAttnDkvLoad, F::ACOLS);
          load_box(sVu + a * F::ATOM, &tm, B(KVF + u), colq + 2 * p.d + F::ACOLS * a, row0 + it.blk * 128,
                   3 * (int64_t)p.h, (int64_t)p.batch * p.seq, p.status, bounds::kSiteAttnDkvLoad, F::ACOLS);
        }
        for (int i = it.blk; i < p.nqb && ok; ++i) {
          for (int qd = 0; qd < 2; ++qd, ++g) {
            const int s = g % BWD_RING, use = g / BWD_RING;
            if (use > 0 && !mbar_wait_bounded(B(RE + s), (use - 1) & 1, p.status, abort_flag)) {
              ok = false;
              break;
            }
            if (qd == 0) {
              // Q(i) with the lse and D of its queries
              mbar_arrive_expect_tx(B(RF + s), TILE + 1024);
              for (int a = 0; a < F::ATOMS; ++a)
                load_box(sR0 + s * TILE + a * F::ATOM, &tm, B(RF + s), colq + F::ACOLS * a, row0 + i * 128,
                         3 * (int64_t)p.h, (int64_t)p.batch * p.seq, p.status, bounds::kSiteAttnDkvQ, F::ACOLS);
              const size_t lo = ((size_t)it.b * p.heads + it.hd) * p.seq + (size_t)i * 128;
              bulk_load(s_ld_u32 + (s >> 1) * 1024, p.lse + lo, 512, B(RF + s));
              bulk_load(s_ld_u32 + (s >> 1) * 1024 + 512, p.dsum + lo, 512, B(RF + s));
            } else {
              mbar_arrive_expect_tx(B(RF + s), TILE);
              for (int a = 0; a < F::ATOMS; ++a)
                load_box(sR0 + s * TILE + a * F::ATOM, &tmdo, B(RF + s), it.hd * p.d + F::ACOLS * a,
                         row0 + i * 128, (int64_t)p.h, (int64_t)p.batch * p.seq, p.status, bounds::kSiteAttnDkvQ,
                         F::ACOLS);
            }
          }
        }
      }
      sched_done(p.sched);
    }
    __syncwarp();
  } else if (warp == 1 || warp == 2) {
    // ---------------------------------- MMA issuers: warp 1 S^T, dP^T; warp 2 dV, dK
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(BWD_LOW_REGS));
    if (lane == 0) {
      const bool first = warp == 1;
      const uint32_t id_s = idesc_bf16_f32(128, 128, false, false);
      const uint32_t id_acc = idesc_bf16_f32(128, D, false, true);
      const uint64_t dK0 = F::kdesc(sK), dR0 = F::kdesc(sR0);
      const uint64_t dRmn0 = F::mndesc(sR0);
      int g = 0, ni = 0, nit = 0, nb = 0;
      bool ok = true;
      auto wait = [&](int bar, int k) -> bool {
        if (!mbar_wait_bounded(B(bar), k & 1, p.status, abort_flag)) ok = false;
        return ok;
      };
      while (ok) {
        int k;
        if (!item_take(iq, ni++, true, k, p.status, abort_flag)) break;
        if (k >= n_items) break;
        const BwdItem it = bwd_item(p, k, false);
        const int nq = p.nqb - it.blk;
        const int u = nit % NKV;
        const uint64_t dKd = desc_add(dK0, 2 * u * TILE), dVd = desc_add(dKd, TILE);
        for (int i = 0; i < nq && ok; ++i, ++nb) {
          const int gq = g + 2 * i, gd = gq + 1;
          const int sq = gq % BWD_RING, sd = gd % BWD_RING;
          if (first) {
            if (i == 0 && !wait(KVF + u, nit / NKV)) break;
            if (!wait(RF + sq, gq / BWD_RING)) break;
            if (nb > 0 && !wait(DPE, nb - 1)) break;   // the rows hold dP^T of the last block
            tc_fence_after();
            const uint64_t dQ = desc_add(dR0, sq * TILE), dDO = desc_add(dR0, sd * TILE);
#pragma unroll
            for (int kk = 0; kk < KS; ++kk)
              tc_mma_bf16(tmem + TK_S, desc_add(dKd, F::koff(kk)), desc_add(dQ, F::koff(kk)), id_s,
                          kk > 0);
            tc_commit(B(SF));
            tc_commit(B(RE + sq));
            if (!wait(RF + sd, gd / BWD_RING) || !wait(SE, nb)) break;   // rows read S^T
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < KS; ++kk)
              tc_mma_bf16(tmem + TK_S, desc_add(dVd, F::koff(kk)), desc_add(dDO, F::koff(kk)), id_s,
                          kk > 0);
            tc_commit(B(DPF));
            tc_commit(B(RE + sd));
            if (i == nq - 1) tc_commit(B(KVE + u));
          } else {
            if (!wait(PF, nb) || !wait(RF + sd, gd / BWD_RING)) break;
            tc_fence_after();
            const uint64_t dDOmn = desc_add(dRmn0, sd * TILE), dQmn = desc_add(dRmn0, sq * TILE);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              tc_mma_bf16_ts(tmem + TK_DV, tmem + TK_P + 8 * kk, desc_add(dDOmn, F::mnoff(kk)),
                             id_acc, (i > 0 || kk > 0) ? 1u : 0u);
            tc_commit(B(PE));
            tc_commit(B(RE + sd));
            if (!wait(DSF, nb) || !wait(RF + sq, gq / BWD_RING)) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              tc_mma_bf16_ts(tmem + TK_DK, tmem + TK_DS + 8 * kk, desc_add(dQmn, F::mnoff(kk)),
                             id_acc, (i > 0 || kk > 0) ? 1u : 0u);
            tc_commit(B(DSE));
            tc_commit(B(RE + sq));
          }
        }
        if (!ok) break;
        g += 2 * nq;
        ++nit;
      }
    }
    __syncwarp();
  } else if (warp == 3) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(BWD_LOW_REGS));
  } else {
    // ---------------------------------------------------------------- row threads
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(BWD_ROW_REGS));
    const int wg = (warp - 4) >> 2;            // query columns 64 wg .. 64 wg + 63
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;              // key row = TMEM lane
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    const float dsc = DROP ? p.drop.scale : 1.0f;
    int ni = 0, nb = 0, g = 0;
    bool pend = false;
    int px = 0, py = 0;                        // dqkv column of the pending dK, the warp's first row
    const uint32_t stage = sStage + (warp - 4) * STAGE_WARP_BYTES;
    auto epilogue = [&]() {
      // warpgroup 0 writes dK (with the 1/sqrt(d) of S), warpgroup 1 dV
      const uint32_t src = tmem + (wg == 0 ? TK_DK : TK_DV) + lane_off;
      const float sc = wg == 0 ? p.scale : 1.0f;
      const int x = px + (wg == 0 ? 0 : D);
      if (!store_box_ok(p.status, x, py, 3 * (int64_t)p.h, (int64_t)p.batch * p.seq, bounds::kSiteAttnDkvOut))
        return;
#pragma unroll 1
      for (int c = 0; c < D; c += 32) store_acc32_tma(src + c, sc, &tmdq, x + c, py, stage, lane);
    };
    bool ok = true;
    while (ok) {
      int k;
      if (!item_take(iq, ni++, lane == 0, k, p.status, abort_flag)) {
        ok = false;
        break;
      }
      if (k >= n_items) break;
      const BwdItem it = bwd_item(p, k, false);
      const int kb = it.blk, nq = p.nqb - kb;
      // the previous item's dK and dV leave while this item's K and V load
      // and its first S^T is computed: its last dV and dK products are done
      if (pend) {
        if (!mbar_wait_bounded(B(PE), (nb - 1) & 1, p.status, abort_flag) ||
            !mbar_wait_bounded(B(DSE), (nb - 1) & 1, p.status, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        epilogue();
        pend = false;
      }
      for (int i = 0; i < nq; ++i, ++nb) {
        const int qb = kb + i;
        const int sq = (g + 2 * i) % BWD_RING;
        uint32_t kword[2] = {0u, 0u};
        if (DROP) {
          // the forward's keep words of queries 64 wg + 32 t + lane over this
          // warp's 32 keys; a warp transpose hands lane k the word over queries
          const uint32_t* mt = mask_tile(p, it.b, it.hd, qb, kb);
          kword[0] = mt[q4 * 128 + 64 * wg + lane];
          kword[1] = mt[q4 * 128 + 64 * wg + 32 + lane];
        }
        if (!mbar_wait_bounded(B(SF), nb & 1, p.status, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        float pr[64];
        {
          uint32_t s0[32], s1[32];
          tmem_ld32(tmem + TK_S + lane_off + 64 * wg, s0);
          tmem_ld32(tmem + TK_S + lane_off + 64 * wg + 32, s1);
          tmem_ld_wait();
          tc_fence_before();
          mbar_arrive(B(SE));                    // dP^T may take the S^T columns
          // lse of this block's queries came with Q(i): observe that load
          if (!mbar_wait_bounded(B(RF + sq), ((g + 2 * i) / BWD_RING) & 1, p.status,
                                 abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t keep0 = DROP ? warp_transpose32(kword[0], lane) : 0xffffffffu;
          const uint32_t keep1 = DROP ? warp_transpose32(kword[1], lane) : 0xffffffffu;
          // P^T is free once the previous dV product is done
          if (nb > 0 && !mbar_wait_bounded(B(PE), (nb - 1) & 1, p.status, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const float* lse = s_ld + (sq >> 1) * 256 + 64 * wg;
          const bool diag = i == 0;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            // 32 query columns: P, and the dropped and scaled P^T stored while the
            // next half is computed
            const uint32_t keep = h ? keep1 : keep0;
#pragma unroll
            for (int c = 32 * h; c < 32 * h + 32; c += 4) {
              const float4 l4 = *reinterpret_cast<const float4*>(lse + c);
              float x0, x1, x2, x3;
              ffma2(x0, x1, __uint_as_float(h ? s1[c - 32] : s0[c]),
                    __uint_as_float(h ? s1[c - 31] : s0[c + 1]), p.scale_log2, p.scale_log2,
                    -l4.x * LOG2E, -l4.y * LOG2E);
              ffma2(x2, x3, __uint_as_float(h ? s1[c - 30] : s0[c + 2]),
                    __uint_as_float(h ? s1[c - 29] : s0[c + 3]), p.scale_log2, p.scale_log2,
                    -l4.z * LOG2E, -l4.w * LOG2E);
              pr[c] = fast_exp2(x0);
              pr[c + 1] = fast_exp2(x1);
              pr[c + 2] = fast_exp2(x2);
              pr[c + 3] = fast_exp2(x3);
#pragma unroll
              for (int e = 0; e < 4; ++e)
                if (diag && 64 * wg + c + e < r) pr[c + e] = 0.f;   // query before the key
            }
            uint32_t pk[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              const int c0 = 32 * h + 2 * c;
              const float t0 = ((keep >> (2 * c)) & 1u) ? pr[c0] * dsc : 0.f;
              const float t1 = ((keep >> (2 * c + 1)) & 1u) ? pr[c0 + 1] * dsc : 0.f;
              pk[c] = pack_bf16x2(t0, t1);
            }
            tmem_st16(tmem + TK_P + lane_off + 32 * wg + 16 * h, pk);
          }
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(B(PF));
          // dP^T
          if (!mbar_wait_bounded(B(DPF), nb & 1, p.status, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          uint32_t d0[32], d1[32];
          tmem_ld32(tmem + TK_S + lane_off + 64 * wg, d0);
          tmem_ld32(tmem + TK_S + lane_off + 64 * wg + 32, d1);
          tmem_ld_wait();
          tc_fence_before();
          mbar_arrive(B(DPE));                   // S^T / dP^T columns free
          // dS^T is free once the previous dK product is done
          if (nb > 0 && !mbar_wait_bounded(B(DSE), (nb - 1) & 1, p.status, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const float* dsum = s_ld + (sq >> 1) * 256 + 128 + 64 * wg;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t keep = h ? keep1 : keep0;
            uint32_t pk[16];
#pragma unroll
            for (int c = 0; c < 32; c += 4) {
              const float4 d4 = *reinterpret_cast<const float4*>(dsum + 32 * h + c);
              const float dvv[4] = {d4.x, d4.y, d4.z, d4.w};
              float v[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int cc = c + e;
                const bool kept = ((keep >> cc) & 1u) != 0;
                const float dp = kept ? __uint_as_float(h ? d1[cc] : d0[cc]) * dsc : 0.f;
                v[e] = pr[32 * h + cc] * (dp - dvv[e]);   // dS^T
              }
              pk[c / 2] = pack_bf16x2(v[0], v[1]);
              pk[c / 2 + 1] = pack_bf16x2(v[2], v[3]);
            }
            tmem_st16(tmem + TK_DS + lane_off + 32 * wg + 16 * h, pk);
          }
        }
        if (!ok) break;
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(B(DSF));
      }
      if (!ok) break;
      g += 2 * nq;
      pend = true;
      px = it.hd * 3 * D + D;
      py = it.b * p.seq + kb * 128 + q4 * 32;
    }
    if (ok && pend && mbar_wait_bounded(B(PE), (nb - 1) & 1, p.status, abort_flag) &&
        mbar_wait_bounded(B(DSE), (nb - 1) & 1, p.status, abort_flag)) {
      tc_fence_after();
      epilogue();
    }
    if (lane == 0) bulk_wait0();   // this warp's stores are done before shared memory goes
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

// A bf16 [rows][cols] tensor in boxes of box_cols x box_rows (64 x box_rows
// with 128-byte swizzle for the operand loads; 32 x 32 with 64-byte swizzle
// for the epilogue stores).
bool make_map(CUtensorMap* m, const void* ptr, uint64_t cols, uint64_t rows, uint32_t box_rows,
              uint32_t box_cols = 64, CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_128B) {
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
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t fwd_smem(uint32_t tile) {
  const size_t need = (size_t)(2 + FWD_RING) * tile + STAGE_BYTES + 256 + 1024;
  return need < 120 * 1024 ? 120 * 1024 : need;   // one CTA per SM (512 TMEM columns)
}
// The backward kernels hold all 512 TMEM columns: their shared memory requests
// keep them at one CTA per SM so a second CTA never waits in tcgen05.alloc.
size_t dq_smem(uint32_t tile) {
  const size_t need = dq_need(tile, dq_q_bufs(tile));
  return need < 120 * 1024 ? 120 * 1024 : need;   // one CTA per SM (512 TMEM columns)
}
size_t dkv_smem(uint32_t tile) {
  const size_t need = dkv_need(tile, dkv_kv_bufs(tile));
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

// (batch, head) pairs per scheduling chunk: pairs whose two streamed operands
// (d bf16 a row each) fit in about 48 MB of L2 together.
int l2_chunk(int batch, int seq, int heads, int d) {
  const size_t per_pair = 2ull * seq * d * 2;
  const size_t c = ((size_t)48 << 20) / per_pair;
  const size_t pairs = (size_t)batch * heads;
  return c < 1 ? 1 : (int)(c > pairs ? pairs : c);
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
  CUtensorMap tm, tmc;
  const bool sw64 = d % 64 != 0;   // the operand tiles' format (Fmt)
  const uint32_t acols = sw64 ? 32 : 64;
  const CUtensorMapSwizzle asw = sw64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
  if (!make_map(&tm, qkv, 3ull * heads * d, (uint64_t)batch * seq, 128, acols, asw) ||
      !make_map(&tmc, ctx, (uint64_t)heads * d, (uint64_t)batch * seq, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  if (drop.on && !mask) return cudaErrorInvalidValue;
  Params p = make_params(batch, seq, heads, d, status, drop);
  p.mask = mask;
  p.ctx = static_cast<bf16*>(ctx);
  p.lse = lse;
  p.sched = status + kSchedFwd;
  p.chunk = l2_chunk(batch, seq, heads, d);
  const int items = ((p.nqb + 1) / 2) * heads * batch;
  const int grid = items < c.num_sms ? items : c.num_sms;
  const double flops = 2.0 * 2.0 * batch * heads * d * ((double)seq * (seq + 1) / 2.0);
  cudaError_t e;
#define FWD_CASE(KS_, DR_)                                                                         \
  {                                                                                                \
    const size_t sm = fwd_smem(Fmt<KS_>::TILE);                                                    \
    if ((e = set_smem(attn_fwd_tc_kernel<KS_, DR_>, sm)) != cudaSuccess) return e;                 \
    if ((e = check_regs(attn_fwd_tc_kernel<KS_, DR_>, FWD_LAUNCH_REGS)) != cudaSuccess)            \
      return e;                                                                                    \
    c.before(KK_ATTN_FWD, flops);                                                                  \
    attn_fwd_tc_kernel<KS_, DR_><<<grid, FWD_THREADS, sm, c.stream>>>(tm, tmc, p);                 \
  }
  if (drop.on) {
    if (d == 64) FWD_CASE(4, true)
    else if (d == 96) FWD_CASE(6, true)
    else FWD_CASE(8, true)
  } else {
    if (d == 64) FWD_CASE(4, false)
    else if (d == 96) FWD_CASE(6, false)
    else FWD_CASE(8, false)
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
  CUtensorMap tm, tmdo, tmo, tmdq;
  const bool sw64 = d % 64 != 0;   // the operand tiles' format (Fmt)
  const uint32_t acols = sw64 ? 32 : 64;
  const CUtensorMapSwizzle asw = sw64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
  if (!make_map(&tm, qkv, 3ull * heads * d, n, 128, acols, asw) ||
      !make_map(&tmdo, dctx, (uint64_t)heads * d, n, 128, acols, asw) ||
      !make_map(&tmo, ctx, (uint64_t)heads * d, n, 128, acols, asw) ||
      !make_map(&tmdq, dqkv, 3ull * heads * d, n, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  if (drop.on && !mask) return cudaErrorInvalidValue;
  Params p = make_params(batch, seq, heads, d, status, drop);
  p.mask = const_cast<uint32_t*>(mask);
  p.ctx = static_cast<bf16*>(const_cast<void*>(ctx));
  p.lse = const_cast<float*>(lse);
  p.dctx = static_cast<const bf16*>(dctx);
  p.dqkv = static_cast<bf16*>(dqkv);
  p.dsum = dsum;
  p.chunk = l2_chunk(batch, seq, heads, d);
  const int items = p.nqb * heads * batch;
  const int grid = items < c.num_sms ? items : c.num_sms;
  const double tri = (double)batch * heads * d * ((double)seq * (seq + 1) / 2.0);
  cudaError_t e;
#define BWD_CASE(KS_, DR_)                                                                         \
  {                                                                                                \
    auto kq = attn_bwd_dq_tc_kernel<KS_, DR_>;                                                     \
    auto kk = attn_bwd_dkv_tc_kernel<KS_, DR_>;                                                    \
    if ((e = set_smem(kq, dq_smem(Fmt<KS_>::TILE))) != cudaSuccess) return e;                      \
    if ((e = set_smem(kk, dkv_smem(Fmt<KS_>::TILE))) != cudaSuccess) return e;                     \
    if ((e = check_regs(kq, BWD_LAUNCH_REGS)) != cudaSuccess) return e;                            \
    if ((e = check_regs(kk, BWD_LAUNCH_REGS)) != cudaSuccess) return e;                            \
    c.before(KK_ATTN_BWD, 2.0 * 3.0 * tri);                                                        \
    p.sched = status + kSchedDq;                                                                   \
    kq<<<grid, BWD_THREADS, dq_smem(Fmt<KS_>::TILE), c.stream>>>(tm, tmdo, tmo, tmdq, p);          \
    c.after();                                                                                     \
    if ((e = cudaGetLastError()) != cudaSuccess) return e;                                         \
    c.before(KK_ATTN_BWD, 2.0 * 4.0 * tri);                                                        \
    p.sched = status + kSchedDkv;                                                                  \
    kk<<<grid, BWD_THREADS, dkv_smem(Fmt<KS_>::TILE), c.stream>>>(tm, tmdo, tmdq, p);              \
    c.after();                                                                                     \
  }
  if (drop.on) {
    if (d == 64) BWD_CASE(4, true)
    else if (d == 96) BWD_CASE(6, true)
    else BWD_CASE(8, true)
  } else {
    if (d == 64) BWD_CASE(4, false)
    else if (d == 96) BWD_CASE(6, false)
    else BWD_CASE(8, false)
  }
#undef BWD_CASE
  return cudaGetLastError();
}

}  // namespace mtl
