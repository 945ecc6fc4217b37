// Internal host-side launchers of the layer's kernels (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace mtl {

enum DType { kF32 = 0, kBF16 = 1 };

// GEMM epilogues (the numbering is the one mtl_gemm exposes).
enum Epi { EPI_STORE = 0, EPI_BIAS = 1, EPI_BIAS_RESID = 2, EPI_BIAS_GELU = 3, EPI_DGELU = 4 };

// Dropout of one site: element e is kept iff word(e) >= thresh and a kept value
// is multiplied by scale = 1 / (1 - p).  word(e) is lane e mod 4 of the
// Philox4x32-10 block at counter (e div 4 as two 32-bit words, site, 0) under
// the key (seed low word, seed high word).  on == 0: no dropout (p = 0).
enum DropSite { SITE_ATTN = 0, SITE_OUT = 1, SITE_FC2 = 2 };
struct Dropout {
  unsigned long long seed;
  uint32_t thresh;   // floor(p * 2^32)
  float scale;       // 1 / (1 - p)
  uint32_t site;
  int on;
  // Philox round keys: rk[2r], rk[2r+1] = the key of round r (seed words plus
  // r times the Weyl increments), precomputed so the kernels read them from
  // parameter space.
  uint32_t rk[20];
};

// A(m,k) = ptr[m*ld + k] when k_major, else ptr[k*ld + m].
struct GemmOperand {
  const void* ptr;
  int64_t ld;
  bool k_major;
};

// C[m][n] = epi( sum over parts p in order of ( sum_{k in part p} A(m,k) B(n,k) ) )
struct GemmArgs {
  int M, N, K, parts;
  GemmOperand A, B;
  int epi;
  const void* bias;       // [N] (EPI_BIAS, EPI_BIAS_RESID, EPI_BIAS_GELU)
  const void* R;          // residual [M][ldr] (EPI_BIAS_RESID)
  int64_t ldr;
  void* Z;                // EPI_BIAS_GELU: pre-activation out; EPI_DGELU: pre-activation in
  int64_t ldz;
  void* C;                // output [M][ldc]
  int64_t ldc;
  bool c_f32;             // C stored as fp32 (else as the operand dtype)
  unsigned* status;       // device status word
  Dropout drop;           // EPI_BIAS_RESID: C = R + dropout(acc + bias), e = row * N + col
  // FP8 (gemm_fp8): A and B are bytes of format fmt_a / fmt_b (0 E4M3, 1 E5M2),
  // K-major; the accumulator is scaled by 1 / (scale_a * scale_b) (device floats).
  int fmt_a, fmt_b;
  const float* scale_a;
  const float* scale_b;
  // Scratch of the tensor-core pair GEMM for the K slices of its last,
  // partial wave of tiles (gemm_split_bytes / gemm_split_counters for the
  // sizes; the counters must be zero before the launch and are left zero).
  // Null: every tile runs whole.
  float* split_ws;
  size_t split_ws_bytes;
  unsigned* split_cnt;
  size_t split_cnt_count;
  // EPI_DGELU on the tensor-core path with N % 32 == 0: the column sums of each
  // 32 rows of C as stored go to colsum_part [ceil(M / 32)][N] (fp32), ready
  // for a finalize into the bias gradient.  Null: not computed.
  float* colsum_part;
};

// Scratch the pair GEMM uses for sliced tail tiles with M x N outputs on
// num_sms SMs, for any K: partial-tile bytes and arrival counters (0 when the
// waves are whole).
size_t gemm_split_bytes(int M, int N, int num_sms);
size_t gemm_split_counters(int M, int N, int num_sms);

// Kernel kinds reported through the profiling hooks.
enum KernelKind {
  KK_GEMM_TC = 1, KK_GEMM_SIMT = 2, KK_ATTN_FWD = 3, KK_ATTN_BWD = 4, KK_LN_FWD = 5,
  KK_LN_BWD = 6, KK_COLSUM = 7, KK_FINALIZE = 8, KK_GEMV_TC = 9, KK_ATTN_DECODE = 10,
  KK_KV_WRITE = 11, KK_GEMM_FP8 = 12, KK_QUANT = 13
};

// Optional per-launch timing: when set, events[2i] / events[2i+1] are recorded
// on the launch stream around the i-th kernel, with its kind and work (flops
// for contractions, bytes for memory-bound kernels).
struct Profiler {
  cudaEvent_t* events;
  int capacity;
  int count;
  int* kinds;
  double* work;
};

struct LaunchCtx {
  cudaStream_t stream;
  int num_sms;
  int* launches;          // incremented per kernel enqueued
  Profiler* prof;         // may be null
  bool pdl = false;       // launch with programmatic stream serialization (the
                          // kernels then overlap their start with the previous
                          // kernel's tail; each calls griddep_wait first)

  void before(int kind, double work) const {
    if (prof && prof->events && prof->count < prof->capacity) {
      cudaEventRecord(prof->events[2 * prof->count], stream);
      prof->kinds[prof->count] = kind;
      prof->work[prof->count] = work;
    }
  }
  void after() const {
    ++*launches;
    if (prof && prof->events && prof->count < prof->capacity) {
      cudaEventRecord(prof->events[2 * prof->count + 1], stream);
      ++prof->count;
    }
  }
};

// Launches `kernel` on c.stream with, when c.pdl, programmatic stream
// serialization and, when cluster_y > 1, a (1, cluster_y, 1) thread-block
// cluster.
template <typename... KArgs, typename... Args>
cudaError_t launch_ex(const LaunchCtx& c, void (*kernel)(KArgs...), dim3 grid, dim3 block,
                      size_t smem, int cluster_y, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = c.stream;
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (c.pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster_y > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = 1;
    attr[n].val.clusterDim.y = cluster_y;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// CUDA-core GEMM, exact fp32 math; dtype of operands kF32 or kBF16.
cudaError_t gemm_simt(int dtype, const GemmArgs& a, const LaunchCtx& c);
// tcgen05 / TMEM / TMA GEMM, bf16 operands, fp32 accumulate.
cudaError_t gemm_tc(const GemmArgs& a, const LaunchCtx& c);
// FP8 GEMM on the pair kernel (tcgen05 kind::f8f6f4): K-major byte operands,
// (K / parts) % 128 == 0, lda / ldb multiples of 16, at least 2 SMs.
bool gemm_fp8_supported(const GemmArgs& a, int num_sms);
cudaError_t gemm_fp8(const GemmArgs& a, const LaunchCtx& c);
// Per-tensor FP8 quantization of a bf16 / fp32 matrix [rows][cols] (row pitch
// ld): amax = max |x| into *amax_bits (as float bits; zeroed first by the
// caller), then scale = fmt_max / amax (1 if amax = 0) into *scale and
// q = fp8(x * scale) [rows][cols] with row pitch ldq (RNE, saturating).
// cols % 16 == 0.
cudaError_t fp8_quantize(int src_dtype, const void* x, int64_t rows, int64_t cols, int64_t ld,
                         int fmt, unsigned* amax_bits, float* scale, void* q, int64_t ldq,
                         const LaunchCtx& c);
// The same with an optional row-major copy q (may be null) and an optional
// transposed copy qT [cols][rows] (row pitch ldqT; may be null): one amax pass
// and, with qT, one kernel writing both.  rows % 16 == 0 and cols % 16 == 0.
cudaError_t fp8_quantize2(int src_dtype, const void* x, int64_t rows, int64_t cols, int64_t ld,
                          int fmt, unsigned* amax_bits, float* scale, void* q, int64_t ldq,
                          void* qT, int64_t ldqT, const LaunchCtx& c);
// The two passes of fp8_quantize2 apart: fp8_amax folds max |x| into
// *amax_bits (atomicMax on the float bits); fp8_cast takes a finished
// *amax_bits (from fp8_amax, or from a kernel that read x anyway, such as
// colsum) and writes the scale, q and / or qT.
cudaError_t fp8_amax(int src_dtype, const void* x, int64_t rows, int64_t cols, int64_t ld,
                     unsigned* amax_bits, const LaunchCtx& c);
cudaError_t fp8_cast(int src_dtype, const void* x, int64_t rows, int64_t cols, int64_t ld,
                     int fmt, const unsigned* amax_bits, float* scale, void* q, int64_t ldq,
                     void* qT, int64_t ldqT, const LaunchCtx& c);

// LayerNorm backward without a residual: dx = LN_bwd(du + du2) where du (fp32,
// may be null) and du2 (layer dtype) are the two parts of the upstream
// gradient (the Post-LN layer).
cudaError_t ln_bwd_sum(int dtype, const float* du, const void* du2, const void* x,
                       const float* mean, const float* rstd, const void* g, void* dx,
                       float* dgamma, float* dbeta, float* partial, int n, int h,
                       const LaunchCtx& c);
// Recomputation: u = LN output from saved statistics (bitwise the forward's),
// a = GeLU(z) elementwise (count a multiple of 8).
cudaError_t ln_apply(int dtype, const void* x, const float* mean, const float* rstd,
                     const void* g, const void* b, void* u, int n, int h, const LaunchCtx& c);
cudaError_t gelu_apply(int dtype, const void* z, void* a, int64_t count, const LaunchCtx& c);

// Host check of the shapes gemm_tc accepts.
bool gemm_tc_supported(const GemmArgs& a);

// LayerNorm forward of x [n][h] -> u [n][h], mean and rstd [n] (fp32).  With
// amax_bits, max |u| (of the stored values) is folded into *amax_bits
// (atomicMax on the float bits; the caller zeroes it).
cudaError_t ln_fwd(int dtype, const void* x, const void* gamma, const void* beta, void* u,
                   float* mean, float* rstd, int n, int h, float eps, const LaunchCtx& c,
                   unsigned* amax_bits = nullptr);
// Column-sum finalizes collected for one launch (finalize_jobs): job k adds
// nblk[k] rows of partial sums part[k] [nblk][N] in row order into out[k] [N],
// the same fixed order a finalize of its own uses.
struct FinalizeJobs {
  static constexpr int kMax = 12;
  int n = 0;
  const float* part[kMax];
  float* out[kMax];
  int nblk[kMax], N[kMax];
  bool add(const float* p, int nb, int cols, float* o);
};
// Launches the collected finalizes (one kernel) and empties the list.
cudaError_t finalize_jobs(FinalizeJobs& j, const LaunchCtx& c);

// LayerNorm backward plus residual gradient: dx = resid + LN_bwd(du); du fp32.
// dgamma / dbeta (fp32 [h]) are reduced in a fixed order through `partial`
// (ln_bwd_partial_floats(n, h, sums) floats); with defer, their finalizes join
// *defer instead of running now.  With dresid and ddx (ln_bwd_can_sum), the
// column sums of resid (as read) and of dx (as stored) go to dresid / ddx the
// same way.
cudaError_t ln_bwd(int dtype, const float* du, const void* x, const float* mean,
                   const float* rstd, const void* gamma, const void* resid, void* dx,
                   float* dgamma, float* dbeta, float* partial, int n, int h,
                   const LaunchCtx& c, FinalizeJobs* defer = nullptr, float* dresid = nullptr,
                   float* ddx = nullptr);
size_t ln_bwd_partial_floats(int n, int h, bool sums = false);
bool ln_bwd_can_sum(int dtype, int h);

// out[j] = sum_i Y[i*ld + j] (fp32, fixed order) for j < N, i < n, through
// `partial` (colsum_partial_floats(n, N) floats).  With amax_bits, max |Y| over
// the same elements is also folded into *amax_bits (atomicMax on the float
// bits; the caller zeroes it).
cudaError_t colsum(int dtype, const void* Y, int64_t ld, int n, int N, float* out,
                   float* partial, const LaunchCtx& c, unsigned* amax_bits = nullptr,
                   FinalizeJobs* defer = nullptr);
size_t colsum_partial_floats(int n, int N);
// Column sums of the dropped-out Y: Ym = Y * keep / (1 - p) (element e = row * N
// + col of site drop.site) is written with row pitch ld, out = column sums of Ym
// (before rounding to the storage type).  N % 4 == 0.
cudaError_t colsum_dropout(int dtype, const void* Y, void* Ym, int64_t ld, int n, int N,
                           const Dropout& drop, float* out, float* partial, const LaunchCtx& c);
size_t colsum_dropout_partial_floats(int n, int N);

// Error text for mtl_last_cuda_error, shared by every entry point.
void record_cuda_error(cudaError_t e, const char* where);
void clear_cuda_error();

// Causal attention over a head-interleaved qkv [batch*seq][3h] -> ctx
// [batch*seq][h], lse [batch][heads][seq] (CUDA-core reference kernels).
// `drop`: attention dropout on the probabilities (site SITE_ATTN).
cudaError_t attn_fwd_simt(int dtype, const void* qkv, void* ctx, float* lse, int batch, int seq,
                          int heads, int d, const Dropout& drop, const LaunchCtx& c);
// Backward: dctx -> dqkv [batch*seq][3h]; dsum [batch][heads][seq] is scratch.
cudaError_t attn_bwd_simt(int dtype, const void* qkv, const void* ctx, const float* lse,
                          const void* dctx, void* dqkv, float* dsum, int batch, int seq,
                          int heads, int d, const Dropout& drop, const LaunchCtx& c);

// Causal attention on tcgen05 tensor cores (bf16; seq % 128 == 0, d in
// {64, 96, 128}).  Forward writes ctx and lse; backward writes dqkv and, as
// scratch, dsum [batch][heads][seq].
bool attn_tc_supported(int seq, int d);
// With dropout the forward writes the keep bits to `mask` (attn_mask_bytes) and
// the backward reads them back.
size_t attn_mask_bytes(int batch, int seq, int heads);
cudaError_t attn_fwd_tc(const void* qkv, void* ctx, float* lse, int batch, int seq, int heads,
                        int d, const Dropout& drop, uint32_t* mask, unsigned* status,
                        const LaunchCtx& c);
cudaError_t attn_bwd_tc(const void* qkv, const void* ctx, const float* lse, const void* dctx,
                        void* dqkv, float* dsum, int batch, int seq, int heads, int d,
                        const Dropout& drop, const uint32_t* mask, unsigned* status,
                        const LaunchCtx& c);

// ---------------------------------------------------------------- inference
// Largest token batch of a decode step, and the SM count the decode GEMMs'
// K split assumes at most (so workspace sizes do not depend on the device).
constexpr int kDecodeMaxBatch = 128;
constexpr int kDecodeSmCap = 160;

// Decode GEMM out[b][n] = epi(sum_k W[n][k] X[b][k]) for a few tokens b
// (tcgen05, weights as the M operand, K split across the CTAs of a cluster,
// slices summed in order through distributed shared memory).  epi: EPI_BIAS,
// EPI_BIAS_RESID (+ R[b][n]) or EPI_BIAS_GELU.
bool gemv_tc_supported(int N, int K, int batch);
cudaError_t gemv_tc(int epi, int N, int K, int batch, const void* W, const void* X,
                    const void* bias, const void* R, void* out, unsigned* status,
                    const LaunchCtx& c);
// Decode attention: appends each sequence's new K, V (from qkv [batch][3h]) at
// position cache_len[b] of the [batch][heads][max_seq][d] caches and attends to
// keys 0..cache_len[b]; ctx [batch][h].  part: batch*heads*attn_decode_splits
// *(d+2) floats; counters: batch*heads ints, zero on entry.
int attn_decode_splits(int max_seq);
cudaError_t attn_decode(int dtype, const void* qkv, void* kcache, void* vcache,
                        const int* cache_len, void* ctx, float* part, int* counters, int batch,
                        int heads, int d, int max_seq, double kv_bytes, unsigned* status,
                        const LaunchCtx& c);
// Prefill: K, V of every prompt token to cache positions 0..seq-1, lengths = seq.
cudaError_t kv_write(int dtype, const void* qkv, void* kcache, void* vcache, int* cache_len,
                     int batch, int seq, int heads, int d, int max_seq, const LaunchCtx& c);
// cache_len[b] += 1 (lengths outside [0, max_seq) are left alone).
cudaError_t kv_advance(int* cache_len, int batch, int max_seq, const LaunchCtx& c);

}  // namespace mtl
