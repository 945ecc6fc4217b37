// The C ABI: argument validation, buffer layouts and the stream-ordered launch
// sequence of one pre-LN GPT layer, forward and backward.
//
// Layer ("Megatron-LM: GPU-Cluster Training Parallelism"; sections "Paper 1: BERT
// LayerNorm Rearrangement", "Paper 1: The f/g Conjugate Operators", "Paper 1: QKV
// Column-Parallel Splitting in Detail", "Fused Transformer Kernels"):
//   u1 = LN1(x); qkv = u1 W_qkv^T + b_qkv            (column-parallel, f = identity)
//   ctx = causal softmax(Q K^T / sqrt d) V per head    (local to a partition)
//   x1 = x + b_o + g( sum_p ctx[:, P_p] W_o[:, P_p]^T )(row-parallel + g)
//   u2 = LN2(x1); z = u2 W_fc1^T + b_fc1; a = GeLU(z)  (column-parallel)
//   y  = x1 + b_fc2 + g( sum_p a[:, F_p] W_fc2[:, F_p]^T )
// Backward mirrors it; f sums the partitions' partial input gradients of the
// two column-parallel GEMMs.  g and f are fixed-order sums inside the GEMMs.
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "../../include/mtl.h"
#include "common.cuh"
#include "kernels.h"

using namespace mtl;

namespace {
thread_local char g_cuda_err[256] = {0};
}  // namespace

namespace mtl {
// Records a CUDA failure for mtl_last_cuda_error (used by entry points that
// live in other translation units).
void record_cuda_error(cudaError_t e, const char* where) {
  snprintf(g_cuda_err, sizeof(g_cuda_err), "%s: %s", where, cudaGetErrorString(e));
}
void clear_cuda_error() { g_cuda_err[0] = 0; }
}  // namespace mtl

namespace {

thread_local int g_launches = 0;
thread_local Profiler g_prof = {nullptr, 0, 0, nullptr, nullptr};

constexpr size_t kAlign = 256;
constexpr size_t kStatusBytes = 256;

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

mtl_status cuda_fail(cudaError_t e, const char* where) {
  snprintf(g_cuda_err, sizeof(g_cuda_err), "%s: %s", where, cudaGetErrorString(e));
  return MTL_ERR_CUDA;
}

int device_sm_count() {
  static int counts[64];
  static std::once_flag once[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::call_once(once[dev], [dev]() {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    counts[dev] = v;
  });
  return counts[dev];
}

struct Dims {
  int64_t h, heads, d, seq, batch, n, f, t;
  int dtype;
  size_t esz;
  float p_attn, p_hidden;
  unsigned long long seed;
  int fp8;        // 1: FP8 (E4M3) forward GEMMs; 2: and E5M2 x E4M3 backward GEMMs
  int post_ln;    // 1: Post-LN layer
  int recompute;  // 1: LayerNorm outputs and GeLU(z) recomputed in the backward
};

// Dropout of one site: keep iff the Philox word >= floor(p * 2^32), scale 1/(1-p).
Dropout make_drop(float p, unsigned long long seed, uint32_t site) {
  Dropout d;
  d.seed = seed;
  d.site = site;
  d.on = p > 0.f ? 1 : 0;
  const double t = floor((double)p * 4294967296.0);
  d.thresh = d.on ? (uint32_t)(t > 4294967295.0 ? 4294967295.0 : t) : 0u;
  d.scale = d.on ? (float)(1.0 / (1.0 - (double)p)) : 1.0f;
  uint32_t k0 = (uint32_t)seed, k1 = (uint32_t)(seed >> 32);
  for (int r = 0; r < 10; ++r) {
    d.rk[2 * r] = k0;
    d.rk[2 * r + 1] = k1;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return d;
}

mtl_status validate(const mtl_layer_desc* desc, Dims* o) {
  if (!desc) return MTL_ERR_INVALID_ARG;
  const mtl_layer_desc& d = *desc;
  if (d.h <= 0 || d.heads <= 0 || d.seq <= 0 || d.batch < 0 || d.ffn <= 0 || d.t <= 0)
    return MTL_ERR_INVALID_ARG;
  if (d.dtype != MTL_F32 && d.dtype != MTL_BF16) return MTL_ERR_INVALID_ARG;
  if (!(d.ln_eps > 0.f)) return MTL_ERR_INVALID_ARG;
  if (!(d.p_attn >= 0.f && d.p_attn < 1.f) || !(d.p_hidden >= 0.f && d.p_hidden < 1.f))
    return MTL_ERR_INVALID_ARG;
  if (d.fp8 < 0 || d.fp8 > 2) return MTL_ERR_INVALID_ARG;
  if ((d.post_ln != 0 && d.post_ln != 1) || (d.recompute != 0 && d.recompute != 1))
    return MTL_ERR_INVALID_ARG;
  if (d.h % d.heads) return MTL_ERR_INVALID_ARG;
  if (d.heads % d.t || d.ffn % d.t) return MTL_ERR_INVALID_ARG;
  const int dh = d.h / d.heads;
  if (dh != 64 && dh != 96 && dh != 128) return MTL_ERR_UNSUPPORTED;
  if (d.causal != 1) return MTL_ERR_UNSUPPORTED;
  if ((int64_t)d.batch * d.seq > (int64_t)1 << 30) return MTL_ERR_UNSUPPORTED;
  if (d.dtype == MTL_BF16) {
    if (d.seq % 128 || d.h % 64 || d.ffn % 64) return MTL_ERR_UNSUPPORTED;
    if ((d.h / d.t) % 64 || ((3 * d.h) / d.t) % 64 || (d.ffn / d.t) % 64) return MTL_ERR_UNSUPPORTED;
  } else {
    if (d.h % 4 || d.ffn % 4) return MTL_ERR_UNSUPPORTED;
    if (d.seq > 8192) return MTL_ERR_UNSUPPORTED;
  }
  o->h = d.h;
  o->heads = d.heads;
  o->d = dh;
  o->seq = d.seq;
  o->batch = d.batch;
  o->n = (int64_t)d.batch * d.seq;
  o->f = d.ffn;
  o->t = d.t;
  o->dtype = d.dtype;
  o->esz = d.dtype == MTL_BF16 ? 2 : 4;
  o->p_attn = d.p_attn;
  o->p_hidden = d.p_hidden;
  o->seed = d.seed;
  o->fp8 = d.fp8;
  o->post_ln = d.post_ln;
  o->recompute = d.recompute;
  // the Post-LN variant runs without dropout and with bf16 / fp32 GEMMs
  if (d.post_ln && (d.p_attn > 0.f || d.p_hidden > 0.f || d.fp8)) return MTL_ERR_UNSUPPORTED;
  if (d.fp8) {
    // FP8 GEMMs: bf16 layers without dropout, K partitions of whole 128s
    if (d.dtype != MTL_BF16 || d.p_attn > 0.f || d.p_hidden > 0.f) return MTL_ERR_UNSUPPORTED;
    if (d.h % 128 || (d.h / d.t) % 128 || (d.ffn / d.t) % 128) return MTL_ERR_UNSUPPORTED;
    // hybrid backward: the QKV input-gradient partitions are whole 128s too
    if (d.fp8 == 2 && ((3 * d.h) / d.t) % 128) return MTL_ERR_UNSUPPORTED;
  }
  return MTL_OK;
}

// FP8 hybrid: the forward's transposed FP8 copies that the backward's weight-
// and data-gradient GEMMs read, and their scales.  Scale slot 2i / 2i+1: the
// activation / weight of forward GEMM i (QKV, out-proj, fc1, fc2).
struct Fp8Saved {
  size_t scales, act[4], wt[4], total;
};

Fp8Saved fp8_saved_layout(const Dims& D) {
  Fp8Saved F;
  memset(&F, 0, sizeof(F));
  if (D.fp8 != 2) return F;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += align_up(bytes);
    return at;
  };
  const size_t n = (size_t)D.n, h = (size_t)D.h, f = (size_t)D.f;
  F.scales = take(16 * 4);
  F.act[0] = take(h * n);      // u1^T  [h][n]
  F.act[1] = take(h * n);      // ctx^T [h][n]
  F.act[2] = take(h * n);      // u2^T  [h][n]
  F.act[3] = take(f * n);      // a^T   [f][n]
  F.wt[0] = take(h * 3 * h);   // W_qkv^T [h][3h]
  F.wt[1] = take(h * h);       // W_o^T   [h][h]
  F.wt[2] = take(h * f);       // W_fc1^T [h][f]
  F.wt[3] = take(f * h);       // W_fc2^T [f][h]
  F.total = off;
  return F;
}

mtl_saved_layout saved_layout(const Dims& D) {
  mtl_saved_layout L;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += align_up(bytes);
    return at;
  };
  const size_t nh = (size_t)D.n * D.h * D.esz;
  const size_t nf = (size_t)D.n * D.f * D.esz;
  const bool pre = !D.post_ln;
  // FP8 hybrid keeps FP8 transposed copies for the backward instead of the
  // bf16 LayerNorm outputs and GeLU(z): they are dropped as with recomputation
  const bool rc = D.recompute != 0 || D.fp8 == 2;
  // Pre-LN saves u1, x1, u2 (u1, u2 recomputable); Post-LN saves h1, x1, h2 (x1
  // recomputable); a = GeLU(z) is recomputable in both.
  L.mu1 = take((size_t)D.n * 4);
  L.rstd1 = take((size_t)D.n * 4);
  L.u1 = take(pre && !rc ? nh : 0);
  L.qkv = take(3 * nh);
  L.ctx = take(nh);
  L.lse = take((size_t)D.batch * D.heads * D.seq * 4);
  L.x1 = take(pre || !rc ? nh : 0);
  L.mu2 = take((size_t)D.n * 4);
  L.rstd2 = take((size_t)D.n * 4);
  L.u2 = take(pre && !rc ? nh : 0);
  L.z = take(nf);
  L.a = take(rc ? 0 : nf);
  L.attn_mask = take(D.dtype == MTL_BF16 && D.p_attn > 0.f
                         ? attn_mask_bytes((int)D.batch, (int)D.seq, (int)D.heads)
                         : 0);
  L.h1 = take(pre ? 0 : nh);
  L.h2 = take(pre ? 0 : nh);
  L.fp8 = take(fp8_saved_layout(D).total);
  L.total = off;
  return L;
}

// FP8 scratch of the forward: amax words and scales of the 8 quantized
// operands, one activation buffer and one weight buffer (reused GEMM by GEMM).
struct Fp8Ws {
  size_t stats, qa, qb, gq, gqT, total;
};

Fp8Ws fp8_ws_layout(const Dims& D) {
  Fp8Ws F{0, 0, 0, 0, 0, 0};
  if (!D.fp8) return F;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += align_up(bytes);
    return at;
  };
  const size_t wide = (size_t)(D.f > D.h ? D.f : D.h);
  const size_t wmax = (size_t)(D.f > 3 * D.h ? D.f : 3 * D.h) * D.h;
  F.stats = take(128);                    // 16 amax words, 16 scales
  F.qa = take((size_t)D.n * wide);        // activation (forward) / its transpose (backward)
  F.qb = take(wmax);                      // weight (forward) / its transpose (backward)
  const size_t gwide = (size_t)(D.f > 3 * D.h ? D.f : 3 * D.h);
  F.gq = take(D.fp8 == 2 ? (size_t)D.n * gwide : 0);     // gradient, and its transpose
  F.gqT = take(D.fp8 == 2 ? (size_t)D.n * gwide : 0);
  F.total = off;
  return F;
}

// Scratch of the pair GEMM's sliced tail tiles for the GEMMs of the current layer
// call on this thread (set by the layer entry points for their duration).
struct SplitScratch {
  float* ws;
  size_t bytes;
  unsigned* cnt;
  size_t count;
};
thread_local SplitScratch g_split = {nullptr, 0, nullptr, 0};

struct SplitScope {
  explicit SplitScope(const SplitScratch& s) { g_split = s; }
  ~SplitScope() { g_split = {nullptr, 0, nullptr, 0}; }
};

// SM count the tail-slice scratch of the layer's GEMMs is sized for: the
// device's, or a GB300's (152) where no device answers (sizes asked for on a
// host without a GPU).
int split_sms() {
  const int n = device_sm_count();
  return n > 0 ? n : 152;
}

// Tail-slice scratch (bytes, counters) that covers every bf16 GEMM of the layer.
void layer_split_sizes(const Dims& D, size_t* bytes, size_t* counters) {
  *bytes = 0;
  *counters = 0;
  if (D.dtype != MTL_BF16) return;
  const int n = (int)D.n, h = (int)D.h, f = (int)D.f, nsm = split_sms();
  const int shapes[7][2] = {{n, 3 * h}, {n, h}, {n, f}, {h, f}, {f, h}, {h, h}, {3 * h, h}};
  for (const auto& mn : shapes) {
    const size_t b = gemm_split_bytes(mn[0], mn[1], nsm);
    const size_t c = gemm_split_counters(mn[0], mn[1], nsm);
    if (b > *bytes) *bytes = b;
    if (c > *counters) *counters = c;
  }
}

// Partial column sums of the Pre-LN backward, all kept until its one finalize
// launch at the end (float offsets into the workspace's partial region): LN2
// (dgamma2, dbeta2 and, folded in, db_fc2 and db_o), LN1 (dgamma1, dbeta1),
// db_fc1 (from the fc2-dgrad epilogue, or a column sum of dz), db_qkv, db_fc2
// and db_o when not folded, and the dropout column sums (finalized at once).
struct PartialLayout {
  size_t ln2, ln1, dz, qkv, b2, bo, drop, total;
};

PartialLayout partial_layout(const Dims& D) {
  PartialLayout P;
  size_t off = 0;
  auto take = [&](size_t floats) {
    const size_t at = off;
    off += (floats + 63) / 64 * 64;
    return at;
  };
  const int n = (int)D.n, h = (int)D.h, f = (int)D.f;
  P.ln2 = take(ln_bwd_partial_floats(n, h, true));
  P.ln1 = take(ln_bwd_partial_floats(n, h, false));
  const size_t dz_epi = (size_t)((n + 31) / 32) * f;
  const size_t dz_col = colsum_partial_floats(n, f);
  P.dz = take(dz_epi > dz_col ? dz_epi : dz_col);
  P.qkv = take(colsum_partial_floats(n, 3 * h));
  P.b2 = take(colsum_partial_floats(n, h));
  P.bo = take(colsum_partial_floats(n, h));
  P.drop = take(colsum_dropout_partial_floats(n, h));
  P.total = off;
  return P;
}

// Backward scratch, after the status word.  The GEMMs' tail-slice counters
// come first, so that one memset clears them with the status word.
struct WsLayout {
  size_t split_cnt, dz, du, dx1, dctx, dqkv, dsum, gmask, partial, fp8, rc_h, rc_f, zero_h,
      split_ws, total;
  size_t split_bytes, split_count;
};

WsLayout ws_layout(const Dims& D) {
  WsLayout W;
  size_t off = kStatusBytes;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += align_up(bytes);
    return at;
  };
  layer_split_sizes(D, &W.split_bytes, &W.split_count);
  W.split_cnt = take(W.split_count * 4);
  const size_t nh = (size_t)D.n * D.h;
  W.dz = take((size_t)D.n * D.f * D.esz);
  W.du = take(nh * 4);
  W.dx1 = take(nh * D.esz);
  W.dctx = take(nh * D.esz);
  W.dqkv = take(3 * nh * D.esz);
  W.dsum = take((size_t)D.batch * D.heads * D.seq * 4);
  // dropped-out gradient of the fc2 output, later of the out-proj output
  W.gmask = take(D.p_hidden > 0.f ? nh * D.esz : 0);
  size_t pf = ln_bwd_partial_floats((int)D.n, (int)D.h);
  for (const int64_t N : {D.h, D.f, 3 * D.h}) {   // the bias-gradient widths
    const size_t pc = colsum_partial_floats((int)D.n, (int)N);
    if (pc > pf) pf = pc;
  }
  const size_t pd = colsum_dropout_partial_floats((int)D.n, (int)D.h);
  if (pd > pf) pf = pd;
  const size_t pl = partial_layout(D).total;   // the Pre-LN backward's deferred finalizes
  W.partial = take((pl > pf ? pl : pf) * 4);
  W.fp8 = take(fp8_ws_layout(D).total);
  // recomputed activations ([n][h] and [n][ffn]); the forward keeps the ones it
  // does not save here too
  const bool rcw = D.recompute || D.fp8 == 2;
  W.rc_h = take(rcw ? nh * D.esz : 0);
  W.rc_f = take(rcw ? (size_t)D.n * D.f * D.esz : 0);
  W.zero_h = take(D.post_ln ? (size_t)D.h * D.esz : 0);   // a zero bias (Post-LN dx GEMM)
  W.split_ws = take(W.split_bytes);
  W.total = off;
  return W;
}


template <typename T>
T* at(void* base, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(base) + off);
}

SplitScratch layer_split(void* workspace, const WsLayout& W) {
  return {W.split_bytes ? at<float>(workspace, W.split_ws) : nullptr, W.split_bytes,
          W.split_count ? at<unsigned>(workspace, W.split_cnt) : nullptr, W.split_count};
}

// Workspace of a standalone GEMM: the status block, the tail-slice counters,
// the tail-slice partials.  Returns the bytes to clear at the start of a call.
size_t standalone_gemm_split(GemmArgs& g, void* workspace, size_t ws_bytes) {
  const int nsm = split_sms();
  const size_t cnt = gemm_split_counters(g.M, g.N, nsm);
  const size_t bytes = gemm_split_bytes(g.M, g.N, nsm);
  const size_t off_ws = kStatusBytes + align_up(cnt * 4);
  if (cnt == 0 || ws_bytes < off_ws + bytes) return kStatusBytes;
  g.split_cnt = at<unsigned>(workspace, kStatusBytes);
  g.split_cnt_count = cnt;
  g.split_ws = at<float>(workspace, off_ws);
  g.split_ws_bytes = bytes;
  return off_ws;
}

template <typename T>
const T* at(const void* base, size_t off) {
  return reinterpret_cast<const T*>(static_cast<const char*>(base) + off);
}

bool weights_ok(const mtl_weights* w) {
  if (!w) return false;
  const void* ps[] = {w->w_qkv, w->b_qkv, w->w_o,   w->b_o,   w->w_fc1, w->b_fc1,
                      w->w_fc2, w->b_fc2, w->ln1_g, w->ln1_b, w->ln2_g, w->ln2_b};
  for (const void* p : ps)
    if (!aligned16(p)) return false;
  return true;
}

bool grads_ok(const mtl_grads* g) {
  if (!g) return false;
  const void* ps[] = {g->w_qkv, g->b_qkv, g->w_o,   g->b_o,   g->w_fc1, g->b_fc1,
                      g->w_fc2, g->b_fc2, g->ln1_g, g->ln1_b, g->ln2_g, g->ln2_b};
  for (const void* p : ps)
    if (!aligned16(p)) return false;
  return true;
}

// One GEMM on the path of the layer's dtype: tcgen05 for bf16, exact fp32 on
// CUDA cores for fp32.
cudaError_t run_gemm(const Dims& D, const GemmArgs& a, const LaunchCtx& c) {
  if (D.dtype == MTL_BF16) return gemm_tc(a, c);
  return gemm_simt(kF32, a, c);
}

GemmArgs gemm_args(int M, int N, int K, int parts, const void* A, int64_t lda, bool ak,
                   const void* B, int64_t ldb, bool bk, int epi, void* C, int64_t ldc, bool cf32,
                   unsigned* status) {
  GemmArgs g;
  memset(&g, 0, sizeof(g));
  g.split_ws = g_split.ws;
  g.split_ws_bytes = g_split.bytes;
  g.split_cnt = g_split.cnt;
  g.split_cnt_count = g_split.count;
  g.M = M;
  g.N = N;
  g.K = K;
  g.parts = parts;
  g.A = {A, lda, ak};
  g.B = {B, ldb, bk};
  g.epi = epi;
  g.C = C;
  g.ldc = ldc;
  g.c_f32 = cf32;
  g.status = status;
  return g;
}

mtl_status attn_validate(int32_t dtype, int32_t batch, int32_t seq, int32_t heads, int32_t d,
                         float p_attn) {
  if (dtype != MTL_F32 && dtype != MTL_BF16) return MTL_ERR_INVALID_ARG;
  if (batch < 0 || seq <= 0 || heads <= 0) return MTL_ERR_INVALID_ARG;
  if (!(p_attn >= 0.f && p_attn < 1.f)) return MTL_ERR_INVALID_ARG;
  if (d != 64 && d != 96 && d != 128) return MTL_ERR_UNSUPPORTED;
  if ((int64_t)batch * seq > (int64_t)1 << 30) return MTL_ERR_UNSUPPORTED;
  if (dtype == MTL_BF16 && seq % 128) return MTL_ERR_UNSUPPORTED;
  if (dtype == MTL_F32 && seq > 8192) return MTL_ERR_UNSUPPORTED;
  return MTL_OK;
}
size_t attn_ws_bytes(int32_t batch, int32_t seq, int32_t heads) {
  return kStatusBytes + align_up((size_t)batch * heads * seq * 4);
}

#define MTL_TRY(expr, where)                     \
  do {                                           \
    cudaError_t _e = (expr);                     \
    if (_e != cudaSuccess) return cuda_fail(_e, where); \
  } while (0)

// The layer forward after validation (shared by mtl_layer_fwd and prefill):
// intermediates go to `saved` at saved_layout(D).
mtl_status forward_core(const Dims& D, float ln_eps, const mtl_weights* w, const void* x, void* y,
                        void* saved, void* fp8ws, void* rc_h, void* rc_f, unsigned* status,
                        const LaunchCtx& c) {
  const mtl_saved_layout L = saved_layout(D);
  // A GEMM of the forward: bf16 (or fp32) as given, or with FP8 layers each
  // operand quantized per tensor to E4M3 (own amax / scale slot) and the FP8
  // pair kernel.
  const Fp8Ws FW = fp8_ws_layout(D);
  int slot = 0;
  if (D.fp8) MTL_TRY(cudaMemsetAsync(at<char>(fp8ws, FW.stats), 0, 128, c.stream), "fp8 stats");
  // the amax slot of the next FP8 GEMM's A operand, for a kernel that writes
  // that operand (LayerNorm) to fill in (null without FP8 layers)
  auto next_amax_a = [&]() -> unsigned* {
    return D.fp8 ? at<unsigned>(fp8ws, FW.stats) + 2 * slot : nullptr;
  };
  // a_amax_done: the producer of A already folded its amax in
  auto fwd_gemm = [&](GemmArgs g, const char* where, bool a_amax_done = false) -> mtl_status {
    if (!D.fp8) {
      MTL_TRY(run_gemm(D, g, c), where);
      return MTL_OK;
    }
    unsigned* amax = at<unsigned>(fp8ws, FW.stats) + 2 * slot;
    if (!a_amax_done) MTL_TRY(fp8_amax(kBF16, g.A.ptr, g.M, g.K, g.A.ld, amax, c), where);
    float* sc = at<float>(fp8ws, FW.stats + 64) + 2 * slot;
    uint8_t* qa = at<uint8_t>(fp8ws, FW.qa);
    uint8_t* qb = at<uint8_t>(fp8ws, FW.qb);
    if (D.fp8 == 2) {
      // hybrid: the same passes also write the transposed copies the backward
      // reads, into `saved` with their scales
      const Fp8Saved FS = fp8_saved_layout(D);
      char* fsv = at<char>(saved, L.fp8);
      sc = at<float>(fsv, FS.scales) + 2 * slot;
      MTL_TRY(fp8_cast(kBF16, g.A.ptr, g.M, g.K, g.A.ld, 0, amax, sc, qa, g.K,
                       at<uint8_t>(fsv, FS.act[slot]), g.M, c),
              where);
      MTL_TRY(fp8_quantize2(kBF16, g.B.ptr, g.N, g.K, g.B.ld, 0, amax + 1, sc + 1, qb, g.K,
                            at<uint8_t>(fsv, FS.wt[slot]), g.N, c),
              where);
    } else {
      MTL_TRY(fp8_cast(kBF16, g.A.ptr, g.M, g.K, g.A.ld, 0, amax, sc, qa, g.K, nullptr, 0, c),
              where);
      MTL_TRY(fp8_quantize(kBF16, g.B.ptr, g.N, g.K, g.B.ld, 0, amax + 1, sc + 1, qb, g.K, c),
              where);
    }
    ++slot;
    g.A = {qa, g.K, true};
    g.B = {qb, g.K, true};
    g.fmt_a = 0;
    g.fmt_b = 0;
    g.scale_a = sc;
    g.scale_b = sc + 1;
    MTL_TRY(gemm_fp8(g, c), where);
    return MTL_OK;
  };
  mtl_status gst;
  const int n = (int)D.n, h = (int)D.h, f = (int)D.f, t = (int)D.t;
  // activations the backward recomputes live in the workspace during the forward
  const bool rcf = D.recompute || D.fp8 == 2;
  void* u1 = rcf ? rc_h : at<char>(saved, L.u1);
  void* qkv = at<char>(saved, L.qkv);
  void* ctx = at<char>(saved, L.ctx);
  void* x1 = (D.post_ln && D.recompute) ? rc_h : at<char>(saved, L.x1);
  void* u2 = rcf ? rc_h : at<char>(saved, L.u2);
  void* z = at<char>(saved, L.z);
  void* a = rcf ? rc_f : at<char>(saved, L.a);
  const bool bf = D.dtype == MTL_BF16;
  const Dropout drop_attn = make_drop(D.p_attn, D.seed, SITE_ATTN);

  if (D.post_ln) {
    // Post-LN: h1 = x + Attn(x); x1 = LN1(h1); h2 = x1 + MLP(x1); y = LN2(h2)
    void* h1 = at<char>(saved, L.h1);
    void* h2 = at<char>(saved, L.h2);
    {
      GemmArgs g = gemm_args(n, 3 * h, h, 1, x, h, true, w->w_qkv, h, true, EPI_BIAS, qkv, 3 * h,
                             false, status);
      g.bias = w->b_qkv;
      MTL_TRY(run_gemm(D, g, c), "qkv gemm");
    }
    if (bf) {
      MTL_TRY(attn_fwd_tc(qkv, ctx, at<float>(saved, L.lse), (int)D.batch, (int)D.seq,
                          (int)D.heads, (int)D.d, drop_attn, nullptr, status, c),
              "attention fwd");
    } else {
      MTL_TRY(attn_fwd_simt(D.dtype, qkv, ctx, at<float>(saved, L.lse), (int)D.batch, (int)D.seq,
                            (int)D.heads, (int)D.d, drop_attn, c),
              "attention fwd");
    }
    {
      GemmArgs g = gemm_args(n, h, h, t, ctx, h, true, w->w_o, h, true, EPI_BIAS_RESID, h1, h,
                             false, status);
      g.bias = w->b_o;
      g.R = x;
      g.ldr = h;
      MTL_TRY(run_gemm(D, g, c), "out-proj gemm");
    }
    MTL_TRY(ln_fwd(D.dtype, h1, w->ln1_g, w->ln1_b, x1, at<float>(saved, L.mu1),
                   at<float>(saved, L.rstd1), n, h, ln_eps, c),
            "ln1 fwd");
    {
      GemmArgs g = gemm_args(n, f, h, 1, x1, h, true, w->w_fc1, h, true, EPI_BIAS_GELU, a, f,
                             false, status);
      g.bias = w->b_fc1;
      g.Z = z;
      g.ldz = f;
      MTL_TRY(run_gemm(D, g, c), "fc1 gemm");
    }
    {
      GemmArgs g = gemm_args(n, h, f, t, a, f, true, w->w_fc2, f, true, EPI_BIAS_RESID, h2, h,
                             false, status);
      g.bias = w->b_fc2;
      g.R = x1;
      g.ldr = h;
      MTL_TRY(run_gemm(D, g, c), "fc2 gemm");
    }
    MTL_TRY(ln_fwd(D.dtype, h2, w->ln2_g, w->ln2_b, y, at<float>(saved, L.mu2),
                   at<float>(saved, L.rstd2), n, h, ln_eps, c),
            "ln2 fwd");
    return MTL_OK;
  }

  // F1 LN1 (with FP8 layers also the amax of u1 for the QKV GEMM)
  MTL_TRY(ln_fwd(D.dtype, x, w->ln1_g, w->ln1_b, u1, at<float>(saved, L.mu1),
                 at<float>(saved, L.rstd1), n, h, ln_eps, c, next_amax_a()),
          "ln1 fwd");
  // F2 QKV, column-parallel: partition p = rows [p*3h/t, (p+1)*3h/t) of w_qkv
  {
    GemmArgs g = gemm_args(n, 3 * h, h, 1, u1, h, true, w->w_qkv, h, true, EPI_BIAS, qkv, 3 * h,
                           false, status);
    g.bias = w->b_qkv;
    if ((gst = fwd_gemm(g, "qkv gemm", true)) != MTL_OK) return gst;
  }
  // F3 attention per head
  if (bf) {
    MTL_TRY(attn_fwd_tc(qkv, ctx, at<float>(saved, L.lse), (int)D.batch, (int)D.seq, (int)D.heads,
                        (int)D.d, drop_attn, at<uint32_t>(saved, L.attn_mask), status, c),
            "attention fwd");
  } else {
    MTL_TRY(attn_fwd_simt(D.dtype, qkv, ctx, at<float>(saved, L.lse), (int)D.batch, (int)D.seq,
                          (int)D.heads, (int)D.d, drop_attn, c),
            "attention fwd");
  }
  // F4 out-proj, row-parallel + g: t partials over K = h, + b_o, dropout, + x
  {
    GemmArgs g = gemm_args(n, h, h, t, ctx, h, true, w->w_o, h, true, EPI_BIAS_RESID, x1, h,
                           false, status);
    g.bias = w->b_o;
    g.drop = make_drop(D.p_hidden, D.seed, SITE_OUT);
    g.R = x;
    g.ldr = h;
    if ((gst = fwd_gemm(g, "out-proj gemm")) != MTL_OK) return gst;
  }
  // F5 LN2 (and the amax of u2 for fc1)
  MTL_TRY(ln_fwd(D.dtype, x1, w->ln2_g, w->ln2_b, u2, at<float>(saved, L.mu2),
                 at<float>(saved, L.rstd2), n, h, ln_eps, c, next_amax_a()),
          "ln2 fwd");
  // F6 fc1, column-parallel + bias + GeLU (saves z and a)
  {
    GemmArgs g = gemm_args(n, f, h, 1, u2, h, true, w->w_fc1, h, true, EPI_BIAS_GELU, a, f, false,
                           status);
    g.bias = w->b_fc1;
    g.Z = z;
    g.ldz = f;
    if ((gst = fwd_gemm(g, "fc1 gemm", true)) != MTL_OK) return gst;
  }
  // F7 fc2, row-parallel + g: t partials over K = ffn, + b_fc2, dropout, + x1
  {
    GemmArgs g = gemm_args(n, h, f, t, a, f, true, w->w_fc2, f, true, EPI_BIAS_RESID, y, h, false,
                           status);
    g.bias = w->b_fc2;
    g.drop = make_drop(D.p_hidden, D.seed, SITE_FC2);
    g.R = x1;
    g.ldr = h;
    if ((gst = fwd_gemm(g, "fc2 gemm")) != MTL_OK) return gst;
  }
  return MTL_OK;
}


// ---------------------------------------------------------------- inference

// Decode validation: the layer rules that concern a token-batch step (seq is
// not used), max_seq >= 1, batch <= kDecodeMaxBatch.
mtl_status validate_decode(const mtl_layer_desc* desc, int32_t max_seq, Dims* o) {
  if (!desc) return MTL_ERR_INVALID_ARG;
  mtl_layer_desc d = *desc;
  if (max_seq <= 0 || d.batch > kDecodeMaxBatch) return max_seq <= 0 ? MTL_ERR_INVALID_ARG
                                                                     : MTL_ERR_UNSUPPORTED;
  d.seq = d.dtype == MTL_BF16 ? 128 : 1;   // a valid stand-in: decode has no sequence axis
  d.p_attn = 0.f;
  d.p_hidden = 0.f;
  d.fp8 = 0;                                // decode GEMMs stay bf16
  d.recompute = 0;
  if (d.post_ln) return MTL_ERR_UNSUPPORTED;  // decode runs the Pre-LN layer
  mtl_status st = validate(&d, o);
  if (st != MTL_OK) return st;
  o->seq = 1;
  o->n = o->batch;
  return MTL_OK;
}

size_t kv_cache_bytes(const Dims& D, int32_t max_seq) {
  return 2 * align_up((size_t)D.batch * D.heads * max_seq * D.d * D.esz);
}

struct DecWs {
  size_t c_att, mean, rstd, u, qkv, ctx, x1, a, z, apart, total;
};

DecWs decode_ws(const Dims& D, int32_t max_seq) {
  DecWs W;
  size_t off = kStatusBytes;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += align_up(bytes);
    return at;
  };
  const int h = (int)D.h, f = (int)D.f, b = (int)D.batch;
  W.c_att = take((size_t)b * D.heads * 4);
  W.mean = take((size_t)b * 4);
  W.rstd = take((size_t)b * 4);
  W.u = take((size_t)b * h * D.esz);
  W.qkv = take((size_t)b * 3 * h * D.esz);
  W.ctx = take((size_t)b * h * D.esz);
  W.x1 = take((size_t)b * h * D.esz);
  W.a = take((size_t)b * f * D.esz);
  W.z = take(D.dtype == MTL_BF16 ? 0 : (size_t)b * f * D.esz);
  W.apart = take((size_t)b * D.heads * attn_decode_splits(max_seq) * (D.d + 2) * 4);
  W.total = off;
  return W;
}
}  // namespace

extern "C" {

const char* mtl_status_str(mtl_status s) {
  switch (s) {
    case MTL_OK: return "ok";
    case MTL_ERR_INVALID_ARG: return "invalid argument";
    case MTL_ERR_UNSUPPORTED: return "unsupported layer shape";
    case MTL_ERR_WORKSPACE: return "workspace too small";
    case MTL_ERR_CUDA: return "CUDA error";
    case MTL_ERR_TIMEOUT: return "device wait timed out";
    case MTL_ERR_BOUNDS: return "device bounds check failed";
  }
  return "unknown status";
}

const char* mtl_last_cuda_error(void) { return g_cuda_err; }

int32_t mtl_last_launch_count(void) { return g_launches; }

void mtl_profile_set(void** events, int32_t capacity, int32_t* kinds, double* work) {
  g_prof.events = reinterpret_cast<cudaEvent_t*>(events);
  g_prof.capacity = events ? capacity : 0;
  g_prof.count = 0;
  g_prof.kinds = kinds;
  g_prof.work = work;
}

int32_t mtl_profile_count(void) { return g_prof.count; }

mtl_status mtl_layer_sizes(const mtl_layer_desc* desc, size_t* saved_bytes,
                           size_t* workspace_bytes) {
  Dims D;
  mtl_status st = validate(desc, &D);
  if (st != MTL_OK) return st;
  if (saved_bytes) *saved_bytes = saved_layout(D).total;
  if (workspace_bytes) *workspace_bytes = ws_layout(D).total;
  return MTL_OK;
}

mtl_status mtl_layer_saved_layout(const mtl_layer_desc* desc, mtl_saved_layout* out) {
  Dims D;
  mtl_status st = validate(desc, &D);
  if (st != MTL_OK) return st;
  if (!out) return MTL_ERR_INVALID_ARG;
  *out = saved_layout(D);
  return MTL_OK;
}

mtl_status mtl_layer_workspace_layout(const mtl_layer_desc* desc, mtl_workspace_layout* out) {
  Dims D;
  mtl_status st = validate(desc, &D);
  if (st != MTL_OK) return st;
  if (!out) return MTL_ERR_INVALID_ARG;
  const WsLayout W = ws_layout(D);
  out->dz = W.dz;
  out->du = W.du;
  out->dx1 = W.dx1;
  out->dctx = W.dctx;
  out->dqkv = W.dqkv;
  out->total = W.total;
  return MTL_OK;
}

mtl_status mtl_layer_fwd(const mtl_layer_desc* desc, const mtl_weights* w, const void* x,
                         void* y, void* saved, void* workspace, size_t ws_bytes,
                         mtl_stream stream) {
  g_launches = 0;
  g_cuda_err[0] = 0;
  Dims D;
  mtl_status st = validate(desc, &D);
  if (st != MTL_OK) return st;
  if (!weights_ok(w) || !aligned16(x) || !aligned16(y) || !aligned16(saved) ||
      !aligned16(workspace) || x == y || y == saved)
    return MTL_ERR_INVALID_ARG;
  const WsLayout W = ws_layout(D);
  if (ws_bytes < W.total) return MTL_ERR_WORKSPACE;
  const int nsm = device_sm_count();
  if (nsm <= 0) return cuda_fail(cudaGetLastError(), "device query");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  LaunchCtx c{s, nsm, &g_launches, &g_prof};
  unsigned* status = static_cast<unsigned*>(workspace);
  // the status word and the GEMMs' tail-slice counters
  MTL_TRY(cudaMemsetAsync(status, 0, W.dz, s), "status reset");
  if (D.n == 0) return MTL_OK;
  const SplitScope split(layer_split(workspace, W));

  return forward_core(D, desc->ln_eps, w, x, y, saved, at<char>(workspace, W.fp8),
                      at<char>(workspace, W.rc_h), at<char>(workspace, W.rc_f), status, c);
}

mtl_status mtl_layer_bwd(const mtl_layer_desc* desc, const mtl_weights* w, const void* x,
                         const void* saved, const void* dy, void* dx, const mtl_grads* gr,
                         void* workspace, size_t ws_bytes, mtl_stream stream) {
  g_launches = 0;
  g_cuda_err[0] = 0;
  Dims D;
  mtl_status st = validate(desc, &D);
  if (st != MTL_OK) return st;
  if (!weights_ok(w) || !grads_ok(gr) || !aligned16(x) || !aligned16(saved) || !aligned16(dy) ||
      !aligned16(dx) || !aligned16(workspace) || dx == dy)
    return MTL_ERR_INVALID_ARG;
  const WsLayout W = ws_layout(D);
  if (ws_bytes < W.total) return MTL_ERR_WORKSPACE;
  const int nsm = device_sm_count();
  if (nsm <= 0) return cuda_fail(cudaGetLastError(), "device query");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  LaunchCtx c{s, nsm, &g_launches, &g_prof};
  unsigned* status = static_cast<unsigned*>(workspace);
  // the status word and the GEMMs' tail-slice counters
  MTL_TRY(cudaMemsetAsync(status, 0, W.dz, s), "status reset");
  const SplitScope split(layer_split(workspace, W));

  const mtl_saved_layout L = saved_layout(D);
  const int n = (int)D.n, h = (int)D.h, f = (int)D.f, t = (int)D.t;
  const void* u1 = at<char>(saved, L.u1);
  const void* qkv = at<char>(saved, L.qkv);
  const void* ctx = at<char>(saved, L.ctx);
  const void* x1 = at<char>(saved, L.x1);
  const void* u2 = at<char>(saved, L.u2);
  const void* z = at<char>(saved, L.z);
  const void* a = at<char>(saved, L.a);
  void* rc_h = at<char>(workspace, W.rc_h);
  void* rc_f = at<char>(workspace, W.rc_f);
  void* dz = at<char>(workspace, W.dz);
  float* du = at<float>(workspace, W.du);
  void* dx1 = at<char>(workspace, W.dx1);
  void* dctx = at<char>(workspace, W.dctx);
  void* dqkv = at<char>(workspace, W.dqkv);
  float* dsum = at<float>(workspace, W.dsum);
  float* partial = at<float>(workspace, W.partial);

  if (D.n == 0) {
    // no tokens: every gradient is zero
    void* zs[] = {gr->w_qkv, gr->b_qkv, gr->w_o, gr->b_o, gr->w_fc1, gr->b_fc1,
                  gr->w_fc2, gr->b_fc2, gr->ln1_g, gr->ln1_b, gr->ln2_g, gr->ln2_b};
    size_t sz[] = {3 * (size_t)h * h, 3 * (size_t)h, (size_t)h * h, (size_t)h,
                   (size_t)f * h,     (size_t)f,     (size_t)h * f, (size_t)h,
                   (size_t)h,         (size_t)h,     (size_t)h,     (size_t)h};
    for (int i = 0; i < 12; ++i) MTL_TRY(cudaMemsetAsync(zs[i], 0, sz[i] * 4, s), "zero grads");
    return MTL_OK;
  }

  if (D.post_ln) {
    // Post-LN backward.  Buffers: dh2 in dctx (dead once dh1 exists), dh1 in dx1.
    const void* h1 = at<char>(saved, L.h1);
    const void* h2 = at<char>(saved, L.h2);
    void* dh2 = dctx;
    void* dh1 = dx1;
    const Dropout no_drop = make_drop(0.f, 0, SITE_ATTN);
    if (D.recompute) {
      MTL_TRY(ln_apply(D.dtype, h1, at<float>(saved, L.mu1), at<float>(saved, L.rstd1), w->ln1_g,
                       w->ln1_b, rc_h, n, h, c),
              "recompute x1");
      MTL_TRY(gelu_apply(D.dtype, z, rc_f, (int64_t)n * f, c), "recompute a");
      x1 = rc_h;
      a = rc_f;
    }
    // P1 dh2 = LN2_bwd(dy); dgamma2, dbeta2
    MTL_TRY(ln_bwd_sum(D.dtype, nullptr, dy, h2, at<float>(saved, L.mu2),
                       at<float>(saved, L.rstd2), w->ln2_g, dh2, static_cast<float*>(gr->ln2_g),
                       static_cast<float*>(gr->ln2_b), partial, n, h, c),
            "ln2 bwd");
    // MLP: dz = (dh2 W2) GeLU'(z); dW2 = dh2^T a; db2; du = sum_p dz W1 (f sum);
    // dW1 = dz^T x1; db1
    {
      GemmArgs g = gemm_args(n, f, h, 1, dh2, h, true, w->w_fc2, f, false, EPI_DGELU, dz, f,
                             false, status);
      g.Z = const_cast<void*>(z);
      g.ldz = f;
      MTL_TRY(run_gemm(D, g, c), "fc2 dgrad");
    }
    MTL_TRY(run_gemm(D, gemm_args(h, f, n, 1, dh2, h, false, a, f, false, EPI_STORE, gr->w_fc2,
                                  f, true, status),
                     c),
            "fc2 wgrad");
    MTL_TRY(colsum(D.dtype, dh2, h, n, h, static_cast<float*>(gr->b_fc2), partial, c), "db_fc2");
    MTL_TRY(run_gemm(D, gemm_args(n, h, f, t, dz, f, true, w->w_fc1, h, false, EPI_STORE, du, h,
                                  true, status),
                     c),
            "fc1 dgrad");
    MTL_TRY(run_gemm(D, gemm_args(f, h, n, 1, dz, f, false, x1, h, false, EPI_STORE, gr->w_fc1, h,
                                  true, status),
                     c),
            "fc1 wgrad");
    MTL_TRY(colsum(D.dtype, dz, f, n, f, static_cast<float*>(gr->b_fc1), partial, c), "db_fc1");
    // P5 dh1 = LN1_bwd(dh2 + du); dgamma1, dbeta1
    MTL_TRY(ln_bwd_sum(D.dtype, du, dh2, h1, at<float>(saved, L.mu1), at<float>(saved, L.rstd1),
                       w->ln1_g, dh1, static_cast<float*>(gr->ln1_g),
                       static_cast<float*>(gr->ln1_b), partial, n, h, c),
            "ln1 bwd");
    // attention block: dW_o = dh1^T ctx; db_o; dctx = dh1 W_o; attention; dW_qkv = dqkv^T x
    MTL_TRY(colsum(D.dtype, dh1, h, n, h, static_cast<float*>(gr->b_o), partial, c), "db_o");
    MTL_TRY(run_gemm(D, gemm_args(h, h, n, 1, dh1, h, false, ctx, h, false, EPI_STORE, gr->w_o, h,
                                  true, status),
                     c),
            "out-proj wgrad");
    MTL_TRY(run_gemm(D, gemm_args(n, h, h, 1, dh1, h, true, w->w_o, h, false, EPI_STORE, dctx, h,
                                  false, status),
                     c),
            "out-proj dgrad");
    if (D.dtype == MTL_BF16) {
      MTL_TRY(attn_bwd_tc(qkv, ctx, at<float>(saved, L.lse), dctx, dqkv, dsum, (int)D.batch,
                          (int)D.seq, (int)D.heads, (int)D.d, no_drop, nullptr, status, c),
              "attention bwd");
    } else {
      MTL_TRY(attn_bwd_simt(D.dtype, qkv, ctx, at<float>(saved, L.lse), dctx, dqkv, dsum,
                            (int)D.batch, (int)D.seq, (int)D.heads, (int)D.d, no_drop, c),
              "attention bwd");
    }
    MTL_TRY(run_gemm(D, gemm_args(3 * h, h, n, 1, dqkv, 3 * h, false, x, h, false, EPI_STORE,
                                  gr->w_qkv, h, true, status),
                     c),
            "qkv wgrad");
    MTL_TRY(colsum(D.dtype, dqkv, 3 * h, n, 3 * h, static_cast<float*>(gr->b_qkv), partial, c),
            "db_qkv");
    // dx = dh1 + sum_p dqkv[:, Q_p] W_qkv[Q_p, :]  (the f sum, residual in the epilogue)
    {
      void* zero_h = at<char>(workspace, W.zero_h);
      MTL_TRY(cudaMemsetAsync(zero_h, 0, (size_t)h * D.esz, s), "zero bias");
      GemmArgs g = gemm_args(n, h, 3 * h, t, dqkv, 3 * h, true, w->w_qkv, h, false,
                             EPI_BIAS_RESID, dx, h, false, status);
      g.bias = zero_h;
      g.R = dh1;
      g.ldr = h;
      MTL_TRY(run_gemm(D, g, c), "qkv dgrad");
    }
    return MTL_OK;
  }

  if (D.fp8 == 2) {
    // FP8 hybrid backward (Pre-LN, no dropout): every GEMM takes an E5M2
    // gradient and an E4M3 activation or weight, both K-major.  The forward left
    // the transposed E4M3 copies of its operands (and their scales) in `saved`;
    // each gradient is quantized once into a row-major and a transposed copy
    // (its amax comes from the bias-gradient column sum, which reads the
    // gradient anyway; then one conversion pass).  Bias and LayerNorm
    // gradients and attention stay bf16 / fp32.
    const Fp8Ws FW = fp8_ws_layout(D);
    const Fp8Saved FS = fp8_saved_layout(D);
    const char* fsv = at<char>(saved, L.fp8);
    const float* fsc = at<float>(fsv, FS.scales);
    auto act = [&](int i) { return at<uint8_t>(fsv, FS.act[i]); };
    auto wtr = [&](int i) { return at<uint8_t>(fsv, FS.wt[i]); };
    char* fb = at<char>(workspace, W.fp8);
    unsigned* amax = at<unsigned>(fb, FW.stats);
    float* gscale = at<float>(fb, FW.stats + 64);
    uint8_t* gq = at<uint8_t>(fb, FW.gq);
    uint8_t* gqT = at<uint8_t>(fb, FW.gqT);
    MTL_TRY(cudaMemsetAsync(amax, 0, 64, s), "fp8 stats");
    int slot = 0;
    // the gradient src [rows][cols] to E5M2: gq row-major, gqT transposed; its
    // amax is in amax[slot], folded in by the column sum that read src
    auto quant_grad = [&](const void* src, int64_t rows, int64_t cols, const float** scale)
        -> cudaError_t {
      *scale = gscale + slot;
      const cudaError_t e = fp8_cast(kBF16, src, rows, cols, cols, MTL_FP8_E5M2, amax + slot,
                                     gscale + slot, gq, cols, gqT, rows, c);
      ++slot;
      return e;
    };
    // C = epi(A B^T) with K-major FP8 A [M][K] (E5M2) and B [N][K] (E4M3)
    auto f8 = [&](int M, int N, int K, int parts, const void* qa, const float* sa, const void* qb,
                  const float* sbb, int epi, void* C, int64_t ldc, bool cf32,
                  const void* Z) -> cudaError_t {
      GemmArgs g = gemm_args(M, N, K, parts, qa, K, true, qb, K, true, epi, C, ldc, cf32, status);
      g.fmt_a = MTL_FP8_E5M2;
      g.fmt_b = MTL_FP8_E4M3;
      g.scale_a = sa;
      g.scale_b = sbb;
      g.Z = const_cast<void*>(Z);
      g.ldz = N;
      return gemm_fp8(g, c);
    };
    const float* s_g;
    // MLP block
    MTL_TRY(colsum(D.dtype, dy, h, n, h, static_cast<float*>(gr->b_fc2), partial, c, amax + slot),
            "db_fc2");
    MTL_TRY(quant_grad(dy, n, h, &s_g), "fp8 dy");
    MTL_TRY(f8(n, f, h, 1, gq, s_g, wtr(3), fsc + 7, EPI_DGELU, dz, f, false, z), "fc2 dgrad");
    MTL_TRY(f8(h, f, n, 1, gqT, s_g, act(3), fsc + 6, EPI_STORE, gr->w_fc2, f, true, nullptr),
            "fc2 wgrad");
    MTL_TRY(colsum(D.dtype, dz, f, n, f, static_cast<float*>(gr->b_fc1), partial, c, amax + slot),
            "db_fc1");
    MTL_TRY(quant_grad(dz, n, f, &s_g), "fp8 dz");
    MTL_TRY(f8(n, h, f, t, gq, s_g, wtr(2), fsc + 5, EPI_STORE, du, h, true, nullptr),
            "fc1 dgrad");
    MTL_TRY(f8(f, h, n, 1, gqT, s_g, act(2), fsc + 4, EPI_STORE, gr->w_fc1, h, true, nullptr),
            "fc1 wgrad");
    MTL_TRY(ln_bwd(D.dtype, du, x1, at<float>(saved, L.mu2), at<float>(saved, L.rstd2), w->ln2_g,
                   dy, dx1, static_cast<float*>(gr->ln2_g), static_cast<float*>(gr->ln2_b),
                   partial, n, h, c),
            "ln2 bwd");
    // attention block
    MTL_TRY(colsum(D.dtype, dx1, h, n, h, static_cast<float*>(gr->b_o), partial, c, amax + slot),
            "db_o");
    MTL_TRY(quant_grad(dx1, n, h, &s_g), "fp8 dx1");
    MTL_TRY(f8(n, h, h, 1, gq, s_g, wtr(1), fsc + 3, EPI_STORE, dctx, h, false, nullptr),
            "out-proj dgrad");
    MTL_TRY(f8(h, h, n, 1, gqT, s_g, act(1), fsc + 2, EPI_STORE, gr->w_o, h, true, nullptr),
            "out-proj wgrad");
    MTL_TRY(attn_bwd_tc(qkv, ctx, at<float>(saved, L.lse), dctx, dqkv, dsum, (int)D.batch,
                        (int)D.seq, (int)D.heads, (int)D.d, make_drop(0.f, 0, SITE_ATTN),
                        nullptr, status, c),
            "attention bwd");
    MTL_TRY(colsum(D.dtype, dqkv, 3 * h, n, 3 * h, static_cast<float*>(gr->b_qkv), partial, c,
                   amax + slot),
            "db_qkv");
    MTL_TRY(quant_grad(dqkv, n, 3 * h, &s_g), "fp8 dqkv");
    MTL_TRY(f8(3 * h, h, n, 1, gqT, s_g, act(0), fsc + 0, EPI_STORE, gr->w_qkv, h, true,
               nullptr),
            "qkv wgrad");
    MTL_TRY(f8(n, h, 3 * h, t, gq, s_g, wtr(0), fsc + 1, EPI_STORE, du, h, true, nullptr),
            "qkv dgrad");
    MTL_TRY(ln_bwd(D.dtype, du, x, at<float>(saved, L.mu1), at<float>(saved, L.rstd1), w->ln1_g,
                   dx1, dx, static_cast<float*>(gr->ln1_g), static_cast<float*>(gr->ln1_b),
                   partial, n, h, c),
            "ln1 bwd");
    (void)u1;
    (void)u2;
    (void)a;
    (void)rc_h;
    (void)rc_f;
    return MTL_OK;
  }

  const bool hid_drop = D.p_hidden > 0.f;
  const Dropout drop_attn = make_drop(D.p_attn, D.seed, SITE_ATTN);
  void* gmask = at<char>(workspace, W.gmask);
  // Bias, gamma and beta gradients: every partial column sum stays in its own
  // region and one launch at the end adds them up (finalize_jobs).  db_fc2 and
  // db_o ride the LN2 backward (it reads dy and writes dx1 anyway) and db_fc1
  // the fc2-dgrad epilogue (it holds every dz) where they can.
  const PartialLayout P = partial_layout(D);
  FinalizeJobs fin;
  const bool fold_ln2 = !hid_drop && ln_bwd_can_sum(D.dtype, h);
  const bool fold_dz = D.dtype == MTL_BF16 && f % 32 == 0;
  // B0 gradient at the fc2 output g2 = dy * keep_2 / (1 - p) (dy itself without
  // dropout) and db2 = sum_rows g2
  const void* g2 = dy;
  if (hid_drop) {
    MTL_TRY(colsum_dropout(D.dtype, dy, gmask, h, n, h, make_drop(D.p_hidden, D.seed, SITE_FC2),
                           static_cast<float*>(gr->b_fc2), partial + P.drop, c),
            "db_fc2");
    g2 = gmask;
  } else if (!fold_ln2) {
    MTL_TRY(colsum(D.dtype, dy, h, n, h, static_cast<float*>(gr->b_fc2), partial + P.b2, c,
                   nullptr, &fin),
            "db_fc2");
  }
  // B1 fc2 dgrad + GeLU': dz = (g2 W_fc2) * GeLU'(z)  (column-local, no reduction)
  {
    GemmArgs g = gemm_args(n, f, h, 1, g2, h, true, w->w_fc2, f, false, EPI_DGELU, dz, f, false,
                           status);
    g.Z = const_cast<void*>(z);
    g.ldz = f;
    if (fold_dz) g.colsum_part = partial + P.dz;
    MTL_TRY(run_gemm(D, g, c), "fc2 dgrad");
    if (fold_dz && !fin.add(partial + P.dz, (n + 31) / 32, f, static_cast<float*>(gr->b_fc1)))
      return cuda_fail(cudaErrorInvalidValue, "finalize list");
  }
  // B2 fc2 wgrad dW2 = g2^T a  (a recomputed as GeLU(z) when not saved)
  if (D.recompute) {
    MTL_TRY(gelu_apply(D.dtype, z, rc_f, (int64_t)n * f, c), "recompute a");
    a = rc_f;
  }
  MTL_TRY(run_gemm(D, gemm_args(h, f, n, 1, g2, h, false, a, f, false, EPI_STORE, gr->w_fc2, f,
                                true, status),
                   c),
          "fc2 wgrad");
  // B3 fc1 dgrad with the f reduction: du2 = sum_p dz[:, F_p] W_fc1[F_p, :]
  MTL_TRY(run_gemm(D, gemm_args(n, h, f, t, dz, f, true, w->w_fc1, h, false, EPI_STORE, du, h,
                                true, status),
                   c),
          "fc1 dgrad");
  // B4 fc1 wgrad dW1 = dz^T u2, db1 = sum_rows dz  (u2 recomputed from x1 and the
  // saved statistics when not saved)
  if (D.recompute) {
    MTL_TRY(ln_apply(D.dtype, x1, at<float>(saved, L.mu2), at<float>(saved, L.rstd2), w->ln2_g,
                     w->ln2_b, rc_h, n, h, c),
            "recompute u2");
    u2 = rc_h;
  }
  MTL_TRY(run_gemm(D, gemm_args(f, h, n, 1, dz, f, false, u2, h, false, EPI_STORE, gr->w_fc1, h,
                                true, status),
                   c),
          "fc1 wgrad");
  if (!fold_dz)
    MTL_TRY(colsum(D.dtype, dz, f, n, f, static_cast<float*>(gr->b_fc1), partial + P.dz, c,
                   nullptr, &fin),
            "db_fc1");
  // B5 LN2 backward + residual: dx1 = dy + LN2_bwd(du2); with the fold also
  // db_fc2 = sum_rows dy and db_o = sum_rows dx1
  MTL_TRY(ln_bwd(D.dtype, du, x1, at<float>(saved, L.mu2), at<float>(saved, L.rstd2), w->ln2_g, dy,
                 dx1, static_cast<float*>(gr->ln2_g), static_cast<float*>(gr->ln2_b),
                 partial + P.ln2, n, h, c, &fin,
                 fold_ln2 ? static_cast<float*>(gr->b_fc2) : nullptr,
                 fold_ln2 ? static_cast<float*>(gr->b_o) : nullptr),
          "ln2 bwd");
  // B6 gradient at the out-proj output go = dx1 * keep_1 / (1 - p) (dx1 without
  // dropout), db_o = sum_rows go; dgrad dctx = go W_o, wgrad dW_o = go^T ctx
  const void* go = dx1;
  if (hid_drop) {
    MTL_TRY(colsum_dropout(D.dtype, dx1, gmask, h, n, h, make_drop(D.p_hidden, D.seed, SITE_OUT),
                           static_cast<float*>(gr->b_o), partial + P.drop, c),
            "db_o");
    go = gmask;
  } else if (!fold_ln2) {
    MTL_TRY(colsum(D.dtype, dx1, h, n, h, static_cast<float*>(gr->b_o), partial + P.bo, c,
                   nullptr, &fin),
            "db_o");
  }
  MTL_TRY(run_gemm(D, gemm_args(n, h, h, 1, go, h, true, w->w_o, h, false, EPI_STORE, dctx, h,
                                false, status),
                   c),
          "out-proj dgrad");
  MTL_TRY(run_gemm(D, gemm_args(h, h, n, 1, go, h, false, ctx, h, false, EPI_STORE, gr->w_o, h,
                                true, status),
                   c),
          "out-proj wgrad");
  // B7 attention backward per head
  if (D.dtype == MTL_BF16) {
    MTL_TRY(attn_bwd_tc(qkv, ctx, at<float>(saved, L.lse), dctx, dqkv, dsum, (int)D.batch,
                        (int)D.seq, (int)D.heads, (int)D.d, drop_attn,
                        at<uint32_t>(saved, L.attn_mask), status, c),
            "attention bwd");
  } else {
    MTL_TRY(attn_bwd_simt(D.dtype, qkv, ctx, at<float>(saved, L.lse), dctx, dqkv, dsum,
                          (int)D.batch, (int)D.seq, (int)D.heads, (int)D.d, drop_attn, c),
            "attention bwd");
  }
  // B8 QKV wgrad dW_qkv = dqkv^T u1, db_qkv = sum_rows dqkv  (u1 recomputed from x
  // and the saved statistics when not saved)
  if (D.recompute) {
    MTL_TRY(ln_apply(D.dtype, x, at<float>(saved, L.mu1), at<float>(saved, L.rstd1), w->ln1_g,
                     w->ln1_b, rc_h, n, h, c),
            "recompute u1");
    u1 = rc_h;
  }
  MTL_TRY(run_gemm(D, gemm_args(3 * h, h, n, 1, dqkv, 3 * h, false, u1, h, false, EPI_STORE,
                                gr->w_qkv, h, true, status),
                   c),
          "qkv wgrad");
  MTL_TRY(colsum(D.dtype, dqkv, 3 * h, n, 3 * h, static_cast<float*>(gr->b_qkv), partial + P.qkv,
                 c, nullptr, &fin),
          "db_qkv");
  // B9 QKV dgrad with the f reduction: du1 = sum_p dqkv[:, Q_p] W_qkv[Q_p, :]
  MTL_TRY(run_gemm(D, gemm_args(n, h, 3 * h, t, dqkv, 3 * h, true, w->w_qkv, h, false, EPI_STORE,
                                du, h, true, status),
                   c),
          "qkv dgrad");
  // B10 LN1 backward + residual: dx = dx1 + LN1_bwd(du1)
  MTL_TRY(ln_bwd(D.dtype, du, x, at<float>(saved, L.mu1), at<float>(saved, L.rstd1), w->ln1_g,
                 dx1, dx, static_cast<float*>(gr->ln1_g), static_cast<float*>(gr->ln1_b),
                 partial + P.ln1, n, h, c, &fin),
          "ln1 bwd");
  // every deferred bias / gamma / beta finalize in one launch
  MTL_TRY(finalize_jobs(fin, c), "finalize");
  return MTL_OK;
}

mtl_status mtl_layer_check(void* workspace, mtl_stream stream) {
  if (!aligned16(workspace)) return MTL_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "stream sync");
  unsigned word = 0;
  e = cudaMemcpy(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "status read");
  if (word) {
    unsigned zero = 0;
    cudaMemcpy(workspace, &zero, sizeof(zero), cudaMemcpyHostToDevice);
  }
  if (word & kDevErrBounds) {
    // a skipped access usually also leaves a bounded wait to time out: the
    // bounds fault is the cause, so it is reported first
    snprintf(g_cuda_err, sizeof(g_cuda_err), "bounds check: fault %u at site %u (word 0x%08x)",
             (word >> 8) & 0xFu, (word >> 16) & 0xFFu, word);
    return MTL_ERR_BOUNDS;
  }
  if (word & kDevErrTimeout) return MTL_ERR_TIMEOUT;
  if (word) return MTL_ERR_INVALID_ARG;
  return MTL_OK;
}

namespace {
// One CTA waits, with the same bounded wait the pipelined kernels use, on an
// mbarrier that nothing will ever arrive at.
__global__ void selftest_wait_kernel(unsigned* status, long long limit) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait_bounded(smem_u32(&bar), 0, status, &abort_flag, limit);
  __syncthreads();
}
}  // namespace

mtl_status mtl_selftest_wait_timeout(void* workspace, int64_t limit_cycles, mtl_stream stream) {
  g_launches = 0;
  g_cuda_err[0] = 0;
  if (!aligned16(workspace)) return MTL_ERR_INVALID_ARG;
  if (limit_cycles < 1000 || limit_cycles > kWaitLimitCycles) return MTL_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  unsigned* status = static_cast<unsigned*>(workspace);
  MTL_TRY(cudaMemsetAsync(status, 0, kStatusBytes, s), "status reset");
  selftest_wait_kernel<<<1, 32, 0, s>>>(status, limit_cycles);
  ++g_launches;
  MTL_TRY(cudaGetLastError(), "selftest launch");
  return MTL_OK;
}

namespace {
__global__ void selftest_empty_kernel() {}
}  // namespace

mtl_status mtl_selftest_launch_error(mtl_stream stream) {
  g_launches = 0;
  g_cuda_err[0] = 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // 2048 threads a block is above the 1024-thread limit of every CUDA device:
  // the runtime rejects the launch configuration and nothing reaches the GPU.
  selftest_empty_kernel<<<1, 2048, 0, s>>>();
  const cudaError_t e = cudaGetLastError();   // returns and clears the launch error
  if (e != cudaSuccess) return cuda_fail(e, "selftest launch");
  ++g_launches;
  return MTL_OK;
}

// ---------------------------------------------------------------- attention alone


mtl_status mtl_attention_ws_bytes(int32_t batch, int32_t seq, int32_t heads, size_t* bytes) {
  if (batch < 0 || seq <= 0 || heads <= 0 || !bytes) return MTL_ERR_INVALID_ARG;
  *bytes = attn_ws_bytes(batch, seq, heads);
  return MTL_OK;
}

mtl_status mtl_attention_mask_bytes(int32_t dtype, int32_t batch, int32_t seq, int32_t heads,
                                    float p_attn, size_t* bytes) {
  if (!bytes) return MTL_ERR_INVALID_ARG;
  mtl_status st = attn_validate(dtype, batch, seq, heads, 64, p_attn);
  if (st != MTL_OK) return st;
  *bytes = dtype == MTL_BF16 && p_attn > 0.f ? attn_mask_bytes(batch, seq, heads) : 0;
  return MTL_OK;
}

mtl_status mtl_attention_fwd(int32_t dtype, int32_t batch, int32_t seq, int32_t heads, int32_t d,
                             const void* qkv, void* ctx, float* lse, void* mask_bits,
                             float p_attn, uint64_t seed, void* workspace, size_t ws_bytes,
                             mtl_stream stream) {
  g_launches = 0;
  g_cuda_err[0] = 0;
  mtl_status st = attn_validate(dtype, batch, seq, heads, d, p_attn);
  if (st != MTL_OK) return st;
  const bool need_mask = dtype == MTL_BF16 && p_attn > 0.f;
  if (!aligned16(qkv) || !aligned16(ctx) || !aligned16(lse) || !aligned16(workspace) ||
      qkv == ctx || (need_mask && !aligned16(mask_bits)))
    return MTL_ERR_INVALID_ARG;
  if (ws_bytes < attn_ws_bytes(batch, seq, heads)) return MTL_ERR_WORKSPACE;
  const int nsm = device_sm_count();
  if (nsm <= 0) return cuda_fail(cudaGetLastError(), "device query");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  LaunchCtx c{s, nsm, &g_launches, &g_prof};
  unsigned* status = static_cast<unsigned*>(workspace);
  MTL_TRY(cudaMemsetAsync(status, 0, kStatusBytes, s), "status reset");
  if (batch == 0) return MTL_OK;
  const Dropout drop = make_drop(p_attn, seed, SITE_ATTN);
  if (dtype == MTL_BF16) {
    MTL_TRY(attn_fwd_tc(qkv, ctx, lse, batch, seq, heads, d, drop, static_cast<uint32_t*>(mask_bits),
                        status, c),
            "attention fwd");
  } else {
    MTL_TRY(attn_fwd_simt(dtype, qkv, ctx, lse, batch, seq, heads, d, drop, c), "attention fwd");
  }
  return MTL_OK;
}

mtl_status mtl_attention_bwd(int32_t dtype, int32_t batch, int32_t seq, int32_t heads, int32_t d,
                             const void* qkv, const void* ctx, const float* lse, const void* dctx,
                             const void* mask_bits, void* dqkv, float p_attn, uint64_t seed,
                             void* workspace, size_t ws_bytes, mtl_stream stream) {
  g_launches = 0;
  g_cuda_err[0] = 0;
  mtl_status st = attn_validate(dtype, batch, seq, heads, d, p_attn);
  if (st != MTL_OK) return st;
  if (!aligned16(qkv) || !aligned16(ctx) || !aligned16(lse) || !aligned16(dctx) ||
      !aligned16(dqkv) || !aligned16(workspace) || dqkv == qkv || dqkv == dctx ||
      (dtype == MTL_BF16 && p_attn > 0.f && !aligned16(mask_bits)))
    return MTL_ERR_INVALID_ARG;
  if (ws_bytes < attn_ws_bytes(batch, seq, heads)) return MTL_ERR_WORKSPACE;
  const int nsm = device_sm_count();
  if (nsm <= 0) return cuda_fail(cudaGetLastError(), "device query");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  LaunchCtx c{s, nsm, &g_launches, &g_prof};
  unsigned* status = static_cast<unsigned*>(workspace);
  MTL_TRY(cudaMemsetAsync(status, 0, kStatusBytes, s), "status reset");
  if (batch == 0) return MTL_OK;
  float* dsum = at<float>(workspace, kStatusBytes);
  const Dropout drop = make_drop(p_attn, seed, SITE_ATTN);
  if (dtype == MTL_BF16) {
    MTL_TRY(attn_bwd_tc(qkv, ctx, lse, dctx, dqkv, dsum, batch, seq, heads, d, drop,
                        static_cast<const uint32_t*>(mask_bits), status, c),
            "attention bwd");
  } else {
    MTL_TRY(attn_bwd_simt(dtype, qkv, ctx, lse, dctx, dqkv, dsum, batch, seq, heads, d, drop, c),
            "attention bwd");
  }
  return MTL_OK;
}

// ---------------------------------------------------------------- inference

mtl_status mtl_infer_sizes(const mtl_layer_desc* desc, int32_t max_seq, size_t* kv_bytes,
                           size_t* prefill_ws_bytes, size_t* decode_ws_bytes) {
  Dims D;
  mtl_status st = validate_decode(desc, max_seq, &D);
  if (st != MTL_OK) return st;
  if (kv_bytes) *kv_bytes = kv_cache_bytes(D, max_seq);
  if (decode_ws_bytes) *decode_ws_bytes = decode_ws(D, max_seq).total;
  if (prefill_ws_bytes) {
    Dims P;
    mtl_layer_desc pd = *desc;
    pd.p_attn = 0.f;
    pd.p_hidden = 0.f;
    pd.recompute = 0;
    st = validate(&pd, &P);
    if (st != MTL_OK) return st;
    if (pd.seq > max_seq) return MTL_ERR_INVALID_ARG;
    *prefill_ws_bytes = kStatusBytes + saved_layout(P).total + fp8_ws_layout(P).total;
  }
  return MTL_OK;
}

mtl_status mtl_layer_prefill(const mtl_layer_desc* desc, const mtl_weights* w, const void* x,
                             void* y, void* kv_cache, int32_t max_seq, int32_t* cache_len,
                             void* workspace, size_t ws_bytes, mtl_stream stream) {
  g_launches = 0;
  g_cuda_err[0] = 0;
  if (!desc) return MTL_ERR_INVALID_ARG;
  if (desc->p_attn != 0.f || desc->p_hidden != 0.f) return MTL_ERR_INVALID_ARG;
  mtl_layer_desc pdesc = *desc;
  pdesc.recompute = 0;   // nothing is kept for a backward
  Dims D;
  mtl_status st = validate(&pdesc, &D);
  if (st != MTL_OK) return st;
  if (max_seq < desc->seq) return MTL_ERR_INVALID_ARG;
  if (!weights_ok(w) || !aligned16(x) || !aligned16(y) || !aligned16(kv_cache) ||
      !aligned16(workspace) || !cache_len || x == y)
    return MTL_ERR_INVALID_ARG;
  const size_t need = kStatusBytes + saved_layout(D).total + fp8_ws_layout(D).total;
  if (ws_bytes < need) return MTL_ERR_WORKSPACE;
  const int nsm = device_sm_count();
  if (nsm <= 0) return cuda_fail(cudaGetLastError(), "device query");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  LaunchCtx c{s, nsm, &g_launches, &g_prof};
  unsigned* status = static_cast<unsigned*>(workspace);
  MTL_TRY(cudaMemsetAsync(status, 0, kStatusBytes, s), "status reset");
  if (D.n == 0) return MTL_OK;
  void* saved = at<char>(workspace, kStatusBytes);
  st = forward_core(D, desc->ln_eps, w, x, y, saved,
                    at<char>(workspace, kStatusBytes + saved_layout(D).total), nullptr, nullptr,
                    status, c);
  if (st != MTL_OK) return st;
  const size_t half = kv_cache_bytes(D, max_seq) / 2;
  MTL_TRY(kv_write(D.dtype, at<char>(saved, saved_layout(D).qkv), kv_cache,
                   at<char>(kv_cache, half), cache_len, (int)D.batch, (int)D.seq, (int)D.heads,
                   (int)D.d, max_seq, c),
          "kv write");
  return MTL_OK;
}

mtl_status mtl_layer_decode(const mtl_layer_desc* desc, const mtl_weights* w, const void* x_tok,
                            void* y_tok, void* kv_cache, int32_t max_seq, int32_t* cache_len,
                            void* workspace, size_t ws_bytes, mtl_stream stream) {
  g_launches = 0;
  g_cuda_err[0] = 0;
  Dims D;
  mtl_status st = validate_decode(desc, max_seq, &D);
  if (st != MTL_OK) return st;
  if (!weights_ok(w) || !aligned16(x_tok) || !aligned16(y_tok) || !aligned16(kv_cache) ||
      !aligned16(workspace) || !cache_len || x_tok == y_tok)
    return MTL_ERR_INVALID_ARG;
  const DecWs W = decode_ws(D, max_seq);
  if (ws_bytes < W.total) return MTL_ERR_WORKSPACE;
  const int nsm = device_sm_count();
  if (nsm <= 0) return cuda_fail(cudaGetLastError(), "device query");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  LaunchCtx c{s, nsm, &g_launches, &g_prof};
  c.pdl = true;   // chain the step's kernels with programmatic dependent launch
  unsigned* status = static_cast<unsigned*>(workspace);
  // status word and the split-KV counters
  MTL_TRY(cudaMemsetAsync(status, 0, W.mean, s), "status reset");
  if (D.batch == 0) return MTL_OK;
  const int b = (int)D.batch, h = (int)D.h, f = (int)D.f;
  const bool bf = D.dtype == MTL_BF16;
  void* u = at<char>(workspace, W.u);
  void* qkv = at<char>(workspace, W.qkv);
  void* ctx = at<char>(workspace, W.ctx);
  void* x1 = at<char>(workspace, W.x1);
  void* a = at<char>(workspace, W.a);
  const size_t half = kv_cache_bytes(D, max_seq) / 2;
  // gemm on the layer's path: the split-K tcgen05 decode GEMM for bf16, the
  // exact fp32 CUDA-core GEMM for fp32
  auto dgemm = [&](int epi, int N, int K, const void* Wt, const void* X, const void* bias,
                   const void* R, void* out) -> cudaError_t {
    if (bf) return gemv_tc(epi, N, K, b, Wt, X, bias, R, out, status, c);
    GemmArgs g = gemm_args(b, N, K, 1, X, K, true, Wt, K, true, epi, out, N, false, status);
    g.bias = bias;
    g.R = R;
    g.ldr = N;
    g.Z = at<char>(workspace, W.z);
    g.ldz = N;
    return gemm_simt(kF32, g, c);
  };
  // D1 LN1
  MTL_TRY(ln_fwd(D.dtype, x_tok, w->ln1_g, w->ln1_b, u, at<float>(workspace, W.mean),
                 at<float>(workspace, W.rstd), b, h, desc->ln_eps, c),
          "ln1");
  // D2 QKV (column-parallel)
  MTL_TRY(dgemm(EPI_BIAS, 3 * h, h, w->w_qkv, u, w->b_qkv, nullptr, qkv), "qkv");
  // D3 attention over the cache; appends K, V
  double kvb = 0;   // algorithmic bytes are not known on the host (lengths live on the device)
  MTL_TRY(attn_decode(D.dtype, qkv, kv_cache, at<char>(kv_cache, half), cache_len, ctx,
                      at<float>(workspace, W.apart), at<int>(workspace, W.c_att), b,
                      (int)D.heads, (int)D.d, max_seq, kvb, status, c),
          "attention");
  // D4 out-proj (row-parallel, ordered K-slice sum) + b_o + x
  MTL_TRY(dgemm(EPI_BIAS_RESID, h, h, w->w_o, ctx, w->b_o, x_tok, x1), "out-proj");
  // D5 LN2
  MTL_TRY(ln_fwd(D.dtype, x1, w->ln2_g, w->ln2_b, u, at<float>(workspace, W.mean),
                 at<float>(workspace, W.rstd), b, h, desc->ln_eps, c),
          "ln2");
  // D6 fc1 + GeLU
  MTL_TRY(dgemm(EPI_BIAS_GELU, f, h, w->w_fc1, u, w->b_fc1, nullptr, a), "fc1");
  // D7 fc2 (row-parallel) + b_fc2 + x1
  MTL_TRY(dgemm(EPI_BIAS_RESID, h, f, w->w_fc2, a, w->b_fc2, x1, y_tok), "fc2");
  // D8 cache lengths + 1
  MTL_TRY(kv_advance(cache_len, b, max_seq, c), "advance");
  return MTL_OK;
}

// ---------------------------------------------------------------- FP8

mtl_status mtl_fp8_quantize(int32_t src_dtype, const void* x, int64_t rows, int64_t cols,
                            int64_t ld, int32_t fmt, void* q, int64_t ldq, void* qT,
                            int64_t ldqT, float* scale, void* workspace, size_t ws_bytes,
                            mtl_stream stream) {
  g_launches = 0;
  g_cuda_err[0] = 0;
  if (src_dtype != MTL_F32 && src_dtype != MTL_BF16) return MTL_ERR_INVALID_ARG;
  if (fmt != MTL_FP8_E4M3 && fmt != MTL_FP8_E5M2) return MTL_ERR_INVALID_ARG;
  if (rows < 0 || cols < 0 || ld < cols || cols % 16 || (!q && !qT)) return MTL_ERR_INVALID_ARG;
  if (q && (ldq < cols || ldq % 16 || !aligned16(q))) return MTL_ERR_INVALID_ARG;
  if (qT && (rows % 16 || ldqT < rows || ldqT % 16 || !aligned16(qT))) return MTL_ERR_INVALID_ARG;
  if (!aligned16(x) || !scale || !aligned16(workspace) ||
      (ld * (src_dtype == MTL_BF16 ? 2 : 4)) % 16)
    return MTL_ERR_INVALID_ARG;
  if (ws_bytes < kStatusBytes) return MTL_ERR_WORKSPACE;
  const int nsm = device_sm_count();
  if (nsm <= 0) return cuda_fail(cudaGetLastError(), "device query");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  LaunchCtx c{s, nsm, &g_launches, &g_prof};
  unsigned* status = static_cast<unsigned*>(workspace);
  MTL_TRY(cudaMemsetAsync(status, 0, kStatusBytes, s), "status reset");
  // the amax word sits in the status block, after the status word
  if (qT) {
    MTL_TRY(fp8_quantize2(src_dtype == MTL_BF16 ? kBF16 : kF32, x, rows, cols, ld, fmt, status + 1,
                          scale, q, ldq, qT, ldqT, c),
            "fp8 quantize");
  } else {
    MTL_TRY(fp8_quantize(src_dtype == MTL_BF16 ? kBF16 : kF32, x, rows, cols, ld, fmt,
                         status + 1, scale, q, ldq, c),
            "fp8 quantize");
  }
  return MTL_OK;
}

mtl_status mtl_gemm_ws_bytes(int32_t M, int32_t N, size_t* bytes) {
  if (M < 0 || N < 0 || !bytes) return MTL_ERR_INVALID_ARG;
  const int nsm = split_sms();
  const size_t split = gemm_split_bytes(M, N, nsm);
  *bytes = split ? kStatusBytes + align_up(gemm_split_counters(M, N, nsm) * 4) + split
                 : kStatusBytes;
  return MTL_OK;
}

mtl_status mtl_gemm_fp8(int32_t M, int32_t N, int32_t K, int32_t k_parts, const void* A,
                        int64_t lda, int32_t fmt_a, const float* scale_a, const void* B,
                        int64_t ldb, int32_t fmt_b, const float* scale_b, int32_t epi,
                        const void* bias, const void* R, int64_t ldr, void* Z, int64_t ldz,
                        void* C, int64_t ldc, int32_t c_f32, void* workspace, size_t ws_bytes,
                        mtl_stream stream) {
  g_launches = 0;
  g_cuda_err[0] = 0;
  if (M < 0 || N < 0 || K <= 0 || k_parts < 1 || K % k_parts) return MTL_ERR_INVALID_ARG;
  if (epi < EPI_STORE || epi > EPI_DGELU) return MTL_ERR_INVALID_ARG;
  if (lda < K || ldb < K || ldc < N) return MTL_ERR_INVALID_ARG;
  if ((fmt_a != MTL_FP8_E4M3 && fmt_a != MTL_FP8_E5M2) ||
      (fmt_b != MTL_FP8_E4M3 && fmt_b != MTL_FP8_E5M2))
    return MTL_ERR_INVALID_ARG;
  if (!aligned16(workspace) || !scale_a || !scale_b || !aligned16(A) || !aligned16(B) ||
      !aligned16(C))
    return MTL_ERR_INVALID_ARG;
  if (ws_bytes < kStatusBytes) return MTL_ERR_WORKSPACE;
  unsigned* status = static_cast<unsigned*>(workspace);
  GemmArgs g = gemm_args(M, N, K, k_parts, A, lda, true, B, ldb, true, epi, C, ldc, c_f32 != 0,
                         status);
  g.bias = bias;
  g.R = R;
  g.ldr = ldr;
  g.Z = Z;
  g.ldz = ldz;
  g.fmt_a = fmt_a;
  g.fmt_b = fmt_b;
  g.scale_a = scale_a;
  g.scale_b = scale_b;
  if (!gemm_fp8_supported(g, 2)) return MTL_ERR_UNSUPPORTED;
  const int nsm = device_sm_count();
  if (nsm <= 0) return cuda_fail(cudaGetLastError(), "device query");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t clear = standalone_gemm_split(g, workspace, ws_bytes);
  LaunchCtx c{s, nsm, &g_launches, &g_prof};
  MTL_TRY(cudaMemsetAsync(status, 0, clear, s), "status reset");
  if (M == 0 || N == 0) return MTL_OK;
  MTL_TRY(gemm_fp8(g, c), "gemm fp8");
  return MTL_OK;
}

mtl_status mtl_gemm(int32_t dtype, int32_t M, int32_t N, int32_t K, int32_t k_parts,
                    const void* A, int64_t lda, int32_t a_k_major, const void* B, int64_t ldb,
                    int32_t b_k_major, int32_t epi, const void* bias, const void* R, int64_t ldr,
                    void* Z, int64_t ldz, void* C, int64_t ldc, int32_t c_f32, void* workspace,
                    size_t ws_bytes, mtl_stream stream) {
  g_launches = 0;
  g_cuda_err[0] = 0;
  if (dtype != MTL_F32 && dtype != MTL_BF16) return MTL_ERR_INVALID_ARG;
  if (M < 0 || N < 0 || K < 0 || k_parts < 1 || K % k_parts) return MTL_ERR_INVALID_ARG;
  if (epi < EPI_STORE || epi > EPI_DGELU) return MTL_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(B) || !aligned16(C) || !aligned16(workspace))
    return MTL_ERR_INVALID_ARG;
  if (ws_bytes < kStatusBytes) return MTL_ERR_WORKSPACE;
  const bool need_bias = epi == EPI_BIAS || epi == EPI_BIAS_RESID || epi == EPI_BIAS_GELU;
  if (need_bias && !aligned16(bias)) return MTL_ERR_INVALID_ARG;
  if (epi == EPI_BIAS_RESID && !aligned16(R)) return MTL_ERR_INVALID_ARG;
  if ((epi == EPI_BIAS_GELU || epi == EPI_DGELU) && !aligned16(Z)) return MTL_ERR_INVALID_ARG;
  const int64_t a_rows = a_k_major ? M : K, b_rows = b_k_major ? N : K;
  const int64_t a_cols = a_k_major ? K : M, b_cols = b_k_major ? K : N;
  if ((a_rows > 0 && lda < a_cols) || (b_rows > 0 && ldb < b_cols) || ldc < N)
    return MTL_ERR_INVALID_ARG;
  if (epi == EPI_BIAS_RESID && ldr < N) return MTL_ERR_INVALID_ARG;
  if ((epi == EPI_BIAS_GELU || epi == EPI_DGELU) && ldz < N) return MTL_ERR_INVALID_ARG;
  unsigned* status = static_cast<unsigned*>(workspace);
  GemmArgs g = gemm_args(M, N, K, k_parts, A, lda, a_k_major != 0, B, ldb, b_k_major != 0, epi, C,
                         ldc, c_f32 != 0, status);
  g.bias = bias;
  g.R = R;
  g.ldr = ldr;
  g.Z = Z;
  g.ldz = ldz;
  if (dtype == MTL_BF16) {
    if (!gemm_tc_supported(g) || K == 0) return MTL_ERR_UNSUPPORTED;
  }
  const int nsm = device_sm_count();
  if (nsm <= 0) return cuda_fail(cudaGetLastError(), "device query");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t clear = dtype == MTL_BF16 ? standalone_gemm_split(g, workspace, ws_bytes)
                                           : kStatusBytes;
  LaunchCtx c{s, nsm, &g_launches, &g_prof};
  MTL_TRY(cudaMemsetAsync(status, 0, clear, s), "status reset");
  if (M == 0 || N == 0) return MTL_OK;
  if (dtype == MTL_BF16) {
    MTL_TRY(gemm_tc(g, c), "gemm");
  } else {
    MTL_TRY(gemm_simt(kF32, g, c), "gemm");
  }
  return MTL_OK;
}

}  // extern "C"
