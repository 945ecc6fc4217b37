/*
 * mtl.h -- C ABI of a GB300-native (sm_103a) pre-LN GPT transformer layer with
 * Megatron's intra-layer tensor-parallel split laid out inside one GPU.
 *
 * The operation (page "Megatron-LM: GPU-Cluster Training Parallelism"):
 *   * "Paper 1: BERT LayerNorm Rearrangement": Pre-LN, x -> LayerNorm ->
 *     sublayer -> added back onto x:
 *         x1 = x  + Attn(LN1(x)),   y = x1 + MLP(LN2(x1)).
 *   * "Paper 1: The f/g Conjugate Operators": the QKV and fc1 GEMMs are split by
 *     columns into t partitions (GeLU and softmax stay local to a partition);
 *     the out-proj and fc2 GEMMs are split by rows and give t partial sums that
 *     g reduces in the forward pass; f reduces the partial input gradients of
 *     the column-split GEMMs in the backward pass.  Two reductions forward, two
 *     backward.
 *   * "Paper 1: QKV Column-Parallel Splitting in Detail": the fused QKV weight is
 *     head-interleaved, so partition p owns heads [p*H/t, (p+1)*H/t) whole.
 *   * "Fused Transformer Kernels": causal scale-mask-softmax, bias+GeLU and
 *     bias+dropout+residual fused into the GEMMs.
 *
 * On one GPU the t partitions are a layout: partition p's shard is a view (a
 * row block of w_qkv / w_fc1, a column block of w_o / w_fc2 and the matching
 * column blocks of the activations).  The g and f all-reduces become fixed-order
 * (p = 0 .. t-1) sums of t separately accumulated fp32 partials inside the GEMM
 * epilogues, so results are bitwise reproducible for a given t and agree across
 * t within rounding.
 *
 * Conventions
 *   * All pointers are DEVICE pointers unless stated; the caller owns all
 *     memory.  The library allocates and frees nothing and keeps no state other
 *     than a once-initialised per-device cache of kernel attributes.
 *   * Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream).  Functions return after enqueueing.
 *   * Layouts are row-major.  x, y, dx, dy: [batch, seq, h].  Weights are
 *     [out, in]: w_qkv [3h][h] with head-interleaved rows
 *     (row = head*3*d + {0:Q,1:K,2:V}*d + channel, d = h/heads); w_o [h][h];
 *     w_fc1 [ffn][h]; w_fc2 [h][ffn].  b_qkv [3h] (same interleaved order),
 *     b_fc1 [ffn]; b_o, b_fc2, ln1_g, ln1_b, ln2_g, ln2_b [h].
 *   * Element type of x, y, dx, dy, weights and saved activations is desc.dtype
 *     (fp32 or bf16).  Gradients of the parameters are always fp32 and are
 *     OVERWRITTEN, not accumulated.  bf16 math accumulates in fp32.
 *   * GeLU is the exact x*Phi(x) (erf) form; the softmax scale is 1/sqrt(d);
 *     keys after the query are excluded (probability 0); LayerNorm uses the
 *     biased variance with desc.ln_eps inside the square root.
 *   * Dropout (desc.p_attn on the attention probabilities, desc.p_hidden after
 *     the out-projection and after fc2, each before its residual add):
 *       x1 = x  + drop_1(ctx W_o^T + b_o),   y = x1 + drop_2(a W_fc2^T + b_fc2),
 *       ctx = (P * keep_0 / (1 - p_attn)) V  (lse stays that of the undropped P).
 *     keep_s(e) = word_s(e) >= floor(p * 2^32) with word_s(e) = output word
 *     (e mod 4) of Philox4x32-10 at counter {e/4 mod 2^32, e/4 >> 32, s, 0} and
 *     key {seed mod 2^32, seed >> 32} (Salmon et al., SC'11).  Site s = 0:
 *     attention, e = ((b*heads + head)*seq + i)*seq + j for query i, key j;
 *     s = 1: out-projection output, s = 2: fc2 output, e = token*h + column.
 *     The hidden-site masks are redrawn from (seed, e) in the backward; the
 *     attention mask of a bf16 layer is drawn once by the forward and kept as
 *     bits in `saved` (fp32 layers redraw it).  mtl_layer_bwd must get the desc
 *     (seed, p) of the forward it follows.
 *   * Every pointer must be 16-byte aligned.  Validation failures return before
 *     anything is enqueued.  No C++ exception crosses this boundary.  Calls are
 *     reentrant; calls on different streams may run concurrently as long as
 *     they use different workspaces.
 *   * Errors: MTL_ERR_INVALID_ARG (null / misaligned pointer, bad sizes),
 *     MTL_ERR_UNSUPPORTED (valid layer outside what the kernels implement),
 *     MTL_ERR_WORKSPACE (ws_bytes too small), MTL_ERR_CUDA (a CUDA call or launch
 *     failed; see mtl_last_cuda_error), MTL_ERR_TIMEOUT (a device-side bounded
 *     wait gave up; reported by mtl_layer_check), MTL_ERR_BOUNDS (a library
 *     built with MTL_DEBUG found a computed TMA coordinate or output index
 *     outside its tensor and skipped that access; reported by mtl_layer_check,
 *     with the fault and call site in mtl_last_cuda_error).
 */
#ifndef MTL_H_
#define MTL_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* mtl_stream;  /* == cudaStream_t */

typedef enum {
  MTL_OK = 0,
  MTL_ERR_INVALID_ARG = 1,
  MTL_ERR_UNSUPPORTED = 2,
  MTL_ERR_WORKSPACE = 3,
  MTL_ERR_CUDA = 4,
  MTL_ERR_TIMEOUT = 5,
  MTL_ERR_BOUNDS = 6
} mtl_status;

typedef enum { MTL_F32 = 0, MTL_BF16 = 1 } mtl_dtype;

/* FP8 formats (OCP 8-bit floating point). */
typedef enum { MTL_FP8_E4M3 = 0, MTL_FP8_E5M2 = 1 } mtl_fp8_format;

/* One layer.  h = heads * d with d in {64, 96, 128}; t divides heads and ffn;
 * causal must be 1.  bf16 layers (tensor-core path) additionally need
 * seq % 128 == 0, h % 64 == 0, ffn % 64 == 0, (h/t) % 64 == 0, (3h/t) % 64 == 0
 * and (ffn/t) % 64 == 0, else MTL_ERR_UNSUPPORTED.  fp32 layers run exact fp32
 * CUDA-core kernels and need only h % 4 == 0 and ffn % 4 == 0. */
typedef struct {
  int32_t h, heads, seq, batch, ffn, t;
  int32_t dtype;     /* mtl_dtype */
  float ln_eps;      /* 1e-5 */
  int32_t causal;    /* 1 */
  float p_attn;      /* attention dropout probability, 0 <= p_attn < 1 */
  float p_hidden;    /* hidden dropout probability, 0 <= p_hidden < 1 */
  uint64_t seed;     /* Philox key of the dropout masks */
  int32_t fp8;       /* 1: the forward's four GEMMs take per-tensor E4M3 operands
                        (bf16 layers without dropout, h, h/t and ffn/t multiples
                        of 128; the backward and decode stay bf16); 2: "hybrid",
                        also the backward's eight GEMMs in FP8, E5M2 gradient x
                        E4M3 activation or weight ((3h)/t a multiple of 128
                        too); 0: bf16 */
  int32_t post_ln;   /* 1: Post-LN layer (original BERT, page section "Paper 1:
                        BERT LayerNorm Rearrangement"): h1 = x + Attn(x),
                        x1 = LN1(h1), h2 = x1 + MLP(x1), y = LN2(h2), with the
                        QKV GEMM on x; no dropout, no FP8, no decode; 0: Pre-LN */
  int32_t recompute; /* 1: selective recomputation: the forward does not save the
                        LayerNorm outputs (Pre-LN u1, u2; Post-LN x1) or
                        a = GeLU(z); the backward recomputes them from the saved
                        inputs and statistics (LayerNorm outputs bit for bit).
                        Smaller `saved`, one elementwise pass each; 0: save all */
} mtl_layer_desc;

typedef struct {
  const void *w_qkv, *b_qkv, *w_o, *b_o, *w_fc1, *b_fc1, *w_fc2, *b_fc2;
  const void *ln1_g, *ln1_b, *ln2_g, *ln2_b;
} mtl_weights;

typedef struct {
  void *w_qkv, *b_qkv, *w_o, *b_o, *w_fc1, *b_fc1, *w_fc2, *b_fc2;
  void *ln1_g, *ln1_b, *ln2_g, *ln2_b;
} mtl_grads;   /* all fp32 */

/* Byte offsets of the activations the forward saves for the backward, inside
 * the caller's `saved` buffer (each 256-byte aligned).  Element types: mu*,
 * rstd*, lse fp32; the rest desc.dtype.  Shapes with n = batch*seq:
 * mu1, rstd1, mu2, rstd2 [n]; u1, ctx, x1, u2 [n][h]; qkv [n][3h] (columns in
 * the head-interleaved order of w_qkv); lse [batch][heads][seq] (log of the
 * softmax normaliser per query row); z (fc1 pre-activation) and a = GeLU(z)
 * [n][ffn]. */
typedef struct {
  size_t mu1, rstd1, u1, qkv, ctx, lse, x1, mu2, rstd2, u2, z, a;
  size_t attn_mask;   /* keep bits of attention dropout (bf16 layers with p_attn > 0;
                         empty otherwise), see mtl_attention_mask_bytes */
  size_t h1, h2;      /* Post-LN: the LayerNorm inputs x + Attn(x) and x1 + MLP(x1)
                         [n][h] (mu1 / rstd1 and mu2 / rstd2 are their statistics;
                         u1, u2 are empty); Pre-LN: empty.  With recompute, u1, u2
                         (Pre-LN), x1 (Post-LN) and a are empty. */
  size_t fp8;         /* FP8 hybrid (desc.fp8 = 2): 16 fp32 scales, then the E4M3
                         transposes of u1, ctx, u2 [h][n] and a [f][n] and of
                         W_qkv [h][3h], W_o [h][h], W_fc1 [h][f], W_fc2 [f][h]
                         (each 256-byte aligned), which the backward reads in
                         place of u1, u2 and a (then empty); otherwise empty. */
  size_t total;
} mtl_saved_layout;

/* Sizes in bytes of the `saved` buffer written by mtl_layer_fwd and read by
 * mtl_layer_bwd, and of the scratch workspace both calls need (the same value
 * serves both).  Returns MTL_ERR_INVALID_ARG / MTL_ERR_UNSUPPORTED for a desc
 * the kernels cannot run. */
mtl_status mtl_layer_sizes(const mtl_layer_desc* desc, size_t* saved_bytes,
                           size_t* workspace_bytes);

/* Offsets of each saved activation inside `saved` (see mtl_saved_layout). */
mtl_status mtl_layer_saved_layout(const mtl_layer_desc* desc, mtl_saved_layout* out);

/* Byte offsets, inside the caller's `workspace`, of the backward's
 * intermediates, which stay there after mtl_layer_bwd (stream-ordered) until
 * the next call using that workspace -- for inspection.  n = batch*seq.
 * Pre-LN layer: dz [n][ffn] (desc.dtype) = (g2 W_fc2) * GeLU'(z); du [n][h]
 * fp32 = the f-summed gradient at the LN1 output (du1; the LN2 one, du2, is
 * written first and overwritten); dx1 [n][h] (desc.dtype), the gradient at
 * the attention block's output; dctx [n][h] (desc.dtype) = go W_o; dqkv
 * [n][3h] (desc.dtype, head-interleaved columns).  Post-LN layer: dctx holds
 * the LN2 input gradient dh2 and dx1 the LN1 input gradient dh1. */
typedef struct {
  size_t dz, du, dx1, dctx, dqkv, total;
} mtl_workspace_layout;
mtl_status mtl_layer_workspace_layout(const mtl_layer_desc* desc, mtl_workspace_layout* out);

/* Forward pass: y = layer(x).  x, y [batch][seq][h] of desc.dtype; `saved`
 * (>= saved_bytes) receives the activations for the backward; `workspace`
 * (>= workspace_bytes, contents not preserved) is scratch.  y must not alias x
 * or saved.  Steps, in stream order: LN1; QKV GEMM (column-parallel, bias
 * epilogue); causal attention per head; out-proj GEMM (row-parallel: t fp32
 * partials summed in order, + b_o + x); LN2; fc1 GEMM (column-parallel, bias +
 * GeLU epilogue, saves z and a); fc2 GEMM (row-parallel, + b_fc2 + x1). */
mtl_status mtl_layer_fwd(const mtl_layer_desc* desc, const mtl_weights* w, const void* x,
                         void* y, void* saved, void* workspace, size_t ws_bytes,
                         mtl_stream stream);

/* Backward pass for upstream gradient dy (the gradient of a loss with respect
 * to y).  Reads x and the `saved` buffer written by mtl_layer_fwd with the same
 * desc and weights; writes dx [batch][seq][h] (desc.dtype) and every pointer in
 * `grads` (fp32, overwritten).  The two f reductions (input gradients of the QKV
 * and fc1 GEMMs) are t fp32 partials summed in partition order. */
mtl_status mtl_layer_bwd(const mtl_layer_desc* desc, const mtl_weights* w, const void* x,
                         const void* saved, const void* dy, void* dx, const mtl_grads* grads,
                         void* workspace, size_t ws_bytes, mtl_stream stream);

/* Waits for `stream`, then reports the device-side status word that the last
 * call using `workspace` left: MTL_OK, or MTL_ERR_TIMEOUT if a bounded
 * device wait gave up (the call's outputs are then undefined).  Resets it. */
mtl_status mtl_layer_check(void* workspace, mtl_stream stream);

/* Utility GEMM on the same kernels, for component tests:
 *   C[m][n] = sum_{p<k_parts} ( sum_{k in part p} A(m,k) * B(n,k) )
 * with the k_parts partial sums accumulated separately in fp32 and added in
 * order p = 0..k_parts-1, then the epilogue:
 *   epi 0: C = acc                      epi 1: C = acc + bias[n]
 *   epi 2: C = acc + bias[n] + R[m][n]  epi 3: Z = acc + bias[n], C = GeLU(Z)
 *   epi 4: C = acc * GeLU'(Z[m][n])
 * A(m,k) = A[m*lda + k] if a_k_major else A[k*lda + m]; likewise B(n,k) with
 * b_k_major.  A, B, bias, R, Z are `dtype`; C is fp32 if c_f32 else `dtype`.
 * Leading dimensions are in elements (C: ldc, R: ldr, Z: ldz).  K must split
 * into k_parts equal parts; bf16 needs (K/k_parts) % 64 == 0 and lda, ldb,
 * ldc, ldr, ldz multiples of 8.
 * workspace: device, 16-byte aligned, at least 256 bytes (the status word).
 * With mtl_gemm_ws_bytes(M, N) bytes, a bf16 GEMM whose 256 x 256 tiles leave
 * the last wave over the SM pairs partly empty cuts each tile of that wave into
 * equal K slices (runs of K-blocks, or of partitions) on separate pairs, whose
 * fp32 partials are added in slice order before the epilogue -- a fixed order
 * for a given shape and SM count, so results stay bitwise reproducible. */
mtl_status mtl_gemm(int32_t dtype, int32_t M, int32_t N, int32_t K, int32_t k_parts,
                    const void* A, int64_t lda, int32_t a_k_major,
                    const void* B, int64_t ldb, int32_t b_k_major,
                    int32_t epi, const void* bias, const void* R, int64_t ldr,
                    void* Z, int64_t ldz, void* C, int64_t ldc, int32_t c_f32,
                    void* workspace, size_t ws_bytes, mtl_stream stream);

/* Workspace bytes for mtl_gemm / mtl_gemm_fp8 with an M x N output (any K)
 * that lets the tiles of the last, partial wave be cut into K slices (at least
 * 256; the count depends on the current device's SM count). */
mtl_status mtl_gemm_ws_bytes(int32_t M, int32_t N, size_t* bytes);

/* Causal multi-head attention, the layer's attention step on its own (same
 * kernels, same dropout numbering with site 0):
 *   qkv [batch*seq][3*heads*d], head-interleaved (column = head*3d +
 *   {0:Q,1:K,2:V}*d + channel); ctx [batch*seq][heads*d]; lse
 *   [batch][heads][seq] fp32 (natural log of the undropped softmax normaliser).
 *   Forward: ctx = (softmax(Q K^T / sqrt d, causal) * keep / (1 - p_attn)) V.
 *   Backward: dqkv [batch*seq][3*heads*d] (same interleave) from dctx, given
 *   the forward's qkv, ctx and lse and the same p_attn and seed.
 * dtype MTL_BF16 (tcgen05 kernels; seq % 128 == 0) or MTL_F32 (CUDA cores;
 * seq <= 8192); d in {64, 96, 128}; 0 <= p_attn < 1.  Device pointers, 16-byte
 * aligned.  mask_bits (mtl_attention_mask_bytes, which is 0 unless dtype is
 * MTL_BF16 and p_attn > 0; may be NULL then): written by the forward with the
 * keep bits it drew, read by the backward.  workspace: >=
 * mtl_attention_ws_bytes (status word and the backward's row sums D_i =
 * dO_i . O_i); check it with mtl_layer_check.  Errors as for the layer calls. */
mtl_status mtl_attention_ws_bytes(int32_t batch, int32_t seq, int32_t heads, size_t* bytes);
mtl_status mtl_attention_mask_bytes(int32_t dtype, int32_t batch, int32_t seq, int32_t heads,
                                    float p_attn, size_t* bytes);
mtl_status mtl_attention_fwd(int32_t dtype, int32_t batch, int32_t seq, int32_t heads, int32_t d,
                             const void* qkv, void* ctx, float* lse, void* mask_bits,
                             float p_attn, uint64_t seed, void* workspace, size_t ws_bytes,
                             mtl_stream stream);
mtl_status mtl_attention_bwd(int32_t dtype, int32_t batch, int32_t seq, int32_t heads, int32_t d,
                             const void* qkv, const void* ctx, const float* lse, const void* dctx,
                             const void* mask_bits, void* dqkv, float p_attn, uint64_t seed,
                             void* workspace, size_t ws_bytes, mtl_stream stream);

/* ---- Inference: prefill and one-token decode with a head-sharded KV cache
 * (page "Megatron-LM: GPU-Cluster Training Parallelism", section "Paper 1: QKV
 * Column-Parallel Splitting in Detail", inference-time behaviour: each
 * partition appends the new token's K and V of its own heads to its local
 * cache shard, so the cache divides evenly by t; the row-parallel outputs are
 * reduced once per token).
 *   kv_cache: K then V, each [batch][heads][max_seq][d] of desc.dtype, the V
 *   block starting kv_bytes/2 into the buffer; partition p's shard is heads
 *   [p*H/t, (p+1)*H/t) of every batch row.  cache_len: DEVICE int32 [batch],
 *   the number of valid positions of each sequence.
 *   mtl_layer_prefill: y = layer(x) for prompts x [batch][desc.seq][h] (no
 *   dropout), K and V of every prompt token written at positions
 *   0..desc.seq-1, cache_len[b] = desc.seq.  Same shape rules as mtl_layer_fwd;
 *   desc.seq <= max_seq.
 *   mtl_layer_decode: one new token per sequence, x_tok / y_tok [batch][h]:
 *   token b sits at position cache_len[b], its K and V are written there, it
 *   attends to keys 0..cache_len[b], and cache_len[b] is incremented, so a
 *   captured CUDA graph of this call can be replayed token after token.
 *   desc.seq is not used; desc.batch <= 128.  A cache_len outside
 *   [0, max_seq) makes the step skip that sequence's attention and report
 *   MTL_ERR_INVALID_ARG through mtl_layer_check (its outputs are undefined).
 *   The bf16 decode GEMMs read every weight once per step (split-K tcgen05,
 *   the K slices of a tile summed in slice order: bitwise reproducible).
 * mtl_infer_sizes: bytes of the cache and of the two calls' workspaces
 * (prefill's holds the layer's intermediates). */
mtl_status mtl_infer_sizes(const mtl_layer_desc* desc, int32_t max_seq, size_t* kv_bytes,
                           size_t* prefill_ws_bytes, size_t* decode_ws_bytes);
mtl_status mtl_layer_prefill(const mtl_layer_desc* desc, const mtl_weights* w, const void* x,
                             void* y, void* kv_cache, int32_t max_seq, int32_t* cache_len,
                             void* workspace, size_t ws_bytes, mtl_stream stream);
mtl_status mtl_layer_decode(const mtl_layer_desc* desc, const mtl_weights* w, const void* x_tok,
                            void* y_tok, void* kv_cache, int32_t max_seq, int32_t* cache_len,
                            void* workspace, size_t ws_bytes, mtl_stream stream);

/* ---- FP8 (the pages list FP8 training, "--fp8-hybrid", without a recipe;
 * read as E4M3 forward operands, E5M2 gradients, per-tensor current scaling).
 * mtl_fp8_quantize: x [rows][cols] (src_dtype, row pitch ld elements) ->
 *   amax = max |x| over the whole matrix, *scale = fmt_max / amax (1 if
 *   amax = 0; fmt_max 448 for E4M3, 57344 for E5M2), q [rows][cols] bytes
 *   (row pitch ldq) = fp8(float32(x * scale)), rounded to nearest even and
 *   saturated to +-fmt_max, and / or its transpose qT [cols][rows] (row pitch
 *   ldqT; for a K-major operand of a transposed use).  Either q or qT may be
 *   NULL, not both.  scale: a DEVICE float.  cols, ldq (and with qT: rows,
 *   ldqT) multiples of 16; workspace >= 256 bytes (status and amax words).
 * mtl_gemm_fp8: as mtl_gemm with K-major FP8 operands A [M][K] (lda) and
 *   B [N][K] (ldb) of formats fmt_a / fmt_b and their DEVICE scales; the
 *   partition partials (k_parts, each a multiple of 128 deep) are summed in
 *   order, multiplied by float32(1 / float32(scale_a * scale_b)), then the
 *   epilogue applies (same epilogue codes and C / R / Z conventions).  lda and
 *   ldb multiples of 16.  Runs on the 2-CTA tcgen05 kernel (kind::f8f6f4). */
mtl_status mtl_fp8_quantize(int32_t src_dtype, const void* x, int64_t rows, int64_t cols,
                            int64_t ld, int32_t fmt, void* q, int64_t ldq, void* qT,
                            int64_t ldqT, float* scale, void* workspace, size_t ws_bytes,
                            mtl_stream stream);
mtl_status mtl_gemm_fp8(int32_t M, int32_t N, int32_t K, int32_t k_parts, const void* A,
                        int64_t lda, int32_t fmt_a, const float* scale_a, const void* B,
                        int64_t ldb, int32_t fmt_b, const float* scale_b, int32_t epi,
                        const void* bias, const void* R, int64_t ldr, void* Z, int64_t ldz,
                        void* C, int64_t ldc, int32_t c_f32, void* workspace, size_t ws_bytes,
                        mtl_stream stream);

/* Bias gradient for callers that cannot allocate device memory:
 *   out[j] = sum_{i < rows} dy[i*ld + j]   (j < cols; fp32, fixed order)
 * -- the sum mtl_layer_bwd uses for b_fc2, b_o, b_fc1 and b_qkv, with the same
 * kernels and the same result.  The paper has no counterpart; this exists for
 * callers whose device memory is planned up front and who may not call the
 * CUDA allocator (a runtime that hands all of HBM to its own pool at start-up,
 * a deployment with a fixed memory plan), and so cannot provide a workspace.
 *   dtype: MTL_F32 or MTL_BF16, the element type of dy; out is fp32.
 *   dy: device, 16-byte aligned; ld and cols multiples of 8 (bf16) or 4 (fp32),
 *   ld >= cols; out: device, cols floats.
 * Scratch: a static device array of 8 MiB (128 x 16384 floats) inside the
 * library, held by every GPU that loads it until the process exits; cols above
 * 16384 return MTL_ERR_UNSUPPORTED.  Nothing is allocated or freed: no
 * cudaMalloc, no cudaFree, no allocating library call.  The first call on a
 * device looks up the array's device address (cudaGetSymbolAddress, with that
 * device current); make that first call before any stream capture.  A failed
 * lookup returns MTL_ERR_CUDA and is not kept: the next call on that device
 * looks the address up again.  All calls
 * on a device share the one array, whose contents persist from the last call:
 * calls that overlap on the GPU (different streams, no ordering) race and give
 * wrong sums, so order them on one stream.  Returns MTL_ERR_INVALID_ARG for
 * bad pointers or sizes and MTL_ERR_CUDA if a launch fails. */
mtl_status mtl_bias_grad_noalloc(int32_t dtype, const void* dy, int64_t ld, int32_t rows,
                                 int32_t cols, void* out, mtl_stream stream);

/* Failure-detection self-test: launches one CTA that waits, with the same
 * bounded device wait the pipelined kernels use, on a barrier nothing signals.
 * After limit_cycles SM cycles (1000 .. 4e9) the wait gives up and records a
 * timeout in the status word of `workspace` (>= 256 bytes), so a following
 * mtl_layer_check returns MTL_ERR_TIMEOUT; the GPU context stays usable. */
mtl_status mtl_selftest_wait_timeout(void* workspace, int64_t limit_cycles, mtl_stream stream);

/* Failure-detection self-test of the launch-error path: enqueues an empty
 * kernel with 2048 threads a block, above the 1024-thread limit of CUDA
 * devices, so the runtime refuses the launch before anything runs on the GPU.
 * Returns MTL_ERR_CUDA, with the runtime's error text in mtl_last_cuda_error,
 * the way every entry point reports a failed launch; the error is not sticky,
 * so the context stays usable. */
mtl_status mtl_selftest_launch_error(mtl_stream stream);

/* Human-readable name of a status. */
const char* mtl_status_str(mtl_status s);

/* Text of the last CUDA error seen by this thread's calls (empty if none). */
const char* mtl_last_cuda_error(void);

/* Number of kernels the last mtl_layer_fwd / mtl_layer_bwd / mtl_gemm call on
 * this thread enqueued. */
int32_t mtl_last_launch_count(void);

/* Per-kernel timing for measurement.  `events` points to 2*capacity caller-
 * created CUDA events (cudaEvent_t); while set, each kernel the calling thread
 * enqueues records events[2i] before and events[2i+1] after itself on its
 * stream, and writes its kind to kinds[i] (1 tensor-core GEMM, 2 CUDA-core
 * GEMM, 3 attention forward, 4 attention backward, 5 LayerNorm forward,
 * 6 LayerNorm backward, 7 column sum, 8 partial-sum finalise) and its
 * algorithmic work to work[i] (flops for GEMMs and attention, bytes moved for
 * the memory-bound kernels).  Launches past `capacity` are not recorded.
 * Passing events = NULL turns recording off.  The library keeps the pointers
 * until the next call; the caller owns and frees everything. */
void mtl_profile_set(void** events, int32_t capacity, int32_t* kinds, double* work);

/* Number of kernels recorded since the last mtl_profile_set. */
int32_t mtl_profile_count(void);

#ifdef __cplusplus
}
#endif

#endif /* MTL_H_ */
