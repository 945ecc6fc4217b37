"""ctypes binding of the C ABI in include/mtl.h (argument marshalling only).

Every step of the layer runs in the CUDA library libmtl.so; this module only
turns torch tensors into device pointers, picks the current CUDA stream and
raises on a non-OK status.  It fails loudly when the library is missing: there
is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

PARAM_NAMES = ("w_qkv", "b_qkv", "w_o", "b_o", "w_fc1", "b_fc1", "w_fc2", "b_fc2",
               "ln1_g", "ln1_b", "ln2_g", "ln2_b")
SAVED_NAMES = ("mu1", "rstd1", "u1", "qkv", "ctx", "lse", "x1", "mu2", "rstd2", "u2", "z", "a",
               "attn_mask", "h1", "h2", "fp8")

F32, BF16 = 0, 1
STATUS = {0: "MTL_OK", 1: "MTL_ERR_INVALID_ARG", 2: "MTL_ERR_UNSUPPORTED",
          3: "MTL_ERR_WORKSPACE", 4: "MTL_ERR_CUDA", 5: "MTL_ERR_TIMEOUT", 6: "MTL_ERR_BOUNDS"}

# The library to load: the in-tree build, or another build of it named by
# MTL_LIBRARY (e.g. the MTL_DEBUG build, libmtl_debug.so).
LIB_PATH = os.environ.get("MTL_LIBRARY") or os.path.join(
    os.path.dirname(os.path.abspath(__file__)), "libmtl.so")


class MtlError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        msg = f"{where}: {STATUS.get(status, status)}"
        if detail:
            msg += f" ({detail})"
        super().__init__(msg)


class LayerDesc(ctypes.Structure):
    _fields_ = [("h", ctypes.c_int32), ("heads", ctypes.c_int32), ("seq", ctypes.c_int32),
                ("batch", ctypes.c_int32), ("ffn", ctypes.c_int32), ("t", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("ln_eps", ctypes.c_float), ("causal", ctypes.c_int32),
                ("p_attn", ctypes.c_float), ("p_hidden", ctypes.c_float), ("seed", ctypes.c_uint64),
                ("fp8", ctypes.c_int32), ("post_ln", ctypes.c_int32), ("recompute", ctypes.c_int32)]


class Weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in PARAM_NAMES]


class Grads(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in PARAM_NAMES]


class WorkspaceLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in ("dz", "du", "dx1", "dctx", "dqkv", "total")]


class SavedLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in SAVED_NAMES] + [("total", ctypes.c_size_t)]


_lib = None


def lib():
    """The loaded libmtl.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "tensor_model_transformer_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        vp, sz, i32, i64 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32, ctypes.c_int64
        pd = ctypes.POINTER(LayerDesc)
        L.mtl_layer_sizes.argtypes = [pd, ctypes.POINTER(sz), ctypes.POINTER(sz)]
        L.mtl_layer_saved_layout.argtypes = [pd, ctypes.POINTER(SavedLayout)]
        L.mtl_layer_workspace_layout.argtypes = [pd, ctypes.POINTER(WorkspaceLayout)]
        L.mtl_layer_fwd.argtypes = [pd, ctypes.POINTER(Weights), vp, vp, vp, vp, sz, vp]
        L.mtl_layer_bwd.argtypes = [pd, ctypes.POINTER(Weights), vp, vp, vp, vp,
                                    ctypes.POINTER(Grads), vp, sz, vp]
        L.mtl_layer_check.argtypes = [vp, vp]
        L.mtl_gemm.argtypes = [i32, i32, i32, i32, i32, vp, i64, i32, vp, i64, i32, i32, vp, vp,
                               i64, vp, i64, vp, i64, i32, vp, sz, vp]
        L.mtl_attention_ws_bytes.argtypes = [i32, i32, i32, ctypes.POINTER(sz)]
        L.mtl_gemm_ws_bytes.argtypes = [i32, i32, ctypes.POINTER(sz)]
        L.mtl_attention_mask_bytes.argtypes = [i32, i32, i32, i32, ctypes.c_float,
                                               ctypes.POINTER(sz)]
        L.mtl_attention_fwd.argtypes = [i32, i32, i32, i32, i32, vp, vp, vp, vp, ctypes.c_float,
                                        ctypes.c_uint64, vp, sz, vp]
        L.mtl_attention_bwd.argtypes = [i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp,
                                        ctypes.c_float, ctypes.c_uint64, vp, sz, vp]
        L.mtl_infer_sizes.argtypes = [pd, i32, ctypes.POINTER(sz), ctypes.POINTER(sz),
                                      ctypes.POINTER(sz)]
        L.mtl_layer_prefill.argtypes = [pd, ctypes.POINTER(Weights), vp, vp, vp, i32, vp, vp, sz,
                                        vp]
        L.mtl_layer_decode.argtypes = [pd, ctypes.POINTER(Weights), vp, vp, vp, i32, vp, vp, sz,
                                       vp]
        L.mtl_fp8_quantize.argtypes = [i32, vp, i64, i64, i64, i32, vp, i64, vp, i64, vp, vp,
                                       sz, vp]
        L.mtl_gemm_fp8.argtypes = [i32, i32, i32, i32, vp, i64, i32, vp, vp, i64, i32, vp, i32,
                                   vp, vp, i64, vp, i64, vp, i64, i32, vp, sz, vp]
        L.mtl_selftest_wait_timeout.argtypes = [vp, i64, vp]
        L.mtl_selftest_wait_timeout.restype = ctypes.c_int
        L.mtl_selftest_launch_error.argtypes = [vp]
        L.mtl_selftest_launch_error.restype = ctypes.c_int
        L.mtl_bias_grad_noalloc.argtypes = [i32, vp, i64, i32, i32, vp, vp]
        L.mtl_bias_grad_noalloc.restype = ctypes.c_int
        L.mtl_status_str.argtypes = [ctypes.c_int]
        L.mtl_status_str.restype = ctypes.c_char_p
        L.mtl_last_cuda_error.restype = ctypes.c_char_p
        L.mtl_last_launch_count.restype = ctypes.c_int32
        for fn in ("mtl_layer_sizes", "mtl_layer_saved_layout", "mtl_layer_fwd", "mtl_layer_bwd",
                   "mtl_layer_check", "mtl_gemm", "mtl_attention_ws_bytes", "mtl_attention_fwd",
                   "mtl_attention_bwd", "mtl_attention_mask_bytes", "mtl_infer_sizes",
                   "mtl_layer_prefill", "mtl_layer_decode", "mtl_fp8_quantize", "mtl_gemm_fp8",
                   "mtl_gemm_ws_bytes", "mtl_layer_workspace_layout"):
            getattr(L, fn).restype = ctypes.c_int
        _lib = L
    return _lib


def _check(status: int, where: str):
    if status != 0:
        detail = lib().mtl_last_cuda_error().decode() if status in (4, 6) else ""
        raise MtlError(status, where, detail)


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


def layer_desc(h, heads, seq, batch, ffn, t, dtype, ln_eps=1e-5, causal=1, p_attn=0.0,
               p_hidden=0.0, seed=0, fp8=0, post_ln=0, recompute=0) -> LayerDesc:
    """mtl_layer_desc; p_attn / p_hidden / seed: dropout probabilities and Philox seed;
    fp8=1: FP8 (E4M3) forward GEMMs; post_ln=1: Post-LN layer; recompute=1:
    selective recomputation of the LayerNorm outputs and GeLU(z)."""
    dt = {"f32": F32, "bf16": BF16, F32: F32, BF16: BF16}[dtype]
    return LayerDesc(h, heads, seq, batch, ffn, t, dt, ln_eps, causal, p_attn, p_hidden, seed,
                     fp8, post_ln, recompute)


def layer_sizes(desc: LayerDesc):
    """(saved_bytes, workspace_bytes) of mtl_layer_sizes."""
    s, w = ctypes.c_size_t(0), ctypes.c_size_t(0)
    _check(lib().mtl_layer_sizes(ctypes.byref(desc), ctypes.byref(s), ctypes.byref(w)),
           "mtl_layer_sizes")
    return s.value, w.value


def layer_saved_layout(desc: LayerDesc) -> dict:
    out = SavedLayout()
    _check(lib().mtl_layer_saved_layout(ctypes.byref(desc), ctypes.byref(out)),
           "mtl_layer_saved_layout")
    return {n: getattr(out, n) for n in SAVED_NAMES + ("total",)}


def _weights(w: dict) -> Weights:
    return Weights(*[_ptr(w[n]) for n in PARAM_NAMES])


def _grads(g: dict) -> Grads:
    return Grads(*[_ptr(g[n]) for n in PARAM_NAMES])


def layer_fwd(desc, weights: dict, x, y, saved, workspace, stream=None):
    """mtl_layer_fwd on torch tensors (device memory)."""
    wt = _weights(weights)
    _check(lib().mtl_layer_fwd(ctypes.byref(desc), ctypes.byref(wt), _ptr(x), _ptr(y),
                               _ptr(saved), _ptr(workspace), workspace.numel() * workspace.element_size(),
                               _stream(stream)), "mtl_layer_fwd")


def layer_bwd(desc, weights: dict, x, saved, dy, dx, grads: dict, workspace, stream=None):
    """mtl_layer_bwd on torch tensors (device memory)."""
    wt, gt = _weights(weights), _grads(grads)
    _check(lib().mtl_layer_bwd(ctypes.byref(desc), ctypes.byref(wt), _ptr(x), _ptr(saved),
                               _ptr(dy), _ptr(dx), ctypes.byref(gt), _ptr(workspace),
                               workspace.numel() * workspace.element_size(), _stream(stream)),
           "mtl_layer_bwd")


def layer_check(workspace, stream=None):
    """mtl_layer_check: waits for the stream, raises MtlError on a device timeout."""
    _check(lib().mtl_layer_check(_ptr(workspace), _stream(stream)), "mtl_layer_check")


def last_launch_count() -> int:
    return lib().mtl_last_launch_count()


def gemm(dtype, M, N, K, parts, A, lda, a_k_major, B, ldb, b_k_major, epi, C, ldc, c_f32,
         workspace, bias=None, R=None, ldr=0, Z=None, ldz=0, stream=None):
    """mtl_gemm on torch tensors."""
    dt = {"f32": F32, "bf16": BF16, F32: F32, BF16: BF16}[dtype]
    _check(lib().mtl_gemm(dt, M, N, K, parts, _ptr(A), lda, int(a_k_major), _ptr(B), ldb,
                          int(b_k_major), epi, _ptr(bias), _ptr(R), ldr, _ptr(Z), ldz, _ptr(C),
                          ldc, int(c_f32), _ptr(workspace),
                          workspace.numel() * workspace.element_size(), _stream(stream)),
           "mtl_gemm")


def gemm_ws_bytes(M, N) -> int:
    """mtl_gemm_ws_bytes: workspace that lets mtl_gemm slice the tiles of its last, partial wave."""
    out = ctypes.c_size_t(0)
    _check(lib().mtl_gemm_ws_bytes(M, N, ctypes.byref(out)), "mtl_gemm_ws_bytes")
    return out.value


def attention_ws_bytes(batch, seq, heads) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().mtl_attention_ws_bytes(batch, seq, heads, ctypes.byref(out)),
           "mtl_attention_ws_bytes")
    return out.value


def _dt(dtype):
    return {"f32": F32, "bf16": BF16, F32: F32, BF16: BF16}[dtype]


def attention_mask_bytes(dtype, batch, seq, heads, p_attn) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().mtl_attention_mask_bytes(_dt(dtype), batch, seq, heads, p_attn,
                                          ctypes.byref(out)), "mtl_attention_mask_bytes")
    return out.value


def attention_fwd(dtype, batch, seq, heads, d, qkv, ctx, lse, workspace, mask=None, p_attn=0.0,
                  seed=0, stream=None):
    """mtl_attention_fwd on torch tensors; mask: attention_mask_bytes bytes or None."""
    _check(lib().mtl_attention_fwd(_dt(dtype), batch, seq, heads, d, _ptr(qkv), _ptr(ctx),
                                   _ptr(lse), _ptr(mask), p_attn, seed, _ptr(workspace),
                                   workspace.numel() * workspace.element_size(), _stream(stream)),
           "mtl_attention_fwd")


def attention_bwd(dtype, batch, seq, heads, d, qkv, ctx, lse, dctx, dqkv, workspace, mask=None,
                  p_attn=0.0, seed=0, stream=None):
    """mtl_attention_bwd on torch tensors (mask: the forward's keep bits)."""
    _check(lib().mtl_attention_bwd(_dt(dtype), batch, seq, heads, d, _ptr(qkv), _ptr(ctx),
                                   _ptr(lse), _ptr(dctx), _ptr(mask), _ptr(dqkv), p_attn, seed,
                                   _ptr(workspace), workspace.numel() * workspace.element_size(),
                                   _stream(stream)),
           "mtl_attention_bwd")


def infer_sizes(desc: LayerDesc, max_seq: int):
    """(kv_cache_bytes, prefill_workspace_bytes, decode_workspace_bytes)."""
    kv, pw, dw = ctypes.c_size_t(0), ctypes.c_size_t(0), ctypes.c_size_t(0)
    _check(lib().mtl_infer_sizes(ctypes.byref(desc), max_seq, ctypes.byref(kv), ctypes.byref(pw),
                                 ctypes.byref(dw)), "mtl_infer_sizes")
    return kv.value, pw.value, dw.value


def layer_prefill(desc, weights: dict, x, y, kv_cache, max_seq, cache_len, workspace,
                  stream=None):
    """mtl_layer_prefill on torch tensors (cache_len: int32 device tensor [batch])."""
    wt = _weights(weights)
    _check(lib().mtl_layer_prefill(ctypes.byref(desc), ctypes.byref(wt), _ptr(x), _ptr(y),
                                   _ptr(kv_cache), max_seq, _ptr(cache_len), _ptr(workspace),
                                   workspace.numel() * workspace.element_size(), _stream(stream)),
           "mtl_layer_prefill")


def layer_decode(desc, weights: dict, x_tok, y_tok, kv_cache, max_seq, cache_len, workspace,
                 stream=None):
    """mtl_layer_decode on torch tensors: one token per sequence, advances cache_len."""
    wt = _weights(weights)
    _check(lib().mtl_layer_decode(ctypes.byref(desc), ctypes.byref(wt), _ptr(x_tok), _ptr(y_tok),
                                  _ptr(kv_cache), max_seq, _ptr(cache_len), _ptr(workspace),
                                  workspace.numel() * workspace.element_size(), _stream(stream)),
           "mtl_layer_decode")


def kv_views(desc: LayerDesc, kv_cache, max_seq):
    """(K, V) views [batch][heads][max_seq][d] of a KV-cache buffer."""
    dt = torch_dtype(desc)
    esz = 2 if desc.dtype == BF16 else 4
    d = desc.h // desc.heads
    cnt = desc.batch * desc.heads * max_seq * d
    half = kv_cache.numel() // 2
    k = kv_cache[:cnt * esz].view(dt).view(desc.batch, desc.heads, max_seq, d)
    v = kv_cache[half:half + cnt * esz].view(dt).view(desc.batch, desc.heads, max_seq, d)
    return k, v


FP8_FORMATS = {"e4m3": 0, "e5m2": 1}


def fp8_quantize(src_dtype, x, rows, cols, ld, fmt, q, ldq, scale, workspace, qT=None, ldqT=0,
                 stream=None):
    """mtl_fp8_quantize on torch tensors (q / qT: uint8 device tensors or None,
    scale: float32 [1])."""
    _check(lib().mtl_fp8_quantize(_dt(src_dtype), _ptr(x), rows, cols, ld, FP8_FORMATS[fmt],
                                  _ptr(q), ldq, _ptr(qT), ldqT, _ptr(scale), _ptr(workspace),
                                  workspace.numel() * workspace.element_size(), _stream(stream)),
           "mtl_fp8_quantize")


def gemm_fp8(M, N, K, parts, A, lda, fmt_a, scale_a, B, ldb, fmt_b, scale_b, epi, C, ldc,
             c_f32, workspace, bias=None, R=None, ldr=0, Z=None, ldz=0, stream=None):
    """mtl_gemm_fp8 on torch tensors."""
    _check(lib().mtl_gemm_fp8(M, N, K, parts, _ptr(A), lda, FP8_FORMATS[fmt_a], _ptr(scale_a),
                              _ptr(B), ldb, FP8_FORMATS[fmt_b], _ptr(scale_b), epi, _ptr(bias),
                              _ptr(R), ldr, _ptr(Z), ldz, _ptr(C), ldc, int(c_f32),
                              _ptr(workspace), workspace.numel() * workspace.element_size(),
                              _stream(stream)),
           "mtl_gemm_fp8")


def selftest_launch_error(stream=None):
    """mtl_selftest_launch_error: a launch the runtime refuses; raises MtlError
    with status MTL_ERR_CUDA and the runtime's error text."""
    _check(lib().mtl_selftest_launch_error(_stream(stream)), "mtl_selftest_launch_error")


def selftest_wait_timeout(workspace, limit_cycles, stream=None):
    """mtl_selftest_wait_timeout: a bounded device wait that is made to run out."""
    _check(lib().mtl_selftest_wait_timeout(_ptr(workspace), limit_cycles, _stream(stream)),
           "mtl_selftest_wait_timeout")


def bias_grad_noalloc(dtype, dy, ld, rows, cols, out, stream=None):
    """mtl_bias_grad_noalloc: out[j] = sum_i dy[i*ld + j] with no workspace.

    For callers that cannot allocate device memory; its scratch is a static
    array inside the library (see include/mtl.h)."""
    import torch
    dt = {"f32": F32, "bf16": BF16, F32: F32, BF16: BF16}[dtype]
    want = torch.bfloat16 if dt == BF16 else torch.float32
    if dy.dtype != want or out.dtype != torch.float32:
        raise MtlError(1, "mtl_bias_grad_noalloc", "dy must match dtype and out must be float32")
    if not (dy.is_cuda and out.is_cuda and out.is_contiguous()):
        raise MtlError(1, "mtl_bias_grad_noalloc", "dy and out must be contiguous device tensors")
    if rows < 0 or cols <= 0 or ld < cols or out.numel() < cols or (
            rows > 0 and dy.numel() < (rows - 1) * ld + cols):
        raise MtlError(1, "mtl_bias_grad_noalloc", "dy or out is smaller than rows, ld and cols")
    _check(lib().mtl_bias_grad_noalloc(dt, _ptr(dy), ld, rows, cols, _ptr(out), _stream(stream)),
           "mtl_bias_grad_noalloc")


# ---------------------------------------------------------------- allocation helpers

def torch_dtype(desc: LayerDesc):
    import torch
    return torch.bfloat16 if desc.dtype == BF16 else torch.float32


def alloc_layer_buffers(desc: LayerDesc, device="cuda"):
    """Device buffers for one layer: saved, workspace (uint8) and the fp32 grads."""
    import torch
    saved_b, ws_b = layer_sizes(desc)
    h, f = desc.h, desc.ffn
    shapes = {"w_qkv": (3 * h, h), "b_qkv": (3 * h,), "w_o": (h, h), "b_o": (h,),
              "w_fc1": (f, h), "b_fc1": (f,), "w_fc2": (h, f), "b_fc2": (h,),
              "ln1_g": (h,), "ln1_b": (h,), "ln2_g": (h,), "ln2_b": (h,)}
    saved = torch.empty(max(saved_b, 16), dtype=torch.uint8, device=device)
    ws = torch.empty(max(ws_b, 256), dtype=torch.uint8, device=device)
    grads = {k: torch.empty(v, dtype=torch.float32, device=device) for k, v in shapes.items()}
    return saved, ws, grads


def workspace_views(desc: LayerDesc, workspace) -> dict:
    """Typed views of the backward's intermediates left in `workspace` after
    mtl_layer_bwd (dz, du, dx1, dctx, dqkv; see mtl_workspace_layout)."""
    import torch
    out = WorkspaceLayout()
    _check(lib().mtl_layer_workspace_layout(ctypes.byref(desc), ctypes.byref(out)),
           "mtl_layer_workspace_layout")
    n, h, f = desc.batch * desc.seq, desc.h, desc.ffn
    dt = torch_dtype(desc)
    esz = 2 if desc.dtype == BF16 else 4

    def view(off, shape, dtype, elsize):
        cnt = shape[0] * shape[1]
        return workspace[off:off + cnt * elsize].view(dtype).view(*shape)

    return {"dz": view(out.dz, (n, f), dt, esz), "du": view(out.du, (n, h), torch.float32, 4),
            "dx1": view(out.dx1, (n, h), dt, esz), "dctx": view(out.dctx, (n, h), dt, esz),
            "dqkv": view(out.dqkv, (n, 3 * h), dt, esz)}


def saved_views(desc: LayerDesc, saved):
    """Typed views of the saved activations inside `saved` (for inspection)."""
    import torch
    lay = layer_saved_layout(desc)
    n, h, f = desc.batch * desc.seq, desc.h, desc.ffn
    dt = torch_dtype(desc)
    esz = 2 if desc.dtype == BF16 else 4

    # fields are laid out in SAVED_NAMES order: a field's bytes end where the next begins
    names = SAVED_NAMES + ("total",)
    size = {k: lay[names[i + 1]] - lay[k] for i, k in enumerate(names[:-1])}

    def view(name, shape, dtype, elsize):
        cnt = 1
        for s in shape:
            cnt *= s
        off = lay[name]
        if size[name] < cnt * elsize:
            return None                       # not saved in this configuration
        return saved[off:off + cnt * elsize].view(dtype).view(*shape)

    views = {
        "mu1": view("mu1", (n,), torch.float32, 4), "rstd1": view("rstd1", (n,), torch.float32, 4),
        "u1": view("u1", (n, h), dt, esz), "qkv": view("qkv", (n, 3 * h), dt, esz),
        "ctx": view("ctx", (n, h), dt, esz),
        "lse": view("lse", (desc.batch, desc.heads, desc.seq), torch.float32, 4),
        "x1": view("x1", (n, h), dt, esz), "mu2": view("mu2", (n,), torch.float32, 4),
        "rstd2": view("rstd2", (n,), torch.float32, 4), "u2": view("u2", (n, h), dt, esz),
        "z": view("z", (n, f), dt, esz), "a": view("a", (n, f), dt, esz),
        "h1": view("h1", (n, h), dt, esz), "h2": view("h2", (n, h), dt, esz),
    }
    return {k: v for k, v in views.items() if v is not None}
