"""Test helpers: run one layer through the C ABI and through the oracle.

Both sides are fed the same seeded inputs from `synthetic`; nothing computed on
the GPU ever reaches the oracle.
"""
from __future__ import annotations

import numpy as np

import oracle
import synthetic

# Tolerances on max|gpu - ref| / max|ref| per tensor.
TOL = {
    "f32": {"fwd": 1e-5, "bwd": 1e-5},
    "bf16": {"fwd": 1.5e-2, "bwd": 3e-2},
}


def rel_err(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    m = float(np.max(np.abs(b))) if b.size else 0.0
    d = float(np.max(np.abs(a - b))) if b.size else 0.0
    return d / m if m > 0 else d


def to_device(arr, dtype):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(arr, dtype=np.float32))
    return t.to(dtype=torch.bfloat16 if dtype == "bf16" else torch.float32).cuda()


def to_np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def f32(v):
    """v rounded to float32: the dropout probabilities cross the C ABI as float."""
    return float(np.float32(v))


def run_gpu(shape, x, p, dy, t, runs=1, want_saved=True, drop=None, fp8=0, post_ln=0,
            recompute=0):
    """Forward + backward through the C ABI.  Returns a dict of float64 arrays.

    drop: optional dict(p_attn, p_hidden, seed) of float32-exact probabilities."""
    import torch
    from tensor_model_transformer_gb300 import mtl
    b = x.shape[0]
    drop = drop or {}
    desc = mtl.layer_desc(shape.h, shape.heads, shape.seq, b, shape.ffn, t, shape.dtype,
                          p_attn=drop.get("p_attn", 0.0), p_hidden=drop.get("p_hidden", 0.0),
                          seed=drop.get("seed", 0), fp8=fp8, post_ln=post_ln,
                          recompute=recompute)
    dev_p = {k: to_device(v, shape.dtype) for k, v in p.items()}
    xd = to_device(x, shape.dtype)
    dyd = to_device(dy, shape.dtype)
    saved, ws, grads = mtl.alloc_layer_buffers(desc)
    y = torch.empty_like(xd)
    dx = torch.empty_like(xd)
    outs = []
    for _ in range(runs):
        mtl.layer_fwd(desc, dev_p, xd, y, saved, ws)
        mtl.layer_check(ws)
        mtl.layer_bwd(desc, dev_p, xd, saved, dyd, dx, grads, ws)
        mtl.layer_check(ws)
        torch.cuda.synchronize()
        out = {"y": to_np(y), "dx": to_np(dx)}
        out.update({"d_" + k: to_np(v) for k, v in grads.items()})
        if want_saved:
            sv = mtl.saved_views(desc, saved)
            out.update({"s_" + k: to_np(v) for k, v in sv.items()})
        outs.append(out)
    return outs if runs > 1 else outs[0]


def run_oracle(shape, x, p, dy, drop=None, fp8=False):
    """The oracle's outputs and intermediates, keyed like run_gpu."""
    y, cache = oracle.layer_fwd(p, x, shape.heads, dropout=drop, fp8=fp8)
    dx, g, _ = oracle.layer_bwd(p, cache, dy)
    out = {"y": y, "dx": dx}
    out.update({"d_" + k: v for k, v in g.items()})
    for k in ("u1", "qkv", "ctx", "lse", "x1", "u2", "z", "a", "mu1", "rstd1", "mu2", "rstd2"):
        out["s_" + k] = cache[k]
    return out


def run_oracle_post_ln(shape, x, p, dy):
    """The oracle's Post-LN layer, keyed like run_gpu (saved x1 = LN1 output)."""
    y, cache = oracle.layer_fwd_post_ln(p, x, shape.heads)
    dx, g, _ = oracle.layer_bwd_post_ln(p, cache, dy)
    out = {"y": y, "dx": dx}
    out.update({"d_" + k: v for k, v in g.items()})
    for k in ("qkv", "ctx", "lse", "x1", "z", "a", "h1", "h2", "mu1", "rstd1", "mu2", "rstd2"):
        out["s_" + k] = cache[k]
    return out


# Tensors whose axis `QKV_AXIS[key]` is the head-interleaved 3h axis of the fused
# QKV (per head: d rows of Q, then K, then V).
QKV_AXIS = {"s_qkv": 1, "d_w_qkv": 0, "d_b_qkv": 0, "dqkv": 1}


def qkv_blocks(a, axis, heads):
    """The (head, part) blocks of a head-interleaved 3h axis: {(head, "qkv"[i]): block}."""
    a = np.asarray(a)
    d = a.shape[axis] // (3 * heads)
    out = {}
    for hd in range(heads):
        for i, part in enumerate("qkv"):
            idx = [slice(None)] * a.ndim
            idx[axis] = slice(hd * 3 * d + i * d, hd * 3 * d + (i + 1) * d)
            out[(hd, part)] = a[tuple(idx)]
    return out


def rel_err_qkv(g, r, axis, heads, zero_k_sum=False):
    """max over heads and Q/K/V blocks of each block's rel_err, so a small block
    (dQ and dK next to a large dV) is judged against its own scale.

    zero_k_sum: r is a sum over key positions of dK (the K part of the QKV bias
    gradient), which is exactly 0 -- softmax does not change when a constant is
    added to every key of a query, so each row of dS sums to zero -- and the
    reference holds only rounding noise; such a block is judged against the
    largest Q/V block of the same tensor instead."""
    gb, rb = qkv_blocks(g, axis, heads), qkv_blocks(r, axis, heads)
    scale_qv = max((float(np.max(np.abs(v))) for k, v in rb.items() if k[1] != "k"), default=0.0)
    worst = 0.0
    for k in rb:
        if zero_k_sum and k[1] == "k":
            e = float(np.max(np.abs(gb[k] - rb[k]))) / scale_qv if scale_qv > 0 else 0.0
        else:
            e = rel_err(gb[k], rb[k])
        worst = max(worst, e)
    return worst


def compare(gpu, ref, dtype, keys=None, heads=None, per_block=True):
    """{key: rel_err} for the outputs present in both.  The fused-QKV tensors
    (s_qkv, d_w_qkv, d_b_qkv, dqkv) are judged per head and per Q/K/V block
    (heads from the argument or from the reference's lse) unless per_block is
    False."""
    keys = keys or [k for k in ref if k in gpu]
    if heads is None and "s_lse" in ref and per_block:
        heads = ref["s_lse"].shape[1]
    res = {}
    for k in keys:
        g = gpu[k].reshape(ref[k].shape)
        if k in QKV_AXIS and heads:
            res[k] = rel_err_qkv(g, ref[k], QKV_AXIS[k], heads, zero_k_sum=(k == "d_b_qkv"))
        else:
            res[k] = rel_err(g, ref[k])
    return res


def tolerance(key, dtype):
    tol = TOL[dtype]
    if key == "y" or key.startswith("s_"):
        return tol["fwd"]
    return tol["bwd"]


def make(shape, seed=0, affine=False, batch=None):
    return synthetic.make_layer(shape, seed=seed, affine=affine, batch=batch)
