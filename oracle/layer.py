"""fp64 CPU oracle of one pre-LN GPT-2-style layer with Megatron's intra-layer split.

TEST INFRASTRUCTURE ONLY.  Nothing in the library imports this module; only the
tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
call it.  It is deliberately plain and slow: numpy float64 arrays, the matrix
product as the only library primitive, and no blocking, fusion or reordering
beyond what the definitions state.

What it follows (page "Megatron-LM: GPU-Cluster Training Parallelism"):
  * "Paper 1: BERT LayerNorm Rearrangement" -- Pre-LN: each sublayer sees
    LayerNorm(x) and its output is added back onto x.
  * "Paper 1: The f/g Conjugate Operators" -- MLP block: first GEMM split by
    columns with GeLU applied per shard, second GEMM split by rows and its
    partial outputs all-reduced (g); self-attention: Q, K, V split by columns so
    each shard owns whole heads, output projection split by rows and reduced.
    f is the identity forward and an all-reduce of input gradients backward; g
    is the reverse.  Two reductions forward, two backward.
  * "Paper 1: QKV Column-Parallel Splitting in Detail" -- the fused QKV weight
    is head-interleaved, [Q0 K0 V0 | Q1 K1 V1 | ...], so a contiguous column
    block holds H/t complete heads.
  * "Fused Transformer Kernels" -- scale-mask-softmax with a causal mask.

Readings where the pages are silent (each is also listed in the design notes):
  * GeLU is the exact x * Phi(x) form (erf), not the tanh approximation.
  * Softmax scale is 1/sqrt(d_head); masked entries (key j > query i) get
    probability exactly 0.
  * LayerNorm uses the biased variance and eps = 1e-5 inside the square root.
  * Row-parallel biases (b_o, b_fc2) are added once, after the partition sum.
  * Activations are [batch, seq, h] row-major; weights are [out, in].
  * Dropout is the identity unless a dropout dict is given (masks as in
    ``oracle/philox.py``).

The unpartitioned functions compute the layer the method reaches exactly (in
exact arithmetic) for any t.  ``layer_fwd_partitioned`` / ``layer_bwd_partitioned``
simulate t ranks literally -- per-rank GEMMs on their shards and explicit g / f
sums over rank partials in rank order, with a counter -- and serve only to pin
the split against the unpartitioned layer.

Parity pins: every function here is pinned by the CPU tests (closed forms,
invariants, special cases, finite differences and an independent autograd
cross-check); the absolute end-to-end values of a full layer are otherwise
"parity unpinned" against the pages, which print no worked numeric example.
"""

from __future__ import annotations

import math

import numpy as np
from scipy.special import erf

from . import philox

LN_EPS = 1e-5


# --------------------------------------------------------------------------
# Elementwise pieces
# --------------------------------------------------------------------------

def gelu(x):
    """GeLU(x) = x * Phi(x), Phi the standard normal CDF (exact erf form).

    The MLP's first GEMM is followed by GeLU ("Paper 1: The f/g Conjugate
    Operators", MLP block); the form is the exact one (reading: erf, not tanh).
    """
    return 0.5 * x * (1.0 + erf(x / math.sqrt(2.0)))


def gelu_grad(x):
    """d/dx GeLU(x) = Phi(x) + x * phi(x), phi the standard normal density."""
    cdf = 0.5 * (1.0 + erf(x / math.sqrt(2.0)))
    pdf = np.exp(-0.5 * x * x) / math.sqrt(2.0 * math.pi)
    return cdf + x * pdf


# --------------------------------------------------------------------------
# LayerNorm (Pre-LN: "Paper 1: BERT LayerNorm Rearrangement")
# --------------------------------------------------------------------------

def layernorm_fwd(x, gamma, beta, eps=LN_EPS):
    """Row LayerNorm of x [n, h]: returns (u, mean [n], rstd [n]).

    mean and variance are per row (biased variance); rstd = 1/sqrt(var + eps);
    u = gamma * (x - mean) * rstd + beta.
    """
    mean = x.mean(axis=1)
    centered = x - mean[:, None]
    var = (centered * centered).mean(axis=1)
    rstd = 1.0 / np.sqrt(var + eps)
    xhat = centered * rstd[:, None]
    return xhat * gamma[None, :] + beta[None, :], mean, rstd


def layernorm_bwd(du, x, mean, rstd, gamma):
    """Gradients of u = LayerNorm(x) given du [n, h].

    Returns (dx [n, h], dgamma [h], dbeta [h]).  With xhat = (x - mean) * rstd
    and g = du * gamma, the input gradient of a normalised row is
    rstd * (g - mean_j(g) - xhat * mean_j(g * xhat)).
    """
    xhat = (x - mean[:, None]) * rstd[:, None]
    g = du * gamma[None, :]
    g_mean = g.mean(axis=1, keepdims=True)
    gx_mean = (g * xhat).mean(axis=1, keepdims=True)
    dx = rstd[:, None] * (g - g_mean - xhat * gx_mean)
    dgamma = (du * xhat).sum(axis=0)
    dbeta = du.sum(axis=0)
    return dx, dgamma, dbeta


# --------------------------------------------------------------------------
# Causal self-attention of one head ("Fused Transformer Kernels": scale-mask-softmax)
# --------------------------------------------------------------------------

def causal_mask(s):
    """Boolean [s, s], True where key j > query i (excluded)."""
    return np.triu(np.ones((s, s), dtype=bool), k=1)


def attention_head_fwd(q, k, v):
    """One head: q, k, v [s, d].  Returns (o [s, d], p [s, s], lse [s]).

    S = q k^T / sqrt(d); entries with j > i are excluded (probability 0);
    P = row softmax of S; o = P v; lse = log sum_j exp(S_ij) over allowed j.
    """
    s, d = q.shape
    scores = (q @ k.T) / math.sqrt(d)
    mask = causal_mask(s)
    scores = np.where(mask, -np.inf, scores)
    row_max = scores.max(axis=1, keepdims=True)
    e = np.exp(scores - row_max)
    e[mask] = 0.0
    denom = e.sum(axis=1, keepdims=True)
    p = e / denom
    lse = row_max[:, 0] + np.log(denom[:, 0])
    return p @ v, p, lse


def attention_head_bwd(q, k, v, p, o, do, keep_scale=None):
    """Gradients of one causal head given do [s, d].  Returns (dq, dk, dv).

    dV = P^T dO; dP = dO V^T; with D_i = sum_j P_ij dP_ij (= sum_c dO_ic O_ic),
    dS = P * (dP - D); dQ = dS K / sqrt(d); dK = dS^T Q / sqrt(d).
    With attention dropout (keep_scale = keep / (1 - p), o = (P * keep_scale) V):
    dV = (P * keep_scale)^T dO, dP = (dO V^T) * keep_scale, and D still equals
    rowsum(dO * O).
    """
    d = q.shape[1]
    if keep_scale is None:
        dv = p.T @ do
        dp = do @ v.T
    else:
        dv = (p * keep_scale).T @ do
        dp = (do @ v.T) * keep_scale
    dsum = (do * o).sum(axis=1, keepdims=True)
    ds = p * (dp - dsum)
    dq = ds @ k / math.sqrt(d)
    dk = ds.T @ q / math.sqrt(d)
    return dq, dk, dv


def split_qkv_columns(qkv_row_block, n_heads, d):
    """Columns of a head-interleaved block -> (q, k, v) each [..., n_heads, d].

    Head-interleaved order ("Paper 1: QKV Column-Parallel Splitting in
    Detail"): column = head * 3d + {0: Q, 1: K, 2: V} * d + channel.
    """
    shp = qkv_row_block.shape[:-1]
    blk = qkv_row_block.reshape(*shp, n_heads, 3, d)
    return blk[..., 0, :], blk[..., 1, :], blk[..., 2, :]


def attention_keep_scale(b, head, heads_total, seq, drop):
    """keep / (1 - p) of the attention probabilities of one head, or None."""
    if not drop or drop.get("p_attn", 0.0) == 0.0:
        return None
    p = drop["p_attn"]
    keep = philox.attention_mask(b, head, heads_total, seq, drop.get("seed", 0), p)
    return keep / (1.0 - p)


def multihead_fwd(qkv, batch, seq, n_heads, d, drop=None, head0=0, heads_total=None):
    """Attention over all heads of a head-interleaved qkv [n, 3 * n_heads * d].

    Returns ctx [n, n_heads * d] (column = head * d + channel), lse
    [batch, n_heads, seq] and the probabilities for the backward.  With
    attention dropout the output is (P * keep / (1 - p)) V; lse and the
    returned probabilities are those of the undropped softmax.  head0 /
    heads_total place these heads among the layer's for the dropout mask.
    """
    heads_total = n_heads if heads_total is None else heads_total
    q, k, v = split_qkv_columns(qkv.reshape(batch, seq, -1), n_heads, d)
    ctx = np.empty((batch, seq, n_heads, d))
    lse = np.empty((batch, n_heads, seq))
    probs = np.empty((batch, n_heads, seq, seq))
    for b in range(batch):
        for hd in range(n_heads):
            o, p, l = attention_head_fwd(q[b, :, hd], k[b, :, hd], v[b, :, hd])
            ks = attention_keep_scale(b, head0 + hd, heads_total, seq, drop)
            if ks is not None:
                o = (p * ks) @ v[b, :, hd]
            ctx[b, :, hd] = o
            lse[b, hd] = l
            probs[b, hd] = p
    return ctx.reshape(batch * seq, n_heads * d), lse, probs


def multihead_bwd(qkv, ctx, probs, dctx, batch, seq, n_heads, d, drop=None, head0=0,
                  heads_total=None):
    """Gradient of multihead_fwd: dctx [n, n_heads*d] -> dqkv [n, 3*n_heads*d]."""
    heads_total = n_heads if heads_total is None else heads_total
    q, k, v = split_qkv_columns(qkv.reshape(batch, seq, -1), n_heads, d)
    o = ctx.reshape(batch, seq, n_heads, d)
    do = dctx.reshape(batch, seq, n_heads, d)
    dqkv = np.empty((batch, seq, n_heads, 3, d))
    for b in range(batch):
        for hd in range(n_heads):
            ks = attention_keep_scale(b, head0 + hd, heads_total, seq, drop)
            dq, dk, dv = attention_head_bwd(q[b, :, hd], k[b, :, hd], v[b, :, hd],
                                            probs[b, hd], o[b, :, hd], do[b, :, hd], ks)
            dqkv[b, :, hd, 0] = dq
            dqkv[b, :, hd, 1] = dk
            dqkv[b, :, hd, 2] = dv
    return dqkv.reshape(batch * seq, 3 * n_heads * d)


# --------------------------------------------------------------------------
# The whole layer, unpartitioned
# --------------------------------------------------------------------------

def _f64(a):
    return np.asarray(a, dtype=np.float64)


def hidden_keep_scale(n, h, drop, site):
    """keep / (1 - p) of a hidden-state dropout site, [n, h], or 1.0."""
    if not drop or drop.get("p_hidden", 0.0) == 0.0:
        return 1.0
    p = drop["p_hidden"]
    return philox.hidden_mask(n, h, drop.get("seed", 0), site, p) / (1.0 - p)


def _lin(u, w, b, fp8, epi=1, R=None):
    """u w^T + b (+ R): in fp64, or as an FP8 GEMM of per-tensor E4M3 operands."""
    if not fp8:
        out = u @ w.T + b
        return out if R is None else out + R
    from . import fp8 as _fp8
    return _fp8.gemm(u, w, "e4m3", "e4m3", epi=epi, bias=b, R=R)[0]


def layer_fwd(params, x, heads, eps=LN_EPS, dropout=None, fp8=False):
    """Pre-LN GPT layer forward.  x [batch, seq, h].  Returns (y, cache).

    u1 = LN1(x); qkv = u1 W_qkv^T + b_qkv; ctx = causal multi-head attention;
    x1 = x + ctx W_o^T + b_o; u2 = LN2(x1); z = u2 W_fc1^T + b_fc1; a = GeLU(z);
    y = x1 + a W_fc2^T + b_fc2.
    dropout = dict(p_attn, p_hidden, seed) (optional): attention dropout on the
    softmax probabilities, and the fused bias + dropout + residual ("Fused
    Transformer Kernels") after the out-projection and after fc2:
    x1 = x + drop(ctx W_o^T + b_o), y = x1 + drop(a W_fc2^T + b_fc2); masks as
    in oracle/philox.py.
    fp8=True (or 1): the four GEMMs take per-tensor E4M3 operands (activation
    and weight quantized as in oracle/fp8.py); LayerNorm, attention, GeLU,
    biases and residuals stay in high precision.  fp8=2 ("hybrid"): the same
    forward, and layer_bwd's eight GEMMs take an E5M2 gradient and an E4M3
    activation or weight.
    """
    if fp8 and dropout:
        raise ValueError("FP8 forward is defined without dropout")
    p = {k: _f64(v) for k, v in params.items()}
    x = _f64(x)
    batch, seq, h = x.shape
    d = h // heads
    n = batch * seq
    xf = x.reshape(n, h)
    u1, mu1, rstd1 = layernorm_fwd(xf, p["ln1_g"], p["ln1_b"], eps)
    qkv = _lin(u1, p["w_qkv"], p["b_qkv"], fp8)
    ctx, lse, probs = multihead_fwd(qkv, batch, seq, heads, d, dropout)
    so = hidden_keep_scale(n, h, dropout, philox.SITE_OUT)
    s2 = hidden_keep_scale(n, h, dropout, philox.SITE_FC2)
    x1 = xf + _lin(ctx, p["w_o"], p["b_o"], fp8) * so
    u2, mu2, rstd2 = layernorm_fwd(x1, p["ln2_g"], p["ln2_b"], eps)
    z = _lin(u2, p["w_fc1"], p["b_fc1"], fp8)
    a = gelu(z)
    y = x1 + _lin(a, p["w_fc2"], p["b_fc2"], fp8) * s2
    cache = dict(x=xf, u1=u1, mu1=mu1, rstd1=rstd1, qkv=qkv, ctx=ctx, lse=lse,
                 probs=probs, x1=x1, u2=u2, mu2=mu2, rstd2=rstd2, z=z, a=a,
                 batch=batch, seq=seq, heads=heads, dropout=dropout, so=so, s2=s2,
                 fp8=int(fp8))
    return y.reshape(batch, seq, h), cache


def layer_bwd(params, cache, dy):
    """Analytic backward of layer_fwd.  dy [batch, seq, h].

    Returns (dx [batch, seq, h], grads) with grads keyed like params.
    """
    p = {k: _f64(v) for k, v in params.items()}
    c = cache
    batch, seq, heads = c["batch"], c["seq"], c["heads"]
    n, h = c["x"].shape
    d = h // heads
    dy = _f64(dy).reshape(n, h)
    drop = c.get("dropout")
    hybrid = c.get("fp8", 0) == 2

    def mm(A, Bt):
        """A Bt^T: in fp64, or (hybrid FP8) with A quantized to E5M2 (the
        gradient side) and Bt to E4M3, each per tensor."""
        if not hybrid:
            return A @ Bt.T
        from . import fp8 as _fp8
        return _fp8.gemm(A, Bt, "e5m2", "e4m3")[0]

    g = {}
    # MLP block: y = x1 + drop(GeLU(u2 W1^T + b1) W2^T + b2)
    g2 = dy * c.get("s2", 1.0)
    g["w_fc2"] = mm(g2.T, c["a"].T)
    g["b_fc2"] = g2.sum(axis=0)
    da = mm(g2, p["w_fc2"].T)
    dz = da * gelu_grad(c["z"])
    g["w_fc1"] = mm(dz.T, c["u2"].T)
    g["b_fc1"] = dz.sum(axis=0)
    du2 = mm(dz, p["w_fc1"].T)
    dx1_ln, g["ln2_g"], g["ln2_b"] = layernorm_bwd(du2, c["x1"], c["mu2"], c["rstd2"],
                                                   p["ln2_g"])
    dx1 = dy + dx1_ln
    # attention block: x1 = x + drop(Attn(u1 W_qkv^T + b_qkv) W_o^T + b_o)
    go = dx1 * c.get("so", 1.0)
    g["w_o"] = mm(go.T, c["ctx"].T)
    g["b_o"] = go.sum(axis=0)
    dctx = mm(go, p["w_o"].T)
    dqkv = multihead_bwd(c["qkv"], c["ctx"], c["probs"], dctx, batch, seq, heads, d, drop)
    g["w_qkv"] = mm(dqkv.T, c["u1"].T)
    g["b_qkv"] = dqkv.sum(axis=0)
    du1 = mm(dqkv, p["w_qkv"].T)
    dx_ln, g["ln1_g"], g["ln1_b"] = layernorm_bwd(du1, c["x"], c["mu1"], c["rstd1"],
                                                  p["ln1_g"])
    dx = dx1 + dx_ln
    inter = dict(da=da, dz=dz, du2=du2, dx1=dx1, dctx=dctx, dqkv=dqkv, du1=du1)
    return dx.reshape(batch, seq, h), g, inter


# --------------------------------------------------------------------------
# Post-LN variant (original BERT)
# --------------------------------------------------------------------------

def layer_fwd_post_ln(params, x, heads, eps=LN_EPS):
    """Post-LN layer ("Paper 1: BERT LayerNorm Rearrangement", the original BERT
    arrangement the Pre-LN layer replaces): LayerNorm after each residual add,
        h1 = x + Attn(x) W_o^T + b_o,    x1 = LN1(h1),
        h2 = x1 + GeLU(x1 W_fc1^T + b_fc1) W_fc2^T + b_fc2,    y = LN2(h2),
    with Attn the same causal multi-head attention over qkv = x W_qkv^T + b_qkv.
    Returns (y, cache)."""
    p = {k: _f64(v) for k, v in params.items()}
    x = _f64(x)
    batch, seq, h = x.shape
    d = h // heads
    xf = x.reshape(batch * seq, h)
    qkv = xf @ p["w_qkv"].T + p["b_qkv"]
    ctx, lse, probs = multihead_fwd(qkv, batch, seq, heads, d)
    h1 = xf + ctx @ p["w_o"].T + p["b_o"]
    x1, mu1, rstd1 = layernorm_fwd(h1, p["ln1_g"], p["ln1_b"], eps)
    z = x1 @ p["w_fc1"].T + p["b_fc1"]
    a = gelu(z)
    h2 = x1 + a @ p["w_fc2"].T + p["b_fc2"]
    y, mu2, rstd2 = layernorm_fwd(h2, p["ln2_g"], p["ln2_b"], eps)
    cache = dict(x=xf, qkv=qkv, ctx=ctx, lse=lse, probs=probs, h1=h1, mu1=mu1, rstd1=rstd1,
                 x1=x1, z=z, a=a, h2=h2, mu2=mu2, rstd2=rstd2, batch=batch, seq=seq,
                 heads=heads, post_ln=True)
    return y.reshape(batch, seq, h), cache


def layer_bwd_post_ln(params, cache, dy):
    """Analytic backward of layer_fwd_post_ln.  Returns (dx, grads, inter)."""
    p = {k: _f64(v) for k, v in params.items()}
    c = cache
    batch, seq, heads = c["batch"], c["seq"], c["heads"]
    n, h = c["x"].shape
    d = h // heads
    dy = _f64(dy).reshape(n, h)
    g = {}
    dh2, g["ln2_g"], g["ln2_b"] = layernorm_bwd(dy, c["h2"], c["mu2"], c["rstd2"], p["ln2_g"])
    g["w_fc2"] = dh2.T @ c["a"]
    g["b_fc2"] = dh2.sum(axis=0)
    dz = (dh2 @ p["w_fc2"]) * gelu_grad(c["z"])
    g["w_fc1"] = dz.T @ c["x1"]
    g["b_fc1"] = dz.sum(axis=0)
    dx1 = dh2 + dz @ p["w_fc1"]
    dh1, g["ln1_g"], g["ln1_b"] = layernorm_bwd(dx1, c["h1"], c["mu1"], c["rstd1"], p["ln1_g"])
    g["w_o"] = dh1.T @ c["ctx"]
    g["b_o"] = dh1.sum(axis=0)
    dctx = dh1 @ p["w_o"]
    dqkv = multihead_bwd(c["qkv"], c["ctx"], c["probs"], dctx, batch, seq, heads, d)
    g["w_qkv"] = dqkv.T @ c["x"]
    g["b_qkv"] = dqkv.sum(axis=0)
    dx = dh1 + dqkv @ p["w_qkv"]
    inter = dict(dh2=dh2, dz=dz, dx1=dx1, dh1=dh1, dctx=dctx, dqkv=dqkv)
    return dx.reshape(batch, seq, h), g, inter


def layer_fwd_post_ln_partitioned(params, x, heads, t, counter, eps=LN_EPS):
    """layer_fwd_post_ln over t simulated ranks: QKV / fc1 split by columns, the
    out-proj / fc2 partials summed in rank order (g) before the residual add and
    the LayerNorm, which stay outside the partitions."""
    p = {k: _f64(v) for k, v in params.items()}
    x = _f64(x)
    batch, seq, h = x.shape
    ffn = p["w_fc1"].shape[0]
    d = h // heads
    xf = x.reshape(batch * seq, h)
    ranks = shard_ranges(h, ffn, heads, t)
    parts = []
    for r, rk in enumerate(ranks):
        qkv_r = xf @ p["w_qkv"][rk["qkv"]].T + p["b_qkv"][rk["qkv"]]
        ctx_r, _, _ = multihead_fwd(qkv_r, batch, seq, rk["heads"], d)
        parts.append(ctx_r @ p["w_o"][:, rk["ctx"]].T)
    h1 = xf + g_allreduce(parts, counter) + p["b_o"]
    x1, _, _ = layernorm_fwd(h1, p["ln1_g"], p["ln1_b"], eps)
    parts = [gelu(x1 @ p["w_fc1"][rk["ffn"]].T + p["b_fc1"][rk["ffn"]]) @ p["w_fc2"][:, rk["ffn"]].T
             for rk in ranks]
    h2 = x1 + g_allreduce(parts, counter) + p["b_fc2"]
    y, _, _ = layernorm_fwd(h2, p["ln2_g"], p["ln2_b"], eps)
    return y.reshape(batch, seq, h)


# --------------------------------------------------------------------------
# The whole layer, partitioned over t simulated ranks
# --------------------------------------------------------------------------

class ReductionCounter:
    """Counts the g (forward) and f (backward) all-reduces a pass performs."""

    def __init__(self):
        self.g = 0
        self.f = 0


def g_allreduce(partials, counter):
    """g forward: the sum of the ranks' partial outputs, in rank order."""
    counter.g += 1
    total = np.zeros_like(partials[0])
    for part in partials:
        total = total + part
    return total


def f_allreduce(partials, counter):
    """f backward: the sum of the ranks' partial input gradients, in rank order."""
    counter.f += 1
    total = np.zeros_like(partials[0])
    for part in partials:
        total = total + part
    return total


def shard_ranges(h, ffn, heads, t):
    """Per-rank index ranges of the column / row splits for t ranks.

    qkv: rank r owns heads [r*H/t, (r+1)*H/t), i.e. the contiguous rows
    [r*3h/t, (r+1)*3h/t) of the head-interleaved W_qkv; ctx / W_o columns
    [r*h/t, (r+1)*h/t); fc1 rows and fc2 columns [r*ffn/t, (r+1)*ffn/t).
    """
    if heads % t or ffn % t:
        raise ValueError("t must divide heads and ffn")
    out = []
    for r in range(t):
        out.append(dict(
            qkv=slice(r * 3 * h // t, (r + 1) * 3 * h // t),
            ctx=slice(r * h // t, (r + 1) * h // t),
            ffn=slice(r * ffn // t, (r + 1) * ffn // t),
            heads=heads // t))
    return out


def layer_fwd_partitioned(params, x, heads, t, counter, eps=LN_EPS, dropout=None):
    """Forward with the layer split over t ranks; returns (y, cache).

    Each rank holds the replicated input (f forward = identity), computes its
    column shard of qkv (its H/t heads), attends locally, and multiplies its
    ctx shard by its row shard of W_o; g sums the t partials, then b_o is added
    once.  The MLP block does the same with the fc1 column shard (GeLU applied
    per shard) and the fc2 row shard.
    """
    p = {k: _f64(v) for k, v in params.items()}
    x = _f64(x)
    batch, seq, h = x.shape
    ffn = p["w_fc1"].shape[0]
    d = h // heads
    xf = x.reshape(batch * seq, h)
    n = batch * seq
    ranks = shard_ranges(h, ffn, heads, t)
    so = hidden_keep_scale(n, h, dropout, philox.SITE_OUT)
    s2 = hidden_keep_scale(n, h, dropout, philox.SITE_FC2)
    u1, mu1, rstd1 = layernorm_fwd(xf, p["ln1_g"], p["ln1_b"], eps)
    parts, rank_cache = [], []
    for r, rk in enumerate(ranks):
        qkv_r = u1 @ p["w_qkv"][rk["qkv"]].T + p["b_qkv"][rk["qkv"]]
        ctx_r, lse_r, probs_r = multihead_fwd(qkv_r, batch, seq, rk["heads"], d, dropout,
                                              r * rk["heads"], heads)
        parts.append(ctx_r @ p["w_o"][:, rk["ctx"]].T)
        rank_cache.append(dict(qkv=qkv_r, ctx=ctx_r, lse=lse_r, probs=probs_r))
    x1 = xf + (g_allreduce(parts, counter) + p["b_o"]) * so
    u2, mu2, rstd2 = layernorm_fwd(x1, p["ln2_g"], p["ln2_b"], eps)
    parts = []
    for rk, rc in zip(ranks, rank_cache):
        z_r = u2 @ p["w_fc1"][rk["ffn"]].T + p["b_fc1"][rk["ffn"]]
        a_r = gelu(z_r)
        parts.append(a_r @ p["w_fc2"][:, rk["ffn"]].T)
        rc.update(z=z_r, a=a_r)
    y = x1 + (g_allreduce(parts, counter) + p["b_fc2"]) * s2
    cache = dict(x=xf, u1=u1, mu1=mu1, rstd1=rstd1, x1=x1, u2=u2, mu2=mu2,
                 rstd2=rstd2, ranks=ranks, rank_cache=rank_cache, batch=batch,
                 seq=seq, heads=heads, t=t, dropout=dropout, so=so, s2=s2)
    return y.reshape(batch, seq, h), cache


def layer_bwd_partitioned(params, cache, dy, counter):
    """Backward over t simulated ranks; returns (dx, grads).

    g backward is the identity (each rank sees the whole dy / dx1); each rank
    forms its shard's weight gradients and a partial input gradient, and f sums
    those partials in rank order before each LayerNorm backward.
    """
    p = {k: _f64(v) for k, v in params.items()}
    c = cache
    batch, seq, heads = c["batch"], c["seq"], c["heads"]
    n, h = c["x"].shape
    ffn = p["w_fc1"].shape[0]
    d = h // heads
    dy = _f64(dy).reshape(n, h)
    drop = c.get("dropout")
    g2 = dy * c.get("s2", 1.0)
    g = {k: np.zeros_like(v) for k, v in p.items()}
    g["b_fc2"] = g2.sum(axis=0)
    parts = []
    for rk, rc in zip(c["ranks"], c["rank_cache"]):
        s = rk["ffn"]
        g["w_fc2"][:, s] = g2.T @ rc["a"]
        dz_r = (g2 @ p["w_fc2"][:, s]) * gelu_grad(rc["z"])
        g["w_fc1"][s] = dz_r.T @ c["u2"]
        g["b_fc1"][s] = dz_r.sum(axis=0)
        parts.append(dz_r @ p["w_fc1"][s])
    du2 = f_allreduce(parts, counter)
    dx1_ln, g["ln2_g"], g["ln2_b"] = layernorm_bwd(du2, c["x1"], c["mu2"], c["rstd2"],
                                                   p["ln2_g"])
    dx1 = dy + dx1_ln
    go = dx1 * c.get("so", 1.0)
    g["b_o"] = go.sum(axis=0)
    parts = []
    for r, (rk, rc) in enumerate(zip(c["ranks"], c["rank_cache"])):
        sc, sq = rk["ctx"], rk["qkv"]
        g["w_o"][:, sc] = go.T @ rc["ctx"]
        dctx_r = go @ p["w_o"][:, sc]
        dqkv_r = multihead_bwd(rc["qkv"], rc["ctx"], rc["probs"], dctx_r, batch, seq,
                               rk["heads"], d, drop, r * rk["heads"], heads)
        g["w_qkv"][sq] = dqkv_r.T @ c["u1"]
        g["b_qkv"][sq] = dqkv_r.sum(axis=0)
        parts.append(dqkv_r @ p["w_qkv"][sq])
    du1 = f_allreduce(parts, counter)
    dx_ln, g["ln1_g"], g["ln1_b"] = layernorm_bwd(du1, c["x"], c["mu1"], c["rstd1"],
                                                  p["ln1_g"])
    dx = dx1 + dx_ln
    return dx.reshape(batch, seq, h), g


# --------------------------------------------------------------------------
# Counting
# --------------------------------------------------------------------------

def layer_flops(h, heads, seq, batch, ffn=None):
    """Algorithmic fwd+bwd flops of one layer (causal attention, no recompute).

    GEMMs: forward 2n(3h*h + h*h + 2*ffn*h), backward twice that.  Attention:
    forward 2 * 2 * batch * heads * d * seq(seq+1)/2 (QK^T and PV over the
    unmasked triangle), backward twice that.
    """
    ffn = 4 * h if ffn is None else ffn
    n = batch * seq
    gemm_fwd = 2 * n * (3 * h * h + h * h + 2 * ffn * h)
    attn_fwd = 2 * batch * seq * (seq + 1) * h
    return 3 * (gemm_fwd + attn_fwd)


# --------------------------------------------------------------------------
# One partitioned GEMM with its fused epilogue (the kernels' unit of work)
# --------------------------------------------------------------------------

def gemm_partitioned(A, B, parts, epi=0, bias=None, R=None, Z=None):
    """C = epi( sum_{p < parts} A[:, K_p] B[:, K_p]^T ), K split into equal parts.

    A [M, K], B [N, K].  The partial products of the parts are summed in part
    order: a row-parallel GEMM's partial outputs and their g / f reduction
    ("Paper 1: The f/g Conjugate Operators").  Epilogues (the fused kernels of
    "Fused Transformer Kernels"):
      0: C = acc            1: C = acc + bias            2: C = acc + bias + R
      3: Z = acc + bias, C = GeLU(Z)                     4: C = acc * GeLU'(Z)
    Returns C, or (C, Z) for epilogue 3.
    """
    A = _f64(A)
    B = _f64(B)
    K = A.shape[1]
    if parts < 1 or K % parts:
        raise ValueError("parts must divide K")
    kp = K // parts
    acc = np.zeros((A.shape[0], B.shape[0]))
    for p in range(parts):
        acc = acc + A[:, p * kp:(p + 1) * kp] @ B[:, p * kp:(p + 1) * kp].T
    if epi == 0:
        return acc
    if epi == 1:
        return acc + _f64(bias)[None, :]
    if epi == 2:
        return acc + _f64(bias)[None, :] + _f64(R)
    if epi == 3:
        z = acc + _f64(bias)[None, :]
        return gelu(z), z
    if epi == 4:
        return acc * gelu_grad(_f64(Z))
    raise ValueError(epi)
