"""fp64 oracle of inference with a head-sharded KV cache: prefill and decode.

TEST INFRASTRUCTURE ONLY (see ``oracle/layer.py``): only the tests,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` use it.

What it follows (page "Megatron-LM: GPU-Cluster Training Parallelism", section
"Paper 1: QKV Column-Parallel Splitting in Detail", its inference-time
behaviour): the column split is the same as in training; prefill runs the
prompt through the layer; at decode time each partition appends the new
token's K and V of its own heads to its local KV-cache shard, so the cache
memory divides evenly by t, while the out-projection and fc2 outputs are still
reduced once per token (two reductions per layer and token).

Readings where the page is silent:
  * The KV cache of one layer holds K and V as [batch][heads][max_seq][d];
    partition p's shard is heads [p*H/t, (p+1)*H/t) of every batch row.
  * Each sequence b has a cache length L_b.  A decode step places the new
    token at position L_b, writes its K and V there, lets it attend causally to
    keys 0..L_b, and leaves L_b + 1.  Prefill of a prompt of length S writes
    positions 0..S-1 and sets L_b = S.
  * By definition the decode output of a token equals the full causal forward
    of its sequence (prompt and every decoded token so far) at that token's
    position; the CPU tests check exactly that, against ``layer_fwd``.
  * No dropout at inference.
"""

from __future__ import annotations

import numpy as np

from .layer import LN_EPS, g_allreduce, gelu, layer_fwd, layernorm_fwd, shard_ranges


def kv_cache(batch, heads, max_seq, d):
    """An empty cache: K, V [batch][heads][max_seq][d] and lengths [batch]."""
    return {"k": np.zeros((batch, heads, max_seq, d)), "v": np.zeros((batch, heads, max_seq, d)),
            "len": np.zeros(batch, dtype=np.int64)}


def _p64(params):
    return {k: np.asarray(v, dtype=np.float64) for k, v in params.items()}


def prefill(params, x, heads, cache, eps=LN_EPS):
    """The layer over prompts x [batch][S][h]; K and V of every prompt token go
    to cache positions 0..S-1.  Returns y [batch][S][h]."""
    batch, seq, h = x.shape
    d = h // heads
    if seq > cache["k"].shape[2]:
        raise ValueError("prompt longer than the cache")
    y, c = layer_fwd(params, x, heads, eps)
    qkv = c["qkv"].reshape(batch, seq, heads, 3, d)
    cache["k"][:, :, :seq] = qkv[:, :, :, 1].transpose(0, 2, 1, 3)
    cache["v"][:, :, :seq] = qkv[:, :, :, 2].transpose(0, 2, 1, 3)
    cache["len"][:] = seq
    return y


def _one_query(q, k, v):
    """Softmax(q k^T / sqrt d) v for one query over all rows of k, v."""
    d = q.shape[0]
    s = k @ q / np.sqrt(d)
    m = np.max(s)
    e = np.exp(s - m)
    return (e / e.sum()) @ v


def decode_step(params, x_tok, heads, cache, eps=LN_EPS):
    """One new token per sequence, x_tok [batch][h]: returns y_tok [batch][h];
    appends K, V at position cache["len"][b] and increments the lengths."""
    p = _p64(params)
    x = np.asarray(x_tok, dtype=np.float64)
    batch, h = x.shape
    d = h // heads
    if np.any(cache["len"] >= cache["k"].shape[2]):
        raise ValueError("cache full")
    u1, _, _ = layernorm_fwd(x, p["ln1_g"], p["ln1_b"], eps)
    qkv = (u1 @ p["w_qkv"].T + p["b_qkv"]).reshape(batch, heads, 3, d)
    ctx = np.empty((batch, heads, d))
    for b in range(batch):
        L = int(cache["len"][b])
        cache["k"][b, :, L] = qkv[b, :, 1]
        cache["v"][b, :, L] = qkv[b, :, 2]
        for hd in range(heads):
            ctx[b, hd] = _one_query(qkv[b, hd, 0], cache["k"][b, hd, :L + 1],
                                    cache["v"][b, hd, :L + 1])
    x1 = x + ctx.reshape(batch, h) @ p["w_o"].T + p["b_o"]
    u2, _, _ = layernorm_fwd(x1, p["ln2_g"], p["ln2_b"], eps)
    y = x1 + gelu(u2 @ p["w_fc1"].T + p["b_fc1"]) @ p["w_fc2"].T + p["b_fc2"]
    cache["len"] += 1
    return y


def shard_caches(batch, heads, max_seq, d, t):
    """t cache shards, partition p holding its H/t heads."""
    if heads % t:
        raise ValueError("t must divide heads")
    return [kv_cache(batch, heads // t, max_seq, d) for _ in range(t)]


def decode_step_partitioned(params, x_tok, heads, t, shards, counter, eps=LN_EPS):
    """decode_step with t literal partitions: partition p computes the QKV
    columns of its heads, appends to its own cache shard, attends locally and
    gives a partial out-projection; g sums the partials (and again after fc2)."""
    p = _p64(params)
    x = np.asarray(x_tok, dtype=np.float64)
    batch, h = x.shape
    ffn = p["w_fc1"].shape[0]
    d = h // heads
    ranks = shard_ranges(h, ffn, heads, t)
    u1, _, _ = layernorm_fwd(x, p["ln1_g"], p["ln1_b"], eps)
    parts = []
    for rk, sh in zip(ranks, shards):
        hp = rk["heads"]
        qkv = (u1 @ p["w_qkv"][rk["qkv"]].T + p["b_qkv"][rk["qkv"]]).reshape(batch, hp, 3, d)
        ctx = np.empty((batch, hp, d))
        for b in range(batch):
            L = int(sh["len"][b])
            sh["k"][b, :, L] = qkv[b, :, 1]
            sh["v"][b, :, L] = qkv[b, :, 2]
            for j in range(hp):
                ctx[b, j] = _one_query(qkv[b, j, 0], sh["k"][b, j, :L + 1], sh["v"][b, j, :L + 1])
        parts.append(ctx.reshape(batch, hp * d) @ p["w_o"][:, rk["ctx"]].T)
        sh["len"] += 1
    x1 = x + g_allreduce(parts, counter) + p["b_o"]
    u2, _, _ = layernorm_fwd(x1, p["ln2_g"], p["ln2_b"], eps)
    parts = [gelu(u2 @ p["w_fc1"][rk["ffn"]].T + p["b_fc1"][rk["ffn"]]) @ p["w_fc2"][:, rk["ffn"]].T
             for rk in ranks]
    return x1 + g_allreduce(parts, counter) + p["b_fc2"]


def decode_bytes(h, heads, ffn, batch, lengths, esz=2):
    """Minimum HBM bytes of one decode step: every weight once, the KV cache
    read up to each sequence's new length, the new K, V written, and the
    token-sized activations (negligible) left out."""
    weights = (3 * h * h + h * h + 2 * h * ffn) * esz + (3 * h + h + ffn + h + 4 * h) * esz
    kv = sum(2 * (int(L) + 1) * h * esz for L in lengths)
    return weights + kv
