"""Pins of the fp64 oracle against what the pages and the mathematics fix.

No GPU.  Each test would fail on a plausible mistake in the oracle: a dropped
term, a wrong sign or index, a transposed operand, a mis-read layout.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
import synthetic

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rel_err(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    m = np.max(np.abs(b))
    return float(np.max(np.abs(a - b)) / (m if m > 0 else 1.0))


def small_layer(h=32, heads=4, seq=12, batch=2, ffn=None, seed=3, affine=True):
    shp = synthetic.tiny(h=h, heads=heads, seq=seq, batch=batch, ffn=ffn, dtype="f32",
                         w_std=0.2, out_std=0.2)
    x, p, dy = synthetic.make_layer(shp, seed=seed, affine=affine)
    return shp, x.astype(np.float64), {k: v.astype(np.float64) for k, v in p.items()}, \
        dy.astype(np.float64)


# ---------------------------------------------------------------- GeLU

def test_gelu_textbook_values():
    tab = json.load(open(os.path.join(GOLDEN, "normal_cdf.json")))["phi"]
    for xs, phi in tab.items():
        x = float(xs)
        assert abs(oracle.gelu(np.array([x]))[0] - x * phi) <= 2e-15 * max(1.0, abs(x))


def test_gelu_identities():
    x = np.linspace(-6, 6, 1201)
    # GeLU(x) - GeLU(-x) = x (since Phi(x) + Phi(-x) = 1)
    assert np.max(np.abs(oracle.gelu(x) - oracle.gelu(-x) - x)) < 1e-14
    assert oracle.gelu(np.array([0.0]))[0] == 0.0
    assert abs(oracle.gelu_grad(np.array([0.0]))[0] - 0.5) < 1e-16
    # far tails: GeLU(x) -> x for x >> 0 and -> 0 for x << 0
    assert abs(oracle.gelu(np.array([12.0]))[0] - 12.0) < 1e-14
    assert abs(oracle.gelu(np.array([-12.0]))[0]) < 1e-14


def test_gelu_grad_central_difference():
    x = np.linspace(-5, 5, 101)
    eps = 1e-5
    fd = (oracle.gelu(x + eps) - oracle.gelu(x - eps)) / (2 * eps)
    assert np.max(np.abs(fd - oracle.gelu_grad(x))) < 1e-9


# ---------------------------------------------------------------- LayerNorm

def test_layernorm_moments():
    rng = np.random.default_rng(7)
    x = rng.standard_normal((9, 40)) * 3.0 + 1.5
    u, mu, rstd = oracle.layernorm_fwd(x, np.ones(40), np.zeros(40))
    var = x.var(axis=1)  # biased variance
    assert np.max(np.abs(u.mean(axis=1))) < 1e-14
    assert np.max(np.abs(u.var(axis=1) - var / (var + oracle.LN_EPS))) < 1e-13
    assert np.max(np.abs(mu - x.mean(axis=1))) < 1e-14
    # gamma / beta act per column
    g = rng.standard_normal(40)
    b = rng.standard_normal(40)
    u2, _, _ = oracle.layernorm_fwd(x, g, b)
    assert np.max(np.abs(u2 - (u * g + b))) < 1e-13


def test_layernorm_bwd_invariants_and_fd():
    rng = np.random.default_rng(8)
    n, h = 5, 24
    x = rng.standard_normal((n, h))
    g = 1 + 0.3 * rng.standard_normal(h)
    b = 0.3 * rng.standard_normal(h)
    du = rng.standard_normal((n, h))
    _, mu, rstd = oracle.layernorm_fwd(x, g, b)
    dx, dg, db = oracle.layernorm_bwd(du, x, mu, rstd, g)
    xhat = (x - mu[:, None]) * rstd[:, None]
    assert np.max(np.abs(dx.sum(axis=1))) < 1e-12
    # sum_j dx_j xhat_j = rstd * h * mean(g xhat) * (1 - mean(xhat^2)), which is
    # eps / (var + eps) times rstd * h * mean(g xhat): zero exactly when eps = 0
    gx = (du * g * xhat).mean(axis=1)
    closed = rstd * h * gx * (1.0 - (xhat * xhat).mean(axis=1))
    assert np.max(np.abs((dx * xhat).sum(axis=1) - closed)) < 1e-12
    _, mu0, rstd0 = oracle.layernorm_fwd(x, g, b, eps=0.0)
    dx0, _, _ = oracle.layernorm_bwd(du, x, mu0, rstd0, g)
    xhat0 = (x - mu0[:, None]) * rstd0[:, None]
    assert np.max(np.abs((dx0 * xhat0).sum(axis=1))) < 1e-12

    def loss(xx, gg, bb):
        return float((oracle.layernorm_fwd(xx, gg, bb)[0] * du).sum())

    eps = 1e-6
    for (arr, grad) in ((x, dx), (g, dg), (b, db)):
        fd = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            old = arr[idx]
            arr[idx] = old + eps
            lp = loss(x, g, b)
            arr[idx] = old - eps
            lm = loss(x, g, b)
            arr[idx] = old
            fd[idx] = (lp - lm) / (2 * eps)
        assert rel_err(fd, grad) < 1e-7


# ---------------------------------------------------------------- attention

def test_softmax_rows_and_mask():
    rng = np.random.default_rng(9)
    s, d = 17, 8
    q, k, v = (rng.standard_normal((s, d)) for _ in range(3))
    o, p, lse = oracle.attention_head_fwd(q, k, v)
    assert np.max(np.abs(p.sum(axis=1) - 1.0)) <= 1e-14
    assert np.all(p[oracle.causal_mask(s)] == 0.0)
    assert np.all(p[~oracle.causal_mask(s)] > 0.0)
    # token 0 sees only itself: its output is its own value row, exactly
    assert np.array_equal(o[0], v[0])
    # lse is the log of the normaliser: P = exp(S - lse) on the allowed entries
    scores = q @ k.T / math.sqrt(d)
    allowed = ~oracle.causal_mask(s)
    assert np.max(np.abs(np.exp(scores - lse[:, None])[allowed] - p[allowed])) < 1e-14


def test_attention_uniform_when_query_zero():
    rng = np.random.default_rng(10)
    s, d = 13, 6
    q = np.zeros((s, d))
    k, v = rng.standard_normal((s, d)), rng.standard_normal((s, d))
    o, _, _ = oracle.attention_head_fwd(q, k, v)
    closed = np.cumsum(v, axis=0) / np.arange(1, s + 1)[:, None]  # mean of v_0..v_i
    assert np.max(np.abs(o - closed)) < 1e-14


def test_attention_scale_is_inverse_sqrt_dhead():
    # two keys, query 1: P[1,0] / P[1,1] = exp((q.k0 - q.k1) / sqrt(d))
    d = 9
    q = np.zeros((2, d)); q[1, 0] = 1.0
    k = np.zeros((2, d)); k[0, 0] = 3.0
    v = np.eye(2, d)
    _, p, _ = oracle.attention_head_fwd(q, k, v)
    assert abs(p[1, 0] / p[1, 1] - math.exp(3.0 / 3.0)) < 1e-14


def test_attention_bwd_finite_difference():
    rng = np.random.default_rng(11)
    s, d = 6, 4
    q, k, v = (rng.standard_normal((s, d)) for _ in range(3))
    do = rng.standard_normal((s, d))
    o, p, _ = oracle.attention_head_fwd(q, k, v)
    dq, dk, dv = oracle.attention_head_bwd(q, k, v, p, o, do)

    def loss():
        return float((oracle.attention_head_fwd(q, k, v)[0] * do).sum())

    eps = 1e-6
    for arr, grad in ((q, dq), (k, dk), (v, dv)):
        fd = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            old = arr[idx]
            arr[idx] = old + eps
            lp = loss()
            arr[idx] = old - eps
            lm = loss()
            arr[idx] = old
            fd[idx] = (lp - lm) / (2 * eps)
        assert rel_err(fd, grad) < 1e-7


def test_head_interleaved_split():
    # column = head*3d + {Q,K,V}*d + channel
    H, d = 3, 2
    cols = np.arange(3 * H * d, dtype=np.float64)[None, :]
    q, k, v = oracle.split_qkv_columns(cols, H, d)
    assert q[0, 1].tolist() == [6.0, 7.0]
    assert k[0, 1].tolist() == [8.0, 9.0]
    assert v[0, 2].tolist() == [16.0, 17.0]


# ---------------------------------------------------------------- the split

def test_shard_layout_matches_pages():
    gold = json.load(open(os.path.join(GOLDEN, "shard_heads.json")))
    h, heads, t = 3072, gold["heads"], gold["t"]
    d = h // heads
    ranks = oracle.shard_ranges(h, 4 * h, heads, t)
    assert all(r["heads"] == gold["heads_per_rank"] for r in ranks)
    for rank, owned in gold["rank_heads"].items():
        sl = ranks[int(rank)]["qkv"]
        assert sl.start == owned[0] * 3 * d and sl.stop == (owned[-1] + 1) * 3 * d
    assert ranks[0]["qkv"].stop - ranks[0]["qkv"].start == 1152
    f = ranks[0]["ffn"]
    assert (f.stop - f.start) / (4 * h) == gold["mlp_fraction_per_rank"]


@pytest.mark.parametrize("case", ["A", "tiny8"])
def test_split_identity(case):
    """partitioned(t) equals the unpartitioned layer; 2 g-sums fwd, 2 f-sums bwd."""
    if case == "A":
        shp = synthetic.CONFIGS["A"]
        ts = (1, 2, 4)
    else:
        shp = synthetic.tiny(h=64, heads=8, seq=16, batch=2, dtype="f32",
                             w_std=0.1, out_std=0.1)
        ts = (1, 2, 4, 8)
    x, p, dy = synthetic.make_layer(shp, seed=0, affine=True)
    y_ref, cache = oracle.layer_fwd(p, x, shp.heads)
    dx_ref, g_ref, _ = oracle.layer_bwd(p, cache, dy)
    gold = json.load(open(os.path.join(GOLDEN, "shard_heads.json")))
    for t in ts:
        cnt = oracle.ReductionCounter()
        y, pc = oracle.layer_fwd_partitioned(p, x, shp.heads, t, cnt)
        assert cnt.g == gold["reductions_forward"] and cnt.f == 0
        dx, g = oracle.layer_bwd_partitioned(p, pc, dy, cnt)
        assert cnt.f == gold["reductions_backward"] and cnt.g == 2
        assert rel_err(y, y_ref) <= 1e-12
        assert rel_err(dx, dx_ref) <= 1e-12
        for k in g_ref:
            assert rel_err(g[k], g_ref[k]) <= 1e-12, (t, k)


def test_split_rejects_bad_t():
    with pytest.raises(ValueError):
        oracle.shard_ranges(64, 256, 6, 4)


def _permute_heads(p, perm, h, heads):
    d = h // heads
    q = dict(p)
    rows = np.concatenate([np.arange(hd * 3 * d, (hd + 1) * 3 * d) for hd in perm])
    cols = np.concatenate([np.arange(hd * d, (hd + 1) * d) for hd in perm])
    q["w_qkv"] = p["w_qkv"][rows]
    q["b_qkv"] = p["b_qkv"][rows]
    q["w_o"] = p["w_o"][:, cols]
    return q


def test_head_and_ffn_permutation_invariance():
    shp, x, p, dy = small_layer(h=32, heads=4)
    y, _ = oracle.layer_fwd(p, x, shp.heads)
    q = _permute_heads(p, [2, 0, 3, 1], shp.h, shp.heads)
    y2, _ = oracle.layer_fwd(q, x, shp.heads)
    assert rel_err(y2, y) < 1e-13
    perm = np.random.default_rng(1).permutation(shp.ffn)
    r = dict(p)
    r["w_fc1"], r["b_fc1"], r["w_fc2"] = p["w_fc1"][perm], p["b_fc1"][perm], p["w_fc2"][:, perm]
    y3, _ = oracle.layer_fwd(r, x, shp.heads)
    assert rel_err(y3, y) < 1e-13
    # a permutation of rows alone (not matched by W_o columns) does change y
    bad = dict(p)
    bad["w_qkv"] = q["w_qkv"]
    y4, _ = oracle.layer_fwd(bad, x, shp.heads)
    assert rel_err(y4, y) > 1e-6


def test_causality_and_batch_independence():
    shp, x, p, dy = small_layer(h=32, heads=4, seq=10, batch=3)
    y, _ = oracle.layer_fwd(p, x, shp.heads)
    x2 = x.copy()
    j = 6
    x2[1, j] += 0.5
    y2, _ = oracle.layer_fwd(p, x2, shp.heads)
    assert np.array_equal(y2[1, :j], y[1, :j])
    assert not np.array_equal(y2[1, j:], y[1, j:])
    assert np.array_equal(y2[0], y[0]) and np.array_equal(y2[2], y[2])


def test_identity_layer():
    shp, x, p, dy = small_layer()
    for k in ("w_o", "b_o", "w_fc2", "b_fc2"):
        p[k] = np.zeros_like(p[k])
    y, _ = oracle.layer_fwd(p, x, shp.heads)
    assert np.array_equal(y, x)


def test_single_token_sequence_closed_form():
    """seq = 1: attention returns the token's own V, so the layer is a plain MLP stack."""
    shp, x, p, dy = small_layer(h=32, heads=4, seq=1, batch=3)
    y, _ = oracle.layer_fwd(p, x, shp.heads)
    xf = x.reshape(3, 32)
    mu = xf.mean(1, keepdims=True)
    sd = np.sqrt(((xf - mu) ** 2).mean(1, keepdims=True) + 1e-5)
    u1 = (xf - mu) / sd * p["ln1_g"] + p["ln1_b"]
    v_cols = np.concatenate([np.arange(hd * 24 + 16, hd * 24 + 24) for hd in range(4)])
    vv = u1 @ p["w_qkv"][v_cols].T + p["b_qkv"][v_cols]
    x1 = xf + vv @ p["w_o"].T + p["b_o"]
    mu2 = x1.mean(1, keepdims=True)
    sd2 = np.sqrt(((x1 - mu2) ** 2).mean(1, keepdims=True) + 1e-5)
    u2 = (x1 - mu2) / sd2 * p["ln2_g"] + p["ln2_b"]
    zz = u2 @ p["w_fc1"].T + p["b_fc1"]
    phi = np.vectorize(lambda v: 0.5 * (1 + math.erf(v / math.sqrt(2))))(zz)
    yy = x1 + (zz * phi) @ p["w_fc2"].T + p["b_fc2"]
    assert rel_err(y.reshape(3, 32), yy) < 1e-13


# ---------------------------------------------------------------- backward

def test_layer_backward_finite_differences():
    """Every input and parameter entry of a tiny layer, central differences."""
    shp = synthetic.tiny(h=16, heads=4, seq=5, batch=2, ffn=64, dtype="f32",
                         w_std=0.3, out_std=0.3)
    x, p, dy = synthetic.make_layer(shp, seed=5, affine=True)
    x = x.astype(np.float64)
    p = {k: v.astype(np.float64) for k, v in p.items()}
    dy = dy.astype(np.float64)
    _, cache = oracle.layer_fwd(p, x, shp.heads)
    dx, g, _ = oracle.layer_bwd(p, cache, dy)

    def loss():
        return float((oracle.layer_fwd(p, x, shp.heads)[0] * dy).sum())

    eps = 1e-6
    for name, arr, grad in [("x", x, dx)] + [(k, p[k], g[k]) for k in synthetic.PARAM_ORDER]:
        fd = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            old = arr[idx]
            arr[idx] = old + eps
            lp = loss()
            arr[idx] = old - eps
            lm = loss()
            arr[idx] = old
            fd[idx] = (lp - lm) / (2 * eps)
        assert rel_err(fd, grad) <= 1e-6, name


def test_backward_is_linear_in_dy():
    shp, x, p, dy = small_layer()
    _, cache = oracle.layer_fwd(p, x, shp.heads)
    dy2 = np.random.default_rng(4).standard_normal(dy.shape)
    d1, g1, _ = oracle.layer_bwd(p, cache, dy)
    d2, g2, _ = oracle.layer_bwd(p, cache, dy2)
    d3, g3, _ = oracle.layer_bwd(p, cache, 2.0 * dy - 3.0 * dy2)
    assert rel_err(d3, 2 * d1 - 3 * d2) < 1e-12
    for k in g1:
        assert rel_err(g3[k], 2 * g1[k] - 3 * g2[k]) < 1e-12


def _torch_layer(p, x, heads):
    """An independent float64 torch forward of the same layer (test-only)."""
    import torch
    import torch.nn.functional as F
    b, s, h = x.shape
    d = h // heads
    u1 = F.layer_norm(x, (h,), p["ln1_g"], p["ln1_b"], eps=1e-5)
    qkv = F.linear(u1, p["w_qkv"], p["b_qkv"]).view(b, s, heads, 3, d)
    q, k, v = (qkv[:, :, :, i].transpose(1, 2) for i in range(3))
    o = F.scaled_dot_product_attention(q, k, v, is_causal=True)
    ctx = o.transpose(1, 2).reshape(b, s, h)
    x1 = x + F.linear(ctx, p["w_o"], p["b_o"])
    u2 = F.layer_norm(x1, (h,), p["ln2_g"], p["ln2_b"], eps=1e-5)
    return x1 + F.linear(F.gelu(F.linear(u2, p["w_fc1"], p["b_fc1"])), p["w_fc2"], p["b_fc2"])


def test_torch_autograd_crosscheck_config_a():
    torch = pytest.importorskip("torch")
    shp = synthetic.CONFIGS["A"]
    x, p, dy = synthetic.make_layer(shp, seed=0, affine=True)
    y_ref, cache = oracle.layer_fwd(p, x, shp.heads)
    dx_ref, g_ref, _ = oracle.layer_bwd(p, cache, dy)
    tp = {k: torch.tensor(v, dtype=torch.float64, requires_grad=True) for k, v in p.items()}
    tx = torch.tensor(x, dtype=torch.float64, requires_grad=True)
    ty = _torch_layer(tp, tx, shp.heads)
    ty.backward(torch.tensor(dy, dtype=torch.float64))
    assert rel_err(ty.detach().numpy(), y_ref) < 1e-12
    assert rel_err(tx.grad.numpy(), dx_ref) < 1e-11
    for k in g_ref:
        assert rel_err(tp[k].grad.numpy(), g_ref[k]) < 1e-11, k


def test_flop_count():
    # 3 * (24 n h^2 + 2 batch seq (seq+1) h) for ffn = 4h
    assert oracle.layer_flops(3072, 32, 1024, 16) == 3 * (24 * 16384 * 3072 ** 2
                                                         + 2 * 16 * 1024 * 1025 * 3072)
    assert abs(oracle.layer_flops(3072, 32, 1024, 16) - 1.144e13) / 1.144e13 < 1e-3


# ---------------------------------------------------------------- the GEMM unit

def test_gemm_partitioned_pins():
    rng = np.random.default_rng(12)
    A = rng.standard_normal((7, 12))
    B = rng.standard_normal((5, 12))
    full = oracle.gemm_partitioned(A, B, 1)
    # identity operand: A I^T = A
    assert np.array_equal(oracle.gemm_partitioned(A, np.eye(12), 3), A)
    # the split identity: any number of parts sums to the same product
    for parts in (2, 3, 4, 6, 12):
        assert rel_err(oracle.gemm_partitioned(A, B, parts), full) < 1e-14
    # entry (i, j) is the dot product of row i of A with row j of B (not a transpose)
    assert abs(full[3, 2] - sum(A[3, k] * B[2, k] for k in range(12))) < 1e-12
    bias = rng.standard_normal(5)
    R = rng.standard_normal((7, 5))
    assert rel_err(oracle.gemm_partitioned(A, B, 2, 1, bias=bias), full + bias) < 1e-14
    assert rel_err(oracle.gemm_partitioned(A, B, 2, 2, bias=bias, R=R), full + bias + R) < 1e-14
    c, z = oracle.gemm_partitioned(A, B, 3, 3, bias=bias)
    assert rel_err(z, full + bias) < 1e-14
    assert np.max(np.abs(c - z * oracle.gelu_grad(0 * z) * 0 - oracle.gelu(z))) == 0.0
    c4 = oracle.gemm_partitioned(A, B, 4, 4, Z=R)
    assert rel_err(c4, full * oracle.gelu_grad(R)) < 1e-14
    with pytest.raises(ValueError):
        oracle.gemm_partitioned(A, B, 5)


# ---------------------------------------------------------------- dropout (Philox masks)

def test_philox_known_answers():
    gold = json.load(open(os.path.join(GOLDEN, "philox_kat.json")))
    for v in gold["vectors"]:
        ctr = np.array([int(c, 16) for c in v["counter"]], dtype=np.uint32)
        key = [int(k, 16) for k in v["key"]]
        out = oracle.philox.philox4x32(ctr, key)
        assert [int(o) for o in out] == [int(o, 16) for o in v["out"]]


def test_philox_word_layout():
    """word(e) is lane e mod 4 of the block at counter (e div 4, site); seed splits into the key."""
    seed = (0x01234567 << 32) | 0x89ABCDEF
    e = np.arange(4 * 3, dtype=np.uint64) + np.uint64((1 << 34) + 8)
    w = oracle.philox.words(e, seed, 2)
    for i, ei in enumerate(e.tolist()):
        ctr = np.array([(ei >> 2) & 0xFFFFFFFF, ei >> 34, 2, 0], dtype=np.uint32)
        blk = oracle.philox.philox4x32(ctr, (0x89ABCDEF, 0x01234567))
        assert int(w[i]) == int(blk[ei & 3])


def test_dropout_mask_statistics():
    """Keep fraction 1 - p within 5 sigma; the words are uniform (mean, decile counts)."""
    n = 1 << 18
    e = np.arange(n, dtype=np.uint64)
    w = oracle.philox.words(e, 1234, 1).astype(np.float64) / 2.0 ** 32
    assert abs(w.mean() - 0.5) < 5 * math.sqrt(1 / 12 / n)
    counts = np.histogram(w, bins=10, range=(0, 1))[0]
    chi2 = float(((counts - n / 10) ** 2 / (n / 10)).sum())
    assert chi2 < 40.0          # 9 degrees of freedom; P(chi2 > 40) < 1e-5
    for p in (0.1, 0.5, 0.9):
        keep = oracle.philox.keep_mask(e, 99, 0, p)
        assert abs(keep.mean() - (1 - p)) < 5 * math.sqrt(p * (1 - p) / n)
    # different sites and seeds give different masks
    a = oracle.philox.keep_mask(e[:4096], 7, 1, 0.5)
    b = oracle.philox.keep_mask(e[:4096], 7, 2, 0.5)
    c = oracle.philox.keep_mask(e[:4096], 8, 1, 0.5)
    assert 0.4 < (a != b).mean() < 0.6 and 0.4 < (a != c).mean() < 0.6
    assert oracle.philox.threshold(0.0) == 0 and oracle.philox.threshold(0.5) == 1 << 31
    with pytest.raises(ValueError):
        oracle.philox.threshold(1.0)


def test_dropout_zero_is_the_plain_layer():
    shp, x, p, dy = small_layer()
    y0, c0 = oracle.layer_fwd(p, x, shp.heads)
    dx0, g0, _ = oracle.layer_bwd(p, c0, dy)
    drop = dict(p_attn=0.0, p_hidden=0.0, seed=5)
    y1, c1 = oracle.layer_fwd(p, x, shp.heads, dropout=drop)
    dx1, g1, _ = oracle.layer_bwd(p, c1, dy)
    assert np.array_equal(y0, y1) and np.array_equal(dx0, dx1)
    for k in g0:
        assert np.array_equal(g0[k], g1[k])


def test_hidden_dropout_zeroes_and_rescales():
    """With only hidden dropout, y - x1 is 0 where dropped and (fc2 out) / (1 - p) where kept."""
    shp, x, p, dy = small_layer()
    drop = dict(p_attn=0.0, p_hidden=0.3, seed=11)
    y, c = oracle.layer_fwd(p, x, shp.heads, dropout=drop)
    n, h = c["x"].shape
    keep = oracle.philox.hidden_mask(n, h, 11, oracle.philox.SITE_FC2, 0.3)
    r = y.reshape(n, h) - c["x1"]
    fc2 = c["a"] @ p["w_fc2"].T + p["b_fc2"]
    assert np.all(r[~keep] == 0.0)
    assert np.allclose(r[keep], fc2[keep] / 0.7, rtol=1e-12, atol=1e-12)
    assert 0.55 < keep.mean() < 0.85


def test_attention_dropout_is_unbiased():
    """Averaged over seeds, dropped attention approaches the undropped output."""
    rng = np.random.default_rng(0)
    seq, d, heads = 8, 4, 2
    qkv = rng.standard_normal((seq, 3 * heads * d))
    ref, _, _ = oracle.multihead_fwd(qkv, 1, seq, heads, d)
    runs = 400
    acc = np.zeros_like(ref)
    for s in range(runs):
        out, _, _ = oracle.multihead_fwd(qkv, 1, seq, heads, d, dict(p_attn=0.2, seed=s))
        acc += out
    assert np.max(np.abs(acc / runs - ref)) < 0.15
    one, _, _ = oracle.multihead_fwd(qkv, 1, seq, heads, d, dict(p_attn=0.2, seed=3))
    assert not np.allclose(one, ref)


def _torch_layer_dropout(p, x, heads, mo, m2, ma, p_attn, p_hidden):
    """Float64 torch forward with the given keep masks (test-only, written independently)."""
    import torch
    import torch.nn.functional as F
    b, s, h = x.shape
    d = h // heads
    u1 = F.layer_norm(x, (h,), p["ln1_g"], p["ln1_b"], eps=1e-5)
    qkv = F.linear(u1, p["w_qkv"], p["b_qkv"]).view(b, s, heads, 3, d)
    q, k, v = (qkv[:, :, :, i].transpose(1, 2) for i in range(3))
    sc = q @ k.transpose(-1, -2) / math.sqrt(d)
    causal = torch.ones(s, s, dtype=torch.bool).tril()
    prob = torch.softmax(sc.masked_fill(~causal, float("-inf")), dim=-1)
    o = (prob * ma / (1 - p_attn)) @ v
    ctx = o.transpose(1, 2).reshape(b, s, h)
    x1 = x + F.linear(ctx, p["w_o"], p["b_o"]) * mo / (1 - p_hidden)
    u2 = F.layer_norm(x1, (h,), p["ln2_g"], p["ln2_b"], eps=1e-5)
    fc2 = F.linear(F.gelu(F.linear(u2, p["w_fc1"], p["b_fc1"])), p["w_fc2"], p["b_fc2"])
    return x1 + fc2 * m2 / (1 - p_hidden)


def test_dropout_layer_matches_torch_autograd():
    torch = pytest.importorskip("torch")
    shp, x, p, dy = small_layer(h=32, heads=4, seq=12, batch=2)
    pa, ph, seed = 0.25, 0.15, 77
    drop = dict(p_attn=pa, p_hidden=ph, seed=seed)
    y_ref, cache = oracle.layer_fwd(p, x, shp.heads, dropout=drop)
    dx_ref, g_ref, _ = oracle.layer_bwd(p, cache, dy)
    b, s, h = x.shape
    ph_ = oracle.philox
    mo = ph_.hidden_mask(b * s, h, seed, ph_.SITE_OUT, ph).reshape(b, s, h)
    m2 = ph_.hidden_mask(b * s, h, seed, ph_.SITE_FC2, ph).reshape(b, s, h)
    ma = np.stack([np.stack([ph_.attention_mask(bb, hd, shp.heads, s, seed, pa)
                             for hd in range(shp.heads)]) for bb in range(b)])
    T = lambda a: torch.tensor(a, dtype=torch.float64)  # noqa: E731
    tp = {k: torch.tensor(v, dtype=torch.float64, requires_grad=True) for k, v in p.items()}
    tx = torch.tensor(x, dtype=torch.float64, requires_grad=True)
    ty = _torch_layer_dropout(tp, tx, shp.heads, T(mo), T(m2), T(ma), pa, ph)
    ty.backward(T(dy))
    assert rel_err(ty.detach().numpy(), y_ref) < 1e-12
    assert rel_err(tx.grad.numpy(), dx_ref) < 1e-11
    for k in g_ref:
        assert rel_err(tp[k].grad.numpy(), g_ref[k]) < 1e-11, k


def test_dropout_layer_backward_finite_differences():
    shp = synthetic.tiny(h=16, heads=4, seq=5, batch=2, ffn=64, dtype="f32",
                         w_std=0.3, out_std=0.3)
    x, p, dy = synthetic.make_layer(shp, seed=6, affine=True)
    x = x.astype(np.float64)
    p = {k: v.astype(np.float64) for k, v in p.items()}
    dy = dy.astype(np.float64)
    drop = dict(p_attn=0.3, p_hidden=0.2, seed=2024)
    _, cache = oracle.layer_fwd(p, x, shp.heads, dropout=drop)
    dx, g, _ = oracle.layer_bwd(p, cache, dy)

    def loss():
        return float((oracle.layer_fwd(p, x, shp.heads, dropout=drop)[0] * dy).sum())

    eps = 1e-6
    for name, arr, grad in [("x", x, dx), ("w_qkv", p["w_qkv"], g["w_qkv"]),
                            ("b_o", p["b_o"], g["b_o"]), ("w_fc2", p["w_fc2"], g["w_fc2"]),
                            ("ln1_g", p["ln1_g"], g["ln1_g"])]:
        fd = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            old = arr[idx]
            arr[idx] = old + eps
            lp = loss()
            arr[idx] = old - eps
            lm = loss()
            arr[idx] = old
            fd[idx] = (lp - lm) / (2 * eps)
        assert rel_err(fd, grad) <= 1e-6, name


@pytest.mark.parametrize("t", [1, 2, 4])
def test_split_identity_with_dropout(t):
    """The partitioned layer draws the same masks: head masks use the layer-wide head index."""
    shp = synthetic.tiny(h=64, heads=8, seq=16, batch=2, dtype="f32", w_std=0.1, out_std=0.1)
    x, p, dy = synthetic.make_layer(shp, seed=1, affine=True)
    drop = dict(p_attn=0.2, p_hidden=0.1, seed=31337)
    y_ref, cache = oracle.layer_fwd(p, x, shp.heads, dropout=drop)
    dx_ref, g_ref, _ = oracle.layer_bwd(p, cache, dy)
    cnt = oracle.ReductionCounter()
    y, pc = oracle.layer_fwd_partitioned(p, x, shp.heads, t, cnt, dropout=drop)
    dx, g = oracle.layer_bwd_partitioned(p, pc, dy, cnt)
    assert rel_err(y, y_ref) <= 1e-12 and rel_err(dx, dx_ref) <= 1e-12
    for k in g_ref:
        assert rel_err(g[k], g_ref[k]) <= 1e-12, (t, k)
