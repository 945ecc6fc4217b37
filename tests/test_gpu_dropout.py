"""GPU parity of dropout: the layer with dropout against the oracle with the
same Philox masks, and exact checks of every mask the kernels draw.

Masks decide values bit for bit, so besides the usual tolerances (fp32 1e-5,
bf16 1.5e-2 forward / 3e-2 gradients) the tests build inputs whose outputs
reveal each keep bit exactly:
  * hidden sites: with a large bias, x1 == x (bitwise) exactly where the
    out-proj output was dropped, y == x1 exactly where the fc2 output was;
  * attention: Q = K = 0 makes P uniform, and one-hot V (or dO, Q, K) columns
    carry the keep bits of two keys (or queries) each, so every drawn bit shows
    up in the output as an integer."""
import numpy as np
import pytest

import oracle
import synthetic
from harness import compare, f32, make, run_gpu, run_oracle, tolerance

pytestmark = pytest.mark.gpu

P_ATTN, P_HIDDEN = f32(0.15), f32(0.1)


def check_layer(shape, t, drop, affine=True, seed=0, batch=None):
    x, p, dy = make(shape, seed=seed, affine=affine, batch=batch)
    gpu = run_gpu(shape, x, p, dy, t, drop=drop)
    ref = run_oracle(shape, x, p, dy, drop=drop)
    errs = compare(gpu, ref, shape.dtype)
    bad = {k: v for k, v in errs.items() if not v <= tolerance(k, shape.dtype)}
    assert not bad, (bad, errs)


@pytest.mark.parametrize("t", [1, 2])
def test_fp32_layer_with_dropout(t):
    drop = dict(p_attn=P_ATTN, p_hidden=P_HIDDEN, seed=1234)
    check_layer(synthetic.CONFIGS["A"], t, drop)


SHAPES = {
    "d64": synthetic.tiny(h=128, heads=2, seq=128, batch=2, dtype="bf16", w_std=0.02,
                          out_std=0.01),
    "d96": synthetic.tiny(h=384, heads=4, seq=256, batch=1, dtype="bf16", w_std=0.02,
                          out_std=0.01),
    "d128": synthetic.tiny(h=256, heads=2, seq=384, batch=2, dtype="bf16", w_std=0.02,
                           out_std=0.01),
}


@pytest.mark.parametrize("name,t", [("d64", 2), ("d96", 1), ("d96", 2), ("d128", 1), ("d128", 2)])
def test_bf16_layer_with_dropout(name, t):
    drop = dict(p_attn=P_ATTN, p_hidden=P_HIDDEN, seed=(1 << 40) + 77)
    check_layer(SHAPES[name], t, drop)


@pytest.mark.parametrize("which", ["attn", "hidden"])
def test_bf16_layer_single_site(which):
    drop = dict(p_attn=P_ATTN if which == "attn" else 0.0,
                p_hidden=P_HIDDEN if which == "hidden" else 0.0, seed=5)
    check_layer(SHAPES["d128"], 2, drop)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_hidden_masks_exact(dtype):
    """x1 != x exactly where site 1 keeps, y != x1 exactly where site 2 keeps."""
    base = SHAPES["d96"]
    shape = synthetic.tiny(h=base.h, heads=base.heads, seq=base.seq, batch=2, dtype=dtype,
                           w_std=0.02, out_std=0.01)
    x, p, dy = make(shape, seed=3, affine=True)
    p = dict(p)
    p["b_o"] = np.ones_like(p["b_o"])
    p["b_fc2"] = np.ones_like(p["b_fc2"])
    seed, ph = 99, f32(0.3)
    gpu = run_gpu(shape, x, p, dy, 2, drop=dict(p_attn=0.0, p_hidden=ph, seed=seed))
    n, h = shape.batch * shape.seq, shape.h
    x1 = gpu["s_x1"].reshape(n, h)
    xs = synthetic.to_storage(x, dtype).reshape(n, h)
    y = gpu["y"].reshape(n, h)
    k1 = oracle.philox.hidden_mask(n, h, seed, oracle.philox.SITE_OUT, ph)
    k2 = oracle.philox.hidden_mask(n, h, seed, oracle.philox.SITE_FC2, ph)
    assert np.array_equal(x1 != xs, k1)
    assert np.array_equal(y != x1, k2)
    assert abs(k1.mean() - 0.7) < 0.02


def _attn_inputs(batch, seq, heads, d, q=None, k=None, v=None):
    """qkv [batch*seq][3*heads*d] with per-head Q, K, V given as [seq][d] arrays."""
    qkv = np.zeros((batch, seq, heads, 3, d))
    for i, a in enumerate((q, k, v)):
        if a is not None:
            qkv[:, :, :, i, :] = a[None, :, None, :]
    return qkv.reshape(batch * seq, 3 * heads * d)


def _onehot_pairs(seq, d):
    """a[r][c] = 1 + (r & 1) if c == r // 2: column c carries rows 2c and 2c+1."""
    a = np.zeros((seq, d))
    r = np.arange(seq)
    a[r, r // 2] = 1 + (r & 1)
    return a


def _gpu_attention(dtype, batch, seq, heads, d, qkv, p_attn, seed, dctx=None):
    import torch
    from tensor_model_transformer_gb300 import mtl
    from harness import to_device, to_np
    tq = to_device(qkv, dtype)
    ctx = torch.empty((batch * seq, heads * d), dtype=tq.dtype, device="cuda")
    lse = torch.empty((batch, heads, seq), dtype=torch.float32, device="cuda")
    ws = torch.empty(mtl.attention_ws_bytes(batch, seq, heads), dtype=torch.uint8, device="cuda")
    mb = mtl.attention_mask_bytes(dtype, batch, seq, heads, p_attn)
    mask = torch.empty(mb, dtype=torch.uint8, device="cuda") if mb else None
    mtl.attention_fwd(dtype, batch, seq, heads, d, tq, ctx, lse, ws, mask=mask, p_attn=p_attn,
                      seed=seed)
    mtl.layer_check(ws)
    out = {"ctx": to_np(ctx), "lse": to_np(lse)}
    if dctx is not None:
        tdo = to_device(dctx, dtype)
        dqkv = torch.empty_like(tq)
        mtl.attention_bwd(dtype, batch, seq, heads, d, tq, ctx, lse, tdo, dqkv, ws, mask=mask,
                          p_attn=p_attn, seed=seed)
        mtl.layer_check(ws)
        out["dqkv"] = to_np(dqkv)
    torch.cuda.synchronize()
    return out


def _oracle_attention(batch, seq, heads, d, qkv, p_attn, seed, dctx=None):
    drop = dict(p_attn=p_attn, seed=seed)
    ctx, lse, probs = oracle.multihead_fwd(qkv, batch, seq, heads, d, drop)
    out = {"ctx": ctx, "lse": lse}
    if dctx is not None:
        out["dqkv"] = oracle.multihead_bwd(qkv, ctx, probs, dctx, batch, seq, heads, d, drop)
    return out


ATTN_CASES = [("bf16", 128, 64), ("bf16", 128, 96), ("bf16", 256, 128), ("f32", 128, 64),
              ("f32", 192, 96)]


@pytest.mark.parametrize("dtype,seq,d", ATTN_CASES)
@pytest.mark.parametrize("p_attn", [0.0, f32(0.25)])
def test_attention_forward_masks_exact(dtype, seq, d, p_attn):
    """Q = K = 0: P_ij = 1/(i+1); V column c holds keys 2c (x1) and 2c+1 (x2), so
    O_ic (i+1)(1-p) = keep(i,2c) + 2 keep(i,2c+1) exactly."""
    batch, heads, seed = 2, 2, 2024
    qkv = _attn_inputs(batch, seq, heads, d, v=_onehot_pairs(seq, d))
    g = _gpu_attention(dtype, batch, seq, heads, d, qkv, p_attn, seed)
    r = _oracle_attention(batch, seq, heads, d, qkv, p_attn, seed)
    i = np.arange(seq)[None, :, None, None]
    scale = (i + 1) * (1 - p_attn)
    kg = g["ctx"].reshape(batch, seq, heads, d) * scale
    kr = r["ctx"].reshape(batch, seq, heads, d) * scale
    assert np.max(np.abs(kg - np.rint(kg))) < 0.1
    assert np.array_equal(np.rint(kg), np.rint(kr))
    assert np.max(np.abs(g["lse"] - r["lse"])) < 1e-5 * np.log(seq)


@pytest.mark.parametrize("dtype,seq,d", ATTN_CASES)
@pytest.mark.parametrize("p_attn", [0.0, f32(0.25)])
def test_attention_dv_masks_exact(dtype, seq, d, p_attn):
    """Q = K = V = 0, dO column c holds queries 2c and 2c+1 scaled by (i+1):
    dV_jc (1-p) = keep(2c,j) + 2 keep(2c+1,j) exactly (zero for queries before j)."""
    batch, heads, seed = 2, 2, 31
    qkv = _attn_inputs(batch, seq, heads, d)
    do = _onehot_pairs(seq, d) * (np.arange(seq) + 1)[:, None]
    dctx = np.broadcast_to(do[None, :, None, :], (batch, seq, heads, d)).reshape(batch * seq, -1)
    g = _gpu_attention(dtype, batch, seq, heads, d, qkv, p_attn, seed, dctx)
    r = _oracle_attention(batch, seq, heads, d, qkv, p_attn, seed, dctx)
    dv_g = g["dqkv"].reshape(batch, seq, heads, 3, d)[:, :, :, 2] * (1 - p_attn)
    dv_r = r["dqkv"].reshape(batch, seq, heads, 3, d)[:, :, :, 2] * (1 - p_attn)
    assert np.max(np.abs(dv_g - np.rint(dv_g))) < 0.1
    assert np.array_equal(np.rint(dv_g), np.rint(dv_r))
    assert np.all(g["dqkv"].reshape(batch, seq, heads, 3, d)[:, :, :, :2] == 0)


@pytest.mark.parametrize("dtype,seq,d", ATTN_CASES)
@pytest.mark.parametrize("grad", ["dq", "dk"])
@pytest.mark.parametrize("p_attn", [0.0, f32(0.25)])
def test_attention_ds_masks(dtype, seq, d, grad, p_attn):
    """S = 0 with one of Q, K one-hot and the other 0; V[:, 0] = 1, dO[:, 0] = i+1:
    dS_ij = (keep(i,j) - cnt_i/(i+1)) / (1-p), so every keep bit moves dQ (dK) by
    at least scale/(1-p) -- far above the rounding (atol a quarter of that)."""
    batch, heads, seed = 2, 2, 8
    oh = _onehot_pairs(seq, d)
    v = np.zeros((seq, d))
    v[:, 0] = 1.0
    qkv = _attn_inputs(batch, seq, heads, d, q=oh if grad == "dk" else None,
                       k=oh if grad == "dq" else None, v=v)
    do = np.zeros((seq, d))
    do[:, 0] = np.arange(seq) + 1
    dctx = np.broadcast_to(do[None, :, None, :], (batch, seq, heads, d)).reshape(batch * seq, -1)
    g = _gpu_attention(dtype, batch, seq, heads, d, qkv, p_attn, seed, dctx)
    r = _oracle_attention(batch, seq, heads, d, qkv, p_attn, seed, dctx)
    part = 0 if grad == "dq" else 1
    a_g = g["dqkv"].reshape(batch, seq, heads, 3, d)[:, :, :, part]
    a_r = r["dqkv"].reshape(batch, seq, heads, 3, d)[:, :, :, part]
    step = (1.0 / np.sqrt(d)) / (1 - p_attn)
    if p_attn > 0:
        assert np.max(np.abs(a_r)) > step      # the design is not degenerate
    assert np.max(np.abs(a_g - a_r)) < 0.25 * step


@pytest.mark.parametrize("seq,d", [(128, 64), (384, 128)])
def test_attention_stored_keep_bits(seq, d):
    """The bits the bf16 forward stores for the backward are the oracle's keep
    mask: tile (qb, kb <= qb) of each (batch, head), word w of row r at w*128+r."""
    import torch
    from tensor_model_transformer_gb300 import mtl
    from harness import to_device
    batch, heads, seed, p_attn = 2, 3, 4242, f32(0.4)
    rng = np.random.default_rng(0)
    qkv = rng.standard_normal((batch * seq, 3 * heads * d)) * 0.5
    tq = to_device(qkv, "bf16")
    ctx = torch.empty((batch * seq, heads * d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((batch, heads, seq), dtype=torch.float32, device="cuda")
    ws = torch.empty(mtl.attention_ws_bytes(batch, seq, heads), dtype=torch.uint8, device="cuda")
    mb = mtl.attention_mask_bytes("bf16", batch, seq, heads, p_attn)
    mask = torch.zeros(mb, dtype=torch.uint8, device="cuda")
    mtl.attention_fwd("bf16", batch, seq, heads, d, tq, ctx, lse, ws, mask=mask, p_attn=p_attn,
                      seed=seed)
    mtl.layer_check(ws)
    words = mask.cpu().numpy().view(np.uint32)
    nqb = seq // 128
    nt = nqb * (nqb + 1) // 2
    assert words.size == batch * heads * nt * 512
    bits = ((words[:, None] >> np.arange(32, dtype=np.uint32)[None, :]) & 1).astype(bool)
    bits = bits.reshape(batch, heads, nt, 4, 128, 32)       # [.., word, row, bit]
    for b in range(batch):
        for hd in range(heads):
            ref = oracle.philox.attention_mask(b, hd, heads, seq, seed, p_attn)
            for qb in range(nqb):
                for kb in range(qb + 1):
                    t = bits[b, hd, qb * (qb + 1) // 2 + kb]          # [4, 128, 32]
                    got = t.transpose(1, 0, 2).reshape(128, 128)      # [row, key]
                    want = ref[qb * 128:(qb + 1) * 128, kb * 128:(kb + 1) * 128]
                    assert np.array_equal(got, want), (b, hd, qb, kb)
