"""Pins of the oracle's Post-LN layer (LayerNorm after each residual add)."""
import math

import numpy as np
import pytest

import oracle
import synthetic


def _layer(seed=0, h=32, heads=4, seq=6, batch=2, ffn=None, std=0.3):
    shp = synthetic.tiny(h=h, heads=heads, seq=seq, batch=batch, ffn=ffn, dtype="f32",
                         w_std=std, out_std=std)
    x, p, dy = synthetic.make_layer(shp, seed=seed, affine=True)
    return shp, x.astype(np.float64), {k: v.astype(np.float64) for k, v in p.items()}, \
        dy.astype(np.float64)


def test_output_rows_are_normalized():
    """With gamma2 = 1, beta2 = 0 every output row has mean 0 and variance
    s^2 / (s^2 + eps) (s^2 the row variance of h2)."""
    shp, x, p, _ = _layer()
    p["ln2_g"][:] = 1.0
    p["ln2_b"][:] = 0.0
    y, c = oracle.layer_fwd_post_ln(p, x, shp.heads)
    y = y.reshape(-1, shp.h)
    s2 = c["h2"].var(axis=1)
    assert np.max(np.abs(y.mean(axis=1))) < 1e-12
    assert np.allclose(y.var(axis=1), s2 / (s2 + 1e-5), rtol=1e-10)


def test_identity_sublayers():
    """W_o = W_fc2 = 0 and b_o = b_fc2 = 0: y = LN2(LN1(x))."""
    shp, x, p, _ = _layer(seed=1)
    for k in ("w_o", "b_o", "w_fc2", "b_fc2"):
        p[k][:] = 0.0
    y, _ = oracle.layer_fwd_post_ln(p, x, shp.heads)
    xf = x.reshape(-1, shp.h)
    u, _, _ = oracle.layernorm_fwd(xf, p["ln1_g"], p["ln1_b"])
    ref, _, _ = oracle.layernorm_fwd(u, p["ln2_g"], p["ln2_b"])
    assert np.max(np.abs(y.reshape(-1, shp.h) - ref)) < 1e-12


def test_differs_from_pre_ln():
    shp, x, p, _ = _layer(seed=2)
    assert not np.allclose(oracle.layer_fwd_post_ln(p, x, shp.heads)[0],
                           oracle.layer_fwd(p, x, shp.heads)[0])


def test_post_ln_backward_finite_differences():
    shp, x, p, dy = _layer(seed=3, h=16, heads=4, seq=5, batch=2, ffn=64)
    _, c = oracle.layer_fwd_post_ln(p, x, shp.heads)
    dx, g, _ = oracle.layer_bwd_post_ln(p, c, dy)

    def loss():
        return float((oracle.layer_fwd_post_ln(p, x, shp.heads)[0] * dy).sum())

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
        assert np.max(np.abs(fd - grad)) <= 1e-6 * max(1.0, np.max(np.abs(grad))), name


def test_post_ln_matches_torch_autograd():
    torch = pytest.importorskip("torch")
    import torch.nn.functional as F
    shp = synthetic.CONFIGS["A"]
    x, p, dy = synthetic.make_layer(shp, seed=4, affine=True)
    y_ref, c = oracle.layer_fwd_post_ln(p, x, shp.heads)
    dx_ref, g_ref, _ = oracle.layer_bwd_post_ln(p, c, dy)
    tp = {k: torch.tensor(v, dtype=torch.float64, requires_grad=True) for k, v in p.items()}
    tx = torch.tensor(x, dtype=torch.float64, requires_grad=True)
    b, s, h = x.shape
    heads = shp.heads
    d = h // heads
    qkv = F.linear(tx, tp["w_qkv"], tp["b_qkv"]).view(b, s, heads, 3, d)
    q, k, v = (qkv[:, :, :, i].transpose(1, 2) for i in range(3))
    o = F.scaled_dot_product_attention(q, k, v, is_causal=True)
    ctx = o.transpose(1, 2).reshape(b, s, h)
    x1 = F.layer_norm(tx + F.linear(ctx, tp["w_o"], tp["b_o"]), (h,), tp["ln1_g"], tp["ln1_b"],
                      eps=1e-5)
    h2 = x1 + F.linear(F.gelu(F.linear(x1, tp["w_fc1"], tp["b_fc1"])), tp["w_fc2"], tp["b_fc2"])
    ty = F.layer_norm(h2, (h,), tp["ln2_g"], tp["ln2_b"], eps=1e-5)
    ty.backward(torch.tensor(dy, dtype=torch.float64))
    rel = lambda a, b_: np.max(np.abs(a - b_)) / np.max(np.abs(b_))  # noqa: E731
    assert rel(ty.detach().numpy(), y_ref) < 1e-12
    assert rel(tx.grad.numpy(), dx_ref) < 1e-10
    for k in g_ref:
        assert rel(tp[k].grad.numpy(), g_ref[k]) < 1e-10, k


@pytest.mark.parametrize("t", [1, 2, 4])
def test_post_ln_split_identity(t):
    shp = synthetic.tiny(h=64, heads=8, seq=12, batch=2, dtype="f32", w_std=0.1, out_std=0.1)
    x, p, _ = synthetic.make_layer(shp, seed=5, affine=True)
    y_ref, _ = oracle.layer_fwd_post_ln(p, x, shp.heads)
    cnt = oracle.ReductionCounter()
    y = oracle.layer_fwd_post_ln_partitioned(p, x, shp.heads, t, cnt)
    assert cnt.g == 2
    assert np.max(np.abs(y - y_ref)) < 1e-12
