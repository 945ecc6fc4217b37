"""Causal attention alone through the C ABI against the oracle, on random inputs.

The shapes give the persistent kernels several work items per CTA (so barrier
phases carry across items, and one-block items run between long ones),
sequences whose last 256-query pair has a single 128-row tile (seq % 256 ==
128), every supported head size, and logits large enough that the running row
maximum jumps and the accumulator is rescaled.
"""
import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.gpu

# batch, seq, heads, d, logit amplitude
CASES = [
    (4, 384, 40, 96, 1.0),
    (2, 640, 20, 64, 1.0),
    (1, 1024, 40, 128, 1.0),
    (2, 384, 24, 96, 4.0),
    (1, 256, 160, 64, 2.0),
    # long items next to one-block items, ~10 items per CTA (the large layer's shape)
    (1, 2048, 96, 128, 0.02),
]


def _bf16(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(
        torch.bfloat16).float().numpy().astype(np.float64)


def _run(batch, seq, heads, d, qkv, dctx):
    import torch
    from tensor_model_transformer_gb300 import mtl
    from harness import to_device, to_np
    tq = to_device(qkv, "bf16")
    ctx = torch.empty((batch * seq, heads * d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((batch, heads, seq), dtype=torch.float32, device="cuda")
    ws = torch.empty(mtl.attention_ws_bytes(batch, seq, heads), dtype=torch.uint8, device="cuda")
    mtl.attention_fwd("bf16", batch, seq, heads, d, tq, ctx, lse, ws)
    mtl.layer_check(ws)
    tdo = to_device(dctx, "bf16")
    dqkv = torch.empty_like(tq)
    mtl.attention_bwd("bf16", batch, seq, heads, d, tq, ctx, lse, tdo, dqkv, ws)
    mtl.layer_check(ws)
    torch.cuda.synchronize()
    return to_np(ctx), to_np(lse), to_np(dqkv)


@pytest.mark.parametrize("batch,seq,heads,d,amp", CASES)
def test_attention_random(batch, seq, heads, d, amp):
    from harness import TOL, rel_err, rel_err_qkv
    rng = np.random.default_rng(seq * 7 + d)
    qkv = _bf16(rng.standard_normal((batch * seq, 3 * heads * d)) * np.sqrt(amp))
    dctx = _bf16(rng.standard_normal((batch * seq, heads * d)))
    ctx_g, lse_g, dqkv_g = _run(batch, seq, heads, d, qkv, dctx)
    ctx_r, lse_r, probs = oracle.multihead_fwd(qkv, batch, seq, heads, d)
    dqkv_r = oracle.multihead_bwd(qkv, ctx_r, probs, dctx, batch, seq, heads, d)
    assert rel_err(ctx_g.reshape(ctx_r.shape), ctx_r) <= TOL["bf16"]["fwd"]
    assert np.max(np.abs(lse_g.reshape(lse_r.shape) - lse_r) / np.maximum(1.0, np.abs(lse_r))) < 1e-3
    # dQ, dK and dV of every head are judged against their own scale: with a
    # near-uniform softmax (amp 0.02) dQ and dK are ~70x smaller than dV
    assert rel_err_qkv(dqkv_g.reshape(dqkv_r.shape), dqkv_r, 1, heads) <= TOL["bf16"]["bwd"]
