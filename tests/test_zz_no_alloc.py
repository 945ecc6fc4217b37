"""The allocation-free bias gradient (mtl_bias_grad_noalloc).

Some callers cannot call cudaMalloc -- their device memory is planned up front
and owned by their own pool -- so they cannot hand the library a workspace.
This entry point computes the same fixed-order bias gradient that
mtl_layer_bwd writes for b_fc2 (the column sum of dy), with its scratch in a
static device array inside the library.  The GPU test compares it, through the
C ABI, with the b_fc2 gradient of the existing mtl_layer_bwd on two calls in a
row with different inputs (the second call must not see the first's scratch).
This file is collected last so that a failure here comes after every other test.
"""
import ctypes

import numpy as np
import pytest

import synthetic
from harness import make, to_device


def _layer_b_fc2_grad(shape, seed, t=2):
    """b_fc2 gradient from mtl_layer_bwd, and the dy it was computed from."""
    import torch
    from tensor_model_transformer_gb300 import mtl
    x, p, dy = make(shape, seed=seed, affine=True)
    desc = mtl.layer_desc(shape.h, shape.heads, shape.seq, shape.batch, shape.ffn, t, shape.dtype)
    w = {k: to_device(v, shape.dtype) for k, v in p.items()}
    xd, dyd = to_device(x, shape.dtype), to_device(dy, shape.dtype)
    saved, ws, grads = mtl.alloc_layer_buffers(desc)
    y = torch.empty_like(xd)
    dx = torch.empty_like(xd)
    mtl.layer_fwd(desc, w, xd, y, saved, ws)
    mtl.layer_bwd(desc, w, xd, saved, dyd, dx, grads, ws)
    mtl.layer_check(ws)
    torch.cuda.synchronize()
    return dyd, grads["b_fc2"].clone()


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_noalloc_bias_grad_matches_layer_backward(dtype):
    import torch
    from tensor_model_transformer_gb300 import mtl
    if dtype == "bf16":
        shape = synthetic.tiny(h=128, heads=2, seq=128, batch=2, dtype="bf16", w_std=0.02,
                               out_std=0.01)
    else:
        shape = synthetic.tiny(h=256, heads=4, seq=64, batch=3, dtype="f32", w_std=0.02,
                               out_std=0.01)
    for seed in (11, 12):   # two calls in a row, different inputs
        dyd, ref = _layer_b_fc2_grad(shape, seed)
        out = torch.full((shape.h,), float("nan"), dtype=torch.float32, device="cuda")
        rows = shape.batch * shape.seq
        mtl.bias_grad_noalloc(dtype, dyd, shape.h, rows, shape.h, out)
        torch.cuda.synchronize()
        got = out.cpu().numpy().astype(np.float64)
        want = ref.cpu().numpy().astype(np.float64)
        err = np.max(np.abs(got - want)) / max(np.max(np.abs(want)), 1e-30)
        assert err <= 1e-6, (seed, err)


def test_noalloc_bias_grad_rejects_oversize():
    # checked on the host before any CUDA call: no GPU needed
    from tensor_model_transformer_gb300 import build, mtl
    import os
    if not os.path.exists(mtl.LIB_PATH):
        build.build()
    L = mtl.lib()
    fake = 0x10000
    assert L.mtl_bias_grad_noalloc(1, fake, 16384 + 64, 256, 16384 + 64, fake, None) == 2
    assert L.mtl_bias_grad_noalloc(1, fake, 64, 256, 100, fake, None) == 1    # ld < cols
    assert L.mtl_bias_grad_noalloc(1, fake + 8, 64, 256, 64, fake, None) == 1  # misaligned
    assert L.mtl_bias_grad_noalloc(3, fake, 64, 256, 64, fake, None) == 1     # bad dtype
