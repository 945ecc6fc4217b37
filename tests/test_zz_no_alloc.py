"""The allocation-free bias gradient (mtl_bias_grad_noalloc).

Some callers cannot call cudaMalloc -- their device memory is planned up front
and owned by their own pool -- so they cannot hand the library a workspace.
This entry point computes the same fixed-order bias gradient that
mtl_layer_bwd writes for b_fc2 (the column sum of dy), with its scratch in a
static device array inside the library.

The GPU tests call it through the C ABI and check it
* against the b_fc2 gradient of the existing mtl_layer_bwd, and against the
  float64 column sum of the host copy of dy, on two calls in a row with
  different inputs (the second call must not see the first's scratch);
* at the sizes that fill the static scratch (bf16, 4096 columns and enough rows
  for the most row blocks; the 16384-column limit), then on a smaller call
  after them, so stale partial sums of a larger call are never read;
* with rows = 0, which must write zeros.
This file is collected last so that a failure here comes after every other test.
"""
import numpy as np
import pytest

import synthetic
from harness import make, to_device

# max|gpu - ref| / max|ref| of a column sum: fp32 accumulation against float64
TOL = 1e-5


def _layer_b_fc2_grad(shape, seed, t=2):
    """b_fc2 gradient from mtl_layer_bwd, the device dy and the host dy."""
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
    return dyd, dy, grads["b_fc2"].clone()


def _rel(got, want):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    return float(np.max(np.abs(got - want)) / max(np.max(np.abs(want)), 1e-30))


def _noalloc(dtype, dyd, ld, rows, cols):
    import torch
    from tensor_model_transformer_gb300 import mtl
    out = torch.full((cols,), float("nan"), dtype=torch.float32, device="cuda")
    mtl.bias_grad_noalloc(dtype, dyd, ld, rows, cols, out)
    torch.cuda.synchronize()
    return out.cpu().numpy().astype(np.float64)


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_noalloc_bias_grad_matches_layer_backward(dtype):
    if dtype == "bf16":
        shape = synthetic.tiny(h=128, heads=2, seq=128, batch=2, dtype="bf16", w_std=0.02,
                               out_std=0.01)
    else:
        shape = synthetic.tiny(h=256, heads=4, seq=64, batch=3, dtype="f32", w_std=0.02,
                               out_std=0.01)
    for seed in (11, 12):   # two calls in a row, different inputs
        dyd, dy_host, ref = _layer_b_fc2_grad(shape, seed)
        rows = shape.batch * shape.seq
        got = _noalloc(dtype, dyd, shape.h, rows, shape.h)
        # the existing entry point's result for the same gradient
        assert _rel(got, ref.cpu().numpy()) <= TOL, seed
        # the float64 column sum of the host dy (what the oracle gives for b_fc2)
        want = dy_host.reshape(rows, shape.h).astype(np.float64).sum(axis=0)
        assert _rel(got, want) <= TOL, seed


def _host_and_device(rng, rows, ld, dtype):
    host = synthetic.to_storage(rng.standard_normal((rows, ld)), dtype)
    return host, to_device(host, dtype)


@pytest.mark.gpu
def test_noalloc_bias_grad_full_scratch_then_smaller():
    """The largest scratch uses, then a smaller call and rows = 0 after them."""
    rng = np.random.default_rng(7)
    cases = [
        ("bf16", 640, 4096, 4096),     # 512 row blocks x 4096 columns: the whole scratch
        ("bf16", 300, 16384, 16384),   # the column limit
        ("f32", 129, 16384, 16384),
        ("bf16", 37, 72, 64),          # smaller, after the larger calls; ld > cols
        ("f32", 5, 8, 8),
    ]
    for dtype, rows, ld, cols in cases:
        host, dev = _host_and_device(rng, rows, ld, dtype)
        got = _noalloc(dtype, dev, ld, rows, cols)
        want = host[:, :cols].astype(np.float64).sum(axis=0)
        assert _rel(got, want) <= TOL, (dtype, rows, cols, _rel(got, want))
    # rows = 0: the sum over no rows is zero in every column
    _, dev = _host_and_device(rng, 1, 256, "bf16")
    got = _noalloc("bf16", dev, 256, 0, 256)
    assert np.all(got == 0.0), got[:8]


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
    assert L.mtl_bias_grad_noalloc(1, fake, 64, -1, 64, fake, None) == 1      # negative rows
