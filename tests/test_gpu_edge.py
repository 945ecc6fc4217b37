"""Edge cases of the layer on the GPU, and the failure-detection path.

* empty batch: the forward enqueues nothing, the backward writes zero grads;
* t equal to the head count (one head per partition);
* one 128-token sequence (one attention block; GEMM M below the pair tile);
* an fp32 layer with a ragged sequence length and three partitions;
* a bounded device wait made to run out reports MTL_ERR_TIMEOUT and leaves
  the context usable (no fault, no hang).
"""
import numpy as np
import pytest

import synthetic
from harness import compare, make, run_gpu, run_oracle, tolerance

pytestmark = pytest.mark.gpu


def check(shape, t, affine=True, seed=0):
    x, p, dy = make(shape, seed=seed, affine=affine)
    gpu = run_gpu(shape, x, p, dy, t)
    ref = run_oracle(shape, x, p, dy)
    errs = compare(gpu, ref, shape.dtype)
    bad = {k: v for k, v in errs.items() if not v <= tolerance(k, shape.dtype)}
    assert not bad, (bad, errs)


def test_empty_batch():
    import torch
    from tensor_model_transformer_gb300 import mtl
    desc = mtl.layer_desc(128, 2, 128, 0, 512, 2, "bf16")
    saved, ws, grads = mtl.alloc_layer_buffers(desc)
    w = {k: torch.ones(v.shape, dtype=torch.bfloat16, device="cuda") for k, v in grads.items()}
    x = torch.empty((16,), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((16,), dtype=torch.bfloat16, device="cuda")
    for g in grads.values():
        g.fill_(7.0)
    mtl.layer_fwd(desc, w, x, y, saved, ws)
    mtl.layer_bwd(desc, w, x, saved, x, y, grads, ws)
    mtl.layer_check(ws)
    torch.cuda.synchronize()
    for k, g in grads.items():
        assert float(g.abs().max()) == 0.0, k


def test_one_head_per_partition():
    check(synthetic.tiny(h=256, heads=4, seq=128, batch=2, dtype="bf16", w_std=0.02,
                         out_std=0.01), t=4)


def test_single_block_sequence():
    check(synthetic.tiny(h=128, heads=2, seq=128, batch=1, dtype="bf16", w_std=0.02,
                         out_std=0.01), t=2)


def test_fp32_ragged_sequence():
    check(synthetic.tiny(h=192, heads=3, seq=100, batch=2, ffn=768, dtype="f32", w_std=0.02,
                       out_std=0.01), t=3)


def test_bounded_wait_times_out_and_context_survives():
    import torch
    from tensor_model_transformer_gb300 import mtl
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    mtl.selftest_wait_timeout(ws, 2_000_000)   # ~1 ms of SM clock
    with pytest.raises(mtl.MtlError) as ei:
        mtl.layer_check(ws)
    assert ei.value.status == 5                # MTL_ERR_TIMEOUT
    mtl.layer_check(ws)                        # the status word was reset
    # the context still runs a layer correctly
    check(synthetic.tiny(h=128, heads=2, seq=128, batch=1, dtype="bf16", w_std=0.02,
                         out_std=0.01), t=1)


def test_launch_failure_maps_to_cuda_error_and_context_survives():
    """A launch the runtime refuses (a block above the 1024-thread limit, checked
    on the host before anything runs) comes back as MTL_ERR_CUDA with the
    runtime's text, and the next layer call runs correctly."""
    from tensor_model_transformer_gb300 import mtl
    with pytest.raises(mtl.MtlError) as ei:
        mtl.selftest_launch_error()
    assert ei.value.status == 4                # MTL_ERR_CUDA
    text = mtl.lib().mtl_last_cuda_error().decode()
    assert text.startswith("selftest launch:") and len(text) > len("selftest launch: "), text
    check(synthetic.tiny(h=128, heads=2, seq=128, batch=1, dtype="bf16", w_std=0.02,
                         out_std=0.01), t=1)
    assert mtl.lib().mtl_last_cuda_error().decode() == ""
