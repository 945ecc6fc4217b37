"""GPU parity of the layer variants: Post-LN (against the oracle's Post-LN
layer) and selective recomputation (against the same layer without it).

Recomputation rebuilds the LayerNorm outputs from the saved inputs and
statistics with the forward's arithmetic, so every result that depends only on
them is bitwise equal; a = GeLU(z) is rebuilt from the stored (rounded) z,
which in bf16 moves dW_fc2 by bf16 rounding only (fp32 layers: bitwise)."""
import numpy as np
import pytest

import synthetic
from harness import (compare, make, rel_err, run_gpu, run_oracle, run_oracle_post_ln,
                     tolerance)

pytestmark = pytest.mark.gpu

SHAPES = {
    "d64": synthetic.tiny(h=128, heads=2, seq=128, batch=2, dtype="bf16", w_std=0.02,
                          out_std=0.01),
    "d96": synthetic.tiny(h=384, heads=4, seq=256, batch=1, dtype="bf16", w_std=0.02,
                          out_std=0.01),
    "d128": synthetic.tiny(h=256, heads=2, seq=256, batch=2, dtype="bf16", w_std=0.02,
                           out_std=0.01),
}


def _check_post_ln(shape, t, recompute=0):
    x, p, dy = make(shape, seed=4, affine=True)
    gpu = run_gpu(shape, x, p, dy, t, post_ln=1, recompute=recompute)
    ref = run_oracle_post_ln(shape, x, p, dy)
    errs = compare(gpu, ref, shape.dtype)
    # A row mean of h1 or h2 nearly cancels (x1 is normalized): its error, set by
    # the bf16 rounding of the row's elements, is measured against the size of
    # those elements rather than against the small means themselves.
    for i in (1, 2):
        k = f"s_mu{i}"
        errs[k] = float(np.max(np.abs(gpu[k] - ref[k])) / np.max(np.abs(ref[f"s_h{i}"])))
    bad = {k: v for k, v in errs.items() if not v <= tolerance(k, shape.dtype)}
    assert not bad, (bad, errs)
    assert "s_u1" not in gpu and "s_h1" in gpu
    return gpu


@pytest.mark.parametrize("t", [1, 2, 4])
def test_post_ln_fp32(t):
    _check_post_ln(synthetic.CONFIGS["A"], t)


@pytest.mark.parametrize("name,t", [("d64", 2), ("d96", 1), ("d128", 2)])
def test_post_ln_bf16(name, t):
    _check_post_ln(SHAPES[name], t)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("post_ln", [0, 1])
def test_recompute_matches_saving(dtype, post_ln):
    shape = synthetic.CONFIGS["A"] if dtype == "f32" else SHAPES["d128"]
    t = 2
    x, p, dy = make(shape, seed=6, affine=True)
    full = run_gpu(shape, x, p, dy, t, post_ln=post_ln)
    rc = run_gpu(shape, x, p, dy, t, post_ln=post_ln, recompute=1)
    gkeys = [k for k in full if k.startswith("d_")] + ["dx"]
    assert np.array_equal(rc["y"], full["y"])
    for k in gkeys:
        if k == "d_w_fc2" and dtype == "bf16":
            assert rel_err(rc[k], full[k]) <= 1e-2
        else:
            assert np.array_equal(rc[k], full[k]), k
    dropped = ["s_u1", "s_u2", "s_a"] if not post_ln else ["s_x1", "s_a"]
    for k in dropped:
        assert k in full and k not in rc, k
    # and against the oracle
    ref = run_oracle_post_ln(shape, x, p, dy) if post_ln else run_oracle(shape, x, p, dy)
    errs = compare(rc, ref, shape.dtype, keys=["y", "dx"] + [k for k in gkeys if k != "dx"])
    assert all(v <= tolerance(k, shape.dtype) for k, v in errs.items()), errs


def test_recompute_saves_memory_at_the_headline_shape():
    from tensor_model_transformer_gb300 import mtl
    s = synthetic.CONFIGS["D"]
    base = mtl.layer_desc(s.h, s.heads, s.seq, s.batch, s.ffn, 8, "bf16")
    rc = mtl.layer_desc(s.h, s.heads, s.seq, s.batch, s.ffn, 8, "bf16", recompute=1)
    n = s.batch * s.seq
    assert mtl.layer_sizes(base)[0] - mtl.layer_sizes(rc)[0] >= n * (2 * s.h + s.ffn) * 2
