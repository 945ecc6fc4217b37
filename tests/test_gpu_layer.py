"""GPU parity of the whole layer (forward, backward, saved intermediates)
through the C ABI against the fp64 oracle, element by element, on seeded inputs.

Tolerances (max|gpu - ref| / max|ref| per tensor): fp32 layers 1e-5; bf16
layers 1.5e-2 for forward outputs and 3e-2 for gradients."""
import numpy as np
import pytest

import synthetic
from harness import compare, make, run_gpu, run_oracle, tolerance

pytestmark = pytest.mark.gpu


def check(shape, t, affine, seed=0, batch=None):
    x, p, dy = make(shape, seed=seed, affine=affine, batch=batch)
    gpu = run_gpu(shape, x, p, dy, t)
    ref = run_oracle(shape, x, p, dy)
    errs = compare(gpu, ref, shape.dtype)
    bad = {k: v for k, v in errs.items() if not v <= tolerance(k, shape.dtype)}
    assert not bad, (bad, errs)
    return errs


@pytest.mark.parametrize("t", [1, 2, 4])
@pytest.mark.parametrize("affine", [False, True])
def test_config_a_fp32(t, affine):
    check(synthetic.CONFIGS["A"], t, affine)


BF16_SHAPES = {
    "d64": synthetic.tiny(h=128, heads=2, seq=128, batch=2, dtype="bf16", w_std=0.02,
                          out_std=0.01),
    "d96_ragged": synthetic.tiny(h=384, heads=4, seq=256, batch=1, dtype="bf16", w_std=0.02,
                                 out_std=0.01),
    "d128": synthetic.tiny(h=256, heads=2, seq=256, batch=2, dtype="bf16", w_std=0.02,
                           out_std=0.01),
}


@pytest.mark.parametrize("name,t", [("d64", 1), ("d64", 2), ("d96_ragged", 2), ("d96_ragged", 1),
                                    ("d128", 2)])
@pytest.mark.parametrize("affine", [False, True])
def test_bf16_small(name, t, affine):
    check(BF16_SHAPES[name], t, affine)


@pytest.mark.parametrize("t", [1, 2])
def test_config_b_batch1(t):
    check(synthetic.CONFIGS["B"], t, affine=False, batch=1)


def test_config_b_batch1_affine():
    check(synthetic.CONFIGS["B"], 2, affine=True, batch=1)


def test_bf16_deterministic():
    shape = BF16_SHAPES["d96_ragged"]
    x, p, dy = make(shape, affine=True)
    a, b = run_gpu(shape, x, p, dy, 2, runs=2, want_saved=False)
    for k in a:
        assert np.array_equal(a[k], b[k]), k


def test_bf16_causality_and_batch_independence():
    shape = BF16_SHAPES["d64"].with_(batch=3)
    x, p, dy = make(shape, affine=True)
    y0 = run_gpu(shape, x, p, dy, 2, want_saved=False)["y"]
    x2 = x.copy()
    j = 77
    x2[1, j] = synthetic.round_bf16(synthetic.round_f32(x2[1, j] + 0.5))
    y1 = run_gpu(shape, x2, p, dy, 2, want_saved=False)["y"]
    assert np.array_equal(y1[1, :j], y0[1, :j])
    assert not np.array_equal(y1[1, j], y0[1, j])
    assert np.array_equal(y1[0], y0[0]) and np.array_equal(y1[2], y0[2])


def test_bf16_identity_layer():
    shape = BF16_SHAPES["d64"]
    x, p, dy = make(shape, affine=True)
    for k in ("w_o", "b_o", "w_fc2", "b_fc2"):
        p[k] = np.zeros_like(p[k])
    y = run_gpu(shape, x, p, dy, 2, want_saved=False)["y"]
    assert np.array_equal(y, x.astype(np.float64))


def test_partitions_agree_across_t():
    shape = BF16_SHAPES["d64"]
    x, p, dy = make(shape, affine=True)
    a = run_gpu(shape, x, p, dy, 1, want_saved=False)
    b = run_gpu(shape, x, p, dy, 2, want_saved=False)
    for k in a:
        m = max(np.max(np.abs(a[k])), 1e-30)
        assert np.max(np.abs(a[k] - b[k])) / m < 1e-2, k
