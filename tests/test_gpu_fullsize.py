"""Parity at the workloads' full sizes, in the launch configuration bench.py
times (same layer descriptor and t).

The oracle cannot run a whole full-size layer in test time, so:
* forward and input gradient: batch element 0 of the full-batch GPU run is
  compared with the oracle run on that element alone (batch elements are
  independent in y and dx);
* parameter gradients: a batch-1 GPU run is compared with the same oracle run,
  and the full-batch GPU gradients must equal the sum of the per-element GPU
  gradients (the gradient of a sum over the batch), a property that holds at
  any size.
"""
import numpy as np
import pytest

import synthetic
from harness import compare, make, rel_err, run_gpu, run_oracle, tolerance

pytestmark = pytest.mark.gpu

GRADS = ["d_" + k for k in synthetic.PARAM_ORDER]


def full_size_check(cfg, t):
    shape = synthetic.CONFIGS[cfg]
    x, p, dy = make(shape)
    full = run_gpu(shape, x, p, dy, t, want_saved=False)
    one = shape.with_(batch=1)
    ref0 = run_oracle(one, x[:1], p, dy[:1])
    errs = {"y[0]": rel_err(full["y"][0], ref0["y"][0]),
            "dx[0]": rel_err(full["dx"][0], ref0["dx"][0])}
    assert errs["y[0]"] <= tolerance("y", "bf16"), errs
    assert errs["dx[0]"] <= tolerance("dx", "bf16"), errs
    acc = None
    for b in range(shape.batch):
        g = run_gpu(one, x[b:b + 1], p, dy[b:b + 1], t, want_saved=(b == 0))
        if b == 0:
            e0 = compare(g, ref0, "bf16", keys=GRADS + ["y", "dx", "s_qkv", "s_ctx", "s_lse",
                                                      "s_x1", "s_z", "s_a"])
            bad = {k: v for k, v in e0.items() if v > tolerance(k, "bf16")}
            assert not bad, bad
        acc = {k: g[k] for k in GRADS} if acc is None else {k: acc[k] + g[k] for k in GRADS}
    for k in GRADS:
        assert rel_err(full[k], acc[k]) <= 2e-3, k
    return errs


@pytest.mark.parametrize("cfg,t", [("B", 1), ("B", 2), ("C", 4), ("D", 8)])
def test_full_size(cfg, t):
    full_size_check(cfg, t)


@pytest.mark.slow
def test_full_size_large_layer():
    full_size_check("E", 8)


@pytest.mark.parametrize("cfg,t", [("D", 8)])
def test_full_size_with_dropout(cfg, t):
    """The headline workload with dropout (bench.py --p-drop 0.1): batch element 0
    of the full run against the oracle on that element (its masks depend only on
    its own batch index, 0 in both runs), and every parameter gradient of a
    batch-1 run against the oracle."""
    from harness import f32
    shape = synthetic.CONFIGS[cfg]
    drop = dict(p_attn=f32(0.1), p_hidden=f32(0.1), seed=1234)
    x, p, dy = make(shape)
    full = run_gpu(shape, x, p, dy, t, want_saved=False, drop=drop)
    one = shape.with_(batch=1)
    ref0 = run_oracle(one, x[:1], p, dy[:1], drop=drop)
    errs = {"y[0]": rel_err(full["y"][0], ref0["y"][0]),
            "dx[0]": rel_err(full["dx"][0], ref0["dx"][0])}
    assert errs["y[0]"] <= tolerance("y", "bf16"), errs
    assert errs["dx[0]"] <= tolerance("dx", "bf16"), errs
    g = run_gpu(one, x[:1], p, dy[:1], t, drop=drop)
    e0 = compare(g, ref0, "bf16", keys=GRADS + ["y", "dx", "s_ctx", "s_x1"])
    bad = {k: v for k, v in e0.items() if v > tolerance(k, "bf16")}
    assert not bad, bad
