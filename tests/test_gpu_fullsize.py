"""Parity at the workloads' full sizes, in the launch configuration bench.py
times (same layer descriptor), and at every partition count t in {1, 2, 4, 8}
of the two largest layers.

Every output of the full-batch GPU run -- y, dx, all twelve parameter
gradients and the saved intermediates -- is compared element by element with
the oracle run on the same full batch.  The fused-QKV tensors are judged per
head and per Q/K/V block (harness.compare).

t changes the kernels that run (the K partition length decides between the
2-CTA pair GEMM and the single-CTA GEMM, and how many fp32 partials the
row-parallel epilogues sum in order) but not the result beyond rounding (the
column / row split identity of page "Megatron-LM: GPU-Cluster Training
Parallelism", section "Paper 1: The f/g Conjugate Operators"), so one oracle
run of a workload serves all of its t.  The tests are ordered by workload and
the oracle result of the previous workload is dropped before the next one is
computed, so the host holds one workload's float64 tensors at a time.
"""
import gc

import numpy as np
import pytest

import synthetic
from harness import compare, make, rel_err, run_gpu, run_oracle, tolerance

pytestmark = pytest.mark.gpu

GRADS = ["d_" + k for k in synthetic.PARAM_ORDER]

_REF = {}


def _oracle(cfg):
    """(shape, x, p, dy, oracle outputs) of a workload's full batch, cached for
    the tests of that workload only."""
    if cfg not in _REF:
        _REF.clear()
        gc.collect()
        shape = synthetic.CONFIGS[cfg]
        x, p, dy = make(shape)
        _REF[cfg] = (shape, x, p, dy, run_oracle(shape, x, p, dy))
    return _REF[cfg]


def full_batch_check(cfg, t):
    shape, x, p, dy, ref = _oracle(cfg)
    gpu = run_gpu(shape, x, p, dy, t, want_saved=True)
    errs = compare(gpu, ref, "bf16")
    del gpu
    bad = {k: v for k, v in errs.items() if v > tolerance(k, "bf16")}
    assert not bad, (cfg, t, bad)
    # every output was compared
    assert set(GRADS) | {"y", "dx", "s_u1", "s_qkv", "s_ctx", "s_lse", "s_x1", "s_u2", "s_z",
                         "s_a"} <= set(errs), sorted(errs)
    return errs


# ordered by workload so that each oracle result is computed once
FULL = [("B", 1), ("B", 2), ("C", 4), ("D", 8), ("D", 1), ("D", 2), ("D", 4)]


@pytest.mark.parametrize("cfg,t", FULL)
def test_full_batch(cfg, t):
    full_batch_check(cfg, t)


@pytest.mark.slow
@pytest.mark.parametrize("t", [8, 1, 2, 4])
def test_full_batch_large_layer(t):
    full_batch_check("E", t)


@pytest.fixture(scope="module", autouse=True)
def _drop_oracle_results():
    yield
    _REF.clear()
    gc.collect()


@pytest.mark.parametrize("cfg,t", [("D", 8)])
def test_full_size_with_dropout(cfg, t):
    """The headline workload with dropout (bench.py --p-drop 0.1): batch element 0
    of the full run against the oracle on that element (its masks depend only on
    its own batch index, 0 in both runs), and every parameter gradient of a
    batch-1 run against the oracle."""
    from harness import f32
    _REF.clear()
    gc.collect()
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
