"""Seeded synthetic inputs for one pre-LN GPT layer.

This module draws random numbers and rounds them to the storage dtype. It holds
none of the layer's arithmetic, and it is the only code that both the fp64 oracle
(through the tests) and the CUDA library (through the tests and the benchmark)
are fed from.

Recipe
------
* Generator: ``numpy.random.Generator(PCG64(seed))`` with ``standard_normal``
  in float64, drawn in a fixed order: x, w_qkv, b_qkv, w_o, b_o, w_fc1, b_fc1,
  w_fc2, b_fc2, ln1_g, ln1_b, ln2_g, ln2_b.  The upstream gradient dy comes from
  a second generator seeded with ``seed + 1``.
* Scales: x ~ N(0, 1); w_qkv, w_fc1 ~ N(0, w_std); w_o, w_fc2 ~ N(0, out_std)
  (the scaled init of the residual-output projections used for GPT-2-style
  models); biases 0, LN gamma 1, beta 0.  With ``affine=True`` the biases are
  N(0, 0.02), gamma 1 + N(0, 0.1), beta N(0, 0.1), so the bias and affine code
  paths carry non-trivial values.  The same normal draws are consumed either
  way, so the weights do not change between the two variants.
* Rounding: values are rounded to float32 (round to nearest even), then, for
  bf16 layers, to bf16 (round to nearest even).  Both sides read the rounded
  values: the oracle as exact float64 numbers, the GPU as its storage dtype.

Layouts: x, dy are [batch, seq, h] row-major; w_qkv is [3h, h] whose rows are
head-interleaved (head-major, then Q/K/V, then the d_h channels of the head);
w_o is [h, h]; w_fc1 is [ffn, h]; w_fc2 is [h, ffn]; all weights [out, in].
"""

from __future__ import annotations

import dataclasses
import math

import numpy as np

PARAM_ORDER = ("w_qkv", "b_qkv", "w_o", "b_o", "w_fc1", "b_fc1", "w_fc2",
               "b_fc2", "ln1_g", "ln1_b", "ln2_g", "ln2_b")


@dataclasses.dataclass(frozen=True)
class LayerShape:
    """Shape and init of one layer workload."""
    name: str
    dtype: str          # "f32" or "bf16"
    h: int
    heads: int
    seq: int
    batch: int
    ffn: int
    t: tuple            # partition counts the workload is run with
    w_std: float
    out_std: float

    @property
    def d_head(self) -> int:
        return self.h // self.heads

    @property
    def n(self) -> int:
        return self.batch * self.seq

    def with_(self, **kw) -> "LayerShape":
        return dataclasses.replace(self, **kw)


# The five workloads: a small fp32 case the oracle finishes in seconds, then
# layers shaped like the 355M, 4.2B and 8.3B GPT models and one large-model layer.
CONFIGS = {
    "A": LayerShape("fp32 h256 H4 s128 b2", "f32", 256, 4, 128, 2, 1024, (2, 1, 4),
                    0.02, 0.02 / math.sqrt(2 * 2)),
    "B": LayerShape("355M-shape h1024 H16 s1024 b8", "bf16", 1024, 16, 1024, 8, 4096, (1, 2),
                    0.02, 0.02 / math.sqrt(48)),
    "C": LayerShape("4.2B-shape h2304 H24 s1024 b8", "bf16", 2304, 24, 1024, 8, 9216, (4,),
                    0.02, 0.02 / math.sqrt(128)),
    "D": LayerShape("8.3B-shape h3072 H32 s1024 b16", "bf16", 3072, 32, 1024, 16, 12288, (8,),
                    0.02, 0.02 / math.sqrt(144)),
    "E": LayerShape("large h12288 H96 s2048 b2", "bf16", 12288, 96, 2048, 2, 49152, (8,),
                    0.006, 0.006 / math.sqrt(192)),
}


def round_f32(a: np.ndarray) -> np.ndarray:
    return np.asarray(a, dtype=np.float64).astype(np.float32)


def round_bf16(a32: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); returns float32."""
    a32 = np.ascontiguousarray(a32, dtype=np.float32)
    b = a32.view(np.uint32).astype(np.uint64)
    lsb = (b >> np.uint64(16)) & np.uint64(1)
    b = (b + np.uint64(0x7FFF) + lsb) & np.uint64(0xFFFF0000)
    return b.astype(np.uint32).view(np.float32).reshape(a32.shape)


def to_storage(a: np.ndarray, dtype: str) -> np.ndarray:
    """float64 draw -> float32 array holding values exactly representable in `dtype`."""
    a32 = round_f32(a)
    if dtype == "bf16":
        return round_bf16(a32)
    if dtype == "f32":
        return a32
    raise ValueError(dtype)


def _normal(rng: np.random.Generator, shape, std: float, dtype: str,
            offset: float = 0.0, chunk: int = 1 << 24) -> np.ndarray:
    """Draw N(offset, std) of `shape` in float64 chunks, rounded to `dtype`."""
    size = int(np.prod(shape))
    out = np.empty(size, dtype=np.float32)
    for lo in range(0, size, chunk):
        hi = min(size, lo + chunk)
        v = rng.standard_normal(hi - lo) * std + offset
        out[lo:hi] = to_storage(v, dtype)
    return out.reshape(shape)


def make_layer(shape: LayerShape, seed: int = 0, affine: bool = False,
               batch: int | None = None):
    """Return (x, params, dy) as float32 arrays holding storage-dtype values.

    `batch` overrides the number of sequences drawn (the weights are drawn
    first-come in the fixed order, so they are the same for any batch only if
    x has the same size; a reduced batch draws a different x).
    """
    b = shape.batch if batch is None else batch
    h, f, dt = shape.h, shape.ffn, shape.dtype
    rng = np.random.Generator(np.random.PCG64(seed))
    x = _normal(rng, (b, shape.seq, h), 1.0, dt)
    p = {}
    bias_std = 0.02 if affine else 0.0
    p["w_qkv"] = _normal(rng, (3 * h, h), shape.w_std, dt)
    p["b_qkv"] = _normal(rng, (3 * h,), bias_std, dt)
    p["w_o"] = _normal(rng, (h, h), shape.out_std, dt)
    p["b_o"] = _normal(rng, (h,), bias_std, dt)
    p["w_fc1"] = _normal(rng, (f, h), shape.w_std, dt)
    p["b_fc1"] = _normal(rng, (f,), bias_std, dt)
    p["w_fc2"] = _normal(rng, (h, f), shape.out_std, dt)
    p["b_fc2"] = _normal(rng, (h,), bias_std, dt)
    g_std, beta_std = (0.1, 0.1) if affine else (0.0, 0.0)
    p["ln1_g"] = _normal(rng, (h,), g_std, dt, offset=1.0)
    p["ln1_b"] = _normal(rng, (h,), beta_std, dt)
    p["ln2_g"] = _normal(rng, (h,), g_std, dt, offset=1.0)
    p["ln2_b"] = _normal(rng, (h,), beta_std, dt)
    rng_dy = np.random.Generator(np.random.PCG64(seed + 1))
    dy = _normal(rng_dy, (b, shape.seq, h), 1.0, dt)
    return x, p, dy


def tiny(h=64, heads=2, seq=128, batch=2, ffn=None, dtype="bf16", t=(1,),
         w_std=0.05, out_std=0.05, name=None) -> LayerShape:
    """A small custom shape for unit tests."""
    ffn = 4 * h if ffn is None else ffn
    return LayerShape(name or f"tiny h{h} H{heads} s{seq} b{batch}", dtype, h, heads,
                      seq, batch, ffn, tuple(t), w_std, out_std)
