"""FP8 (E4M3 / E5M2) rounding, per-tensor scaling and the FP8 GEMM, in fp64.

TEST INFRASTRUCTURE ONLY (see ``oracle/layer.py``).

The pages list FP8 training ("--fp8-hybrid", FP8 on Hopper, Ada and Blackwell
GPUs) without a recipe.  Readings:
  * Formats (OCP 8-bit floating point): E4M3 = sign, 4 exponent bits (bias 7),
    3 mantissa bits, no infinities, largest finite 448, smallest subnormal
    2^-9; E5M2 = sign, 5 exponent bits (bias 15), 2 mantissa bits, largest
    finite 57344, smallest subnormal 2^-16.
  * "hybrid": forward GEMM operands (activations and weights) in E4M3,
    gradient operands in E5M2.
  * Per-tensor current scaling: amax = max |x| over the whole tensor (all t
    partitions together), scale = fmt_max / amax in float32 (1 when amax = 0),
    q = fp8(float32(x * scale)) with round-to-nearest-even and saturation to
    +-fmt_max; the value q represents is q / scale.
  * An FP8 GEMM accumulates the products of the FP8 values exactly (fp32 on the
    GPU) and multiplies by descale = float32(1 / float32(scale_a * scale_b)),
    then applies the epilogue (bias, residual, GeLU) in fp32.
"""

from __future__ import annotations

import numpy as np

FORMATS = {
    # name: (exponent bits, mantissa bits, bias, largest finite)
    "e4m3": (4, 3, 7, 448.0),
    "e5m2": (5, 2, 15, 57344.0),
}


def decode(code, fmt):
    """The value of an 8-bit code (uint8 array) from the format's bit fields;
    NaN (and, for E5M2, +-inf) where the format defines them."""
    ebits, mbits, bias, _ = FORMATS[fmt]
    c = np.asarray(code, dtype=np.int64)
    sign = np.where(c >> 7, -1.0, 1.0)
    e = (c >> mbits) & ((1 << ebits) - 1)
    m = c & ((1 << mbits) - 1)
    sub = e == 0
    val = np.where(sub, m * 2.0 ** (1 - bias - mbits),
                   (1.0 + m / 2.0 ** mbits) * np.exp2(e.astype(np.float64) - bias))
    top = e == (1 << ebits) - 1
    if fmt == "e4m3":
        val = np.where(top & (m == (1 << mbits) - 1), np.nan, val)
    else:
        val = np.where(top & (m == 0), np.inf, val)
        val = np.where(top & (m != 0), np.nan, val)
    return sign * val


def round_to(v, fmt):
    """Round float values to the nearest FP8 value (ties to even), saturating
    to +-largest finite.  Returns float64 values on the FP8 grid."""
    ebits, mbits, bias, maxv = FORMATS[fmt]
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    emin = 1 - bias
    # exponent of the binade: frexp gives a = f * 2^x with f in [0.5, 1)
    _, x = np.frexp(np.where(a > 0, a, 1.0))
    e = np.maximum(x - 1, emin)
    quantum = np.exp2((e - mbits).astype(np.float64))
    r = np.round(a / quantum) * quantum          # numpy rounds halves to even
    r = np.minimum(r, maxv)
    return np.where(a > 0, np.sign(v) * r, 0.0 * v)


def quantize(x, fmt):
    """Per-tensor scaled FP8 of x: (q on the FP8 grid, scale as float32)."""
    _, _, _, maxv = FORMATS[fmt]
    x32 = np.asarray(x, dtype=np.float32)
    amax = np.float32(np.max(np.abs(x32))) if x32.size else np.float32(0)
    scale = np.float32(1.0) if amax == 0 else np.float32(maxv) / amax
    y = (x32 * scale).astype(np.float32)
    return round_to(y.astype(np.float64), fmt), scale


def descale(scale_a, scale_b):
    """The epilogue's factor: float32(1 / float32(scale_a * scale_b))."""
    return np.float64(np.float32(1.0) / (np.float32(scale_a) * np.float32(scale_b)))


def gemm(A, B, fmt_a="e4m3", fmt_b="e4m3", parts=1, epi=0, bias=None, R=None):
    """C[m][n] = epi(descale * sum_k qa[m][k] qb[n][k]) with A, B quantized per
    tensor; the t = parts partition partials are summed in order before the
    epilogue (which adds bias / residual or applies GeLU like gemm_partitioned).
    Returns (C, qa, qb, scale_a, scale_b)."""
    from .layer import gemm_partitioned
    qa, sa = quantize(A, fmt_a)
    qb, sb = quantize(B, fmt_b)
    acc = gemm_partitioned(qa, qb, parts) * descale(sa, sb)
    C = acc
    if epi in (1, 2, 3):
        C = C + np.asarray(bias, dtype=np.float64)[None, :]
    if epi == 2:
        C = C + np.asarray(R, dtype=np.float64)
    if epi == 3:
        from .layer import gelu
        C = gelu(C)
    return C, qa, qb, sa, sb
