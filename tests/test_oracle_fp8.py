"""Pins of the FP8 oracle (E4M3 / E5M2 rounding, per-tensor scaling, FP8 GEMM).

The bit-level decode and the rounding are checked against torch's float8
dtypes, an implementation independent of this one; saturation, the scaling
rule and the GEMM against what the format definitions fix."""
import numpy as np
import pytest

import oracle

FP8 = oracle.fp8


def _torch_dtype(fmt):
    torch = pytest.importorskip("torch")
    return torch, (torch.float8_e4m3fn if fmt == "e4m3" else torch.float8_e5m2)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_decode_table_matches_torch(fmt):
    torch, dt = _torch_dtype(fmt)
    codes = np.arange(256, dtype=np.uint8)
    ours = FP8.decode(codes, fmt)
    theirs = torch.from_numpy(codes).view(dt).to(torch.float64).numpy()
    same = (ours == theirs) | (np.isnan(ours) & np.isnan(theirs))
    assert same.all(), codes[~same]


def test_format_constants():
    vals = FP8.decode(np.arange(256, dtype=np.uint8), "e4m3")
    fin = vals[np.isfinite(vals)]
    assert fin.max() == 448.0 and np.min(fin[fin > 0]) == 2.0 ** -9
    assert np.isnan(vals).sum() == 2                      # S.1111.111
    vals = FP8.decode(np.arange(256, dtype=np.uint8), "e5m2")
    fin = vals[np.isfinite(vals)]
    assert fin.max() == 57344.0 and np.min(fin[fin > 0]) == 2.0 ** -16
    assert np.isinf(vals).sum() == 2 and np.isnan(vals).sum() == 6


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_rounding_matches_torch_in_range(fmt):
    """Random values across every binade, exact midpoints (ties to even) and
    their neighbours, all inside the finite range."""
    torch, dt = _torch_dtype(fmt)
    maxv = FP8.FORMATS[fmt][3]
    rng = np.random.default_rng(0)
    grid = np.unique(np.abs(FP8.decode(np.arange(256, dtype=np.uint8), fmt)))
    grid = grid[np.isfinite(grid)]
    mids = (grid[:-1] + grid[1:]) / 2
    x = np.concatenate([
        np.exp2(rng.uniform(-20, np.log2(maxv), 20000)) * rng.choice([-1, 1], 20000),
        mids, -mids, np.nextafter(mids, 0), np.nextafter(mids, np.inf), grid, -grid,
    ]).astype(np.float32)
    x = x[np.abs(x) <= maxv]
    ours = FP8.round_to(x.astype(np.float64), fmt)
    theirs = torch.from_numpy(x).to(dt).to(torch.float64).numpy()
    assert np.array_equal(ours, theirs)
    assert np.all(np.isin(np.abs(ours), grid))


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_saturation_and_error_bound(fmt):
    ebits, mbits, bias, maxv = FP8.FORMATS[fmt]
    assert FP8.round_to(np.array([1e9, -1e9, maxv * 1.04]), fmt).tolist() == [maxv, -maxv, maxv]
    rng = np.random.default_rng(1)
    x = np.exp2(rng.uniform(1 - bias, np.log2(maxv), 5000))   # normal range
    r = FP8.round_to(x, fmt)
    assert np.all(np.abs(r - x) <= 2.0 ** -(mbits + 1) * x * (1 + 1e-12))
    assert np.array_equal(FP8.round_to(r, fmt), r)             # idempotent
    assert np.all(np.diff(FP8.round_to(np.sort(x), fmt)) >= 0)  # monotone


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_quantize_scaling(fmt):
    maxv = FP8.FORMATS[fmt][3]
    rng = np.random.default_rng(2)
    x = (rng.standard_normal((64, 48)) * 3.0).astype(np.float32)
    q, s = FP8.quantize(x, fmt)
    assert s == np.float32(maxv) / np.float32(np.max(np.abs(x)))
    i = np.unravel_index(np.argmax(np.abs(x)), x.shape)
    assert abs(q[i]) == maxv                                  # amax lands on the top code
    assert np.max(np.abs(q)) == maxv
    back = q / np.float64(s)
    mbits = FP8.FORMATS[fmt][1]
    big = np.abs(x) * s >= 2.0 ** (1 - FP8.FORMATS[fmt][2])    # normal range after scaling
    assert np.all(np.abs(back - x)[big] <= 2.0 ** -(mbits + 1) * np.abs(x)[big] * 1.0001)
    z, s0 = FP8.quantize(np.zeros((3, 3)), fmt)
    assert s0 == 1.0 and not z.any()


def test_gemm_on_grid_inputs_is_exact():
    """Inputs already on the E4M3 grid with amax = 448 get scale 1: the FP8
    GEMM is then the plain GEMM of the inputs, for every epilogue."""
    rng = np.random.default_rng(3)
    grid = FP8.decode(np.arange(256, dtype=np.uint8), "e4m3")
    grid = grid[np.isfinite(grid)]
    A = rng.choice(grid, (32, 64))
    B = rng.choice(grid, (48, 64))
    A[0, 0], B[0, 0] = 448.0, -448.0
    bias = rng.standard_normal(48)
    R = rng.standard_normal((32, 48))
    C, qa, qb, sa, sb = FP8.gemm(A, B, parts=2, epi=2, bias=bias, R=R)
    assert sa == 1 and sb == 1 and np.array_equal(qa, A) and np.array_equal(qb, B)
    assert np.allclose(C, A @ B.T + bias + R, rtol=1e-13, atol=1e-9)
    C3, *_ = FP8.gemm(A, B, epi=3, bias=bias)
    assert np.allclose(C3, oracle.gelu(A @ B.T + bias), rtol=1e-12, atol=1e-9)


def test_gemm_descale_and_hybrid():
    """An E4M3 x E5M2 GEMM equals the product of the dequantized operands."""
    rng = np.random.default_rng(4)
    A = rng.standard_normal((16, 96))
    B = rng.standard_normal((24, 96)) * 1e-3
    C, qa, qb, sa, sb = FP8.gemm(A, B, "e4m3", "e5m2")
    ref = (qa / np.float64(sa)) @ (qb / np.float64(sb)).T
    assert np.max(np.abs(C - ref)) <= 1e-6 * np.max(np.abs(ref))
    assert np.max(np.abs(C - A @ B.T)) <= 0.15 * np.max(np.abs(A @ B.T))


def test_fp8_layer_forward():
    """fp8=True quantizes exactly the four GEMMs' operands: rebuilding the layer
    by hand from oracle.fp8.gemm gives the same y; and y stays within FP8
    error of the high-precision layer."""
    import synthetic
    shp = synthetic.tiny(h=64, heads=4, seq=16, batch=2, dtype="f32", w_std=0.1, out_std=0.1)
    x, p, _ = synthetic.make_layer(shp, seed=5, affine=True)
    y8, c = oracle.layer_fwd(p, x, shp.heads, fp8=True)
    y, _ = oracle.layer_fwd(p, x, shp.heads)
    xf = x.reshape(-1, shp.h).astype(np.float64)
    P = {k: np.asarray(v, np.float64) for k, v in p.items()}
    qkv = FP8.gemm(c["u1"], P["w_qkv"], epi=1, bias=P["b_qkv"])[0]
    assert np.array_equal(qkv, c["qkv"])
    x1 = FP8.gemm(c["ctx"], P["w_o"], epi=2, bias=P["b_o"], R=xf)[0]
    assert np.array_equal(x1, c["x1"])
    z = FP8.gemm(c["u2"], P["w_fc1"], epi=1, bias=P["b_fc1"])[0]
    assert np.array_equal(z, c["z"])
    y_hand = FP8.gemm(c["a"], P["w_fc2"], epi=2, bias=P["b_fc2"], R=x1)[0]
    assert np.array_equal(y_hand, y8.reshape(-1, shp.h))
    assert 0 < np.max(np.abs(y8 - y)) <= 0.05 * np.max(np.abs(y))


def test_fp8_hybrid_backward():
    """fp8=2: the backward's GEMMs quantize the gradient side to E5M2 and the
    other side to E4M3 (rebuilt by hand for two of them); the result stays
    within FP8 error of the high-precision backward of the same forward."""
    import synthetic
    shp = synthetic.tiny(h=64, heads=4, seq=16, batch=2, dtype="f32", w_std=0.1, out_std=0.1)
    x, p, dy = synthetic.make_layer(shp, seed=7, affine=True)
    _, c2 = oracle.layer_fwd(p, x, shp.heads, fp8=2)
    _, c1 = oracle.layer_fwd(p, x, shp.heads, fp8=1)
    dx2, g2, _ = oracle.layer_bwd(p, c2, dy)
    dx1, g1, _ = oracle.layer_bwd(p, c1, dy)
    dyf = np.asarray(dy, np.float64).reshape(-1, shp.h)
    assert np.array_equal(g2["w_fc2"], FP8.gemm(dyf.T, c2["a"].T, "e5m2", "e4m3")[0])
    assert np.array_equal(g2["b_fc2"], g1["b_fc2"])             # bias gradients unquantized
    for k in g1:
        scale = np.max(np.abs(g1[k]))
        assert np.max(np.abs(g2[k] - g1[k])) <= 0.25 * scale, k
    assert 0 < np.max(np.abs(dx2 - dx1)) <= 0.25 * np.max(np.abs(dx1))
