"""GPU parity of the GEMM kernels (mtl_gemm through the C ABI) against the
oracle's partitioned GEMM, element by element, on seeded inputs.  Covers both
operand majors, ragged M / N / K tails, several partitions (the g / f sums) and
every fused epilogue, on the tcgen05 path (bf16) and the fp32 CUDA-core path."""
import numpy as np
import pytest

import oracle
import synthetic

pytestmark = pytest.mark.gpu

EPI_STORE, EPI_BIAS, EPI_BIAS_RESID, EPI_BIAS_GELU, EPI_DGELU = range(5)


def _dev(a, dtype):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()
    return t.to(torch.bfloat16) if dtype == "bf16" else t


def _host(t):
    return t.float().cpu().numpy().astype(np.float64)


def run_case(dtype, M, N, K, parts, a_k, b_k, epi, c_f32, seed=0, split=False, raw=False):
    """split: a workspace that lets the tiles of the last, partial wave be sliced;
    raw: also return the device output tensor."""
    import torch
    from tensor_model_transformer_gb300 import mtl
    rng = np.random.default_rng(seed)
    st = lambda a: synthetic.to_storage(a, dtype)  # noqa: E731
    A = st(rng.standard_normal((M, K)))
    B = st(rng.standard_normal((N, K)))
    bias = st(rng.standard_normal(N))
    R = st(rng.standard_normal((M, N)))
    Zin = st(rng.standard_normal((M, N)))
    Ad = _dev(A if a_k else A.T.copy(), dtype)
    Bd = _dev(B if b_k else B.T.copy(), dtype)
    lda = K if a_k else M
    ldb = K if b_k else N
    Cd = torch.zeros((M, N), dtype=torch.float32 if c_f32 else Ad.dtype, device="cuda")
    Zd = _dev(Zin, dtype) if epi == EPI_DGELU else torch.zeros((M, N), dtype=Ad.dtype, device="cuda")
    nws = mtl.gemm_ws_bytes(M, N) if split else 256
    ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
    mtl.gemm(dtype, M, N, K, parts, Ad, lda, a_k, Bd, ldb, b_k, epi, Cd, N, c_f32, ws,
             bias=_dev(bias, dtype), R=_dev(R, dtype), ldr=N, Z=Zd, ldz=N)
    mtl.layer_check(ws)
    torch.cuda.synchronize()
    if raw:
        return Cd.clone(), Zd.clone()
    if epi == EPI_BIAS_GELU:
        ref, zref = oracle.gemm_partitioned(A, B, parts, epi, bias=bias)
        return _host(Cd), ref, _host(Zd), zref
    ref = oracle.gemm_partitioned(A, B, parts, epi, bias=bias, R=R, Z=Zin)
    return _host(Cd), ref, None, None


def rel(a, b):
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-30))


def tol(dtype, c_f32):
    if dtype == "f32":
        return 2e-6
    return 2e-6 if c_f32 else 8e-3


@pytest.mark.parametrize("a_k,b_k", [(1, 1), (1, 0), (0, 0), (0, 1)])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_operand_majors_ragged(dtype, a_k, b_k):
    # M, N not multiples of the 128 x 256 tile; K spans several 64-deep blocks
    c, ref, _, _ = run_case(dtype, 296, 320, 256, 1, a_k, b_k, EPI_STORE, True)
    assert rel(c, ref) < tol(dtype, True)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_ragged_k(dtype):
    c, ref, _, _ = run_case(dtype, 128, 256, 200, 1, 1, 1, EPI_STORE, True)
    assert rel(c, ref) < tol(dtype, True)


@pytest.mark.parametrize("parts", [2, 4, 8])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_partition_sums(dtype, parts):
    c, ref, _, _ = run_case(dtype, 256, 512, 512, parts, 1, 0, EPI_STORE, True)
    assert rel(c, ref) < tol(dtype, True)


@pytest.mark.parametrize("epi", [EPI_BIAS, EPI_BIAS_RESID, EPI_BIAS_GELU, EPI_DGELU])
@pytest.mark.parametrize("parts", [1, 2])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_epilogues(dtype, epi, parts):
    c, ref, z, zref = run_case(dtype, 256, 384, 256, parts, 1, 1, epi, False)
    assert rel(c, ref) < tol(dtype, False)
    if z is not None:
        assert rel(z, zref) < tol(dtype, False)


@pytest.mark.parametrize("epi", [EPI_BIAS, EPI_BIAS_RESID, EPI_BIAS_GELU, EPI_DGELU])
@pytest.mark.parametrize("parts", [1, 2])
def test_epilogues_fp32_output(epi, parts):
    # every fused epilogue with an fp32 C on the tensor-core path; N = 336 ends
    # in a half chunk (whole chunks leave through TMA stores, the last one
    # element by element) and M = 296 in a partial tile
    c, ref, z, zref = run_case("bf16", 296, 336, 256, parts, 1, 1, epi, True)
    assert rel(c, ref) < 2e-6
    if z is not None:
        assert rel(z, zref) < tol("bf16", False)


def test_many_tiles_per_cta():
    # more tiles than SMs: the persistent loop and the TMEM double buffer cycle
    c, ref, _, _ = run_case("bf16", 4096, 2048, 512, 1, 1, 1, EPI_STORE, True)
    assert rel(c, ref) < 2e-6
    c, ref, _, _ = run_case("bf16", 4096, 2048, 512, 4, 1, 0, EPI_BIAS_RESID, False)
    assert rel(c, ref) < 8e-3


def test_gemm_is_deterministic():
    a = run_case("bf16", 1024, 768, 1024, 4, 1, 0, EPI_STORE, True, seed=3)[0]
    b = run_case("bf16", 1024, 768, 1024, 4, 1, 0, EPI_STORE, True, seed=3)[0]
    assert np.array_equal(a, b)


@pytest.mark.parametrize("epi", [EPI_BIAS_GELU, EPI_DGELU])
def test_gelu_epilogue_accuracy(epi):
    """GeLU and GeLU' of the fused epilogues against the exact functions.  The
    fp32 GEMM with one nonzero product per output (A[:, 0] = 1) puts a known
    value z into every accumulator (EPI_BIAS_GELU: B[n, 0] = z_n; EPI_DGELU: the
    product is 1 and Z holds z), so C is the epilogue's function of z alone.
    Bound: 6e-7 * max(1, |z|) absolute (the erfc approximation's 1.5e-7 on erf,
    halved for Phi, plus fp32 rounding of a few operations)."""
    import torch
    from tensor_model_transformer_gb300 import mtl
    from scipy.special import erf
    M, N, K = 64, 4096, 16
    z = np.concatenate([np.linspace(-9.0, 9.0, N - 8),
                        [0.0, 1e-3, -1e-3, 0.5, -0.5, 30.0, -30.0, 3.0]]).astype(np.float32)
    A = np.zeros((M, K), np.float32)
    A[:, 0] = 1.0
    B = np.zeros((N, K), np.float32)
    B[:, 0] = z if epi == EPI_BIAS_GELU else 1.0
    Zd = torch.from_numpy(np.broadcast_to(z, (M, N)).copy()).cuda()
    Cd = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    mtl.gemm("f32", M, N, K, 1, _dev(A, "f32"), K, 1, _dev(B, "f32"), K, 1, epi, Cd, N, True, ws,
             bias=torch.zeros(N, dtype=torch.float32, device="cuda"), Z=Zd, ldz=N)
    mtl.layer_check(ws)
    torch.cuda.synchronize()
    c = _host(Cd)
    zz = z.astype(np.float64)
    cdf = 0.5 * (1.0 + erf(zz / np.sqrt(2.0)))
    pdf = np.exp(-0.5 * zz * zz) / np.sqrt(2.0 * np.pi)
    want = zz * cdf if epi == EPI_BIAS_GELU else cdf + zz * pdf
    err = np.abs(c - want[None, :]) / np.maximum(1.0, np.abs(zz))[None, :]
    assert float(err.max()) <= 6e-7, (float(err.max()), float(zz[np.argmax(err.max(axis=0))]))
    if epi == EPI_BIAS_GELU:                  # the saved pre-activation is z itself
        assert np.array_equal(_host(Zd)[0], zz)


# Tail slices: 90 or 160 output tiles of 256 x 256 leave a partial last wave
# over the SM pairs, so each of its tiles is cut into equal K slices (runs of
# K-blocks, or of partitions) computed on separate pairs, whose fp32 partials
# are added in slice order before the epilogue.  Ragged M and N.
SPLIT_SHAPES = [
    # M, N, K, parts (tiles of at least 48 K-blocks of 128 are sliced)
    (2550, 2296, 6144, 1),    # 14 tail tiles, 5 slices of 9-10 K-blocks
    (2550, 2304, 6144, 8),    # partition sums: 5 slices of 1-2 partitions
    (4096, 2560, 6144, 2),    # 160 tiles: two whole waves, then 2 slices
    (4096, 2560, 8192, 1),    # 8 tail tiles, 9 slices of 7-8 K-blocks
]


@pytest.mark.parametrize("M,N,K,parts", SPLIT_SHAPES)
@pytest.mark.parametrize("epi,c_f32", [(EPI_STORE, True), (EPI_BIAS, False),
                                       (EPI_BIAS_RESID, False), (EPI_BIAS_GELU, False),
                                       (EPI_DGELU, False), (EPI_BIAS_RESID, True)])
def test_tail_slices(M, N, K, parts, epi, c_f32):
    import torch
    from tensor_model_transformer_gb300 import mtl
    assert mtl.gemm_ws_bytes(M, N) > 256            # this shape slices its tail tiles
    c, ref, z, zref = run_case("bf16", M, N, K, parts, 1, 1, epi, c_f32, seed=3, split=True)
    # fp32 outputs: the fp32 accumulation error grows with K (the other tests'
    # 2e-6 holds up to K = 1024; these shapes go to 8192)
    t32 = 2e-6 * max(1.0, K / 1024)
    assert rel(c, ref) < (t32 if c_f32 else tol("bf16", False)), rel(c, ref)
    if epi == EPI_BIAS_GELU:
        assert rel(z, zref) < tol("bf16", False)
    # bitwise reproducible; equal to the unsliced launch up to fp32 rounding
    c1, _ = run_case("bf16", M, N, K, parts, 1, 1, epi, c_f32, seed=3, split=True, raw=True)
    c2, _ = run_case("bf16", M, N, K, parts, 1, 1, epi, c_f32, seed=3, split=True, raw=True)
    assert torch.equal(c1, c2)
    c0, _ = run_case("bf16", M, N, K, parts, 1, 1, epi, c_f32, seed=3, split=False, raw=True)
    d = (c1.float() - c0.float()).abs().max().item() / max(c0.float().abs().max().item(), 1e-30)
    assert d < (t32 if c_f32 else 8e-3), d


def test_tail_slices_mn_major():
    """Both operands MN-major (the weight-gradient form), sliced tail tiles."""
    c, ref, _, _ = run_case("bf16", 2304, 2560, 6144, 1, 0, 0, EPI_STORE, True, seed=5, split=True)
    assert rel(c, ref) < 2e-6 * 6144 / 1024
