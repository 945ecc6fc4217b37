"""Host-only checks of the C ABI: the library loads, exports every declared
symbol, and rejects bad arguments before touching the GPU.  No GPU needed."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def mtl():
    from tensor_model_transformer_gb300 import build, mtl as m
    if not os.path.exists(m.LIB_PATH):
        build.build()
    m.lib()
    return m


def declared_functions():
    src = open(os.path.join(ROOT, "include", "mtl.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mtl_[a-z_0-9]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(mtl):
    names = declared_functions()
    assert "mtl_layer_fwd" in names and "mtl_layer_bwd" in names
    lib = ctypes.CDLL(mtl.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(mtl):
    for s in range(7):
        assert mtl.lib().mtl_status_str(s)


def good_desc(mtl, **kw):
    d = dict(h=256, heads=4, seq=128, batch=2, ffn=1024, t=2, dtype="bf16")
    d.update(kw)
    return mtl.layer_desc(**d)


@pytest.mark.parametrize("kw,status", [
    (dict(h=0), 1), (dict(heads=0), 1), (dict(seq=0), 1), (dict(t=0), 1),
    (dict(h=250), 1),                     # heads does not divide h
    (dict(t=3), 1),                       # t does not divide heads
    (dict(ffn=1000, t=8), 1),             # t does not divide ffn
    (dict(h=128, heads=4), 2),            # d = 32 unsupported
    (dict(seq=100), 2),                   # bf16 needs seq % 128 == 0
    (dict(h=384, heads=4, ffn=1536, t=4), 2),  # h/t = 96 not a multiple of 64
    (dict(dtype=7), 1),
])
def test_layer_sizes_rejects(mtl, kw, status):
    if "dtype" in kw and kw["dtype"] == 7:
        d = good_desc(mtl)
        d.dtype = 7
    else:
        d = good_desc(mtl, **kw)
    s, w = ctypes.c_size_t(), ctypes.c_size_t()
    assert mtl.lib().mtl_layer_sizes(ctypes.byref(d), ctypes.byref(s), ctypes.byref(w)) == status


def test_causal_required(mtl):
    d = good_desc(mtl)
    d.causal = 0
    assert mtl.lib().mtl_layer_sizes(ctypes.byref(d), None, None) == 2


def test_fp32_path_accepts_small_shapes(mtl):
    d = good_desc(mtl, dtype="f32", seq=100, h=192, heads=3, ffn=300, t=3)
    saved, ws = mtl.layer_sizes(d)
    assert saved > 0 and ws > 0


def test_saved_layout_is_aligned_and_sized(mtl):
    d = good_desc(mtl)
    lay = mtl.layer_saved_layout(d)
    n, h, f = 256, 256, 1024
    assert all(v % 256 == 0 for v in lay.values())
    assert lay["qkv"] - lay["u1"] >= n * h * 2
    assert lay["a"] - lay["z"] >= n * f * 2
    assert lay["total"] >= lay["a"] + n * f * 2
    assert lay["total"] == mtl.layer_sizes(d)[0]


FAKE = 0x10000  # an aligned, never dereferenced host-side stand-in


def _weights(mtl, base=FAKE):
    return mtl.Weights(*[base + 256 * i for i in range(12)])


def _grads(mtl, base=FAKE):
    return mtl.Grads(*[base + 256 * i for i in range(12)])


def test_fwd_rejects_null_and_misaligned_pointers(mtl):
    d = good_desc(mtl)
    _, ws_b = mtl.layer_sizes(d)
    w = _weights(mtl)
    L = mtl.lib()
    ok = (FAKE, FAKE + 4096, FAKE + 8192, FAKE + 12288)
    assert L.mtl_layer_fwd(ctypes.byref(d), ctypes.byref(w), None, ok[1], ok[2], ok[3], ws_b, None) == 1
    assert L.mtl_layer_fwd(ctypes.byref(d), ctypes.byref(w), ok[0] + 8, ok[1], ok[2], ok[3], ws_b,
                           None) == 1
    assert L.mtl_layer_fwd(ctypes.byref(d), None, ok[0], ok[1], ok[2], ok[3], ws_b, None) == 1
    w.b_o = None
    assert L.mtl_layer_fwd(ctypes.byref(d), ctypes.byref(w), *ok, ws_b, None) == 1
    # y aliasing x
    w = _weights(mtl)
    assert L.mtl_layer_fwd(ctypes.byref(d), ctypes.byref(w), ok[0], ok[0], ok[2], ok[3], ws_b,
                           None) == 1


def test_fwd_and_bwd_reject_small_workspace(mtl):
    d = good_desc(mtl)
    _, ws_b = mtl.layer_sizes(d)
    w, g = _weights(mtl), _grads(mtl)
    L = mtl.lib()
    assert L.mtl_layer_fwd(ctypes.byref(d), ctypes.byref(w), FAKE, FAKE + 4096, FAKE + 8192,
                           FAKE + 12288, ws_b - 1, None) == 3
    assert L.mtl_layer_bwd(ctypes.byref(d), ctypes.byref(w), FAKE, FAKE + 4096, FAKE + 8192,
                           FAKE + 12288, ctypes.byref(g), FAKE + 16384, ws_b - 1, None) == 3


def test_bwd_rejects_null_grad(mtl):
    d = good_desc(mtl)
    _, ws_b = mtl.layer_sizes(d)
    w, g = _weights(mtl), _grads(mtl)
    g.ln2_b = None
    assert mtl.lib().mtl_layer_bwd(ctypes.byref(d), ctypes.byref(w), FAKE, FAKE + 4096,
                                   FAKE + 8192, FAKE + 12288, ctypes.byref(g), FAKE + 16384,
                                   ws_b, None) == 1


def test_gemm_rejects_bad_arguments(mtl):
    L = mtl.lib()
    args = dict(dtype=1, M=128, N=128, K=128, parts=1, A=FAKE, lda=128, ak=1, B=FAKE, ldb=128,
                bk=1, epi=0, bias=None, R=None, ldr=0, Z=None, ldz=0, C=FAKE, ldc=128, cf=1,
                ws=FAKE, wsb=256)

    def call(**kw):
        a = dict(args)
        a.update(kw)
        return L.mtl_gemm(a["dtype"], a["M"], a["N"], a["K"], a["parts"], a["A"], a["lda"],
                          a["ak"], a["B"], a["ldb"], a["bk"], a["epi"], a["bias"], a["R"],
                          a["ldr"], a["Z"], a["ldz"], a["C"], a["ldc"], a["cf"], a["ws"],
                          a["wsb"], None)

    assert call(parts=3) == 1                  # parts must divide K
    assert call(epi=9) == 1
    assert call(epi=1) == 1                    # bias missing
    assert call(A=FAKE + 2) == 1               # misaligned
    assert call(wsb=16) == 3
    assert call(lda=64) == 1                   # lda < K
    assert call(ldc=8) == 1
    assert call(parts=2, K=192, lda=192, ldb=192) == 2  # bf16: K/parts must be a multiple of 64


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    from tensor_model_transformer_gb300 import mtl as m
    monkeypatch.setattr(m, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(m, "_lib", None)
    with pytest.raises(RuntimeError):
        m.lib()


def test_dropout_probabilities_validated(mtl):
    for kw in (dict(p_attn=1.0), dict(p_attn=-0.1), dict(p_hidden=1.0), dict(p_hidden=-1e-3),
               dict(p_attn=float("nan")), dict(p_hidden=float("nan"))):
        d = good_desc(mtl, **kw)
        assert mtl.lib().mtl_layer_sizes(ctypes.byref(d), None, None) == 1, kw
    d0, d1 = good_desc(mtl), good_desc(mtl, p_attn=0.1, p_hidden=0.1, seed=(1 << 63) + 5)
    assert d1.seed == (1 << 63) + 5
    s0, w0 = mtl.layer_sizes(d0)
    s1, w1 = mtl.layer_sizes(d1)
    # saved grows by the attention keep bits (2 KB per causal 128 x 128 tile of
    # each (batch, head)); the workspace holds one dropped-out [n][h] gradient
    tiles = 2 * 4 * 1                       # batch 2, heads 4, seq 128: one tile
    assert mtl.attention_mask_bytes("bf16", 2, 128, 4, 0.1) == tiles * 2048
    assert mtl.attention_mask_bytes("bf16", 2, 128, 4, 0.0) == 0
    assert mtl.attention_mask_bytes("f32", 2, 128, 4, 0.1) == 0
    assert mtl.attention_mask_bytes("bf16", 1, 512, 1, 0.1) == 10 * 2048
    lay = mtl.layer_saved_layout(d1)
    assert lay["total"] - lay["attn_mask"] >= tiles * 2048 and s1 == lay["total"]
    assert s1 == s0 + tiles * 2048 and w1 >= w0 + 256 * 256 * 2
    # fp32 layers redraw the attention mask: nothing saved
    f0, f1 = good_desc(mtl, dtype="f32"), good_desc(mtl, dtype="f32", p_attn=0.1)
    assert mtl.layer_sizes(f0)[0] == mtl.layer_sizes(f1)[0]


def test_layer_desc_layout_matches_header(mtl, tmp_path):
    """The ctypes mirror of mtl_layer_desc has the C struct's size and offsets."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "probe.c"
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "mtl.h"\n'
                   'int main(void) { printf("%zu %zu %zu %zu %zu %zu\\n", sizeof(mtl_layer_desc),'
                   ' offsetof(mtl_layer_desc, causal), offsetof(mtl_layer_desc, p_attn),'
                   ' offsetof(mtl_layer_desc, p_hidden), offsetof(mtl_layer_desc, seed),'
                   ' offsetof(mtl_layer_desc, fp8));'
                   ' return 0; }\n')
    exe = tmp_path / "probe"
    subprocess.run([gcc, "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True)
    got = [int(v) for v in subprocess.run([str(exe)], capture_output=True, text=True,
                                          check=True).stdout.split()]
    D = mtl.LayerDesc
    assert got == [ctypes.sizeof(D), D.causal.offset, D.p_attn.offset, D.p_hidden.offset,
                   D.seed.offset, D.fp8.offset]


def test_attention_entry_points_reject(mtl):
    L = mtl.lib()
    ws = mtl.attention_ws_bytes(2, 256, 4)
    assert ws >= 256 + 2 * 4 * 256 * 4
    a = (FAKE, FAKE + 4096, FAKE + 8192)
    ok = dict(dtype=1, batch=2, seq=256, heads=4, d=64)

    def fwd(**kw):
        c = dict(ok, p=0.1, ws=ws, qkv=a[0], ctx=a[1], lse=a[2], mask=FAKE + 24576,
                 wsp=FAKE + 16384)
        c.update(kw)
        return L.mtl_attention_fwd(c["dtype"], c["batch"], c["seq"], c["heads"], c["d"], c["qkv"],
                                   c["ctx"], c["lse"], c["mask"], c["p"], 7, c["wsp"], c["ws"],
                                   None)

    assert fwd(p=1.0) == 1 and fwd(p=-0.5) == 1 and fwd(dtype=3) == 1 and fwd(heads=0) == 1
    assert fwd(d=32) == 2 and fwd(seq=200) == 2          # bf16 needs seq % 128 == 0
    assert fwd(qkv=FAKE + 8) == 1 and fwd(lse=None) == 1 and fwd(ctx=a[0]) == 1
    assert fwd(mask=None) == 1                           # bf16 with dropout needs the bits
    assert fwd(ws=ws - 1) == 3
    assert L.mtl_attention_bwd(1, 2, 256, 4, 64, a[0], a[1], a[2], FAKE + 12288, FAKE + 24576,
                               a[0], 0.0, 0, FAKE + 16384, ws, None) == 1    # dqkv aliases qkv
    assert L.mtl_attention_bwd(1, 2, 256, 4, 64, a[0], a[1], a[2], FAKE + 12288, None,
                               FAKE + 20480, 0.1, 0, FAKE + 16384, ws, None) == 1
    assert L.mtl_attention_bwd(1, 2, 256, 4, 64, a[0], a[1], a[2], FAKE + 12288, None,
                               FAKE + 20480, 0.0, 0, FAKE + 16384, 255, None) == 3


def test_infer_sizes_and_rejects(mtl):
    d = good_desc(mtl, seq=256, batch=3)
    kv, pw, dw = mtl.infer_sizes(d, 512)
    assert kv == 2 * 3 * 4 * 512 * 64 * 2                  # K and V, bf16
    assert pw >= mtl.layer_sizes(d)[0] and dw > 256
    s, p, w = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    L = mtl.lib()
    assert L.mtl_infer_sizes(ctypes.byref(d), 0, ctypes.byref(s), None, None) == 1
    assert L.mtl_infer_sizes(ctypes.byref(d), 128, None, ctypes.byref(p), None) == 1  # prompt > cache
    big = good_desc(mtl, batch=129)
    assert L.mtl_infer_sizes(ctypes.byref(big), 512, ctypes.byref(s), None, None) == 2
    # decode does not need seq % 128: a bf16 desc with seq = 1 still sizes a decode
    one = good_desc(mtl, seq=1)
    assert L.mtl_infer_sizes(ctypes.byref(one), 64, ctypes.byref(s), None, ctypes.byref(w)) == 0
    wt = _weights(mtl)
    ok = (FAKE, FAKE + 4096, FAKE + 8192, FAKE + 12288)
    assert L.mtl_layer_decode(ctypes.byref(one), ctypes.byref(wt), ok[0], ok[1], ok[2], 64, None,
                              ok[3], w.value, None) == 1              # no cache_len
    assert L.mtl_layer_decode(ctypes.byref(one), ctypes.byref(wt), ok[0], ok[0], ok[2], 64, FAKE,
                              ok[3], w.value, None) == 1              # y aliases x
    assert L.mtl_layer_decode(ctypes.byref(one), ctypes.byref(wt), ok[0], ok[1], ok[2], 64, FAKE,
                              ok[3], w.value - 1, None) == 3
    dd = good_desc(mtl, p_attn=0.1)
    assert L.mtl_layer_prefill(ctypes.byref(dd), ctypes.byref(wt), ok[0], ok[1], ok[2], 512, FAKE,
                               ok[3], 1 << 30, None) == 1             # no dropout at inference


def test_fp8_entry_points_reject(mtl):
    L = mtl.lib()
    ok = (FAKE, FAKE + 4096, FAKE + 8192, FAKE + 12288)
    def q(src, x, rows, cols, ld, fmt, qq, ldq, scale, ws, wsb, st, qT=None, ldqT=0):
        return L.mtl_fp8_quantize(src, x, rows, cols, ld, fmt, qq, ldq, qT, ldqT, scale, ws, wsb,
                                  st)

    assert q(1, ok[0], 64, 250, 256, 0, ok[1], 256, ok[2], ok[3], 256, None) == 1   # cols % 16
    assert q(1, ok[0], 64, 256, 256, 2, ok[1], 256, ok[2], ok[3], 256, None) == 1   # format
    assert q(1, ok[0], 64, 256, 256, 0, ok[1], 256, None, ok[3], 256, None) == 1    # no scale
    assert q(1, ok[0], 64, 256, 256, 0, ok[1], 256, ok[2], ok[3], 255, None) == 3
    assert q(1, ok[0], 64, 256, 256, 0, None, 0, ok[2], ok[3], 256, None) == 1      # no output
    assert q(1, ok[0], 60, 256, 256, 0, None, 0, ok[2], ok[3], 256, None,
             qT=ok[1], ldqT=64) == 1                                              # rows % 16
    g = L.mtl_gemm_fp8
    args = dict(M=256, N=256, K=512, parts=1, A=ok[0], lda=512, fa=0, sa=ok[2], B=ok[1], ldb=512,
                fb=0, sb=ok[2], epi=0, C=ok[3], ldc=256)

    def call(**kw):
        a = dict(args)
        a.update(kw)
        return g(a["M"], a["N"], a["K"], a["parts"], a["A"], a["lda"], a["fa"], a["sa"], a["B"],
                 a["ldb"], a["fb"], a["sb"], a["epi"], None, None, 0, None, 0, a["C"], a["ldc"], 1,
                 FAKE + 16384, 256, None)

    assert call(fa=3) == 1 and call(sb=None) == 1 and call(K=0) == 1 and call(parts=3) == 1
    assert call(A=FAKE + 8) == 1
    assert call(K=576, lda=576, ldb=576, parts=2) == 2        # 288-deep parts: not whole 128s
    assert call(lda=520) == 2                                  # row pitch not a multiple of 16


def test_fp8_layer_validation(mtl):
    ok = good_desc(mtl, fp8=1)                                  # h 256, t 2: 128-wide parts
    assert mtl.layer_sizes(good_desc(mtl, fp8=2))[1] > mtl.layer_sizes(ok)[1]
    assert mtl.layer_sizes(ok)[1] > mtl.layer_sizes(good_desc(mtl))[1]
    L = mtl.lib()
    for kw, st in ((dict(fp8=3), 1), (dict(fp8=1, dtype="f32"), 2), (dict(fp8=1, p_attn=0.1), 2),
                   (dict(fp8=1, t=4), 2)):                      # h/t = 64: not whole 128s
        d = good_desc(mtl, **kw)
        assert L.mtl_layer_sizes(ctypes.byref(d), None, None) == st, kw


def test_variant_validation(mtl):
    L = mtl.lib()
    for kw, st in ((dict(post_ln=2), 1), (dict(recompute=-1), 1),
                   (dict(post_ln=1, p_hidden=0.1), 2), (dict(post_ln=1, fp8=1), 2)):
        d = good_desc(mtl, **kw)
        assert L.mtl_layer_sizes(ctypes.byref(d), None, None) == st, kw
    base, rc = good_desc(mtl), good_desc(mtl, recompute=1)
    n, h, f = 256, 256, 1024
    assert mtl.layer_sizes(base)[0] - mtl.layer_sizes(rc)[0] == (2 * n * h + n * f) * 2
    post = mtl.layer_saved_layout(good_desc(mtl, post_ln=1))
    assert post["qkv"] == post["u1"] and post["h2"] - post["h1"] >= n * h * 2
    d = good_desc(mtl, post_ln=1)
    s = ctypes.c_size_t()
    assert L.mtl_infer_sizes(ctypes.byref(d), 512, ctypes.byref(s), None, None) == 2  # no decode
