"""The MTL_DEBUG build (device-side checks of every computed TMA coordinate and
output index of the GEMM and attention kernels, reporting MTL_ERR_BOUNDS instead
of faulting) on valid work: a layer forward and backward, the FP8 hybrid layer,
GEMMs with sliced tail tiles in both operand majors, and attention alone.  No
check may fire, and since the checks add no arithmetic the outputs must equal
the release build's bit for bit.  Each build runs in a process of its own
(MTL_LIBRARY selects the library)."""
import os
import subprocess
import sys

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r"""
import sys
import numpy as np
import torch
sys.path.insert(0, ".")
sys.path.insert(0, "tests")
import synthetic
from harness import make, to_device
from tensor_model_transformer_gb300 import mtl

out = {}

def layer(tag, shape, t, fp8=0):
    x, p, dy = make(shape, seed=4, affine=True)
    desc = mtl.layer_desc(shape.h, shape.heads, shape.seq, shape.batch, shape.ffn, t, "bf16", fp8=fp8)
    w = {k: to_device(v, "bf16") for k, v in p.items()}
    xd, dyd = to_device(x, "bf16"), to_device(dy, "bf16")
    saved, ws, grads = mtl.alloc_layer_buffers(desc)
    y, dx = torch.empty_like(xd), torch.empty_like(xd)
    mtl.layer_fwd(desc, w, xd, y, saved, ws)
    mtl.layer_check(ws)
    mtl.layer_bwd(desc, w, xd, saved, dyd, dx, grads, ws)
    mtl.layer_check(ws)
    out[tag + "y"] = y.float().cpu().numpy()
    out[tag + "dx"] = dx.float().cpu().numpy()
    for k, v in grads.items():
        out[tag + k] = v.cpu().numpy()

layer("l_", synthetic.tiny(h=256, heads=4, seq=256, batch=2, dtype="bf16", w_std=0.02, out_std=0.01), 2)
layer("f_", synthetic.tiny(h=256, heads=2, seq=256, batch=2, dtype="bf16", w_std=0.02, out_std=0.01), 2, fp8=2)

rng = np.random.default_rng(9)
for tag, (M, N, K, parts, ak, bk) in {"g1_": (2550, 2296, 6144, 1, 1, 1),
                                      "g2_": (2304, 2560, 6144, 1, 0, 0),
                                      "g3_": (2550, 2304, 6144, 8, 1, 1)}.items():
    A = torch.from_numpy(rng.standard_normal((M, K) if ak else (K, M)).astype(np.float32)).to(torch.bfloat16).cuda()
    B = torch.from_numpy(rng.standard_normal((N, K) if bk else (K, N)).astype(np.float32)).to(torch.bfloat16).cuda()
    bias = torch.from_numpy(rng.standard_normal(N).astype(np.float32)).to(torch.bfloat16).cuda()
    R = torch.from_numpy(rng.standard_normal((M, N)).astype(np.float32)).to(torch.bfloat16).cuda()
    C = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(mtl.gemm_ws_bytes(M, N), dtype=torch.uint8, device="cuda")
    mtl.gemm("bf16", M, N, K, parts, A, K if ak else M, ak, B, K if bk else N, bk, 2, C, N, False,
             ws, bias=bias, R=R, ldr=N)
    mtl.layer_check(ws)
    out[tag + "C"] = C.float().cpu().numpy()

batch, seq, heads, d = 2, 384, 4, 96
qkv = torch.from_numpy(rng.standard_normal((batch * seq, 3 * heads * d)).astype(np.float32)).to(torch.bfloat16).cuda()
do = torch.from_numpy(rng.standard_normal((batch * seq, heads * d)).astype(np.float32)).to(torch.bfloat16).cuda()
ctx = torch.empty((batch * seq, heads * d), dtype=torch.bfloat16, device="cuda")
lse = torch.empty((batch, heads, seq), dtype=torch.float32, device="cuda")
ws = torch.empty(mtl.attention_ws_bytes(batch, seq, heads), dtype=torch.uint8, device="cuda")
mtl.attention_fwd("bf16", batch, seq, heads, d, qkv, ctx, lse, ws)
mtl.layer_check(ws)
dqkv = torch.empty_like(qkv)
mtl.attention_bwd("bf16", batch, seq, heads, d, qkv, ctx, lse, do, dqkv, ws)
mtl.layer_check(ws)
out["a_ctx"] = ctx.float().cpu().numpy()
out["a_lse"] = lse.cpu().numpy()
out["a_dqkv"] = dqkv.float().cpu().numpy()
np.savez(sys.argv[1], **out)
"""


def _run(path, env_lib=None):
    env = dict(os.environ)
    env.pop("MTL_LIBRARY", None)
    if env_lib:
        env["MTL_LIBRARY"] = env_lib
    r = subprocess.run([sys.executable, "-c", SCRIPT, str(path)], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    return dict(np.load(path))


def test_debug_build_runs_clean_and_matches_release(tmp_path):
    from tensor_model_transformer_gb300 import build
    dbg = build.build(debug=True)
    got = _run(tmp_path / "debug.npz", dbg)
    want = _run(tmp_path / "release.npz")
    assert set(got) == set(want)
    diff = [k for k in want if not np.array_equal(got[k], want[k])]
    assert not diff, diff
