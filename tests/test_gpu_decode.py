"""GPU parity of inference: prefill and decode with the KV cache through the C
ABI against the oracle (``oracle.decode``), element by element.

Tolerances as for the forward: fp32 layers 1e-5, bf16 1.5e-2 of the largest
reference value, per decoded token and per cache tensor.  Cache lengths are
integers and must match exactly."""
import numpy as np
import pytest

import oracle
import synthetic
from harness import rel_err, to_device, to_np

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-5, "bf16": 1.5e-2}


def _setup(shape, max_seq, seed=0, t=1, affine=True):
    import torch
    from tensor_model_transformer_gb300 import mtl
    x, p, _ = synthetic.make_layer(shape, seed=seed, affine=affine)
    desc = mtl.layer_desc(shape.h, shape.heads, shape.seq, shape.batch, shape.ffn, t, shape.dtype)
    kvb, pwb, dwb = mtl.infer_sizes(desc, max_seq)
    dev = {k: to_device(v, shape.dtype) for k, v in p.items()}
    kv = torch.zeros(kvb, dtype=torch.uint8, device="cuda")
    pws = torch.empty(pwb, dtype=torch.uint8, device="cuda")
    dws = torch.empty(dwb, dtype=torch.uint8, device="cuda")
    lens = torch.zeros(shape.batch, dtype=torch.int32, device="cuda")
    return x, p, desc, dev, kv, pws, dws, lens


def _tokens(shape, steps, seed):
    rng = np.random.default_rng(seed)
    return synthetic.to_storage(rng.standard_normal((steps, shape.batch, shape.h)).astype(np.float32),
                                shape.dtype)


def run_case(shape, max_seq, steps, seed=0, t=1, check=None, affine=True):
    """Prefill and `steps` decode steps of every sequence on the GPU; the
    sequences `check` (default: all) are run through the oracle on their own
    (sequences are independent) and compared."""
    import torch
    from tensor_model_transformer_gb300 import mtl
    x, p, desc, dev, kv, pws, dws, lens = _setup(shape, max_seq, seed, t, affine)
    sel = list(range(shape.batch)) if check is None else list(check)
    toks = _tokens(shape, steps, seed + 7)
    xd = to_device(x, shape.dtype)
    y = torch.empty_like(xd)
    mtl.layer_prefill(desc, dev, xd, y, kv, max_seq, lens, pws)
    mtl.layer_check(pws)
    cache = oracle.decode.kv_cache(len(sel), shape.heads, max_seq, shape.h // shape.heads)
    y_ref = oracle.decode.prefill(p, x[sel], shape.heads, cache)
    tol = TOL[shape.dtype]
    assert rel_err(to_np(y)[sel], y_ref) <= tol
    assert lens.cpu().tolist() == [shape.seq] * shape.batch
    for i in range(steps):
        xt = to_device(toks[i], shape.dtype)
        yt = torch.empty_like(xt)
        mtl.layer_decode(desc, dev, xt, yt, kv, max_seq, lens, dws)
        mtl.layer_check(dws)
        yr = oracle.decode.decode_step(p, toks[i][sel], shape.heads, cache)
        assert rel_err(to_np(yt)[sel], yr) <= tol, (i, rel_err(to_np(yt)[sel], yr))
    assert lens.cpu().tolist() == [shape.seq + steps] * shape.batch
    k, v = mtl.kv_views(desc, kv, max_seq)
    L = shape.seq + steps
    k, v = to_np(k), to_np(v)
    assert rel_err(k[sel][:, :, :L], cache["k"][:, :, :L]) <= tol
    assert rel_err(v[sel][:, :, :L], cache["v"][:, :, :L]) <= tol
    assert np.all(k[:, :, L:] == 0)
    # partition p's shard of the cache: heads [p*H/t, (p+1)*H/t) of every sequence
    for part in range(t):
        hs = slice(part * shape.heads // t, (part + 1) * shape.heads // t)
        assert rel_err(k[sel][:, hs, :L], cache["k"][:, hs, :L]) <= tol, part


CASES = {
    # name: (shape, max_seq, decode steps)
    "f32_d64_ragged": (synthetic.tiny(h=256, heads=4, seq=100, batch=2, dtype="f32", w_std=0.05,
                                      out_std=0.05), 160, 3),
    "f32_cross_chunk": (synthetic.tiny(h=192, heads=2, seq=254, batch=2, dtype="f32",
                                       w_std=0.05, out_std=0.05), 300, 4),
    "bf16_d64": (synthetic.tiny(h=256, heads=4, seq=128, batch=3, dtype="bf16", w_std=0.02,
                                out_std=0.01), 256, 3),
    "bf16_d96_batch17": (synthetic.tiny(h=384, heads=4, seq=128, batch=17, dtype="bf16",
                                        w_std=0.02, out_std=0.01), 160, 2),
    "bf16_d128_two_chunks": (synthetic.tiny(h=256, heads=2, seq=384, batch=2, dtype="bf16",
                                            w_std=0.02, out_std=0.01), 640, 3),
    "bf16_batch1": (synthetic.tiny(h=512, heads=8, seq=128, batch=1, dtype="bf16", w_std=0.02,
                                   out_std=0.01), 130, 2),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_prefill_and_decode(name):
    shape, max_seq, steps = CASES[name]
    run_case(shape, max_seq, steps)


# name: (shape, max_seq, decode steps, t)
SHARDED = {
    "bf16_d64_t2": (synthetic.tiny(h=256, heads=4, seq=128, batch=3, dtype="bf16", w_std=0.02,
                                   out_std=0.01), 256, 3, 2),
    "bf16_d96_t8": (synthetic.tiny(h=1536, heads=16, seq=256, batch=4, dtype="bf16",
                                   w_std=0.02, out_std=0.01), 384, 3, 8),
    "f32_d64_t2": (synthetic.tiny(h=256, heads=4, seq=100, batch=2, dtype="f32", w_std=0.05,
                                  out_std=0.05), 160, 2, 2),
}


@pytest.mark.parametrize("name", sorted(SHARDED))
def test_prefill_and_decode_head_sharded(name):
    """t > 1: the prefill runs the t-partitioned forward, every partition's heads
    fill its own shard of the cache, and decode reads the shards."""
    shape, max_seq, steps, t = SHARDED[name]
    run_case(shape, max_seq, steps, t=t)


def test_decode_at_the_benchmarked_shape():
    """bench.py --workload decode: the 8.3B-shape layer (h 3072, 32 heads, t = 8),
    16 sequences with a 1024-token context, the same seeded inputs.  The GPU
    prefills and decodes all 16; sequences 0, 7 and 15 are checked."""
    shape = synthetic.CONFIGS["D"]
    run_case(shape, shape.seq + 8, 2, seed=0, t=8, check=[0, 7, 15], affine=False)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_ragged_cache_lengths(dtype):
    """Sequences at different lengths: shortening cache_len of a sequence makes
    its decode equal the forward of its shorter prompt plus the new token."""
    import torch
    from tensor_model_transformer_gb300 import mtl
    shape = synthetic.tiny(h=256, heads=4, seq=128, batch=3, dtype=dtype, w_std=0.02, out_std=0.01)
    max_seq = 200
    x, p, desc, dev, kv, pws, dws, lens = _setup(shape, max_seq, seed=3)
    xd = to_device(x, dtype)
    mtl.layer_prefill(desc, dev, xd, torch.empty_like(xd), kv, max_seq, lens, pws)
    short = [128, 77, 5]
    lens.copy_(torch.tensor(short, dtype=torch.int32))
    tok = _tokens(shape, 1, 11)[0]
    xt = to_device(tok, dtype)
    yt = torch.empty_like(xt)
    mtl.layer_decode(desc, dev, xt, yt, kv, max_seq, lens, dws)
    mtl.layer_check(dws)
    assert lens.cpu().tolist() == [L + 1 for L in short]
    for b, L in enumerate(short):
        seq = np.concatenate([x[b, :L], tok[b][None]], axis=0)[None]
        y_full, _ = oracle.layer_fwd(p, seq, shape.heads)
        assert rel_err(to_np(yt)[b], y_full[0, -1]) <= TOL[dtype], b


def test_decode_deterministic_and_graph_replay():
    """Two decode runs are bitwise equal; a captured CUDA graph of one decode
    call, replayed with new tokens, advances the cache like eager calls."""
    import torch
    from tensor_model_transformer_gb300 import mtl
    shape = synthetic.tiny(h=384, heads=4, seq=128, batch=4, dtype="bf16", w_std=0.02,
                           out_std=0.01)
    max_seq, steps = 192, 3
    toks = _tokens(shape, steps, 5)

    def prefilled():
        x, p, desc, dev, kv, pws, dws, lens = _setup(shape, max_seq, seed=1)
        xd = to_device(x, "bf16")
        mtl.layer_prefill(desc, dev, xd, torch.empty_like(xd), kv, max_seq, lens, pws)
        return desc, dev, kv, dws, lens

    outs = []
    for _ in range(2):
        desc, dev, kv, dws, lens = prefilled()
        ys = []
        for i in range(steps):
            xt = to_device(toks[i], "bf16")
            yt = torch.empty_like(xt)
            mtl.layer_decode(desc, dev, xt, yt, kv, max_seq, lens, dws)
            ys.append(yt.clone())
        mtl.layer_check(dws)
        outs.append((torch.stack(ys), kv.clone()))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])

    desc, dev, kv, dws, lens = prefilled()
    torch.cuda.synchronize()
    x_in = to_device(toks[0], "bf16")
    y_out = torch.empty_like(x_in)
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side, capture_error_mode="relaxed"):
            mtl.layer_decode(desc, dev, x_in, y_out, kv, max_seq, lens, dws, stream=side)
    torch.cuda.synchronize()
    assert lens.cpu().tolist() == [128] * shape.batch      # capture ran nothing
    ys = []
    for i in range(steps):
        x_in.copy_(to_device(toks[i], "bf16"))
        g.replay()
        ys.append(y_out.clone())
    torch.cuda.synchronize()
    mtl.layer_check(dws)
    assert lens.cpu().tolist() == [128 + steps] * shape.batch
    assert torch.equal(torch.stack(ys), outs[0][0])
    assert torch.equal(kv, outs[0][1])


def test_full_cache_is_reported():
    """A sequence whose cache is full: the step reports MTL_ERR_INVALID_ARG
    and writes nothing into the cache."""
    import torch
    from tensor_model_transformer_gb300 import mtl
    shape = synthetic.tiny(h=256, heads=4, seq=128, batch=2, dtype="bf16", w_std=0.02,
                           out_std=0.01)
    max_seq = 128
    x, p, desc, dev, kv, pws, dws, lens = _setup(shape, max_seq)
    xd = to_device(x, "bf16")
    mtl.layer_prefill(desc, dev, xd, torch.empty_like(xd), kv, max_seq, lens, pws)
    mtl.layer_check(pws)
    before = kv.clone()
    xt = to_device(_tokens(shape, 1, 2)[0], "bf16")
    mtl.layer_decode(desc, dev, xt, torch.empty_like(xt), kv, max_seq, lens, dws)
    with pytest.raises(mtl.MtlError) as e:
        mtl.layer_check(dws)
    assert e.value.status == 1
    assert torch.equal(kv, before)
    assert lens.cpu().tolist() == [128, 128]
