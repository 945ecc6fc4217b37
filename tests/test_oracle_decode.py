"""Pins of the inference oracle (prefill / decode with a KV cache), no GPU.

The decode step is pinned against its definition: the full causal forward of
the extended sequence (``oracle.layer_fwd``), which computes attention through
a different path (whole causal matrix, not one cached query)."""
import numpy as np
import pytest

import oracle
import synthetic


def _tiny(seed=0, h=64, heads=4, ffn=256):
    shp = synthetic.tiny(h=h, heads=heads, seq=8, batch=2, ffn=ffn, dtype="f32", w_std=0.2,
                         out_std=0.2)
    x, p, _ = synthetic.make_layer(shp, seed=seed, affine=True)
    rng = np.random.default_rng(seed + 100)
    return shp, p, rng


def test_prefill_then_decode_is_the_full_forward():
    shp, p, rng = _tiny()
    batch, S, steps, h, heads = 2, 5, 4, shp.h, shp.heads
    d = h // heads
    seqs = rng.standard_normal((batch, S + steps, h))
    cache = oracle.decode.kv_cache(batch, heads, 16, d)
    y_pre = oracle.decode.prefill(p, seqs[:, :S], heads, cache)
    assert np.all(cache["len"] == S)
    ys = [oracle.decode.decode_step(p, seqs[:, S + i], heads, cache) for i in range(steps)]
    assert np.all(cache["len"] == S + steps)
    y_full, c_full = oracle.layer_fwd(p, seqs, heads)
    assert np.max(np.abs(y_pre - y_full[:, :S])) < 1e-12
    for i, y in enumerate(ys):
        assert np.max(np.abs(y - y_full[:, S + i])) < 1e-11 * max(1.0, np.max(np.abs(y))), i
    qkv = c_full["qkv"].reshape(batch, S + steps, heads, 3, d)
    assert np.max(np.abs(cache["k"][:, :, :S + steps] - qkv[:, :, :, 1].transpose(0, 2, 1, 3))) < 1e-12
    assert np.max(np.abs(cache["v"][:, :, :S + steps] - qkv[:, :, :, 2].transpose(0, 2, 1, 3))) < 1e-12
    assert np.all(cache["k"][:, :, S + steps:] == 0)


def test_ragged_cache_lengths():
    """Sequences at different cache lengths decode independently."""
    shp, p, rng = _tiny(seed=1)
    h, heads = shp.h, shp.heads
    d = h // heads
    lens = [6, 3]
    seqs = [rng.standard_normal((1, L + 2, h)) for L in lens]
    cache = oracle.decode.kv_cache(2, heads, 12, d)
    for b, L in enumerate(lens):
        one = oracle.decode.kv_cache(1, heads, 12, d)
        oracle.decode.prefill(p, seqs[b][:, :L], heads, one)
        cache["k"][b], cache["v"][b], cache["len"][b] = one["k"][0], one["v"][0], L
    for step in range(2):
        x_tok = np.stack([seqs[b][0, lens[b] + step] for b in range(2)])
        y = oracle.decode.decode_step(p, x_tok, heads, cache)
        for b, L in enumerate(lens):
            y_full, _ = oracle.layer_fwd(p, seqs[b][:, :L + step + 1], heads)
            assert np.max(np.abs(y[b] - y_full[0, -1])) < 1e-11, (step, b)
    assert list(cache["len"]) == [8, 5]


@pytest.mark.parametrize("t", [1, 2, 4])
def test_partitioned_decode_matches_and_shards_evenly(t):
    shp, p, rng = _tiny(seed=2, h=64, heads=8)
    batch, S, h, heads = 2, 4, shp.h, shp.heads
    d = h // heads
    seqs = rng.standard_normal((batch, S + 3, h))
    full = oracle.decode.kv_cache(batch, heads, 10, d)
    oracle.decode.prefill(p, seqs[:, :S], heads, full)
    shards = oracle.decode.shard_caches(batch, heads, 10, d, t)
    for r, sh in enumerate(shards):
        hp = heads // t
        sh["k"][:] = full["k"][:, r * hp:(r + 1) * hp]
        sh["v"][:] = full["v"][:, r * hp:(r + 1) * hp]
        sh["len"][:] = full["len"]
        assert sh["k"].size * t == full["k"].size      # the cache splits evenly by t
    cnt = oracle.ReductionCounter()
    for i in range(3):
        y_ref = oracle.decode.decode_step(p, seqs[:, S + i], heads, full)
        y = oracle.decode.decode_step_partitioned(p, seqs[:, S + i], heads, t, shards, cnt)
        assert np.max(np.abs(y - y_ref)) < 1e-12
        assert cnt.g == 2 * (i + 1) and cnt.f == 0
    hp = heads // t
    for r, sh in enumerate(shards):
        assert np.max(np.abs(sh["k"] - full["k"][:, r * hp:(r + 1) * hp])) < 1e-12


def test_cache_limits():
    shp, p, rng = _tiny()
    d = shp.h // shp.heads
    cache = oracle.decode.kv_cache(2, shp.heads, 4, d)
    with pytest.raises(ValueError):
        oracle.decode.prefill(p, rng.standard_normal((2, 5, shp.h)), shp.heads, cache)
    oracle.decode.prefill(p, rng.standard_normal((2, 4, shp.h)), shp.heads, cache)
    with pytest.raises(ValueError):
        oracle.decode.decode_step(p, rng.standard_normal((2, shp.h)), shp.heads, cache)


def test_decode_bytes_counts():
    # h = 8, ffn = 32: weights 3*64 + 64 + 2*256 = 768 elements, small vectors
    # 3h + h + ffn + h + 4h = 104; cache of lengths [2, 0] -> (3 + 1) rows of K and V
    b = oracle.decode.decode_bytes(8, 2, 32, 2, [2, 0], esz=2)
    assert b == (768 + 104) * 2 + 2 * (3 + 1) * 8 * 2
