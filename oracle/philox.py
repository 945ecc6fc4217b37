"""Philox4x32-10 counter-based generator and the dropout masks built from it.

TEST INFRASTRUCTURE ONLY (see oracle/layer.py).

Philox4x32 (J. K. Salmon, M. A. Moraes, R. O. Dror, D. E. Shaw, "Parallel random
numbers: as easy as 1, 2, 3", SC'11): a 4 x 32-bit counter and a 2 x 32-bit key;
each of the 10 rounds multiplies counter words 0 and 2 by the Philox constants
(full 64-bit products), mixes the high halves with the other two words and the
round key, and the key is bumped by the Weyl constants between rounds.

Dropout masks (the pages name dropout in the fused bias + dropout + residual
kernel and attention dropout, without a generator; this is the reading used by
the oracle and the CUDA kernels alike):
  key       = (seed mod 2^32, seed div 2^32)
  counter   = (e div 4 mod 2^32, e div 4 div 2^32, site, 0)
  word(e)   = Philox4x32-10(counter, key)[e mod 4]
  keep(e)   = word(e) >= floor(p * 2^32)      (drop with probability p)
  value     = x * keep / (1 - p)
for element index e and site 0 = attention probabilities
(e = ((b * heads + head) * seq + i) * seq + j), 1 = out-projection output and
2 = fc2 output (e = token * h + column).
"""

from __future__ import annotations

import numpy as np

M0, M1 = 0xD2511F53, 0xCD9E8D57
W0, W1 = 0x9E3779B9, 0xBB67AE85
MASK32 = np.uint64(0xFFFFFFFF)

SITE_ATTN, SITE_OUT, SITE_FC2 = 0, 1, 2


def philox4x32(counter, key, rounds=10):
    """Philox4x32 of counters [..., 4] (uint32) under key (k0, k1); returns [..., 4] uint32."""
    c = np.asarray(counter, dtype=np.uint64)
    c0, c1, c2, c3 = c[..., 0], c[..., 1], c[..., 2], c[..., 3]
    k0 = np.uint64(int(key[0]) & 0xFFFFFFFF)
    k1 = np.uint64(int(key[1]) & 0xFFFFFFFF)
    for r in range(rounds):
        if r > 0:
            k0 = (k0 + np.uint64(W0)) & MASK32
            k1 = (k1 + np.uint64(W1)) & MASK32
        p0 = c0 * np.uint64(M0)
        p1 = c2 * np.uint64(M1)
        hi0, lo0 = p0 >> np.uint64(32), p0 & MASK32
        hi1, lo1 = p1 >> np.uint64(32), p1 & MASK32
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
    return np.stack([c0, c1, c2, c3], axis=-1).astype(np.uint32)


def threshold(p):
    """floor(p * 2^32) as an integer, for 0 <= p < 1."""
    if not 0.0 <= p < 1.0:
        raise ValueError("dropout probability must be in [0, 1)")
    return min(int(np.floor(p * 4294967296.0)), 0xFFFFFFFF)


def words(e, seed, site):
    """The 32-bit random word of each element index in e (uint64 array)."""
    e = np.asarray(e, dtype=np.uint64)
    q = e >> np.uint64(2)
    ctr = np.stack([q & MASK32, q >> np.uint64(32), np.full_like(q, site),
                    np.zeros_like(q)], axis=-1)
    out = philox4x32(ctr, (seed & 0xFFFFFFFF, seed >> 32))
    lane = (e & np.uint64(3)).astype(np.int64)
    return np.take_along_axis(out, lane[..., None], axis=-1)[..., 0]


def keep_mask(e, seed, site, p):
    """Boolean keep mask of the elements with indices e."""
    if p == 0.0:
        return np.ones(np.shape(e), dtype=bool)
    return words(e, seed, site) >= np.uint32(threshold(p))


def hidden_mask(n, h, seed, site, p):
    """[n, h] keep mask of a hidden-state dropout site (e = token * h + column)."""
    e = np.arange(n, dtype=np.uint64)[:, None] * np.uint64(h) + np.arange(h, dtype=np.uint64)[None, :]
    return keep_mask(e, seed, site, p)


def attention_mask(b, head, heads, seq, seed, p):
    """[seq, seq] keep mask of the attention probabilities of one (batch, head)."""
    base = (np.uint64(b) * np.uint64(heads) + np.uint64(head)) * np.uint64(seq)
    e = (base + np.arange(seq, dtype=np.uint64)[:, None]) * np.uint64(seq) + \
        np.arange(seq, dtype=np.uint64)[None, :]
    return keep_mask(e, seed, SITE_ATTN, p)
