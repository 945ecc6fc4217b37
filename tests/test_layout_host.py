"""The shared-memory tile layout of the attention kernels (csrc/tile_layout.h),
run on the CPU.

The header is plain C++ (host and device); a small program compiled with g++
prints its offsets, and the tests hold them against the swizzle rule as the
tensor-copy unit states it on byte addresses (the 16-byte piece index, offset
bits 4.., XORed with offset bits 7..), against the tile's logical layout
(row-major atoms of ACOLS columns), and against the shared-memory bank rule
(32 banks of 4 bytes: a warp's 16-byte accesses take one wavefront per 128
bytes when no two of them share a bank group).
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "tensor_model_transformer_gb300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include "tile_layout.h"
using namespace mtl::layout;
template <int KS> void tile() {
  using T = TileFmt<KS>;
  printf("tile %d %u %d %u %u\n", KS, T::TILE, T::ACOLS, T::ATOM, T::ROWB);
  for (int kk = 0; kk < KS; ++kk) printf("koff %d %d %u %u\n", KS, kk, T::koff(kk), T::mnoff(kk));
  for (int r = 0; r < 128; ++r)
    for (int c = 0; c < T::D / 8; ++c) printf("chunk %d %d %d %u\n", KS, r, c, T::chunk(r, c));
}
int main() {
  for (int r = 0; r < 32; ++r)
    for (int p = 0; p < 4; ++p) printf("sw64 %d %d %u\n", r, p, sw64_off(r, p));
  for (int r = 0; r < 16; ++r)
    for (int p = 0; p < 8; ++p) printf("sw128 %d %d %u\n", r, p, sw128_off(r, p));
  tile<4>();
  tile<6>();
  tile<8>();
  return 0;
}
"""


@pytest.fixture(scope="module")
def out(tmp_path_factory):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("g++ not found")
    d = tmp_path_factory.mktemp("layout")
    src = d / "layout.cpp"
    src.write_text(PROGRAM)
    exe = d / "layout"
    subprocess.run([gxx, "-std=c++17", "-O1", "-I", CSRC, str(src), "-o", str(exe)], check=True)
    lines = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    res = {"sw64": {}, "sw128": {}, "tile": {}, "koff": {}, "chunk": {}}
    for ln in lines:
        if not ln:
            continue
        f = ln.split()
        vals = [int(v) for v in f[1:]]
        if f[0] in ("sw64", "sw128"):
            res[f[0]][(vals[0], vals[1])] = vals[2]
        elif f[0] == "tile":
            res["tile"][vals[0]] = dict(TILE=vals[1], ACOLS=vals[2], ATOM=vals[3], ROWB=vals[4])
        elif f[0] == "koff":
            res["koff"][(vals[0], vals[1])] = (vals[2], vals[3])
        else:
            res["chunk"][(vals[0], vals[1], vals[2])] = vals[3]
    return res


def swizzle(off, span):
    """The copy unit's swizzle of a byte offset inside a box whose base is
    1024-byte aligned: 16-byte piece bits XOR the bits just above the span."""
    if span == 64:
        return off ^ (((off >> 7) & 3) << 4)
    if span == 128:
        return off ^ (((off >> 7) & 7) << 4)
    raise ValueError(span)


def test_staging_offsets_follow_the_swizzle_rule(out):
    for (r, p), v in out["sw64"].items():
        assert v == swizzle(r * 64 + p * 16, 64), (r, p)
    for (r, p), v in out["sw128"].items():
        assert v == swizzle(r * 128 + p * 16, 128), (r, p)
    # every 16-byte piece of the 2 KB staging buffer is used exactly once
    assert sorted(out["sw64"].values()) == list(range(0, 2048, 16))


def wavefronts(offsets):
    """Shared-memory wavefronts of one warp access of 16 bytes a lane: the
    most lanes that fall on the same group of four banks."""
    groups = {}
    for o in offsets:
        groups[(o // 16) % 8] = groups.get((o // 16) % 8, 0) + 1
    return max(groups.values())


def test_staging_accesses_take_four_wavefronts(out):
    sw = out["sw64"]
    for q in range(4):
        # the row-wise write: lane l writes piece q of its own row
        assert wavefronts([sw[(lane, q)] for lane in range(32)]) == 4
        # the store-side read: lane l reads piece l % 4 of row 8q + l / 4
        assert wavefronts([sw[(8 * q + lane // 4, lane % 4)] for lane in range(32)]) == 4


@pytest.mark.parametrize("ks,tile,acols", [(4, 16384, 64), (6, 24576, 32), (8, 32768, 64)])
def test_tile_format(out, ks, tile, acols):
    t = out["tile"][ks]
    assert t["TILE"] == tile and t["ACOLS"] == acols
    assert t["ROWB"] == 2 * acols and t["ATOM"] == 128 * t["ROWB"]
    span = t["ROWB"]
    d = 16 * ks
    seen = set()
    for r in range(128):
        for c in range(d // 8):
            atom, q = divmod(8 * c, acols)
            want = atom * t["ATOM"] + swizzle(r * span + (q // 8) * 16, span)
            got = out["chunk"][(ks, r, c)]
            assert got == want, (ks, r, c, got, want)
            seen.add(got)
    # the tile's chunks fill it exactly
    assert sorted(seen) == list(range(0, tile, 16))


@pytest.mark.parametrize("ks", [4, 6, 8])
def test_kstep_offsets(out, ks):
    t = out["tile"][ks]
    for kk in range(ks):
        koff, mnoff = out["koff"][(ks, kk)]
        # K-major: columns 16 kk .. 16 kk + 15 begin in atom 16 kk / ACOLS, at
        # byte 2 (16 kk % ACOLS) of its (unswizzled) first row
        atom, col = divmod(16 * kk, t["ACOLS"])
        assert koff == atom * t["ATOM"] + 2 * col
        # MN-major: rows 16 kk .. 16 kk + 15 of every atom
        assert mnoff == 16 * kk * t["ROWB"]
