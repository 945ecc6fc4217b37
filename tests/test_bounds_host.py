"""The coordinate checks of the MTL_DEBUG build (csrc/bounds.h), run on the CPU.

The header is plain C++ (host and device); a small program compiled with g++
runs every rule on cases whose answers follow from the tensor-copy rules: the
innermost coordinate times the element size a multiple of 16 bytes; a load may
start outside the tensor but not lie wholly outside it; a store may not start
at a negative coordinate nor past the end; indices inside [0, n)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "tensor_model_transformer_gb300", "csrc")

# (kind, ext_x, ext_y, box_x, box_y, elem_bytes, x, y, expected fault)
CASES = [
    ("load", 256, 512, 64, 128, 2, 0, 0, 0),
    ("load", 256, 512, 64, 128, 2, 8, 0, 0),       # 16 bytes
    ("load", 256, 512, 64, 128, 2, 4, 0, 1),       # 8 bytes: misaligned
    ("load", 256, 512, 128, 128, 1, 8, 0, 1),      # FP8: 8 bytes
    ("load", 256, 512, 128, 128, 1, 16, 0, 0),
    ("load", 256, 512, 32, 32, 4, 2, 0, 1),        # fp32: 8 bytes
    ("load", 256, 512, 32, 32, 4, 4, 0, 0),
    ("load", 256, 512, 64, 128, 2, -8, 0, 0),      # starts before the tensor, partly inside
    ("load", 256, 512, 64, 128, 2, -64, 0, 2),     # wholly before it
    ("load", 256, 512, 64, 128, 2, 256, 0, 2),     # starts at the end
    ("load", 256, 512, 64, 128, 2, 248, 0, 0),     # ragged tail, partly inside
    ("load", 256, 512, 64, 128, 2, 0, 512, 2),
    ("load", 256, 512, 64, 128, 2, 0, -127, 0),
    ("load", 256, 512, 64, 128, 2, 0, -128, 2),
    ("load", 256, 512, 64, 128, 2, -3, -200, 1),   # misalignment is reported first
    ("store", 256, 512, 32, 32, 2, 0, 0, 0),
    ("store", 256, 512, 32, 32, 2, 224, 480, 0),
    ("store", 256, 512, 32, 32, 2, 240, 500, 0),   # ragged: the box's bounds drop the rest
    ("store", 256, 512, 32, 32, 2, -8, 0, 3),      # aligned but negative
    ("store", 256, 512, 32, 32, 2, 0, -1, 3),
    ("store", 256, 512, 32, 32, 2, 256, 0, 4),
    ("store", 256, 512, 32, 32, 2, 0, 512, 4),
    ("store", 256, 512, 32, 32, 2, 12, 0, 1),
]
INDEX_CASES = [(0, 10, 0), (9, 10, 0), (10, 10, 5), (-1, 10, 5), (1 << 40, 1 << 41, 0)]

PROGRAM = r"""
#include <cstdio>
#include "bounds.h"
using namespace mtl::bounds;
int main() {
  long long kind, ex, ey, bx, by, eb, x, y;
  char k[16];
  while (scanf("%15s", k) == 1) {
    if (k[0] == 'i') {
      scanf("%lld %lld", &x, &ex);
      printf("%u\n", check_index(x, ex));
    } else if (k[0] == 's' && k[1] == 'b') {
      scanf("%lld %lld", &x, &y);
      printf("%u\n", status_bits((uint32_t)x, (uint32_t)y));
    } else {
      scanf("%lld %lld %lld %lld %lld %lld %lld", &ex, &ey, &bx, &by, &eb, &x, &y);
      const Box2 b = {ex, ey, (int32_t)bx, (int32_t)by, (int32_t)eb};
      printf("%u\n", k[0] == 'l' ? check_tma_load(b, x, y) : check_tma_store(b, x, y));
    }
  }
  (void)kind;
  return 0;
}
"""


@pytest.fixture(scope="module")
def checker(tmp_path_factory):
    gxx = shutil.which("g++") or shutil.which("c++")
    if not gxx:
        pytest.skip("no C++ compiler")
    d = tmp_path_factory.mktemp("bounds")
    src = d / "bounds_cases.cc"
    src.write_text(PROGRAM)
    exe = d / "bounds_cases"
    subprocess.run([gxx, "-std=c++17", "-O1", "-I", CSRC, str(src), "-o", str(exe)], check=True)
    return exe


def run(exe, lines):
    out = subprocess.run([str(exe)], input="\n".join(lines) + "\n", capture_output=True,
                         text=True, check=True).stdout.split()
    return [int(v) for v in out]


def test_tma_rules(checker):
    lines = [f"{c[0]} {' '.join(str(v) for v in c[1:8])}" for c in CASES]
    got = run(checker, lines)
    assert got == [c[8] for c in CASES], [(c, g) for c, g in zip(CASES, got) if g != c[8]]


def test_index_rule(checker):
    got = run(checker, [f"i {i} {n}" for i, n, _ in INDEX_CASES])
    assert got == [e for _, _, e in INDEX_CASES]


def test_status_bits(checker):
    got = run(checker, ["sb 0 7", "sb 2 7", "sb 5 13"])
    assert got == [0, 4 | (2 << 8) | (7 << 16), 4 | (5 << 8) | (13 << 16)]
