"""The debug build's bounds and alignment predicates, on the host.

csrc/fa_checks.h holds the predicates that libfa_debug.so's kernels evaluate
before every TMA load, shared-memory operand, tensor-memory access and bulk
copy.  They are plain integer functions, so this test compiles the header
with the host C++ compiler and checks them against hand-worked cases at and
around every boundary (the 16-byte rule for a TMA's innermost coordinate, the
last box of a tensor, the last columns of the 512-column allocation, operand
alignment).  It also checks that the debug library exports the same entry
points as the release library and says which one it is.
"""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "exact_tiled_attention_12_gb300", "csrc")

# (expression, expected) — each a call of one predicate.
CASES = [
    ("tma_x_ok(0, 64, 128)", True),
    ("tma_x_ok(64, 64, 128)", True),
    ("tma_x_ok(8, 64, 128)", True),        # 16 bytes of 16-bit elements
    ("tma_x_ok(4, 64, 128)", False),       # 8 bytes: off the 16-byte boundary
    ("tma_x_ok(1, 64, 128)", False),
    ("tma_x_ok(-8, 64, 128)", False),
    ("tma_x_ok(128, 64, 128)", False),     # starts past the row
    ("tma_rows_ok(0, 128, 128)", True),
    ("tma_rows_ok(896, 128, 1024)", True),
    ("tma_rows_ok(960, 128, 1024)", False),
    ("tma_rows_ok(-1, 128, 1024)", False),
    ("tma_rows_ok(0, 128, 127)", False),
    ("tma_rows_ok(4294967296LL, 128, 4294967424LL)", True),   # 64-bit row counts
    ("tma_head_ok(0, 200, 0, 2)", True),
    ("tma_head_ok(128, 200, 1, 2)", True),  # the ragged last tile starts inside the head
    ("tma_head_ok(200, 200, 1, 2)", False),
    ("tma_head_ok(0, 200, 2, 2)", False),
    ("tma_head_ok(-128, 200, 0, 2)", False),
    ("smem_ok(0, 16384, 65536, 1024)", True),
    ("smem_ok(49152, 16384, 65536, 1024)", True),
    ("smem_ok(49153, 16384, 65536, 1)", False),
    ("smem_ok(512, 16384, 65536, 1024)", False),
    ("smem_ok(65536, 16, 65536, 16)", False),
    ("smem_ok(0, 0, 65536, 16)", False),
    ("tmem_ok(0, 512, 512)", True),
    ("tmem_ok(384, 128, 512)", True),
    ("tmem_ok(448, 128, 512)", False),
    ("tmem_ok(512, 1, 512)", False),
    ("tmem_ok(4294967295u, 2, 512)", False),   # wrap-around cannot pass
    ("bulk_ok(256, 1024, 512)", True),
    ("bulk_ok(264, 1024, 512)", False),
    ("bulk_ok(256, 1032, 512)", False),
    ("bulk_ok(256, 1024, 500)", False),
    ("is_check_code(check_code(kChkTmem, 7))", True),
    ("is_check_code(0x0201u)", False),         # a timed-out wait's site code
    ("check_code(kChkTmaX, 0x1F1) == 0xC1F1u", True),
]


def test_predicates_at_their_boundaries(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    body = "\n".join(f'  if ((bool)({e}) != {str(w).lower()}) {{ std::printf("FAIL %d\\n", {i}); bad = 1; }}'
                     for i, (e, w) in enumerate(CASES))
    src = tmp_path / "checks.cc"
    src.write_text(f'''#include <cstdio>
#include "fa_checks.h"
using namespace fa;
int main() {{
  int bad = 0;
{body}
  std::printf("done %d\\n", bad);
  return bad;
}}
''')
    exe = tmp_path / "checks"
    r = subprocess.run([cxx, "-std=c++17", "-O1", "-I", CSRC, str(src), "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip().endswith("done 0")


def test_debug_library_exports_the_same_entry_points():
    import __graft_entry__

    __graft_entry__.build()
    from exact_tiled_attention_12_gb300 import binding

    rel, dbg = binding.lib(), binding.debug_lib()
    for name in binding.SIGNATURES:
        assert hasattr(dbg, name), name
    assert rel.fa_debug_checks_enabled() == 0
    assert dbg.fa_debug_checks_enabled() == 1
    # The release library has no checks to test; argument errors come first in both.
    assert rel.fa_selftest_bounds_check(None, None) == 2    # FA_ERR_UNSUPPORTED
    assert dbg.fa_selftest_bounds_check(None, None) == 1    # FA_ERR_INVALID_ARG
    assert binding.status_string(7).startswith("FA_ERR_BOUNDS")
