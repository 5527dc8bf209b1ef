"""The boundary from C: include/muon.h compiles as strict C99 and as C++17, and
a plain C program links against libmuon.so and calls it (CPU only: every call
below returns before any CUDA call)."""

import os
import shutil
import subprocess

import pytest

import muon_newton_schulz_expert_gb300 as mk
from muon_newton_schulz_expert_gb300 import build as mkbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")

PROGRAM = r"""
#include <stdio.h>
#include "muon.h"

int main(void) {
  const float c3[3] = {3.4445f, -4.775f, 2.0315f};
  muon_stream_t s = NULL;
  printf("%d\n", muon_ns_batched(NULL, 1, 8, 8, 5, c3, 1e-7f, s));          /* null X */
  printf("%d\n", muon_ns_batched(NULL, 0, 8, 8, 5, c3, 1e-7f, s));          /* empty batch */
  printf("%d\n", muon_momentum_update(NULL, NULL, NULL, 0, 0.95f, 1, s));   /* nothing to do */
  printf("%d\n", muon_momentum_update(NULL, NULL, NULL, -1, 0.95f, 1, s));  /* bad size */
  printf("%d\n", muon_apply_update(NULL, NULL, 1, 8, 8, 0.02f, 0.1f, 0.0f, s));
  printf("%zu\n", muon_ns_workspace_bytes(96, 1792, 6144));
  printf("%zu\n", muon_step_workspace_bytes(64, 6144, 1792));
  printf("%s\n", muon_status_string(MUON_ERR_NO_MEMORY));
  printf("%.6f\n", (double)muon_default_scale(6144, 1792));
  return 0;
}
"""


@pytest.fixture(scope="module")
def libdir():
    if shutil.which("gcc") is None or shutil.which("g++") is None:
        pytest.skip("no host C compiler")
    mkbuild.build()
    return os.path.dirname(mkbuild.LIB)


def test_header_compiles_as_c99_and_cxx17(tmp_path, libdir):
    src = tmp_path / "h.c"
    src.write_text('#include "muon.h"\nint main(void) { return MUON_OK; }\n')
    for cc, std, lang in (("gcc", "-std=c99", "c"), ("g++", "-std=c++17", "c++")):
        r = subprocess.run([cc, std, "-x", lang, "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", INCLUDE,
                            "-fsyntax-only", str(src)], capture_output=True, text=True)
        assert r.returncode == 0, (cc, r.stderr)


def test_c_program_links_and_calls_the_library(tmp_path, libdir):
    src, exe = tmp_path / "client.c", tmp_path / "client"
    src.write_text(PROGRAM)
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", INCLUDE, str(src),
                        "-L", libdir, "-lmuon", f"-Wl,-rpath,{libdir}", "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, out.stderr
    lines = out.stdout.split()
    lib = mk.lib()
    assert [int(v) for v in lines[:5]] == [-1, 0, 0, -1, -1]
    assert int(lines[5]) == lib.muon_ns_workspace_bytes(96, 1792, 6144)
    assert int(lines[6]) == lib.muon_step_workspace_bytes(64, 6144, 1792) > 0
    assert lines[7] == lib.muon_status_string(-4).decode() == "MUON_ERR_NO_MEMORY"
    assert float(lines[8]) == pytest.approx((6144 / 1792) ** 0.5, rel=1e-6)
