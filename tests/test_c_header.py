"""The C ABI is usable from plain C: the header compiles as C99 and as
C++17 with warnings as errors, and a C program linked against the built
library calls its host-only entry points (version, status strings, argument
checks, the host work plan).  No GPU is involved."""

import os
import shutil
import subprocess

import pytest

import mla_decode_paged_gb300 as mla

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")

PROGRAM = r"""
#include <stdio.h>
#include <stdint.h>
#include "mla_decode.h"

int main(void) {
    int32_t lengths[3] = {256, 128, 1};
    int32_t plan[64];
    int used = 0;
    int64_t n;
    printf("version %s\n", mla_version());
    printf("invalid %s\n", mla_status_string(MLA_ERR_INVALID));
    /* a null pointer fails the host checks before anything is launched */
    printf("merge %d\n", (int)mla_merge_splits(NULL, NULL, 2, 4, 12, NULL, NULL, NULL));
    n = mla_plan_units(3, 1, 12, lengths, 4, 2, plan, 64, &used);
    printf("plan %lld used %d:", (long long)n, used);
    for (int64_t i = 0; i < n; ++i) printf(" %d", (int)plan[i]);
    printf("\n");
    return 0;
}
"""


def _cc(kind):
    exe = shutil.which({"c": "gcc", "c++": "g++"}[kind])
    if exe is None:
        pytest.skip("no %s compiler" % kind)
    return exe


@pytest.mark.parametrize("kind,std", [("c", "-std=c99"), ("c++", "-std=c++17")])
def test_header_compiles_cleanly(tmp_path, kind, std):
    src = tmp_path / ("h.c" if kind == "c" else "h.cpp")
    src.write_text('#include "mla_decode.h"\nint main(void) { return MLA_OK; }\n')
    r = subprocess.run([_cc(kind), std, "-Wall", "-Wextra", "-Werror", "-pedantic", "-fsyntax-only",
                        "-I", INCLUDE, str(src)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_c_program_calls_the_host_entry_points(tmp_path):
    lib = mla.build()
    src = tmp_path / "use.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "use"
    libdir = os.path.dirname(lib)
    r = subprocess.run([_cc("c"), "-std=c99", "-Wall", "-Werror", "-I", INCLUDE, str(src), "-o", str(exe),
                        lib, "-Wl,-rpath," + libdir], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, out.stderr
    lines = out.stdout.splitlines()
    assert lines[0].startswith("version ") and "sm_103a" in lines[0]
    assert lines[1] == "invalid invalid argument"
    assert lines[2] == "merge %d" % mla.MLA_ERR_INVALID
    # [256, 128, 1] tokens on 2 CTAs: request 0 alone, then requests 1 and 2 (budget 30 tenths of a
    # tile); then each CTA's first item again
    one = 1 << 9
    assert lines[3] == "plan 24 used 1: " + " ".join(str(x) for x in
                                                   [2, 0, 1, 3, 0, one, 0, 256, 1, one, 0, 128, 2, one, 0, 1,
                                                    0, one, 0, 256, 1, one, 0, 128])
