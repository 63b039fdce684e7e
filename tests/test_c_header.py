"""The public headers are plain C: a C99 program (and the same file as
C++17) that includes them compiles without warnings, links against
libhisparse.so and runs its host-only calls (no GPU is needed for these)."""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "hierarchical_sparse_kv_request_gb300")

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "hisparse.h"
#include "hisparse_measure.h"

int main(void)
{
    if (hisparse_version() != 201) return 1;
    if (strcmp(hisparse_error_string(HISPARSE_OK), "ok") != 0) return 2;
    if (hisparse_swap_in(NULL, 0, NULL, NULL, NULL, NULL, NULL) != HISPARSE_ERR_INVALID_ARG) return 3;
    if (hisparse_create(NULL, NULL) != HISPARSE_ERR_INVALID_ARG) return 4;
    if (hisparse_link_probe(NULL, NULL, 16, 0, NULL) != HISPARSE_ERR_INVALID_ARG) return 5;
    hisparse_plan plan;
    plan.rows = NULL;
    plan.counts = NULL;
    hisparse_layout layout;
    memset(&layout, 0, sizeof layout);
    if (hisparse_create(&layout, NULL) != HISPARSE_ERR_INVALID_ARG) return 6;
    (void)plan;
    printf("ok %d\n", HISPARSE_RESIDENT_FLAG);
    return 0;
}
"""


@pytest.fixture(scope="module")
def lib_built():
    import __graft_entry__
    __graft_entry__.build()
    return os.path.join(PKG, "libhisparse.so")


@pytest.mark.parametrize("compiler,flags", [("gcc", ["-x", "c", "-std=c99"]),
                                            ("g++", ["-x", "c++", "-std=c++17"])])
def test_headers_compile_link_and_run(tmp_path, lib_built, compiler, flags):
    if shutil.which(compiler) is None:
        pytest.skip(f"{compiler} not found")
    src = tmp_path / "use_hisparse.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "use_hisparse"
    cmd = [compiler, *flags, "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
           str(src), "-x", "none", lib_built, "-o", str(exe), f"-Wl,-rpath,{PKG}"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert run.returncode == 0, (run.returncode, run.stderr)
    assert run.stdout.strip() == f"ok {1 << 30}"
