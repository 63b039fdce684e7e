"""The resolve kernel's shared-memory plan, checked on the host: every region
that is staged or copied in 16-byte units (cp.async, vector stores to the
copier CTAs, bulk copies) starts on a 16-byte boundary, and the mbarrier on
an 8-byte one, for a grid of shapes that covers every option (staged
slot->token row, inverse table, resident-token bitmap, paged block table,
staged rows).  A region
off its boundary would be a misaligned-address fault on the GPU; this finds
it without one.  The check compiles the kernel's source file into a host
program (nvcc; no GPU needed) and calls its plan function."""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "hierarchical_sparse_kv_request_gb300", "csrc")

PROGRAM = r"""
#include "resolve.cu"
#include <cstdio>
int main()
{
    long bad = 0, n = 0;
    for (int k : {1, 3, 7, 100, 255, 1023, 1025, 2047, 2048, 4099, 8192})
        for (int D : {k, k + 1, k + 3, k + 7, k + 299, 6144, 32768})
            for (int cap : {1, 31, 33, 100, 4097, 40064, 82000, 700000})
                for (int s2t = 0; s2t < 2; ++s2t)
                    for (int inv = 0; inv < 3; ++inv)
                        for (int tbl : {0, 4, 8, 1252})
                            for (int sr : {0, 1, 5})
                                for (long B : {16L, 48L, 656L, 1152L}) {
                                    if (D < k) continue;
                                    const hs::SmemPlan p = hs::plan_smem(k, D, cap, s2t, inv, tbl, sr, B);
                                    ++n;
                                    const size_t a16[] = {p.lru, p.s2t, p.inv, p.res, p.tbl,
                                                          p.lrow, p.avict, p.stage, p.total};
                                    for (size_t x : a16)
                                        if (x % 16) ++bad;
                                    if (p.bar % 8) ++bad;
                                }
    std::printf("%ld plans, %ld misaligned\n", n, bad);
    return bad != 0;
}
"""


def test_shared_memory_regions_are_aligned(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    src = tmp_path / "plan_check.cu"
    src.write_text(PROGRAM)
    exe = tmp_path / "plan_check"
    res = subprocess.run([nvcc, "-std=c++17", "-O1", "-gencode", "arch=compute_103a,code=sm_103a",
                          "-I" + CSRC, "-I" + os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                         capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True)
    assert run.returncode == 0, run.stdout + run.stderr
    assert " 0 misaligned" in run.stdout
