"""The allocation-free swap-in (hisparse_swap_in_noalloc) against the regular
one (hisparse_swap_in), through the C ABI, on the GPU.

Some callers may not allocate device memory at all -- a serving process whose
device memory is owned up front by one pool, or a call site where allocation
is forbidden.  For them the library keeps the plan that passes misses from
its resolve grid to its copy grid in a fixed per-GPU array.  This checks that
such calls give exactly what the regular entry point gives, two calls in a
row (the array keeps the previous call's contents), that a handle too
large for the array is refused, and that the first such call of a fresh
process does not change the device's free memory even when CUDA loads the
library's code lazily.  The file is named to be collected last.
"""

import os
import subprocess
import sys
import textwrap

import numpy as np
import pytest
import torch

from hierarchical_sparse_kv_request_gb300 import hisparse as H
from hierarchical_sparse_kv_request_gb300 import workload as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    yield


def _handle(w):
    g = H.HiSparse.for_workload(w)
    for r in range(w.num_requests):
        W.fill_host_rows(w, 0, r, g.host_rows(0, r), int(w.seq_lens0[r]))
    g.prefill(torch.from_numpy(w.seq_lens0).cuda())
    return g


def test_noalloc_matches_regular_swap_in_two_calls_in_a_row():
    lens = [5000, 700, 3000, 9000, 1024, 4000, 2500, 6000]
    w = W.custom(8, 512, 1024, lens, row_bytes=64)
    regular, noalloc = _handle(w), _handle(w)
    seq = torch.from_numpy(w.seq_lens0).cuda()
    R, k = w.num_requests, w.top_k
    out_a = torch.empty((R, k), dtype=torch.int32, device="cuda")
    out_b = torch.empty((R, k), dtype=torch.int32, device="cuda")
    rng = np.random.default_rng(2)
    prev = None
    for call in range(2):
        rows = np.empty((R, k), dtype=np.int32)
        for r in range(R):
            if prev is None:
                rows[r] = rng.choice(lens[r], k, replace=False)
            else:   # the second call reuses half of the first call's tokens
                kept = rng.choice(prev[r], k // 2, replace=False)
                rest = rng.choice(np.setdiff1d(np.arange(lens[r]), kept), k - k // 2, replace=False)
                rows[r] = rng.permutation(np.concatenate([kept, rest]))
        prev = rows
        topk = torch.from_numpy(rows).cuda()
        regular.swap_in(0, topk, seq, out_a)
        noalloc.swap_in_noalloc(0, topk, seq, out_b)
        torch.cuda.synchronize()
        assert torch.equal(out_a, out_b), f"slot ids differ on call {call}"
        assert torch.equal(regular.status(), noalloc.status())
        for a, b in zip(regular.read_state(0), noalloc.read_state(0)):
            assert np.array_equal(a, b), f"hot state differs on call {call}"
        assert torch.equal(regular.device_buffer(0), noalloc.device_buffer(0)), \
            f"device rows differ on call {call}"
    regular.close()
    noalloc.close()


def test_noalloc_refuses_a_handle_larger_than_its_array():
    # (2 * 2048 + 1) * 512 int32 values = 8,390,656 B > the 8 MiB array
    w = W.custom(512, 2048, 2048, [2049] * 512, row_bytes=16)
    g = H.HiSparse.for_workload(w)
    t = torch.zeros((512, 2048), dtype=torch.int32, device="cuda")
    seq = torch.from_numpy(w.seq_lens0).cuda()
    out = torch.empty_like(t)
    with pytest.raises(H.HiSparseError) as e:
        g.swap_in_noalloc(0, t, seq, out)
    assert e.value.code == H.ERR_UNSUPPORTED
    g.close()


_FIRST_CALL = textwrap.dedent("""
    import sys
    import numpy as np
    import torch
    sys.path.insert(0, {root!r})
    from hierarchical_sparse_kv_request_gb300 import hisparse as H
    from hierarchical_sparse_kv_request_gb300 import workload as W
    torch.cuda.set_device(0)
    w = W.custom(4, 256, 512, [3000, 400, 5000, 2000], row_bytes=64)
    g = H.HiSparse.for_workload(w)
    for r in range(w.num_requests):
        W.fill_host_rows(w, 0, r, g.host_rows(0, r), int(w.seq_lens0[r]))
    seq = torch.from_numpy(w.seq_lens0).cuda()
    g.prefill(seq)
    rng = np.random.default_rng(5)
    rows = np.stack([rng.choice(int(n), 256, replace=False) for n in w.seq_lens0]).astype(np.int32)
    topk = torch.from_numpy(rows).cuda()
    out = torch.empty((4, 256), dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    g.swap_in_noalloc(0, topk, seq, out)
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    g.swap_in_noalloc(0, topk, seq, out)
    torch.cuda.synchronize()
    free2 = torch.cuda.mem_get_info()[0]
    assert int(g.status().cpu().sum()) == 0
    print(free0, free1, free2)
""")


def test_first_noalloc_call_of_a_fresh_process_changes_no_free_memory():
    """With lazy module loading (CUDA's default, forced here) nothing the
    allocation-free call needs may be loaded on its first call: the handle's
    creation already loaded the array and looked its address up, so the
    device's free memory is the same before and after the first two calls."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, CUDA_MODULE_LOADING="LAZY")
    res = subprocess.run([sys.executable, "-c", _FIRST_CALL.format(root=root)], env=env,
                         capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stderr[-2000:]
    free0, free1, free2 = (int(x) for x in res.stdout.split()[-3:])
    assert free0 == free1 == free2, f"free device memory moved: {free0} -> {free1} -> {free2}"
