"""Host-checked errors of calls on a live handle: each returns its code
before any GPU work, and the handle keeps working afterwards (a swap-in that
follows matches the oracle)."""

import ctypes

import numpy as np
import pytest
import torch

from harness import Pair, assert_call_equal
from hierarchical_sparse_kv_request_gb300 import hisparse as H
from hierarchical_sparse_kv_request_gb300 import workload as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def code_of(fn, *args, **kw):
    with pytest.raises(H.HiSparseError) as e:
        fn(*args, **kw)
    return e.value.code


def test_argument_errors_leave_the_handle_usable():
    R, k, D = 3, 16, 32
    lens = [20, 200, 300]
    w = W.custom(R, k, D, lens, row_bytes=64, layers=2, anchor_of_layer=[-1, 0], seed=4)
    p = Pair(w, track_bytes=True)
    g, lib = p.gpu, p.gpu.lib
    plan, cnt = p.plan, p.cnt
    rows = torch.zeros((2, R, 64), dtype=torch.uint8, device="cuda")
    topk = torch.zeros((R, k), dtype=torch.int32, device="cuda")

    assert code_of(g.set_copy_mode, 5) == H.ERR_INVALID_ARG
    assert code_of(g.set_copy_mode, 0) == H.ERR_INVALID_ARG
    assert code_of(g.set_protected_calls, -1) == H.ERR_INVALID_ARG
    # layers: out of range, a skip layer where state is needed
    assert code_of(g.swap_in, 2, topk, p.seq_d, p.out, plan, cnt) == H.ERR_LAYER
    assert code_of(g.swap_in, -1, topk, p.seq_d, p.out, plan, cnt) == H.ERR_LAYER
    assert code_of(g.swap_in, 1, topk, p.seq_d, p.out, plan, cnt) == H.ERR_LAYER
    assert code_of(g.read_state, 1) == H.ERR_LAYER
    s2t = np.full((R, D), -1, dtype=np.int32)
    lu = np.zeros((R, D), dtype=np.uint32)
    ticks = np.zeros(R, dtype=np.uint32)
    assert code_of(g.write_state, 1, s2t, lu, ticks) == H.ERR_LAYER
    assert code_of(g.backup, 2, rows[0], p.seq_d) == H.ERR_LAYER
    # replays: no layers, too many, a layer out of range
    assert code_of(g.replay_plan_layers, plan, cnt, []) == H.ERR_INVALID_ARG
    assert code_of(g.replay_plan_layers, plan, cnt, [1] * 17) == H.ERR_INVALID_ARG
    assert code_of(g.replay_plan_layers, plan, cnt, [1, 5]) == H.ERR_LAYER
    # backups: the same layer twice; rows not 16-byte aligned
    assert code_of(g.backup_layers, [0, 0], rows, p.seq_d) == H.ERR_INVALID_ARG
    odd = rows.view(-1)[8:8 + R * 64]
    assert code_of(g.backup, 0, odd, p.seq_d) == H.ERR_ALIGNMENT
    # resident pages: bad block size or table width
    tab = torch.full((R, 4), -1, dtype=torch.int32, device="cuda")
    assert code_of(g.swap_in_resident, 0, topk, p.seq_d, tab, 0, p.out, plan, cnt) == H.ERR_INVALID_ARG
    # paged-pool calls on a contiguous pool; guard check without guard bands
    assert code_of(g.host_reserve, [0], [10]) == H.ERR_INVALID_ARG
    assert code_of(g.host_release, [0]) == H.ERR_INVALID_ARG
    assert code_of(g.check_guards) == H.ERR_UNSUPPORTED
    # null pointers straight through the C ABI
    assert lib.hisparse_swap_in(g.h, 0, None, None, None, None, None) == H.ERR_INVALID_ARG
    assert lib.hisparse_prefill(g.h, None, None) == H.ERR_INVALID_ARG
    assert lib.hisparse_backup(g.h, 0, None, None, None) == H.ERR_INVALID_ARG
    torch.cuda.synchronize()

    # nothing above launched anything: the next calls match the oracle
    rng = np.random.default_rng(5)
    for c in range(3):
        t = np.stack([rng.choice(S, k, replace=False) for S in lens]).astype(np.int32)
        got, want = p.swap_in(0, t)
        assert_call_equal(got, want, f"call {c}")
    p.close()


def test_paged_handle_refuses_contiguous_pool_calls():
    w = W.custom(2, 8, 16, [10, 40], row_bytes=16, capacity=[40, 60], seed=6)
    g = H.HiSparse.for_workload(w, host_block_tokens=8)
    assert code_of(g.host_rows, 0, 0) == H.ERR_INVALID_ARG
    assert code_of(g.host_block_rows, 0, 10 ** 6) == H.ERR_INVALID_ARG
    assert code_of(g.host_block_rows, 3, 0) == H.ERR_LAYER
    assert code_of(g.host_reserve, [2], [8]) == H.ERR_INVALID_ARG      # no request 2
    assert code_of(g.host_reserve, [0], [41]) == H.ERR_INVALID_ARG     # past its capacity
    g.close()
