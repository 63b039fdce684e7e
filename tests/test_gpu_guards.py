"""Out-of-bounds writes, checked without a sanitizer (compute-sanitizer is
not available on this machine).

Every handle here is created with HISPARSE_DEBUG_GUARDS=1: each device array
the library owns, and its pinned pool, carry a 4 KB band of a known byte on
each side, and hisparse_check_guards counts the bands that changed.  The
caller-owned outputs (slot IDs, plans, miss counts) get canary rows on both
sides in the tests themselves.  The workloads mix every path: the three copy
modes, resident pages, protected rows, a paged pool with reservations and
releases, replays onto skip layers, backups and the largest shapes.
"""

import os

import numpy as np
import pytest
import torch

from harness import Pair, assert_call_equal
from hierarchical_sparse_kv_request_gb300 import hisparse as H
from hierarchical_sparse_kv_request_gb300 import workload as W

pytestmark = pytest.mark.gpu

CANARY = -123456789


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    old = os.environ.get("HISPARSE_DEBUG_GUARDS")
    os.environ["HISPARSE_DEBUG_GUARDS"] = "1"
    yield
    if old is None:
        del os.environ["HISPARSE_DEBUG_GUARDS"]
    else:
        os.environ["HISPARSE_DEBUG_GUARDS"] = old


class Canaried:
    """Caller buffers with one canary row before and after the payload."""

    def __init__(self, R, k):
        self.R = R
        self.out = torch.full((R + 2, k), CANARY, dtype=torch.int32, device="cuda")
        self.plan = torch.full((R + 2, k, 2), CANARY, dtype=torch.int32, device="cuda")
        self.cnt = torch.full((R + 2,), CANARY, dtype=torch.int32, device="cuda")

    def views(self):
        R = self.R
        return self.out[1:R + 1], self.plan[1:R + 1], self.cnt[1:R + 1]

    def intact(self):
        R = self.R
        return bool((self.out[0] == CANARY).all() and (self.out[R + 1] == CANARY).all()
                    and (self.plan[0] == CANARY).all() and (self.plan[R + 1] == CANARY).all()
                    and self.cnt[0] == CANARY and self.cnt[R + 1] == CANARY)


@pytest.mark.parametrize("mode", [H.COPY_FUSED, H.COPY_SPLIT, H.COPY_AUTO])
def test_guards_tiny_workload_resident_and_protected(mode):
    w = W.make_config(1)
    sched = W.topk_schedule(w)[0]
    p = Pair(w, track_bytes=True, copy_mode=mode)
    p.gpu.set_protected_calls(1)
    p.orc.set_protected_calls(1)
    R, k = w.num_requests, w.top_k
    c = Canaried(R, k)
    p.out, plan, cnt = c.views()
    rng = np.random.default_rng(4)
    for step in range(w.steps):
        tab = None
        if step % 2:
            tab = np.where(rng.random((R, 1200)) < 0.1, rng.integers(0, 900, (R, 1200)), -1)
            tab = tab.astype(np.int32)
        g, o = p.swap_in(0, sched[step], plan=plan, cnt=cnt, resident=tab,
                         block_size=7 if tab is not None else 0)
        assert_call_equal(g, o, f"call {step}")
        assert c.intact(), f"caller canaries at call {step}"
        assert p.gpu.check_guards() == 0, f"library guard bands at call {step}"
    p.close()


def test_guards_shared_index_replays_and_backups():
    w = W.make_config(4, steps=3, num_requests=8)
    w.top_k, w.device_buffer_size, w.keep = 256, 512, 180
    w.seq_lens0 = np.array([300, 2000, 5000, 512, 513, 8000, 400, 3000], dtype=np.int32)
    w.capacity = (w.seq_lens0 + 8).astype(np.int64)
    sched = W.topk_schedule(w)[0]
    p = Pair(w, track_bytes=True)
    R, k = w.num_requests, w.top_k
    c = Canaried(R, k)
    p.out, plan, cnt = c.views()
    for step in range(w.steps):
        g, o = p.swap_in(0, sched[step], plan=plan, cnt=cnt)
        assert_call_equal(g, o, f"call {step}")
        p.gpu.replay_plan_layers(plan, cnt, [1, 2, 3])
        rows = np.random.default_rng(step).integers(0, 256, (4, R, w.row_bytes), dtype=np.uint8)
        p.gpu.backup_layers([0, 1, 2, 3], torch.from_numpy(rows).cuda(), p.seq_d)
        for l in range(4):
            assert (p.orc.backup(l, rows[l], p.seq) == 0).all()
        p.advance()
        torch.cuda.synchronize()
        assert c.intact()
        assert p.gpu.check_guards() == 0, f"library guard bands at step {step}"
    p.close()


def test_guards_paged_pool_program():
    from test_gpu_paged import PagedProgram
    prog = PagedProgram(6, 64, 24, 5, 2, 500, 64, copy_mode=H.COPY_SPLIT, seed=5,
                        resident_bs=7, protect=1)
    gpu = prog.gpu
    for step in range(12):
        prog.admit()
        prog.call()
        prog.grow()
        prog.release()
        assert gpu.check_guards() == 0, f"library guard bands at step {step}"
    gpu.close()


def test_guards_largest_shapes():
    """k 8192 and D 32768, the largest accepted: one request on the slow path
    at S 700,000 and one short one."""
    R, k, D = 2, 8192, 32768
    lens = [700_000, 20_000]
    w = W.custom(R, k, D, lens, row_bytes=16, seed=3, ratio=100)
    p = Pair(w, track_bytes=False)
    c = Canaried(R, k)
    p.out, plan, cnt = c.views()
    rng = np.random.default_rng(1)
    for step in range(3):
        topk = np.stack([rng.choice(S, k, replace=False) for S in lens]).astype(np.int32)
        g, o = p.swap_in(0, topk, plan=plan, cnt=cnt)
        assert_call_equal(g, o, f"call {step}")
        assert c.intact()
        assert p.gpu.check_guards() == 0
    p.close()


def test_guards_report_a_planted_overwrite():
    """The check does see a change: write one byte into a band of the
    pinned pool (host memory, so no device access goes out of bounds)."""
    w = W.custom(2, 8, 16, [10, 20], row_bytes=16, capacity=[40, 40], seed=2)
    g = H.HiSparse.for_workload(w)
    assert g.check_guards() == 0
    import ctypes
    base = g.host_rows_ptr(0, 0)
    ctypes.memset(base - 1, 0, 1)         # the last byte of the band before the pool
    assert g.check_guards() == 1
    ctypes.memset(base - 1, 0xA5, 1)
    assert g.check_guards() == 0
    g.close()
