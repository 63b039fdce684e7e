"""Parity of the CUDA library (called through its C ABI) with the CPU oracle.

Every comparison is exact (tolerance 0): slot IDs, statuses, miss plans,
slot<->token maps, LRU stamps and order, ticks and device buffer bytes.
"""

import numpy as np
import pytest
import torch

import oracle as O
from golden_trace import load, names
from harness import (Pair, assert_call_equal, assert_device_bytes_equal_oracle,
                     assert_device_rows, assert_state_equal, status_bits)
from hierarchical_sparse_kv_request_gb300 import hisparse as H
from hierarchical_sparse_kv_request_gb300 import workload as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    yield


# ----------------------------------------------------------------------------
# hand-derived golden traces, on the GPU
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("name", names())
def test_golden_trace_gpu(name):
    layout, ops = load(name)
    S0 = ops[0][1]["S"]
    w = W.custom(1, layout["k"], layout["D"], [S0], capacity=[layout["cap"]])
    p = Pair(w, track_bytes=True)
    if layout.get("protect"):
        p.gpu.set_protected_calls(layout["protect"])
        p.orc.set_protected_calls(layout["protect"])
    # a trace that states status words keeps them across its ops (cleared
    # only by its own `clear` lines); the others clear them before each op
    words = any(op == "clear" or "word" in a or "word" in a.get("expect", {})
                for op, a in ops)
    resident = None
    for i, (op, a) in enumerate(ops[1:]):
        if op == "resident":
            resident = np.array([a["ids"]], dtype=np.int32)
            continue
        if op == "clear":
            p.gpu.status_clear()
            p.orc.status_clear()
            continue
        if op in ("backup", "prefill"):
            if op == "backup":
                st = p.backup(0, np.array([a["pos"]], dtype=np.int32), clear_status=not words)
            else:
                p.gpu.prefill(torch.tensor([a["S"]], dtype=torch.int32, device="cuda"))
                st = p.orc.prefill([a["S"]])
                torch.cuda.synchronize()
            assert st[0] == a["status"]
            if "word" in a:
                assert int(p.gpu.status().cpu()[0]) == a["word"] == int(p.orc.status_word()[0])
            continue
        if a["S"] != p.seq[0]:                # grown by backups since the last call
            p.advance(a["S"] - int(p.seq[0]))
        g, o = p.swap_in(0, np.array([a["topk"]], dtype=np.int32), resident=resident,
                         block_size=layout.get("bs", 0), clear_status=not words)
        e = a["expect"]
        out, plan, cnt, st = g
        if words:
            assert int(st[0]) == e["word"] == int(p.orc.status_word()[0])
            assert int(o[3][0]) == e["status"]
            g = (out, plan, cnt, status_bits(o[3]))   # the rest of the call, compared below
        assert_call_equal(g, o, f"{name} op {i}")
        assert out[0].tolist() == e["out"]
        if not words:
            assert int(st[0]) == (1 << e["status"] if e["status"] else 0)
        assert [tuple(x) for x in plan[0, : cnt[0]].tolist()] == e["plan"]
        s2t = assert_state_equal(p, 0, f"{name} op {i}")
        assert s2t[0].tolist() == e["slot2tok"]
        lu = p.gpu.read_state(0)[1]
        assert lu[0].tolist() == e["last_used"]
        assert_device_bytes_equal_oracle(p, 0, f"{name} op {i}")
    p.close()


# ----------------------------------------------------------------------------
# the tiny workload, every byte every call
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("mode", [H.COPY_FUSED, H.COPY_SPLIT, H.COPY_AUTO])
def test_tiny_workload_full_parity(mode):
    w = W.make_config(1)
    sched = W.topk_schedule(w)[0]
    p = Pair(w, track_bytes=True, copy_mode=mode)
    for c in range(w.steps):
        g, o = p.swap_in(0, sched[c])
        assert_call_equal(g, o, f"call {c}")
        assert_state_equal(p, 0, f"call {c}")
        assert_device_bytes_equal_oracle(p, 0, f"call {c}")
    assert g[2][0] == 0                  # the short request never misses
    assert g[2][1:].sum() > 0
    p.close()


@pytest.mark.parametrize("mode", [H.COPY_FUSED, H.COPY_SPLIT])
def test_arguments_in_pinned_host_memory(mode):
    """Top-k rows, sequence lengths, slot IDs and plans may live in pinned
    host memory: the kernels read and write them over the host link.  Eager
    calls and calls replayed from a CUDA graph both match the oracle."""
    w = W.make_config(1)
    sched = W.topk_schedule(w)[0]
    p = Pair(w, track_bytes=True, copy_mode=mode)
    R, k = w.num_requests, w.top_k
    topk_h = torch.empty((R, k), dtype=torch.int32).pin_memory()
    seq_h = torch.from_numpy(p.seq.copy()).pin_memory()
    out_h = torch.empty((R, k), dtype=torch.int32).pin_memory()
    plan_h = torch.empty((R, k, 2), dtype=torch.int32).pin_memory()
    cnt_h = torch.empty(R, dtype=torch.int32).pin_memory()

    def check(c):
        o = p.orc.swap_in(0, sched[c], p.seq)
        torch.cuda.synchronize()
        g = (out_h.numpy().copy(), plan_h.numpy().copy(), cnt_h.numpy().copy(),
             p.gpu.status().cpu().numpy())
        assert_call_equal(g, o, f"call {c}")

    half = w.steps // 2
    for c in range(half):
        topk_h.numpy()[:] = sched[c]
        p.gpu.swap_in(0, topk_h.data_ptr(), seq_h.data_ptr(), out_h.data_ptr(),
                      plan_h.data_ptr(), cnt_h.data_ptr())
        check(c)
    graph = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(graph):
        p.gpu.swap_in(0, topk_h.data_ptr(), seq_h.data_ptr(), out_h.data_ptr(),
                      plan_h.data_ptr(), cnt_h.data_ptr())
    for c in range(half, w.steps):
        topk_h.numpy()[:] = sched[c]
        graph.replay()
        check(c)
    assert_state_equal(p, 0, "end")
    assert_device_bytes_equal_oracle(p, 0, "end")
    p.close()


@pytest.mark.parametrize("protect,mode,resident", [(1, H.COPY_FUSED, False),
                                                    (2, H.COPY_FUSED, False),
                                                    (2, H.COPY_SPLIT, False),
                                                    (3, H.COPY_AUTO, False),
                                                    (2, H.COPY_FUSED, True)])
def test_protected_slots_parity(protect, mode, resident):
    """Slots of each request's last P calls are kept; calls that would need
    them fail with CAPACITY on both sides, everything else matches."""
    R, k, D, S = 12, 24, 64, 300
    lens = [S] * (R - 2) + [40, 64]          # two requests on the fast path
    w = W.custom(R, k, D, lens, row_bytes=64, seed=21)
    p = Pair(w, track_bytes=True, copy_mode=mode)
    p.gpu.set_protected_calls(protect)
    p.orc.set_protected_calls(protect)
    rng = np.random.default_rng(protect * 10 + mode)
    failed = 0
    for c in range(24):
        topk = np.full((R, k), -1, dtype=np.int32)
        for r in range(R):
            n = min(k, lens[r])
            # half the picks among the last 2D tokens, so hits also occur
            pool = rng.choice(lens[r], n, replace=False) if rng.random() < 0.5 else \
                lens[r] - 1 - rng.choice(min(lens[r], 2 * D), n, replace=False)
            topk[r, :n] = pool
        if resident:     # resident pages of 5 tokens, about a quarter of them
            tab = np.where(rng.random((R, 64)) < 0.25, rng.integers(0, 500, (R, 64)), -1)
            g, o = p.swap_in(0, topk, resident=tab.astype(np.int32), block_size=5)
        else:
            g, o = p.swap_in(0, topk)
        assert_call_equal(g, o, f"call {c}")
        failed += int((o[3] == H.STATUS_CAPACITY).sum())
        assert_state_equal(p, 0, f"call {c}")
        assert_device_bytes_equal_oracle(p, 0, f"call {c}")
    if protect >= 2 and not resident:
        assert failed > 0
    p.close()


@pytest.mark.parametrize("record_plan", [True, False])
def test_auto_copy_defers_requests_with_many_misses(record_plan):
    """Auto copy mode: requests whose misses exceed 256 KB leave them to the
    full-GPU copy grid, the others copy their own; results are unchanged.
    (Deferral applies to batches of fewer than 8 requests.)"""
    R, k, D = 4, 512, 1024
    lens = [600, 20000, 20000, 5000]           # short / cold / cold / cold
    w = W.custom(R, k, D, lens, row_bytes=1152)
    p = Pair(w, track_bytes=True, copy_mode=H.COPY_AUTO)
    rng = np.random.default_rng(21)
    topk = _random_rows(rng, R, k, lens)
    topk[3] = np.arange(5000 - k, 5000)        # request 3 hits everything
    for c in range(4):
        g, o = p.swap_in(0, topk, record_plan=record_plan)
        assert_call_equal(g, o, f"call {c}")
        assert_state_equal(p, 0, f"call {c}")
        assert_device_bytes_equal_oracle(p, 0, f"call {c}")
        if c == 0:   # requests 1 and 2 missed > 256 KB and were deferred
            assert (o[2][1:3] * w.row_bytes > 256 << 10).all() and o[2][3] == 0
        topk = _reuse_rows(rng, topk, lens, keep=0.9 if c else 0.5)
    p.close()


@pytest.mark.parametrize("R,k,D,B,lens_of", [
    # one request misses ~all of k = 2048 rows of 1152 B, the others are on
    # the fast path or miss little
    (16, 2048, 4096, 1152, lambda R: [60000] + [3000] * 7 + [9000] * (R - 8)),
    # more requests than SMs: the CTAs run in two waves
    (200, 128, 256, 1152, lambda R: [600 + 30 * (r % 7) for r in range(R)]),
])
def test_unbalanced_misses(R, k, D, B, lens_of):
    """Requests whose miss volumes differ by orders of magnitude, eager and
    from a CUDA graph, match the oracle byte for byte."""
    lens = lens_of(R)
    w = W.custom(R, k, D, lens, row_bytes=B, seed=31)
    p = Pair(w, track_bytes=True)
    rng = np.random.default_rng(32)
    topk = _random_rows(rng, R, k, lens)
    for c in range(5):
        g, o = p.swap_in(0, topk, record_plan=c % 2 == 0)
        assert_call_equal(g, o, f"call {c}")
        assert_state_equal(p, 0, f"call {c}")
        assert_device_bytes_equal_oracle(p, 0, f"call {c}")
        topk = _reuse_rows(rng, topk, lens, keep=0.3 if c < 2 else 0.8)
        topk[0] = _random_rows(rng, 1, k, lens[:1])[0]     # request 0 keeps missing
    t = torch.from_numpy(topk).cuda()
    graph = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(graph):
        p.gpu.swap_in(0, t, p.seq_d, p.out, p.plan, p.cnt)
    for c in range(5, 9):
        t.copy_(torch.from_numpy(topk))
        graph.replay()
        o = p.orc.swap_in(0, topk, p.seq)
        torch.cuda.synchronize()
        g = (p.out.cpu().numpy(), p.plan.cpu().numpy(), p.cnt.cpu().numpy(),
             p.gpu.status().cpu().numpy())
        assert_call_equal(g, o, f"graph call {c}")
        topk = _reuse_rows(rng, topk, lens, keep=0.5)
        topk[0] = _random_rows(rng, 1, k, lens[:1])[0]
    assert_state_equal(p, 0, "end")
    assert_device_bytes_equal_oracle(p, 0, "end")
    p.close()


def test_split_copy_with_the_librarys_own_plan():
    """Split copy mode without a caller plan: the resolve grid records the
    misses in the handle's internal plan and the copy grid reads them."""
    w = W.make_config(1)
    sched = W.topk_schedule(w)[0]
    p = Pair(w, track_bytes=True, copy_mode=H.COPY_SPLIT)
    for c in range(w.steps):
        g, o = p.swap_in(0, sched[c], record_plan=False)
        assert_call_equal(g, o, f"call {c}")
        assert_state_equal(p, 0, f"call {c}")
        assert_device_bytes_equal_oracle(p, 0, f"call {c}")
    p.close()


def test_swap_in_replayed_from_a_cuda_graph():
    """A swap-in (plus a skip-layer replay and a backup) captured once in a
    CUDA graph and replayed with new inputs written into the captured
    buffers gives, call after call, what the oracle gives: the tick lives on
    the device, so every replay advances the LRU ([Arch] Performance
    invariants: top-k resolution stays graph-capturable)."""
    w = W.make_config(1, steps=8)
    w.num_layers, w.anchor_of_layer = 2, [-1, 0]
    w.capacity = w.seq_lens0.astype(np.int64) + w.steps
    sched = W.topk_schedule(w)[0]
    p = Pair(w, track_bytes=True)
    R, k, B = w.num_requests, w.top_k, w.row_bytes
    topk_d = torch.empty((R, k), dtype=torch.int32, device="cuda")
    rows_d = torch.empty((R, B), dtype=torch.uint8, device="cuda")
    pos_d = torch.empty(R, dtype=torch.int32, device="cuda")
    one_d = torch.ones(R, dtype=torch.int32, device="cuda")
    topk_d.copy_(torch.from_numpy(sched[0]))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        p.gpu.swap_in(0, topk_d, p.seq_d, p.out, p.plan, p.cnt)
        p.gpu.replay_plan(p.plan, p.cnt, 1, num_ctas=4)
        p.gpu.backup(0, rows_d, pos_d)
        p.gpu.backup(1, rows_d, pos_d)
        p.seq_d.add_(one_d)
    for c in range(w.steps):
        topk_d.copy_(torch.from_numpy(sched[c]))
        pos = p.seq.copy()
        rows = np.stack([W.kv_rows(w, 0, r, [int(pos[r])])[0] for r in range(R)])
        rows_d.copy_(torch.from_numpy(rows))
        pos_d.copy_(torch.from_numpy(pos))
        graph.replay()
        o = p.orc.swap_in(0, sched[c], p.seq)
        p.orc.replay(o[1], o[2], 1)
        p.orc.backup(0, rows, pos)
        p.orc.backup(1, rows, pos)      # the skip layer backs up the same rows here
        p.seq += 1
        torch.cuda.synchronize()
        g = (p.out.cpu().numpy(), p.plan.cpu().numpy(), p.cnt.cpu().numpy(),
             p.gpu.status().cpu().numpy())
        assert_call_equal(g, o, f"graph replay {c}")
        assert_state_equal(p, 0, f"graph replay {c}")
        assert_device_bytes_equal_oracle(p, 0, f"graph replay {c}")
        assert_device_bytes_equal_oracle(p, 1, f"graph replay {c}")
    p.close()


@pytest.mark.parametrize("bs,frac,lens", [
    (16, 0.3, [3000, 400, 5000, 2100]),       # mixed fast and slow requests
    (1, 0.5, [2000, 2000, 2000, 2000]),       # one-token pages
    (64, 0.0, [3000, 3000, 3000, 3000]),      # a table with nothing resident
    (64, 1.0, [3000, 9000, 3000, 512]),       # everything resident
])
def test_resident_tier_parity(bs, frac, lens):
    """Resident pages first: random block tables per call, reuse between calls."""
    rng = np.random.default_rng(int(bs * 100 + frac * 10))
    R, k, D = 4, 256, 512
    w = W.custom(R, k, D, lens, row_bytes=48)
    p = Pair(w, track_bytes=True)
    nb = -(-max(lens) // bs) - 3                 # a table a little shorter than S
    topk = _random_rows(rng, R, k, lens)
    for c in range(6):
        tab = np.where(rng.random((R, nb)) < frac, rng.integers(0, 3000, (R, nb)), -1)
        g, o = p.swap_in(0, topk, resident=tab.astype(np.int32), block_size=bs)
        assert_call_equal(g, o, f"call {c}")
        assert_state_equal(p, 0, f"call {c}")
        assert_device_bytes_equal_oracle(p, 0, f"call {c}")
        topk = _reuse_rows(rng, topk, lens, keep=0.6)
    # a malformed id in a looked-up block sets BAD_RESIDENT and touches nothing
    before = p.gpu.read_state(0)
    tab = np.full((R, nb), -1, dtype=np.int32)
    inside = topk[1][topk[1] // bs < nb]          # a position whose block is in the table
    tab[1, inside[0] // bs] = -3
    g, o = p.swap_in(0, topk, resident=tab, block_size=bs)
    assert_call_equal(g, o, "malformed")
    assert g[3][1] == H.STATUS_BIT(H.STATUS_BAD_RESIDENT) and (g[0][1] == -1).all()
    after = p.gpu.read_state(0)
    assert np.array_equal(before[0][1], after[0][1]) and np.array_equal(before[1][1], after[1][1])
    p.close()


# ----------------------------------------------------------------------------
# edge cases
# ----------------------------------------------------------------------------

def _random_rows(rng, R, k, lens, pad=0.0):
    rows = np.empty((R, k), dtype=np.int32)
    for r in range(R):
        rows[r] = rng.choice(int(lens[r]), k, replace=False)
        if pad:
            rows[r][rng.random(k) < pad] = -1
    return rows


def _reuse_rows(rng, prev, lens, keep=0.6, pad=0.0):
    """Keep a fraction of each previous row's tokens, draw the rest anew."""
    R, k = prev.shape
    rows = np.empty_like(prev)
    for r in range(R):
        old = prev[r][prev[r] >= 0]
        kept = rng.choice(old, min(old.size, int(keep * k)), replace=False)
        pool = np.setdiff1d(np.arange(int(lens[r])), kept)
        rows[r] = rng.permutation(np.concatenate([kept, rng.choice(pool, k - kept.size, replace=False)]))
        if pad:
            rows[r][rng.random(k) < pad] = -1
    return rows


@pytest.mark.parametrize("R,k,D,lens,pad", [
    (3, 1500, 2000, [2500, 2000, 2001], 0.1),     # ragged k, S == D and D + 1
    (2, 64, 64, [64, 65], 0.0),                   # top_k == D at both sides of the edge
    (5, 1, 7, [8, 9, 100, 7, 3], 0.0),            # k = 1, odd D, tiny S
    (4, 300, 999, [5000, 1000, 999, 4321], 0.3),  # odd D, heavy padding
    (1, 4096, 8192, [200000], 0.0),               # KT = 4, long context
    (2, 8192, 8192, [9000, 8192], 0.0),           # maximum top_k, KT = 8
])
def test_edge_shapes(R, k, D, lens, pad):
    rng = np.random.default_rng(R * 7919 + k)
    w = W.custom(R, k, D, lens, row_bytes=32)
    p = Pair(w, track_bytes=True)
    topk = _random_rows(rng, R, k, lens, pad)
    for c in range(6):
        g, o = p.swap_in(0, topk)
        assert_call_equal(g, o, f"call {c}")
        assert_state_equal(p, 0, f"call {c}")
        assert_device_bytes_equal_oracle(p, 0, f"call {c}")
        topk = _reuse_rows(rng, topk, lens, keep=0.5, pad=pad)
    p.close()


def test_all_hits_then_all_misses():
    R, k, D, S = 4, 256, 512, 5000
    w = W.custom(R, k, D, [S] * R, row_bytes=64)
    p = Pair(w, track_bytes=True)
    # all hits: the newest k tokens are in the buffer after prefill
    topk = np.tile(np.arange(S - k, S, dtype=np.int32)[::-1], (R, 1))
    g, o = p.swap_in(0, topk)
    assert_call_equal(g, o)
    assert (g[2] == 0).all()
    # all misses: k tokens never resident
    topk = np.tile(np.arange(0, k, dtype=np.int32), (R, 1))
    g, o = p.swap_in(0, topk)
    assert_call_equal(g, o)
    assert (g[2] == k).all()
    assert_state_equal(p, 0)
    assert_device_bytes_equal_oracle(p, 0)
    # empty rows: all padding
    g, o = p.swap_in(0, np.full((R, k), -1, dtype=np.int32))
    assert_call_equal(g, o)
    assert (g[0] == -1).all() and (g[2] == 0).all()
    assert_state_equal(p, 0)
    p.close()


def test_malformed_rows_set_status_and_leave_state():
    R, k, D = 6, 8, 16
    lens = [100, 100, 100, 100, 10, 100]
    w = W.custom(R, k, D, lens, row_bytes=16, capacity=[120] * R)
    p = Pair(w, track_bytes=True)
    good = np.array([np.arange(8) * 3 + 1] * R, dtype=np.int32)
    good[4] = np.arange(8)   # request 4 is short (S = 10)
    g, o = p.swap_in(0, good)
    before = p.gpu.read_state(0)
    bad = good.copy()
    bad[0, 3] = 100          # == S: out of range
    bad[1, 5] = bad[1, 2]    # duplicate
    bad[2, 0] = -5           # negative, not padding
    bad[3, 1] = 7; bad[3, 2] = 7; bad[3, 7] = 500   # both: out of range wins
    bad[4, 4] = 10           # fast path, out of range (S = 10)
    g, o = p.swap_in(0, bad)
    assert_call_equal(g, o)
    assert g[3].tolist() == [1 << O.BAD_INDEX, 1 << O.DUPLICATE, 1 << O.BAD_INDEX,
                             1 << O.BAD_INDEX, 1 << O.BAD_INDEX, 0]
    assert (g[0][:5] == -1).all()
    after = p.gpu.read_state(0)
    # requests 0..4 untouched: their slot maps, stamps and LRU order
    for a, b in ((before[0], after[0]), (before[1], after[1]), (before[3], after[3])):
        assert np.array_equal(a[:5], b[:5])
    assert np.array_equal(before[2][: 5 * 120], after[2][: 5 * 120])
    assert (after[4] == 2).all()          # every request's tick advances on every call
    assert_state_equal(p, 0)
    # seq_len beyond the host capacity
    p.seq[5] = 121
    p.seq_d.copy_(torch.from_numpy(p.seq))
    g, o = p.swap_in(0, good)
    assert_call_equal(g, o)
    assert g[3][5] == 1 << O.BAD_SEQ_LEN
    assert_state_equal(p, 0)
    p.close()


@pytest.mark.parametrize("paged", [False, True])
def test_checkpoint_and_resume_with_write_state(paged):
    """hisparse_read_state -> hisparse_write_state restores a layer's hot
    state and, with rebuild_rows, its hot rows (anchor and skip layer): the
    calls that follow give what they gave the first time."""
    R, k, D, S = 6, 16, 48, 400
    lens = [S] * (R - 1) + [40]
    w = W.custom(R, k, D, lens, row_bytes=64, layers=2, anchor_of_layer=[-1, 0], seed=13)
    p = Pair(w, track_bytes=True, host_block_tokens=8 if paged else 0)
    rng = np.random.default_rng(6)
    progs = [np.stack([rng.choice(L, k, replace=False) for L in lens]).astype(np.int32)
             for _ in range(10)]
    for c in range(4):
        g, o = p.swap_in(0, progs[c])
        assert_call_equal(g, o, f"call {c}")
    saved = p.gpu.read_state(0)
    dev_saved = [p.gpu.device_buffer(l).cpu().numpy().copy() for l in range(2)]
    first = []
    for c in range(4, 10):
        g, o = p.swap_in(0, progs[c])
        assert_call_equal(g, o, f"call {c}")
        first.append(g)
    # lose the state, then restore it
    p.gpu.prefill(torch.from_numpy(np.array(lens, dtype=np.int32) // 2).cuda())
    torch.cuda.synchronize()
    s2t, lu, t2s, lru, ticks = saved
    p.gpu.write_state(0, s2t, lu, ticks, rebuild_rows=True)
    again = p.gpu.read_state(0)
    for a, b in zip(saved, again):
        assert np.array_equal(a, b)
    # the anchor's rows are back as they were, and the skip layer now holds
    # the rows of the same tokens (nothing had replayed onto it)
    dev = p.gpu.device_buffer(0).cpu().numpy()
    for r in range(R):
        filled = s2t[r] >= 0
        assert np.array_equal(dev[r][filled], dev_saved[0][r][filled]), f"anchor r{r}"
    for l in range(2):
        assert_device_rows(p, l, s2t, ctx=f"layer {l} after the rebuild")
    out = torch.empty((R, k), dtype=torch.int32, device="cuda")
    plan = torch.empty((R, k, 2), dtype=torch.int32, device="cuda")
    cnt = torch.empty(R, dtype=torch.int32, device="cuda")
    seq = torch.from_numpy(np.array(lens, dtype=np.int32)).cuda()
    for i, c in enumerate(range(4, 10)):
        p.gpu.swap_in(0, torch.from_numpy(progs[c]).cuda(), seq, out, plan, cnt)
        torch.cuda.synchronize()
        g = (out.cpu().numpy(), plan.cpu().numpy(), cnt.cpu().numpy(), p.gpu.status().cpu().numpy())
        assert_call_equal(g, first[i], f"resumed call {c}")
    bad = s2t.copy()
    bad[1, 0] = bad[1, 1] = 5                        # a token in two slots
    with pytest.raises(H.HiSparseError):
        p.gpu.write_state(0, bad, lu, ticks)
    late = lu.copy()
    late[2, 3] = ticks[2] + 1                        # a stamp from a call not made yet
    with pytest.raises(H.HiSparseError):
        p.gpu.write_state(0, s2t, late, ticks)
    p.close()


def test_backup_layers_in_one_launch():
    """hisparse_backup_layers on an anchor and two skip layers equals one
    backup per layer: host rows, device rows of short requests, maps and
    statuses (bad positions included)."""
    R, k, D = 4, 8, 32
    lens = [20, 31, 100, 300]
    w = W.custom(R, k, D, lens, row_bytes=64, layers=3, anchor_of_layer=[-1, 0, 0],
                 capacity=[40, 33, 120, 310], seed=8)
    p = Pair(w, track_bytes=True)
    rng = np.random.default_rng(2)
    for step in range(6):
        pos = p.seq.copy()
        if step == 3:
            pos[1] = 40                      # past request 1's capacity: BAD_POSITION
        if step == 4:
            pos[2] = -1                      # skipped
        rows = rng.integers(0, 256, (3, R, 64), dtype=np.uint8)
        p.gpu.status_clear()
        p.orc.status_clear()
        p.gpu.backup_layers([0, 1, 2], torch.from_numpy(rows).cuda(),
                            torch.from_numpy(pos.astype(np.int32)).cuda())
        st = [p.orc.backup(l, rows[l], pos) for l in range(3)]
        torch.cuda.synchronize()
        got = p.gpu.status().cpu().numpy()
        assert np.array_equal(got, p.orc.status_word()), f"step {step}: status words"
        assert np.array_equal(got, status_bits(st[0]))
        for l in range(3):
            assert_device_bytes_equal_oracle(p, l, f"step {step} layer {l}")
        assert_state_equal(p, 0, f"step {step}")
        p.advance()
    p.close()


def test_fast_path_grows_into_slow_path_with_backups():
    R, k, D = 3, 16, 40
    lens = [30, 38, 70]
    steps = 12
    w = W.custom(R, k, D, lens, row_bytes=48, capacity=[l + steps for l in lens])
    p = Pair(w, track_bytes=True)
    rng = np.random.default_rng(11)
    for c in range(steps):
        topk = _random_rows(rng, R, k, p.seq)
        g, o = p.swap_in(0, topk)
        assert_call_equal(g, o, f"call {c}")
        st = p.backup(0, p.seq.copy())
        assert (st == 0).all()
        p.advance()
        assert_state_equal(p, 0, f"call {c}")
        assert_device_bytes_equal_oracle(p, 0, f"call {c}")
    assert (p.seq > D).all()
    # a position outside the host capacity is reported, nothing written
    pos = np.array([-1, 10_000, -1], dtype=np.int32)
    st = p.backup(0, pos)
    assert st.tolist() == [0, O.BAD_POSITION, 0]
    assert p.gpu.status().cpu().numpy()[1] == 1 << O.BAD_POSITION
    p.close()


def test_replay_on_skip_layers_side_stream():
    R, k, D = 4, 128, 256
    lens = [3000, 256, 5000, 4000]
    w = W.custom(R, k, D, lens, row_bytes=656, layers=4,
                 anchor_of_layer=[-1, 0, 0, 0])
    p = Pair(w, track_bytes=True)
    rng = np.random.default_rng(3)
    side = torch.cuda.Stream()
    for c in range(6):
        topk = _random_rows(rng, R, k, lens)
        t = torch.from_numpy(topk).cuda()
        p.gpu.swap_in(0, t, p.seq_d, p.out, p.plan, p.cnt)
        ev = torch.cuda.Event()
        ev.record()
        side.wait_event(ev)
        if c % 2 == 0:
            for l, ctas in ((1, 1), (2, 16), (3, 152)):
                p.gpu.replay_plan(p.plan, p.cnt, l, num_ctas=ctas, stream=side)
        else:
            p.gpu.replay_plan_layers(p.plan, p.cnt, [3, 1, 2], num_ctas=3 + c, stream=side)
        done = torch.cuda.Event()
        done.record(side)
        torch.cuda.current_stream().wait_event(done)
        o_out, o_plan, o_cnt, _ = p.orc.swap_in(0, topk, p.seq)
        for l in (1, 2, 3):
            p.orc.replay(o_plan, o_cnt, l)
        torch.cuda.synchronize()
        assert np.array_equal(p.out.cpu().numpy(), o_out)
        for l in range(4):
            assert_device_bytes_equal_oracle(p, l, f"call {c} layer {l}")
    with pytest.raises(H.HiSparseError):
        p.gpu.swap_in(1, t, p.seq_d, p.out, p.plan, p.cnt)   # skip layers own no state
    p.close()


def test_largest_supported_shapes():
    # the biggest top-k / buffer / context the kernels accept
    R, k, D, S = 2, 8192, 32768, 700_000
    w = W.custom(R, k, D, [S, D], row_bytes=16)
    p = Pair(w, track_bytes=True)
    rng = np.random.default_rng(5)
    for c in range(3):
        topk = _random_rows(rng, R, k, [S, D])
        g, o = p.swap_in(0, topk)
        assert_call_equal(g, o, f"call {c}")
        assert_state_equal(p, 0, f"call {c}")
    assert_device_bytes_equal_oracle(p, 0)
    p.close()
    # 2^20 tokens with the guide's top_k / buffer
    w = W.custom(1, 2048, 6144, [1 << 20], row_bytes=16)
    p = Pair(w, track_bytes=False)
    for c in range(3):
        g, o = p.swap_in(0, _random_rows(rng, 1, 2048, [1 << 20]))
        assert_call_equal(g, o)
    s2t = assert_state_equal(p, 0)
    assert_device_rows(p, 0, s2t)
    p.close()


def test_layout_errors_through_abi():
    with pytest.raises(H.HiSparseError) as e:
        H.HiSparse(2, 1, 16, 64, 32, 10, [100, 100])            # top_k > D
    assert e.value.code == H.ERR_LAYOUT
    with pytest.raises(H.HiSparseError) as e:
        H.HiSparse(2, 1, 16, 16, 32, 1, [100, 100])             # ratio exceeded
    assert e.value.code == H.ERR_CAPACITY
    with pytest.raises(H.HiSparseError) as e:
        H.HiSparse(1, 1, 16, 8192, 32768, 1000, [1 << 20])      # shared memory
    assert e.value.code == H.ERR_UNSUPPORTED
