"""Full-size parity of the four larger workloads, in the launch configuration
the benchmark times (fused resolve + copy; 16-CTA replays on a side stream
next to the stand-in compute kernel; separate plans per verification
sub-step; eager backups).

Every call's slot IDs, statuses, miss counts and plans are compared with the
oracle in full.  The hot state (maps, stamps, LRU order, ticks) is compared
in full at checkpoints, and device rows against the generator's rows of the
tokens the oracle maps there: a sample during the run, every slot at the end.
"""

import numpy as np
import pytest
import torch

from harness import Pair, assert_call_equal, assert_device_rows, assert_state_equal, status_bits
from hierarchical_sparse_kv_request_gb300 import hisparse as H
from hierarchical_sparse_kv_request_gb300 import workload as W

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    yield


@pytest.mark.parametrize("copy_ctas", [1, 2, 4])
def test_decode_40k_all_steps(copy_ctas):
    """32 x 40000 tokens, k 2048, D 6144, 656 B rows, 64 decode steps; the
    copy in the resolving CTA, or in 1 or 3 copier CTAs per request."""
    w = W.make_config(2)
    sched = W.topk_schedule(w)[0]
    p = Pair(w, track_bytes=False)
    p.gpu.set_copy_ctas(copy_ctas)
    misses = 0
    for c in range(w.steps):
        g, o = p.swap_in(0, sched[c])
        assert_call_equal(g, o, f"call {c}")
        misses += int(g[2].sum())
        if c % 16 == 15:
            s2t = assert_state_equal(p, 0, f"call {c}")
            assert_device_rows(p, 0, s2t, sample=256, seed=c, ctx=f"call {c}")
    assert_device_rows(p, 0, s2t, ctx="end")
    assert misses > 0
    p.close()


def test_decode_40k_with_resident_recent_pages():
    """decode_40k with the newest 4096 tokens of every request still in
    resident pages of 64 tokens (ids scattered over a shared pool)."""
    w = W.make_config(2, steps=16)
    sched = W.topk_schedule(w)[0]
    p = Pair(w, track_bytes=False)
    p.gpu.set_copy_ctas(2)
    R, bs = w.num_requests, 64
    nb = 40000 // bs + 1
    rng = np.random.default_rng(9)
    tab = np.full((R, nb), -1, dtype=np.int32)
    first = (40000 - 4096) // bs
    ids = rng.permutation(R * (nb - first)).reshape(R, nb - first)
    tab[:, first:] = ids
    resident_hits = 0
    for c in range(w.steps):
        g, o = p.swap_in(0, sched[c], resident=tab, block_size=bs)
        assert_call_equal(g, o, f"call {c}")
        resident_hits += int((g[0] >= H.RESIDENT_FLAG).sum())
        if c % 8 == 7:
            s2t = assert_state_equal(p, 0, f"call {c}")
            assert_device_rows(p, 0, s2t, sample=128, seed=c, ctx=f"call {c}")
    assert resident_hits > 0
    p.close()


def test_mixed_lengths_four_layers_with_backups():
    """128 requests of U[2048, 81920] tokens, 4 layers, backups every step."""
    w = W.make_config(3)
    sched = W.topk_schedule(w)
    p = Pair(w, track_bytes=False)
    assert (w.seq_lens0 <= w.device_buffer_size).any()      # some take the fast path
    for step in range(w.steps):
        for l in range(w.num_layers):
            g, o = p.swap_in(l, sched[l][step])
            assert_call_equal(g, o, f"step {step} layer {l}")
        for l in range(w.num_layers):
            st = p.backup(l, p.seq.copy())
            assert (st == 0).all()
        p.advance()
        if step % 8 == 7:
            for l in range(w.num_layers):
                s2t = assert_state_equal(p, l, f"step {step} layer {l}")
                assert_device_rows(p, l, s2t, sample=64, seed=step, ctx=f"step {step} layer {l}")
    for l in range(w.num_layers):
        s2t = assert_state_equal(p, l, f"end layer {l}")
        assert_device_rows(p, l, s2t, ctx=f"end layer {l}")
    p.close()


def test_shared_index_replay_beside_compute():
    """1 anchor + 3 skip layers, 64 x 65536 tokens: the skip layers replay
    the anchor's plan in one 16-CTA launch on a side stream while the
    stand-in compute kernel (many short CTAs) runs on the main stream."""
    w = W.make_config(4)
    sched = W.topk_schedule(w)[0]
    p = Pair(w, track_bytes=False)
    side = torch.cuda.Stream(priority=-1)
    buf = torch.zeros(64 << 20, dtype=torch.bfloat16, device="cuda")
    for c in range(w.steps):
        t = torch.from_numpy(sched[c]).cuda()
        p.gpu.swap_in(0, t, p.seq_d, p.out, p.plan, p.cnt)
        ev = torch.cuda.Event()
        ev.record()
        side.wait_event(ev)
        p.gpu.replay_plan_layers(p.plan, p.cnt, [1, 2, 3], num_ctas=16, stream=side)
        done = torch.cuda.Event()
        done.record(side)
        H.synthetic_compute(buf, 4)
        torch.cuda.current_stream().wait_event(done)
        o = p.orc.swap_in(0, sched[c], p.seq)
        torch.cuda.synchronize()
        g = (p.out.cpu().numpy(), p.plan.cpu().numpy(), p.cnt.cpu().numpy(),
             p.gpu.status().cpu().numpy())
        assert_call_equal(g, o, f"call {c}")
        if c % 8 == 7:
            s2t = assert_state_equal(p, 0, f"call {c}")
            for l in range(4):
                assert_device_rows(p, l, s2t, sample=64, seed=c, ctx=f"call {c} layer {l}")
    s2t = assert_state_equal(p, 0, "end")
    for l in range(4):
        assert_device_rows(p, l, s2t, ctx=f"end layer {l}")
    p.close()


def test_pipelined_index_share_graph_double_buffered_plans():
    """The 16-layer pipelined index-sharing schedule (4 anchors x 3 skip
    layers) with double-buffered plans, each decode step captured once in a
    CUDA graph: replays pre-issued on a side stream between stand-in compute
    launches.  After every step the anchors' outputs, hot state and all 16
    layers' device rows match the oracle."""
    w = W.make_config(6, steps=5, num_requests=6)
    sched = W.topk_schedule(w)
    p = Pair(w, track_bytes=False)
    R, k = w.num_requests, w.top_k
    plans = [torch.empty((R, k, 2), dtype=torch.int32, device="cuda") for _ in range(2)]
    cnts = [torch.zeros(R, dtype=torch.int32, device="cuda") for _ in range(2)]
    outs = {a: torch.empty((R, k), dtype=torch.int32, device="cuda") for a in w.anchors}
    tk = {a: torch.empty((R, k), dtype=torch.int32, device="cuda") for a in w.anchors}
    side = torch.cuda.Stream(priority=-1)
    buf = torch.zeros(8 << 20, dtype=torch.bfloat16, device="cuda")
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for gi, a in enumerate(w.anchors):
            P, C = plans[gi % 2], cnts[gi % 2]
            p.gpu.swap_in(a, tk[a], p.seq_d, outs[a], P, C)
            ev = torch.cuda.Event()
            ev.record()
            side.wait_event(ev)
            p.gpu.replay_plan_layers(P, C, [a + 1, a + 2, a + 3], num_ctas=16, stream=side)
            done = torch.cuda.Event()
            done.record(side)
            H.synthetic_compute(buf, 1)
            torch.cuda.current_stream().wait_event(done)
            H.synthetic_compute(buf, 3)
    for step in range(w.steps):
        for a in w.anchors:
            tk[a].copy_(torch.from_numpy(sched[a][step]))
        graph.replay()
        torch.cuda.synchronize()
        for a in w.anchors:
            o = p.orc.swap_in(a, sched[a][step], p.seq)
            g = (outs[a].cpu().numpy(), o[1], o[2], p.gpu.status().cpu().numpy())
            assert_call_equal(g, o, f"step {step} anchor {a}")
            s2t = assert_state_equal(p, a, f"step {step} anchor {a}")
            for l in (a, a + 1, a + 2, a + 3):
                assert_device_rows(p, l, s2t, sample=None if step == w.steps - 1 else 48,
                                   seed=step, ctx=f"step {step} layer {l}")
    p.close()


def test_pipelined_index_share_full_size():
    """The benchmark's launch shape of the pipelined 16-layer schedule at full
    size: 32 requests x 40000 tokens, 4 anchors each followed by 3 skip
    layers, plans double-buffered between the groups, the whole decode step
    one CUDA graph with the replays pre-issued on a side stream next to the
    stand-in compute.  Every step: every anchor's slot IDs, statuses and miss
    counts and its hot state against the oracle; the plans left in the two
    buffers (anchors 2 and 3, which write them last) pair by pair; and the
    skip layers' device rows, a sample per layer (every slot at the end), so
    the plans of anchors 0 and 1, overwritten within the step, are checked
    by what their replays copied."""
    w = W.make_config(6, steps=10)
    sched = W.topk_schedule(w)
    p = Pair(w, track_bytes=False)
    R, k = w.num_requests, w.top_k
    plans = [torch.empty((R, k, 2), dtype=torch.int32, device="cuda") for _ in range(2)]
    cnts = [torch.zeros(R, dtype=torch.int32, device="cuda") for _ in range(2)]
    outs = {a: torch.empty((R, k), dtype=torch.int32, device="cuda") for a in w.anchors}
    tk = {a: torch.empty((R, k), dtype=torch.int32, device="cuda") for a in w.anchors}
    side = torch.cuda.Stream(priority=-1)
    buf = torch.zeros(160 << 20, dtype=torch.bfloat16, device="cuda")
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for gi, a in enumerate(w.anchors):
            P, C = plans[gi % 2], cnts[gi % 2]
            p.gpu.swap_in(a, tk[a], p.seq_d, outs[a], P, C)
            ev = torch.cuda.Event()
            ev.record()
            side.wait_event(ev)
            p.gpu.replay_plan_layers(P, C, [a + 1, a + 2, a + 3], num_ctas=16, stream=side)
            done = torch.cuda.Event()
            done.record(side)
            H.synthetic_compute(buf, 1)
            torch.cuda.current_stream().wait_event(done)
            H.synthetic_compute(buf, 3)
    misses = 0
    for step in range(w.steps):
        for a in w.anchors:
            tk[a].copy_(torch.from_numpy(sched[a][step]))
        graph.replay()
        torch.cuda.synchronize()
        assert (p.gpu.status().cpu().numpy() == 0).all(), f"step {step}: status words"
        last = {}
        for gi, a in enumerate(w.anchors):
            o = p.orc.swap_in(a, sched[a][step], p.seq)
            last[gi % 2] = o
            g = (outs[a].cpu().numpy(), o[1], o[2], status_bits(np.zeros(R)))
            assert_call_equal(g, o, f"step {step} anchor {a}")
            misses += int(o[2].sum())
            s2t = assert_state_equal(p, a, f"step {step} anchor {a}")
            final = step == w.steps - 1
            for l in (a, a + 1, a + 2, a + 3):
                assert_device_rows(p, l, s2t, sample=None if final else 32, seed=step,
                                   ctx=f"step {step} layer {l}")
        for b, o in last.items():             # anchors 2 and 3 wrote the buffers last
            g = (o[0], plans[b].cpu().numpy(), cnts[b].cpu().numpy(), status_bits(o[3]))
            assert_call_equal(g, o, f"step {step} plan buffer {b}")
    assert misses > 0
    p.close()


@pytest.mark.parametrize("protect", [0, 1])
def test_speculative_substeps_with_backups(protect):
    """256 x 32768 tokens, D 4096, 1152 B rows: 3 verification sub-steps per
    decode step, each with its own plan, then one backup per step.  With
    protect = 1 each sub-step also keeps the previous sub-step's rows."""
    w = W.make_config(5, steps=16 if protect == 0 else 6)
    sched = W.topk_schedule(w)[0]
    p = Pair(w, track_bytes=False)
    p.gpu.set_protected_calls(protect)
    p.orc.set_protected_calls(protect)
    R, k = w.num_requests, w.top_k
    plans = [torch.empty((R, k, 2), dtype=torch.int32, device="cuda") for _ in range(3)]
    cnts = [torch.empty(R, dtype=torch.int32, device="cuda") for _ in range(3)]
    for step in range(w.steps):
        oracle_calls = []
        for sub in range(w.substeps):
            g, o = p.swap_in(0, sched[step * w.substeps + sub], plan=plans[sub], cnt=cnts[sub])
            assert_call_equal(g, o, f"step {step} sub {sub}")
            oracle_calls.append(o)
        # each sub-step's plan row is still intact after the later sub-steps
        for sub, o in enumerate(oracle_calls):
            g = (o[0], plans[sub].cpu().numpy(), cnts[sub].cpu().numpy(), status_bits(o[3]))
            assert_call_equal(g, o, f"step {step} plan {sub} after the step")
        st = p.backup(0, p.seq.copy())
        assert (st == 0).all()
        p.advance()
        if step % 4 == 3:
            s2t = assert_state_equal(p, 0, f"step {step}")
            assert_device_rows(p, 0, s2t, sample=64, seed=step, ctx=f"step {step}")
    s2t = assert_state_equal(p, 0, "end")
    assert_device_rows(p, 0, s2t, ctx="end")
    p.close()
