"""Decode steps whose launches follow each other on one stream with no host
synchronisation in between, as a serving loop issues them: the swap-ins of
every layer (or every verification sub-step), each into its own output and
plan buffers, then one backup launch of all layers.  With programmatic
launch on, the grids overlap on the device: a swap-in on another layer than
the launch before it reads its inputs and state while that launch still
runs, and waits for it only before its first write (one of the paths of
hisparse_set_programmatic_launch); a swap-in on the same layer waits first.
Every call's slot IDs, plans and counts, the status words, the hot state and
the device rows must equal the oracle's, bit for bit."""

import numpy as np
import pytest
import torch

from harness import Pair, assert_call_equal, assert_device_rows, assert_state_equal, status_bits
from hierarchical_sparse_kv_request_gb300 import workload as W

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    yield


def new_rows(w, seq):
    """The step's new row of every layer and request (generator rows at
    position seq[r]), as the [L][R][B] block one backup launch takes."""
    rows = np.stack([np.concatenate([W.kv_rows(w, l, r, [int(seq[r])]) for r in range(w.num_requests)])
                     for l in range(w.num_layers)])
    return rows


def run_steps(p, calls_of_step, steps, sched):
    """Launch each step's swap-ins and its backup back to back, then compare.
    calls_of_step(s) lists (layer, schedule index) per call."""
    w = p.w
    R, k = w.num_requests, w.top_k
    ncalls = len(calls_of_step(0))
    outs = [torch.empty((R, k), dtype=torch.int32, device="cuda") for _ in range(ncalls)]
    plans = [torch.empty((R, k, 2), dtype=torch.int32, device="cuda") for _ in range(ncalls)]
    cnts = [torch.empty(R, dtype=torch.int32, device="cuda") for _ in range(ncalls)]
    layers = list(range(w.num_layers))
    for s in range(steps):
        calls = calls_of_step(s)
        topks = [torch.from_numpy(np.ascontiguousarray(sched[l][c], dtype=np.int32)).cuda()
                 for l, c in calls]
        rows = new_rows(w, p.seq)
        rows_d = torch.from_numpy(rows).cuda()
        pos_d = torch.from_numpy(p.seq.copy()).cuda()
        p.gpu.status_clear()
        p.orc.status_clear()
        torch.cuda.synchronize()
        for i, (l, c) in enumerate(calls):
            p.gpu.swap_in(l, topks[i], p.seq_d, outs[i], plans[i], cnts[i])
        p.gpu.backup_layers(layers, rows_d, pos_d)
        torch.cuda.synchronize()
        want_words = np.zeros(R, dtype=np.int32)
        for i, (l, c) in enumerate(calls):
            o = p.orc.swap_in(l, sched[l][c], p.seq)
            g = (outs[i].cpu().numpy(), plans[i].cpu().numpy(), cnts[i].cpu().numpy(),
                 status_bits(o[3]))
            assert_call_equal(g, o, f"step {s} call {i} (layer {l})")
            want_words |= status_bits(o[3])
        for l in layers:
            st = p.orc.backup(l, rows[l], p.seq.copy())
            want_words |= status_bits(st)
        assert np.array_equal(p.gpu.status().cpu().numpy(), want_words), f"step {s}: status words"
        p.advance()
    for l in sorted(set(l for l, _ in calls_of_step(0))):
        s2t = assert_state_equal(p, l, f"end layer {l}")
        assert_device_rows(p, l, s2t, ctx=f"end layer {l}")


@pytest.mark.parametrize("programmatic", [False, True])
def test_mixed_len_steps_back_to_back(programmatic):
    """mixed_len (128 requests of U[2048, 81920] tokens, 4 independent
    layers): per step 4 swap-ins and a 4-layer backup, back to back."""
    w = W.make_config(3, steps=8)
    sched = W.topk_schedule(w)
    p = Pair(w, track_bytes=False)
    p.gpu.set_programmatic_launch(programmatic)
    run_steps(p, lambda s: [(l, s) for l in range(w.num_layers)], w.steps, sched)
    p.close()


@pytest.mark.parametrize("programmatic", [False, True])
def test_spec_verify_steps_back_to_back(programmatic):
    """spec_verify (256 x 32768 tokens, D 4096, 1152 B rows): per step 3
    verification sub-steps on one layer, each with its own plan, and a
    backup, back to back."""
    w = W.make_config(5, steps=4)
    sched = W.topk_schedule(w)
    p = Pair(w, track_bytes=False)
    p.gpu.set_programmatic_launch(programmatic)
    run_steps(p, lambda s: [(0, s * w.substeps + sub) for sub in range(w.substeps)], w.steps, sched)
    p.close()


@pytest.mark.parametrize("copy_ctas", [1, 4])
def test_decode_40k_layers_back_to_back(copy_ctas):
    """decode_40k shapes with 4 independent layers (32 x 40000 tokens,
    k 2048, D 6144): 4 swap-ins and a backup per step, programmatic launch
    on, the copy in the resolving CTA or in 3 copier CTAs per request."""
    w = W.make_config(2, steps=6)
    w.num_layers = 4
    w.anchor_of_layer = [-1] * 4
    w.backup = True                 # host room for the backed-up rows
    sched = W.topk_schedule(w)
    p = Pair(w, track_bytes=False)
    p.gpu.set_programmatic_launch(True)
    p.gpu.set_copy_ctas(copy_ctas)
    run_steps(p, lambda s: [(l, s) for l in range(w.num_layers)], w.steps, sched)
    p.close()
