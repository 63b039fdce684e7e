"""The per-request status word on the GPU ([Arch] "HiSparse local KV offload
architecture", Performance invariants: no device readback on the decode
path, so a data error has to stay recorded on the device until the caller
reads it).

Bit c of request r's word is set by every call that meets error code c for
r -- swap-ins on any layer, prefills, backups -- and stays set, whatever
later calls return, until hisparse_status_clear.  Here a whole decode step of
the mixed-lengths workload (4 layers, then one backup launch for all of
them) is one CUDA graph, and errors planted on early layers must still be in
the words after the graph has run; the words are compared with the oracle's
after every step, and the rest of every call element by element.
"""

import numpy as np
import pytest
import torch

import oracle as O
from harness import Pair, assert_call_equal, assert_state_equal, status_bits
from hierarchical_sparse_kv_request_gb300 import workload as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    yield


def test_layer0_error_survives_a_captured_four_layer_step():
    w = W.make_config(3, steps=7, num_requests=24)
    sched = W.topk_schedule(w)
    p = Pair(w, track_bytes=False)
    R, k, L, B = w.num_requests, w.top_k, w.num_layers, w.row_bytes
    slow = [r for r in range(R) if w.seq_lens0[r] > w.device_buffer_size]
    fast = [r for r in range(R) if w.seq_lens0[r] <= w.device_buffer_size]
    tk = [torch.empty((R, k), dtype=torch.int32, device="cuda") for _ in range(L)]
    outs = [torch.empty((R, k), dtype=torch.int32, device="cuda") for _ in range(L)]
    plans = [torch.empty((R, k, 2), dtype=torch.int32, device="cuda") for _ in range(L)]
    cnts = [torch.empty(R, dtype=torch.int32, device="cuda") for _ in range(L)]
    rows_d = torch.empty((L, R, B), dtype=torch.uint8, device="cuda")
    pos_d = torch.empty(R, dtype=torch.int32, device="cuda")
    one = torch.ones(R, dtype=torch.int32, device="cuda")
    # the layers' swap-ins and the backup follow each other with programmatic
    # dependencies inside the graph
    p.gpu.set_programmatic_launch(True)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for l in range(L):
            p.gpu.swap_in(l, tk[l], p.seq_d, outs[l], plans[l], cnts[l])
        p.gpu.backup_layers(list(range(L)), rows_d, pos_d)
        p.seq_d.add_(one)
    p.gpu.status_clear()
    p.orc.status_clear()
    planted = {}
    for step in range(w.steps):
        rows = [sched[l][step].copy() for l in range(L)]
        pos = p.seq.copy()
        if step == 1:                       # layer 0 only: a duplicate in request slow[0]
            rows[0][slow[0], 5] = rows[0][slow[0], 2]
            planted[slow[0]] = 1 << O.DUPLICATE
        if step == 3:                       # layer 0, a fast-path request: out of range
            rows[0][fast[0], 0] = p.seq[fast[0]]
            planted[fast[0]] = 1 << O.BAD_INDEX
        if step == 4:                       # a backup past the capacity, every layer
            pos[slow[1]] = int(w.host_capacity[slow[1]])
            planted[slow[1]] = 1 << O.BAD_POSITION
        for l in range(L):
            tk[l].copy_(torch.from_numpy(rows[l]))
        bk = np.stack([np.stack([W.kv_rows(w, l, r, [max(int(pos[r]), 0)])[0] for r in range(R)])
                       for l in range(L)])
        rows_d.copy_(torch.from_numpy(bk))
        pos_d.copy_(torch.from_numpy(pos))
        graph.replay()
        codes = []
        for l in range(L):
            o = p.orc.swap_in(l, rows[l], p.seq)
            codes.append(o[3])
            torch.cuda.synchronize()
            g = (outs[l].cpu().numpy(), plans[l].cpu().numpy(), cnts[l].cpu().numpy(),
                 status_bits(o[3]))
            assert_call_equal(g, o, f"step {step} layer {l}")
        for l in range(L):
            p.orc.backup(l, bk[l], pos)
        p.seq += 1
        torch.cuda.synchronize()
        got = p.gpu.status().cpu().numpy()
        want = p.orc.status_word()
        assert np.array_equal(got, want), f"step {step}: words {got} != oracle {want}"
        # every planted error is still there after the later layers and steps
        for r, bit in planted.items():
            assert got[r] & bit, f"step {step}: request {r} lost bit {bit}"
        assert got[[r for r in range(R) if r not in planted]].sum() == 0
        if step == 1:   # the later layers of the same step resolved request slow[0]
            assert all(codes[l][slow[0]] == 0 for l in range(1, L))
        if step == 5:
            p.gpu.status_clear()
            p.orc.status_clear()
            planted.clear()
            torch.cuda.synchronize()
            assert (p.gpu.status().cpu().numpy() == 0).all()
    for l in range(L):
        assert_state_equal(p, l, f"end layer {l}")
    p.close()


def test_prefill_and_swap_in_errors_accumulate_until_cleared():
    """A bad prefill length and errors of several swap-ins land in one word,
    resident-tier errors included; successful calls leave it; a clear
    empties it."""
    R, k, D = 4, 8, 32
    lens = [100, 20, 300, 100]
    w = W.custom(R, k, D, lens, row_bytes=32, capacity=[120, 40, 310, 120], seed=4)
    p = Pair(w, track_bytes=True)
    rng = np.random.default_rng(7)
    good = np.stack([rng.choice(S, k, replace=False) for S in lens]).astype(np.int32)
    g, o = p.swap_in(0, good, clear_status=False)
    assert (g[3] == 0).all()
    seq = np.array([-1, 41, -1, -1], dtype=np.int32)        # 41 > capacity 40
    p.gpu.prefill(torch.from_numpy(seq).cuda())
    assert p.orc.prefill(seq)[1] == O.BAD_SEQ_LEN
    bad = good.copy()
    bad[2, 1] = bad[2, 0]
    g, o = p.swap_in(0, bad, clear_status=False)
    assert np.array_equal(g[3], p.orc.status_word())
    tab = np.full((R, 8), -1, dtype=np.int32)
    tab[3, good[3, 0] // 16] = -7                            # a malformed resident id
    g, o = p.swap_in(0, good, resident=tab, block_size=16, clear_status=False)
    want = [0, 1 << O.BAD_SEQ_LEN, 1 << O.DUPLICATE, 1 << O.BAD_RESIDENT]
    assert g[3].tolist() == want == p.orc.status_word().tolist()
    g, o = p.swap_in(0, good, clear_status=False)            # all fine: nothing changes
    assert g[3].tolist() == want
    p.gpu.status_clear()
    torch.cuda.synchronize()
    assert (p.gpu.status().cpu().numpy() == 0).all()
    assert_state_equal(p, 0)
    p.close()
