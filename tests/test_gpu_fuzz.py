"""Random configurations, every feature mixed: request counts, top-k and
buffer sizes (D % 8 != 0 included), row sizes, skip layers, copy modes, the
allocation-free swap-in, paged host pools, protected rows, resident pages,
padding, malformed rows, backups on every layer and growth from the fast
path into the slow one.  Each call's outputs,
the hot state and every device byte are compared with the oracle."""

import numpy as np
import pytest
import torch

from harness import (Pair, assert_call_equal, assert_device_bytes_equal_oracle, assert_state_equal,
                     status_bits)
from hierarchical_sparse_kv_request_gb300 import hisparse as H
from hierarchical_sparse_kv_request_gb300 import workload as W

pytestmark = pytest.mark.gpu

CALLS = 5


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def draw_config(rng):
    # mostly small shapes; some with one, two, four and eight top-k entries
    # per thread of the 1024-thread resolver
    u = rng.random()
    if u < 0.7:
        R, k = int(rng.integers(1, 25)), int(rng.integers(1, 200))
    elif u < 0.9:
        R, k = int(rng.integers(1, 9)), int(rng.integers(200, 2100))
    else:
        R, k = int(rng.integers(1, 5)), int(rng.integers(2100, 5000))
    D = k + int(rng.integers(0, 300))
    B = int(rng.choice([16, 48, 656, 1152]))
    L = int(rng.integers(1, 4))
    anchors = [-1] + [int(rng.choice([-1, 0])) for _ in range(L - 1)]
    # short and long requests, some right at the fast-path boundary
    lens = []
    for _ in range(R):
        u = rng.random()
        S = D - int(rng.integers(0, 3)) if u < 0.2 else int(rng.integers(1, 4 * D + 2))
        lens.append(max(1, S))
    return R, k, D, B, L, anchors, lens


def draw_topk(rng, seq, k, prev):
    R = len(seq)
    topk = np.full((R, k), -1, dtype=np.int32)
    for r in range(R):
        S = int(seq[r])
        n = min(k, S)
        old = prev[r][(prev[r] >= 0) & (prev[r] < S)] if prev is not None else np.empty(0, np.int32)
        kept = rng.choice(old, min(old.size, int(rng.random() * n)), replace=False) if old.size else old
        rest = np.setdiff1d(np.arange(S), kept)
        new = rng.choice(rest, n - kept.size, replace=False)
        row = np.concatenate([kept, new]).astype(np.int32)
        if rng.random() < 0.2:                      # some padding
            row[rng.random(row.size) < 0.2] = -1
        topk[r, :n] = row
        topk[r] = rng.permutation(topk[r])
    if rng.random() < 0.3:                          # one malformed row
        r = int(rng.integers(0, R))
        valid = np.nonzero(topk[r] >= 0)[0]
        kind = rng.integers(0, 3)
        if kind == 0 and valid.size >= 2:
            topk[r, valid[1]] = topk[r, valid[0]]   # a duplicate
        elif kind == 1 and valid.size:
            topk[r, valid[0]] = int(seq[r]) + 3     # past seq_len
        elif valid.size:
            topk[r, valid[0]] = -5                  # below -1
    return topk


def check_call(p, g, o, cleared, ctx):
    """The call's results against the oracle's: the status words equal the
    oracle's words always, and the bits of the call's own codes when they
    were cleared before it."""
    assert np.array_equal(g[3], p.orc.status_word()), f"{ctx}: status words"
    if not cleared:
        g = (g[0], g[1], g[2], status_bits(o[3]))
    assert_call_equal(g, o, ctx)


@pytest.mark.parametrize("seed", range(48))
def test_random_configuration(seed):
    rng = np.random.default_rng(1000 + seed)
    R, k, D, B, L, anchors, lens = draw_config(rng)
    caps = [S + CALLS + 2 for S in lens]
    w = W.custom(R, k, D, lens, row_bytes=B, layers=L, anchor_of_layer=anchors, capacity=caps,
                 seed=seed)
    mode = [H.COPY_FUSED, H.COPY_SPLIT, H.COPY_AUTO][seed % 3]
    hb = int(rng.choice([0, 0, 1, 7, 64]))         # paged host pool, whole capacity reserved
    p = Pair(w, track_bytes=True, copy_mode=mode, host_block_tokens=hb)
    noalloc_ok = R * (2 * k + 1) * 4 <= H.NOALLOC_SCRATCH_BYTES
    protect = int(rng.choice([0, 0, 1, 2]))
    p.gpu.set_protected_calls(protect)
    p.orc.set_protected_calls(protect)
    owners = [l for l in range(L) if anchors[l] == -1]      # layer 0 first
    skips = [l for l in range(L) if anchors[l] == 0]
    ctx = f"seed {seed} (R {R} k {k} D {D} B {B} L {L} mode {mode} protect {protect} hb {hb})"
    prev = {l: None for l in owners}
    for c in range(CALLS):
        for l0 in owners:
            topk = draw_topk(rng, p.seq, k, prev[l0])
            prev[l0] = topk
            tab, bs = None, 0
            if rng.random() < 0.3:
                bs = int(rng.integers(1, 17))
                nb = int(rng.integers(1, max(2, max(caps) // bs + 2)))
                tab = np.where(rng.random((R, nb)) < 0.3, rng.integers(0, 1000, (R, nb)), -1)
                tab = tab.astype(np.int32)
            # the status words are cleared before some calls only; they must
            # equal the oracle's after every call either way
            clear = rng.random() < 0.5
            # the copy in the resolving CTA (with staged rows through shared
            # memory: none, a few, or as many as fit) or in copier CTAs
            ctas = int(rng.choice([1, 1, 2, 3, 4]))
            p.gpu.set_copy_ctas(ctas)
            p.gpu.set_stage_rows(int(rng.choice([-1, -1, 0, 1, 5])) if ctas == 1 else 0)
            p.gpu.set_programmatic_launch(bool(rng.random() < 0.5))
            if tab is None and noalloc_ok and rng.random() < 0.25:
                # the allocation-free swap-in: no plan comes back, so no replay
                if clear:
                    p.gpu.status_clear()
                    p.orc.status_clear()
                p.gpu.swap_in_noalloc(l0, torch.from_numpy(topk).cuda(), p.seq_d, p.out)
                o = p.orc.swap_in(l0, topk, p.seq)
                torch.cuda.synchronize()
                g = (p.out.cpu().numpy(), o[1], o[2], p.gpu.status().cpu().numpy())
                check_call(p, g, o, clear, f"{ctx} call {c} layer {l0} (noalloc)")
                assert_state_equal(p, l0, f"{ctx} call {c} layer {l0} (noalloc)")
                continue
            g, o = p.swap_in(l0, topk, resident=tab, block_size=bs, clear_status=clear)
            check_call(p, g, o, clear, f"{ctx} call {c} layer {l0}")
            assert_state_equal(p, l0, f"{ctx} call {c} layer {l0}")
            if l0 == 0 and skips:       # the skip layers replay layer 0's plan
                p.gpu.replay_plan_layers(p.plan, p.cnt, skips, num_ctas=int(rng.integers(1, 40)))
                for l in skips:
                    p.orc.replay(o[1], o[2], l)
                torch.cuda.synchronize()
        for l in range(L):
            assert_device_bytes_equal_oracle(p, l, f"{ctx} call {c} layer {l}")
        if rng.random() < 0.6:                      # the step's new rows, then S + 1
            for l in range(L):
                p.backup(l, p.seq.copy())
            p.advance()
            for l in range(L):
                assert_device_bytes_equal_oracle(p, l, f"{ctx} backup {c} layer {l}")
    p.close()
