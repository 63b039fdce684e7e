"""Parity of the paged host pool on the GPU (through the C ABI) with the oracle.

- random programs at small and medium sizes: admissions that reserve host
  blocks and restart one request, swap-ins (some asking for rows no block
  holds), growth by reserve + backup, releases, and a pool that runs out;
  after every phase the slot IDs, plans, statuses, the whole hot state, the
  block tables, the device buffers and the pinned pool are compared in full;
- the decode workload at full size (32 x 40000, k 2048, D 6144) and the
  mixed-length and shared-index workloads with every request's blocks
  scattered over the pool, in the launch shapes the benchmark times.
"""

import numpy as np
import pytest
import torch

import oracle as O
from harness import Pair, assert_call_equal, assert_device_rows, assert_state_equal, status_bits
from hierarchical_sparse_kv_request_gb300 import hisparse as H
from hierarchical_sparse_kv_request_gb300 import workload as W
from hierarchical_sparse_kv_request_gb300.hisparse import HiSparse, HiSparseError

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    yield


def _reserve(gpu, orc, reqs, ntoks):
    """Both sides; returns the oracle's code after checking the GPU's."""
    want = orc.reserve(reqs, ntoks)
    try:
        gpu.host_reserve(reqs, ntoks)
        got = 0
    except HiSparseError as e:
        got = {H.ERR_CAPACITY: -2, H.ERR_INVALID_ARG: -1}.get(e.code, e.code)
    assert got == want, (reqs, ntoks, got, want)
    return want


class PagedProgram:
    """GPU handle and oracle side by side on one layer, driven by a seeded
    random program of admissions, calls, backups and releases."""

    def __init__(self, R, D, k, hb, ratio, cap, B, copy_mode=None, seed=0, resident_bs=0,
                 noalloc=False, protect=0):
        self.R, self.D, self.k, self.hb, self.B = R, D, k, hb, B
        self.cap = [cap] * R
        self.w = W.custom(R, k, D, [1] * R, row_bytes=B, capacity=self.cap, ratio=ratio,
                          seed=100 + seed)
        self.gpu = HiSparse.for_workload(self.w, host_block_tokens=hb)
        if copy_mode is not None:
            self.gpu.set_copy_mode(copy_mode)
        self.orc = O.Oracle.for_workload(self.w, track_bytes=True, host_block_tokens=hb)
        assert self.gpu.host_pool_info() == (hb, self.orc.pool_blocks, self.orc.pool_blocks)
        self.rng = np.random.default_rng(seed)
        self.rng_words = np.random.default_rng(seed + 7919)   # when to clear the status words
        self.resident_bs = resident_bs      # > 0: resident page tables on half the calls
        self.noalloc = noalloc              # calls through hisparse_swap_in_noalloc
        if protect:
            self.gpu.set_protected_calls(protect)
            self.orc.set_protected_calls(protect)
        self.active = [False] * R
        self.S = [0] * R
        self.gen = [0] * R          # admissions of each request index so far
        self.out = torch.empty((R, k), dtype=torch.int32, device="cuda")
        self.plan = torch.empty((R, k, 2), dtype=torch.int32, device="cuda")
        self.cnt = torch.empty(R, dtype=torch.int32, device="cuda")
        self.seen = {"admit": 0, "pool_full": 0, "no_host_row": 0, "backup_no_row": 0,
                     "slow": 0, "misses": 0, "release": 0}

    def rows(self, r, tokens):
        # a request index's rows differ between admissions
        return W.kv_rows(self.w, 0, r + self.R * self.gen[r], np.asarray(tokens))

    def write_rows(self, r, t0, t1):
        if t1 <= t0:
            return
        rows = self.rows(r, np.arange(t0, t1))
        table = self.gpu.host_block_table(r)
        hb = self.hb
        for b in range(t0 // hb, (t1 + hb - 1) // hb):
            a, e = max(b * hb, t0), min((b + 1) * hb, t1)
            self.gpu.host_block_rows(0, int(table[b]))[a - b * hb:e - b * hb] = rows[a - t0:e - t0]
            self.orc.block_rows(0, int(table[b]))[a - b * hb:e - b * hb] = rows[a - t0:e - t0]

    def check(self, ctx):
        torch.cuda.synchronize()
        s2t, lu, t2s, lru, ticks = self.gpu.read_state(0)
        o_s2t, o_lu, o_t2s, o_ticks = self.orc.state(0)
        assert np.array_equal(s2t, o_s2t), ctx
        assert np.array_equal(lu, o_lu), ctx
        assert np.array_equal(t2s, o_t2s), ctx
        assert np.array_equal(ticks, o_ticks), ctx
        key = o_lu.astype(np.int64) * (self.D + 1) + np.arange(self.D)[None, :]
        assert np.array_equal(lru, np.argsort(key, axis=1, kind="stable")), ctx
        dev = self.gpu.device_buffer(0).cpu().numpy()
        for r in range(self.R):
            assert np.array_equal(dev[r], self.orc.dev_rows(0, r)), f"{ctx}: device rows r{r}"
            assert np.array_equal(self.gpu.host_block_table(r), self.orc.block_table(r)), ctx
        info = self.gpu.host_pool_info()
        assert info[2] == self.orc.free_blocks(), ctx
        for b in range(info[1]):
            assert np.array_equal(self.gpu.host_block_rows(0, b), self.orc.block_rows(0, b)), \
                f"{ctx}: pool block {b}"

    def check_words(self, ctx):
        """The status words, never cleared by the program except before
        some calls, equal the oracle's on both sides of every phase."""
        got = self.gpu.status().cpu().numpy()
        want = self.orc.status_word()
        assert np.array_equal(got, want), f"{ctx}: status words {got} != {want}"

    def admit(self):
        for r in range(self.R):
            if self.active[r] or self.rng.random() >= 0.5:
                continue
            S0 = int(self.rng.integers(self.k // 2, min(self.cap[r] - 1, 3 * self.D)))
            if _reserve(self.gpu, self.orc, [r], [S0 + 1]) == -2:
                self.seen["pool_full"] += 1
                continue
            self.gen[r] += 1
            self.write_rows(r, 0, S0)
            seq = np.full(self.R, -1, dtype=np.int32)
            seq[r] = S0
            self.gpu.prefill(torch.from_numpy(seq).cuda())
            ost = self.orc.prefill(seq)
            torch.cuda.synchronize()
            assert ost[r] == 0
            self.check_words("admit")
            self.active[r] = True
            self.S[r] = S0
            self.seen["admit"] += 1

    def call(self):
        R, k = self.R, self.k
        topk = np.full((R, k), -1, dtype=np.int32)
        seq = np.zeros(R, dtype=np.int32)
        for r in range(R):
            if not self.active[r]:
                continue
            # sometimes a length past the reserved blocks, with its last
            # position asked for: no block holds that row
            held = len(self.gpu.host_block_table(r)) * self.hb
            lie = held + 3 <= self.cap[r] and self.rng.random() < 0.15
            Sc = held + 1 + int(self.rng.integers(0, 3)) if lie else self.S[r]
            seq[r] = Sc
            kk = min(k, Sc)
            if lie:
                topk[r, 0] = Sc - 1
                topk[r, 1:kk] = self.rng.choice(Sc - 1, kk - 1, replace=False)
            else:
                # mostly recent tokens, as an indexer's picks tend to be
                recent = self.rng.random(kk) < 0.6
                cand = np.where(recent, Sc - 1 - self.rng.integers(0, min(Sc, 2 * self.D), kk),
                                self.rng.integers(0, Sc, kk))
                picked = list(dict.fromkeys(cand.tolist()))
                if len(picked) < kk:
                    rest = np.setdiff1d(np.arange(Sc), picked)
                    picked += self.rng.choice(rest, kk - len(picked), replace=False).tolist()
                topk[r, :kk] = picked[:kk]
            if self.rng.random() < 0.2:
                topk[r, self.rng.integers(0, k)] = -1
        t = torch.from_numpy(topk).cuda()
        cleared = self.rng_words.random() < 0.5
        if cleared:
            self.gpu.status_clear()
            self.orc.status_clear()
        if self.resident_bs and self.rng.random() < 0.5:
            bs = self.resident_bs
            nb = -(-max(self.cap) // bs)
            tab = np.where(self.rng.random((R, nb)) < 0.2,
                           self.rng.integers(0, 1000, (R, nb)), -1).astype(np.int32)
            self.gpu.swap_in_resident(0, t, torch.from_numpy(seq).cuda(),
                                      torch.from_numpy(tab).cuda(), bs, self.out, self.plan,
                                      self.cnt)
            o = self.orc.swap_in(0, topk, seq, tab, bs)
            self.seen["resident_calls"] = self.seen.get("resident_calls", 0) + 1
        elif self.noalloc:
            self.gpu.swap_in_noalloc(0, t, torch.from_numpy(seq).cuda(), self.out)
            o = self.orc.swap_in(0, topk, seq)
        else:
            self.gpu.swap_in(0, t, torch.from_numpy(seq).cuda(), self.out, self.plan, self.cnt)
            o = self.orc.swap_in(0, topk, seq)
        torch.cuda.synchronize()
        if self.noalloc:       # no plan comes back: compare what does
            g = (self.out.cpu().numpy(), o[1], o[2], self.gpu.status().cpu().numpy())
        else:
            g = (self.out.cpu().numpy(), self.plan.cpu().numpy(), self.cnt.cpu().numpy(),
                 self.gpu.status().cpu().numpy())
        self.check_words("paged call")
        if cleared:
            assert_call_equal(g, o, "paged call")
        else:        # the words keep earlier errors: compare the rest of the call
            assert_call_equal((g[0], g[1], g[2], status_bits(o[3])), o, "paged call")
        self.seen["no_host_row"] += int((o[3] == H.STATUS_NO_HOST_ROW).sum())
        self.seen["slow"] += int(((seq > self.D) & np.array(self.active)).sum())
        self.seen["misses"] += int(g[2].sum())

    def grow(self):
        R = self.R
        pos = np.full(R, -1, dtype=np.int32)
        for r in range(R):
            if not self.active[r]:
                continue
            held = len(self.gpu.host_block_table(r)) * self.hb
            if self.rng.random() < 0.1 and held < self.cap[r]:
                pos[r] = held          # a scheduler that forgot to reserve
                continue
            if self.S[r] + 1 <= self.cap[r]:
                if _reserve(self.gpu, self.orc, [r], [self.S[r] + 1]) == -2:
                    self.seen["pool_full"] += 1
            if self.S[r] < self.cap[r]:
                pos[r] = self.S[r]
        rows = np.zeros((R, self.B), dtype=np.uint8)
        for r in range(R):
            if pos[r] >= 0:
                rows[r] = self.rows(r, [int(pos[r])])[0]
        self.gpu.backup(0, torch.from_numpy(rows).cuda(), torch.from_numpy(pos).cuda())
        ost = self.orc.backup(0, rows, pos)
        torch.cuda.synchronize()
        self.check_words("backup")
        for r in range(R):
            if pos[r] < 0:
                continue
            if ost[r] == O.NO_HOST_ROW:
                self.seen["backup_no_row"] += 1
                continue
            assert ost[r] == 0 and pos[r] == self.S[r]
            self.S[r] += 1

    def release(self):
        for r in range(self.R):
            if self.active[r] and (self.S[r] >= self.cap[r] or self.rng.random() < 0.08):
                self.gpu.host_release([r])
                assert self.orc.release([r]) == 0
                self.active[r] = False
                self.seen["release"] += 1

    def run(self, steps):
        for step in range(steps):
            self.admit()
            self.check(f"step {step} admit")
            self.call()
            self.check(f"step {step} call")
            self.grow()
            self.check(f"step {step} grow")
            self.release()
        self.gpu.close()
        return self.seen


@pytest.mark.parametrize("R,D,k,hb,ratio,cap,B,mode", [
    (8, 64, 24, 5, 2, 600, 64, None),             # odd block size, tight pool
    (8, 64, 24, 16, 1, 600, 64, H.COPY_SPLIT),
    (4, 64, 24, 16, 1, 600, 64, H.COPY_AUTO),
    (4, 1200, 1100, 64, 2, 4000, 656, None),      # two top-k entries per thread
    (3, 1002, 900, 32, 3, 3500, 144, None),       # D % 8 != 0: LRU list read directly
])
def test_random_paged_program(R, D, k, hb, ratio, cap, B, mode):
    prog = PagedProgram(R, D, k, hb, ratio, cap, B, copy_mode=mode, seed=R * 1000 + hb)
    seen = prog.run(24 if D < 1000 else 10)
    assert seen["admit"] > 0 and seen["slow"] > 0 and seen["misses"] > 0 and seen["release"] > 0, seen
    if D < 1000:
        assert seen["pool_full"] > 0 and seen["no_host_row"] > 0 and seen["backup_no_row"] > 0, seen


def test_random_paged_program_with_resident_pages():
    """The resident-page tier in front of a paged host pool: resident
    positions need no host row, so a request can resolve even where its
    blocks are missing, as long as every miss has one."""
    prog = PagedProgram(6, 64, 24, 8, 2, 500, 64, seed=77, resident_bs=7)
    seen = prog.run(24)
    assert seen.get("resident_calls", 0) > 0 and seen["misses"] > 0 and seen["slow"] > 0, seen


@pytest.mark.parametrize("noalloc,protect", [(True, 0), (False, 2), (True, 1)])
def test_random_paged_program_noalloc_and_protected(noalloc, protect):
    """The allocation-free split copy and protected rows on a paged pool."""
    prog = PagedProgram(6, 64, 24, 8, 2, 500, 64, seed=91 + protect, noalloc=noalloc,
                        protect=protect)
    seen = prog.run(20)
    assert seen["misses"] > 0 and seen["slow"] > 0, seen


def test_paged_graph_capture_and_reserve_on_stream():
    """Swap-ins captured in a CUDA graph read the block table the stream
    ordered before them, and a reservation enqueued on a side stream is seen
    by a swap-in ordered after it by an event."""
    R, D, k, hb = 4, 64, 16, 8
    w = W.custom(R, k, D, [300] * R, row_bytes=64, capacity=[400] * R, ratio=8, seed=5)
    gpu = HiSparse.for_workload(w, host_block_tokens=hb)
    orc = O.Oracle.for_workload(w, track_bytes=True, host_block_tokens=hb)
    side = torch.cuda.Stream()
    ev = torch.cuda.Event()
    with torch.cuda.stream(side):
        gpu.host_reserve(list(range(R)), [300] * R, stream=side)
        ev.record(side)
    torch.cuda.current_stream().wait_event(ev)
    assert orc.reserve(list(range(R)), [300] * R) == 0
    for r in range(R):
        table = gpu.host_block_table(r)
        rows = W.kv_rows(w, 0, r, np.arange(300))
        for b, blk in enumerate(table):
            part = rows[b * hb:(b + 1) * hb]
            gpu.host_block_rows(0, int(blk))[:len(part)] = part
            orc.block_rows(0, int(blk))[:len(part)] = part
    seq = torch.full((R,), 300, dtype=torch.int32, device="cuda")
    gpu.prefill(seq)
    orc.prefill([300] * R)
    rng = np.random.default_rng(3)
    topk_d = torch.empty((R, k), dtype=torch.int32, device="cuda")
    out = torch.empty((R, k), dtype=torch.int32, device="cuda")
    plan = torch.empty((R, k, 2), dtype=torch.int32, device="cuda")
    cnt = torch.empty(R, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        gpu.swap_in(0, topk_d, seq, out, plan, cnt, stream=s)
    for c in range(6):
        topk = np.stack([rng.choice(300, k, replace=False) for _ in range(R)]).astype(np.int32)
        topk_d.copy_(torch.from_numpy(topk))
        g.replay()
        o = orc.swap_in(0, topk, [300] * R)
        torch.cuda.synchronize()
        assert_call_equal((out.cpu().numpy(), plan.cpu().numpy(), cnt.cpu().numpy(),
                           gpu.status().cpu().numpy()), o, f"graph call {c}")
    dev = gpu.device_buffer(0).cpu().numpy()
    for r in range(R):
        assert np.array_equal(dev[r], orc.dev_rows(0, r))
    gpu.close()


def test_reserve_and_release_host_errors():
    """Host-side checks of the pool calls, and that they change nothing."""
    w = W.custom(2, 4, 8, [10, 10], row_bytes=16, capacity=[40, 40], ratio=1, seed=1)
    gpu = HiSparse.for_workload(w, host_block_tokens=4)       # 16 rows: 4 blocks
    assert gpu.host_pool_info() == (4, 4, 4)
    with pytest.raises(HiSparseError) as e:
        gpu.host_reserve([0], [17])                           # 5 blocks wanted
    assert e.value.code == H.ERR_CAPACITY
    assert gpu.host_pool_info()[2] == 4 and gpu.host_block_table(0).size == 0
    for bad in ([2], [-1]):
        with pytest.raises(HiSparseError) as e:
            gpu.host_reserve(bad, [1])
        assert e.value.code == H.ERR_INVALID_ARG
    with pytest.raises(HiSparseError):
        gpu.host_reserve([0], [41])                           # past the capacity
    gpu.host_reserve([1, 0], [5, 4])
    assert gpu.host_block_table(1).tolist() == [0, 1] and gpu.host_block_table(0).tolist() == [2]
    with pytest.raises(HiSparseError):
        gpu.host_release([0, 5])
    assert gpu.host_pool_info()[2] == 1
    gpu.host_release([1])
    assert gpu.host_pool_info()[2] == 3 and gpu.host_block_table(1).size == 0
    with pytest.raises(HiSparseError):
        gpu.host_rows(0, 0)                                   # no per-request region
    with pytest.raises(HiSparseError):
        gpu.host_block_rows(0, 4)
    gpu.close()
    flat = HiSparse.for_workload(W.custom(2, 4, 8, [8, 8], row_bytes=16, capacity=[8, 8],
                                          ratio=1, seed=1))
    with pytest.raises(HiSparseError):
        flat.host_reserve([0], [1])
    assert flat.host_pool_info() == (0, 0, 0)
    flat.close()


# ---- full-size workloads with scattered blocks --------------------------------

@pytest.mark.slow
def test_decode_40k_paged():
    """decode_40k with 64-token host blocks scattered over the pool."""
    w = W.make_config(2, steps=24)
    sched = W.topk_schedule(w)[0]
    p = Pair(w, track_bytes=False, host_block_tokens=64)
    t0 = p.gpu.host_block_table(0)
    assert (np.diff(t0) != 1).any()                           # not one run of ids
    misses = 0
    for c in range(w.steps):
        g, o = p.swap_in(0, sched[c])
        assert_call_equal(g, o, f"call {c}")
        misses += int(g[2].sum())
        if c % 8 == 7:
            s2t = assert_state_equal(p, 0, f"call {c}")
            assert_device_rows(p, 0, s2t, sample=256, seed=c, ctx=f"call {c}")
    assert_device_rows(p, 0, s2t, ctx="end")
    assert misses > 0
    p.close()


@pytest.mark.slow
def test_mixed_lengths_paged_with_backups():
    """32 requests of U[2048, 81920] tokens, 4 layers, backups every step,
    host blocks of 32 tokens."""
    w = W.make_config(3, steps=6, num_requests=32)
    sched = W.topk_schedule(w)
    p = Pair(w, track_bytes=False, host_block_tokens=32)
    for step in range(w.steps):
        for l in w.anchors:
            g, o = p.swap_in(l, sched[l][step])
            assert_call_equal(g, o, f"step {step} layer {l}")
        for l in range(w.num_layers):
            st = p.backup(l, p.seq.copy())
            assert (st == 0).all()
        p.advance()
    for l in w.anchors:
        s2t = assert_state_equal(p, l, "end")
        assert_device_rows(p, l, s2t, sample=64, seed=l, ctx=f"layer {l}")
    p.close()


@pytest.mark.slow
def test_shared_index_paged_replay():
    """The anchor's plan (pool rows) replayed onto three skip layers."""
    w = W.make_config(4, steps=4, num_requests=16)
    sched = W.topk_schedule(w)[0]
    p = Pair(w, track_bytes=False, host_block_tokens=64)
    side = torch.cuda.Stream()
    for c in range(w.steps):
        g, o = p.swap_in(0, sched[c])
        assert_call_equal(g, o, f"call {c}")
        ev = torch.cuda.Event()
        ev.record()
        side.wait_event(ev)
        p.gpu.replay_plan_layers(p.plan, p.cnt, [1, 2, 3], stream=side)
        torch.cuda.synchronize()
    s2t = assert_state_equal(p, 0, "end")
    for l in range(w.num_layers):
        assert_device_rows(p, l, s2t, sample=128, seed=l, ctx=f"layer {l}")
    p.close()
