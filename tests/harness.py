"""Run a workload through the CUDA library (via its C ABI) and the CPU oracle
side by side, and compare everything they produce bit for bit."""

from __future__ import annotations

from typing import Optional

import numpy as np
import torch

import oracle as O
from hierarchical_sparse_kv_request_gb300 import workload as W
from hierarchical_sparse_kv_request_gb300.hisparse import HiSparse


def reserve_interleaved(gpu, orc, caps, hb: int, blocks_per_round: int = 8, seed: int = 0):
    """Reserve every request's whole capacity on both sides in rounds of a
    few blocks per request, requests in a seeded random order each round, so
    each request's blocks are scattered over the pool."""
    rng = np.random.default_rng(seed)
    caps = [int(c) for c in caps]
    done = [0] * len(caps)
    while any(d < c for d, c in zip(done, caps)):
        reqs = [int(r) for r in rng.permutation(len(caps)) if done[r] < caps[r]]
        ntok = [min(caps[r], done[r] + blocks_per_round * hb) for r in reqs]
        gpu.host_reserve(reqs, ntok)
        assert orc.reserve(reqs, ntok) == 0
        for r, n in zip(reqs, ntok):
            done[r] = n


def fill_paged_rows(w: W.Workload, gpu, orc, layer: int, r: int, upto: int,
                    track_bytes: bool, chunk: int = 8192):
    """Generator rows of tokens [0, upto) of (layer, r) into the pool blocks
    the request holds, on both sides."""
    hb = gpu.hb
    table = gpu.host_block_table(r)
    for t0 in range(0, upto, chunk):
        t1 = min(upto, t0 + chunk)
        rows = W.kv_rows(w, layer, r, np.arange(t0, t1))
        for b in range(t0 // hb, (t1 + hb - 1) // hb):
            a, e = max(b * hb, t0), min((b + 1) * hb, t1)
            gpu.host_block_rows(layer, int(table[b]))[a - b * hb:e - b * hb] = rows[a - t0:e - t0]
            if track_bytes:
                orc.block_rows(layer, int(table[b]))[a - b * hb:e - b * hb] = rows[a - t0:e - t0]


class Pair:
    """One workload on the GPU library and on the oracle.  host_block_tokens
    > 0 runs both with a paged host pool, each request's whole capacity
    reserved up front in interleaved rounds."""

    def __init__(self, w: W.Workload, track_bytes: bool, copy_mode: Optional[int] = None,
                 host_block_tokens: int = 0):
        self.w = w
        self.track = track_bytes
        self.hb = host_block_tokens
        self.gpu = HiSparse.for_workload(w, host_block_tokens=host_block_tokens)
        if copy_mode is not None:
            self.gpu.set_copy_mode(copy_mode)
        self.orc = O.Oracle.for_workload(w, track_bytes=track_bytes,
                                         host_block_tokens=host_block_tokens)
        R, k = w.num_requests, w.top_k
        if self.hb:
            reserve_interleaved(self.gpu, self.orc, w.host_capacity, self.hb)
            for r in range(R):
                assert np.array_equal(self.gpu.host_block_table(r), self.orc.block_table(r))
        for l in range(w.num_layers):
            for r in range(R):
                n = int(w.seq_lens0[r])
                if self.hb:
                    fill_paged_rows(w, self.gpu, self.orc, l, r, n, track_bytes)
                    continue
                dst = self.gpu.host_rows(l, r)
                W.fill_host_rows(w, l, r, dst, n)
                if track_bytes:
                    self.orc.host_rows(l, r)[:n] = dst[:n]
        self.seq = w.seq_lens0.astype(np.int32).copy()
        self.seq_d = torch.from_numpy(self.seq).cuda()
        self.gpu.prefill(self.seq_d)
        self.orc.prefill(self.seq)
        self.out = torch.empty((R, k), dtype=torch.int32, device="cuda")
        self.plan = torch.empty((R, k, 2), dtype=torch.int32, device="cuda")
        self.cnt = torch.empty(R, dtype=torch.int32, device="cuda")
        self.last = None

    def close(self):
        self.gpu.close()
        self.orc.close()

    def swap_in(self, layer: int, topk: np.ndarray, plan=None, cnt=None, record_plan=True,
                resident=None, block_size: int = 0, clear_status: bool = True):
        """One call on both sides; returns (gpu results, oracle results): the
        GPU's fourth item is the library's status words, the oracle's its
        per-call status codes.  With clear_status (the default) both sides'
        status words are cleared first, so each GPU word is exactly the bit
        of the call's own code (see assert_call_equal).  With
        record_plan=False the library gets no plan to fill; the GPU
        plan/count results are then the oracle's (nothing to compare).
        resident: optional int32 [R][max_blocks] resident block table."""
        plan = self.plan if plan is None else plan
        cnt = self.cnt if cnt is None else cnt
        if clear_status:
            self.gpu.status_clear()
            self.orc.status_clear()
        t = torch.from_numpy(np.ascontiguousarray(topk, dtype=np.int32)).cuda()
        if resident is not None:
            rb = torch.from_numpy(np.ascontiguousarray(resident, dtype=np.int32)).cuda()
            self.gpu.swap_in_resident(layer, t, self.seq_d, rb, block_size, self.out,
                                      plan if record_plan else None, cnt if record_plan else None)
        elif record_plan:
            self.gpu.swap_in(layer, t, self.seq_d, self.out, plan, cnt)
        else:
            self.gpu.swap_in(layer, t, self.seq_d, self.out)
        o = self.orc.swap_in(layer, topk, self.seq, resident, block_size)
        torch.cuda.synchronize()
        if record_plan:
            g = (self.out.cpu().numpy(), plan.cpu().numpy(), cnt.cpu().numpy(),
                 self.gpu.status().cpu().numpy())
        else:
            g = (self.out.cpu().numpy(), o[1], o[2], self.gpu.status().cpu().numpy())
        self.last = (g, o)
        return g, o

    def backup(self, layer: int, positions: np.ndarray, clear_status: bool = True):
        """Back up each request's row at `positions` (generator rows); returns
        the oracle's per-call status codes.  With clear_status (the default)
        both status words are cleared first and the library's words are
        checked against the bits of those codes."""
        w = self.w
        rows = np.zeros((w.num_requests, w.row_bytes), dtype=np.uint8)
        for r in range(w.num_requests):
            if positions[r] >= 0:
                rows[r] = W.kv_rows(w, layer, r, [int(positions[r])])[0]
        rows_d = torch.from_numpy(rows).cuda()
        pos_d = torch.from_numpy(np.ascontiguousarray(positions, dtype=np.int32)).cuda()
        if clear_status:
            self.gpu.status_clear()
            self.orc.status_clear()
        self.gpu.backup(layer, rows_d, pos_d)
        st = self.orc.backup(layer, rows, positions)
        torch.cuda.synchronize()
        if clear_status:
            got = self.gpu.status().cpu().numpy()
            assert np.array_equal(got, status_bits(st)), f"backup status words {got} != {st}"
        return st

    def advance(self, delta: int = 1):
        self.seq += delta
        self.seq_d.copy_(torch.from_numpy(self.seq))


def status_bits(codes) -> np.ndarray:
    """The status word each per-call code gives on a cleared word (bit c for
    code c, 0 for OK)."""
    c = np.asarray(codes, dtype=np.int64)
    return np.where(c != 0, np.left_shift(1, c), 0).astype(np.int32)


def assert_call_equal(g, o, ctx=""):
    """g: the library's (out, plan, count, status words); o: the oracle's
    (out, plan, count, per-call codes).  The words must be the bits of the
    codes: the words were cleared before the call, or no error was recorded
    since they last were."""
    out, plan, cnt, st = g
    o_out, o_plan, o_cnt, o_st = o
    assert np.array_equal(st, status_bits(o_st)), f"{ctx}: status words {st} != codes {o_st}"
    assert np.array_equal(cnt, o_cnt), f"{ctx}: miss counts differ"
    assert np.array_equal(out, o_out), f"{ctx}: slot ids differ"
    for r in range(out.shape[0]):
        n = int(o_cnt[r])
        assert np.array_equal(plan[r, :n], o_plan[r, :n]), f"{ctx}: plan of request {r} differs"


def assert_state_equal(p: Pair, layer: int, ctx=""):
    s2t, lu, t2s, lru, ticks = p.gpu.read_state(layer)
    o_s2t, o_lu, o_t2s, o_tick = p.orc.state(layer)
    assert np.array_equal(s2t, o_s2t), f"{ctx}: slot->token maps differ"
    assert np.array_equal(lu, o_lu), f"{ctx}: LRU stamps differ"
    assert np.array_equal(t2s, o_t2s), f"{ctx}: token->slot maps differ"
    assert (ticks == o_tick).all(), f"{ctx}: ticks {set(ticks.tolist())} != {o_tick}"
    # the kernel's LRU list must be the slots sorted by the oracle's (last_used, slot)
    D = p.w.device_buffer_size
    key = o_lu.astype(np.int64) * (D + 1) + np.arange(D)[None, :]
    want = np.argsort(key, axis=1, kind="stable")
    assert np.array_equal(lru, want), f"{ctx}: LRU order differs"
    return o_s2t


def assert_device_rows(p: Pair, layer: int, slot2tok: np.ndarray, sample: Optional[int] = None,
                       seed: int = 0, ctx=""):
    """Device slots hold the generator's row of the token the oracle maps
    there (every filled slot, or a random sample of them)."""
    w = p.w
    dev = p.gpu.device_buffer(layer)
    rng = np.random.default_rng(seed)
    for r in range(w.num_requests):
        filled = np.nonzero(slot2tok[r] >= 0)[0]
        if sample is not None and filled.size > sample:
            filled = np.sort(rng.choice(filled, sample, replace=False))
        if filled.size == 0:
            continue
        got = dev[r][torch.from_numpy(filled).cuda()].cpu().numpy()
        want = W.kv_rows(w, layer, r, slot2tok[r][filled])
        bad = np.nonzero((got != want).any(axis=1))[0]
        assert bad.size == 0, f"{ctx}: request {r} slot {filled[bad[0]]} holds wrong bytes"


def assert_device_bytes_equal_oracle(p: Pair, layer: int, ctx=""):
    dev = p.gpu.device_buffer(layer).cpu().numpy()
    for r in range(p.w.num_requests):
        assert np.array_equal(dev[r], p.orc.dev_rows(layer, r)), f"{ctx}: device bytes of request {r}"
