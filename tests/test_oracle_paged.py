"""Pins of the oracle's paged host pool (CPU only).

- a hand-worked reservation sequence, and the pool size rounded down to
  whole blocks;
- the special case that reduces to contiguous per-request regions: blocks
  reserved in request order on a fresh pool give every request consecutive
  rows, and the paged oracle must then agree with the contiguous one;
- brute force against two independent models on random programs with
  admissions, growth by backups, releases, a pool that runs out, and calls
  that need rows no block holds: the recency-list LRU (tests/lru_model.py)
  for the hot buffer and a heap-based block pool (tests/paged_model.py) plus
  a row-by-row byte model for the host pool and the device buffer.
"""

import numpy as np
import pytest

import oracle as O
from lru_model import ListLRU
from paged_model import PagedPool
from hierarchical_sparse_kv_request_gb300 import workload as W


def pin_paged_pool_rounds_down(lib_path=None):
    # ratio 3 x 2 requests x 8 slots = 48 rows of budget; blocks of 5 rows
    orc = O.Oracle(2, 1, 16, 4, 8, [-1], [30, 30], host_block_tokens=5, ratio=3,
                   lib_path=lib_path)
    assert orc.pool_blocks == 9 and orc.free_blocks() == 9
    orc = O.Oracle(1, 1, 16, 2, 8, [-1], [100], host_block_tokens=3, ratio=1,
                   lib_path=lib_path)
    assert orc.pool_blocks == 2


def pin_reserve_worked_example(lib_path=None):
    """Worked by hand: 3 requests, ratio 1, D 8 -> 24 rows -> 6 blocks of 4."""
    orc = O.Oracle(3, 1, 16, 2, 8, [-1], [40, 40, 40], host_block_tokens=4, ratio=1,
                   lib_path=lib_path)
    assert orc.pool_blocks == 6
    assert orc.reserve([0, 1], [5, 4]) == 0          # r0 <- 0, 1; r1 <- 2
    assert orc.block_table(0).tolist() == [0, 1] and orc.block_table(1).tolist() == [2]
    assert orc.reserve([2], [13]) == -2              # 4 blocks wanted, 3 free
    assert orc.block_table(2).tolist() == [] and orc.free_blocks() == 3
    assert orc.reserve([2], [12]) == 0               # r2 <- 3, 4, 5
    assert orc.block_table(2).tolist() == [3, 4, 5] and orc.free_blocks() == 0
    assert orc.release([0]) == 0                     # 0 and 1 come back
    assert orc.reserve([1, 1], [6, 8]) == 0          # r1 grows by one block: 0
    assert orc.block_table(1).tolist() == [2, 0]
    assert orc.reserve([0], [1]) == 0                # r0 <- 1
    assert orc.block_table(0).tolist() == [1]
    assert orc.reserve([0], [-1]) == -1 and orc.reserve([3], [1]) == -1
    assert orc.reserve([0], [41]) == -1              # beyond the request's capacity
    assert orc.reserve([0], [0]) == 0 and orc.block_table(0).tolist() == [1]


def pin_prefill_needs_the_newest_rows(lib_path=None):
    """A prefill whose newest min(S, D) tokens are not all in reserved blocks
    reports NO_HOST_ROW and leaves the request as it was; other requests in
    the same call proceed."""
    D, hb = 4, 2
    orc = O.Oracle(2, 1, 16, 2, D, [-1], [20, 20], host_block_tokens=hb, ratio=4,
                   lib_path=lib_path)
    assert orc.reserve([0, 1], [3, 6]) == 0        # r0 holds tokens 0..3, r1 0..5
    for blk in range(orc.pool_blocks):
        orc.block_rows(0, blk)[:] = _rows_of_ids([100 + 2 * blk, 101 + 2 * blk])
    before = orc.state(0)
    dev0 = orc.dev_rows(0, 0).copy()
    st = orc.prefill([6, 6])                       # r0 needs tokens 2..5
    assert st.tolist() == [O.NO_HOST_ROW, O.OK]
    after = orc.state(0)
    assert np.array_equal(before[0][0], after[0][0]) and np.array_equal(dev0, orc.dev_rows(0, 0))
    assert after[0][1].tolist() == [2, 3, 4, 5]
    # r1's blocks are 2, 3, 4: token t sits in row (2 + t // 2) * 2 + t % 2 = 4 + t
    assert orc.dev_rows(0, 1).view(np.uint32)[:, 0].tolist() == [106, 107, 108, 109]
    assert orc.reserve([0], [6]) == 0
    assert orc.prefill([6, -1]).tolist() == [O.OK, O.OK]
    assert orc.state(0)[0][0].tolist() == [2, 3, 4, 5]


def _rows_of_ids(ids, B=16):
    return np.repeat(np.asarray(ids, dtype=np.uint32)[:, None], B // 4, axis=1).view(np.uint8)


def pin_paged_in_request_order_equals_contiguous(lib_path=None):
    """Reserving whole requests in order on a fresh pool lays them out
    exactly like contiguous regions: same outputs and state, and plan host
    slots that differ only by the request's region offset."""
    w = W.make_config(1)
    hb = 8
    assert all(int(c) % hb == 0 for c in w.host_capacity)
    a = O.Oracle.for_workload(w, track_bytes=True, lib_path=lib_path)
    p = O.Oracle.for_workload(w, track_bytes=True, lib_path=lib_path, host_block_tokens=hb)
    assert p.reserve(list(range(w.num_requests)), w.host_capacity.tolist()) == 0
    for r in range(w.num_requests):
        rows = W.kv_rows(w, 0, r, np.arange(int(w.host_capacity[r])))
        a.host_rows(0, r)[:] = rows
        for b, blk in enumerate(p.block_table(r)):
            p.block_rows(0, int(blk))[:] = rows[b * hb:(b + 1) * hb]
    a.prefill(w.seq_lens0)
    p.prefill(w.seq_lens0)
    sched = W.topk_schedule(w)[0]
    for c in range(w.steps):
        seq = w.seq_lens_at(c)
        oa, pa, ca, sa = a.swap_in(0, sched[c], seq)
        op, pp, cp, sp = p.swap_in(0, sched[c], seq)
        assert np.array_equal(oa, op) and np.array_equal(ca, cp) and np.array_equal(sa, sp)
        for r in range(w.num_requests):
            n = int(ca[r])
            assert np.array_equal(pp[r, :n, 1], pa[r, :n, 1])
            assert np.array_equal(pp[r, :n, 0], pa[r, :n, 0] + a.host_off[r])
    for x, y in zip(a.state(0), p.state(0)):
        assert np.array_equal(x, y)
    for r in range(w.num_requests):
        assert np.array_equal(a.dev_rows(0, r), p.dev_rows(0, r))


def run_random_paged_program(seed, lib_path=None, steps=40):
    """Random admissions, calls, backups and releases on a tight pool; the
    oracle must match the models after every operation.  Returns counters
    of the cases that occurred."""
    rng = np.random.default_rng(seed)
    R, D, k, hb, ratio, B = 5, 8, 4, 3, 2, 16
    cap = [45] * R
    orc = O.Oracle(R, 1, B, k, D, [-1], cap, track_bytes=True, lib_path=lib_path,
                   host_block_tokens=hb, ratio=ratio)
    pool = PagedPool(R, D, ratio, hb, cap)
    assert orc.pool_blocks == pool.num_blocks
    pool_ids = np.zeros(pool.num_blocks * hb, dtype=np.int64)   # id of each pool row
    dev_ids = np.zeros((R, D), dtype=np.int64)                  # id of each device slot
    models = [None] * R
    S = [0] * R
    next_id = [1]
    seen = {"no_host_row_call": 0, "no_host_row_backup": 0, "pool_full": 0,
            "slow_calls": 0, "releases": 0, "admissions": 0}

    def new_id():
        next_id[0] += 1
        return next_id[0]

    def write_rows(r, tokens):
        for t in tokens:
            row = pool.row(r, t)
            if row is None:
                continue
            i = new_id()
            pool_ids[row] = i
            blk = orc.block_table(r)[t // hb]
            orc.block_rows(0, int(blk))[t % hb] = _rows_of_ids([i])[0]

    def check_state(ctx):
        s2t, lu, t2s, _ = orc.state(0)
        for r in range(R):
            if models[r] is None:
                continue
            assert s2t[r].tolist() == models[r].slot2tok(), ctx
            if S[r] > D:
                order = sorted(range(D), key=lambda s_: (int(lu[r, s_]), s_))
                assert order == models[r].recency, ctx
            got = orc.dev_rows(0, r).view(np.uint32)[:, 0]
            assert got.tolist() == dev_ids[r].tolist(), ctx
        for r in range(R):
            assert orc.block_table(r).tolist() == pool.tables[r], ctx

    for step in range(steps):
        # admissions of idle requests
        for r in range(R):
            if models[r] is None and rng.random() < 0.5:
                S0 = int(rng.integers(1, 30))
                want = pool.reserve([r], [S0 + 1])
                assert orc.reserve([r], [S0 + 1]) == want
                if want == -2:
                    seen["pool_full"] += 1
                    continue
                write_rows(r, range(S0))
                seq = [-1] * R
                seq[r] = S0
                st = orc.prefill(seq)
                assert st[r] == 0
                models[r] = ListLRU(D, S0)
                S[r] = S0
                n = min(S0, D)
                for i in range(n):
                    dev_ids[r, i] = pool_ids[pool.row(r, S0 - n + i)]
                seen["admissions"] += 1
        check_state(f"seed {seed} step {step} admit")

        # one swap-in call over all requests (idle ones: padding, S = 0)
        topk = np.full((R, k), -1, dtype=np.int32)
        seq = np.zeros(R, dtype=np.int32)
        for r in range(R):
            if models[r] is None:
                continue
            # sometimes a length past the rows held, with its last position asked for
            lie = S[r] + 2 <= cap[r] and rng.random() < 0.15
            Sc = S[r] + 2 if lie else S[r]
            seq[r] = Sc
            kk = min(k, Sc)
            if lie:
                topk[r, 0] = Sc - 1
                topk[r, 1:kk] = rng.choice(Sc - 1, kk - 1, replace=False)
            else:
                topk[r, :kk] = rng.choice(Sc, kk, replace=False)
        out, plan, cnt, st = orc.swap_in(0, topk, seq)
        for r in range(R):
            if models[r] is None:
                assert st[r] == 0 and (out[r] == -1).all() and cnt[r] == 0
                continue
            row = topk[r].tolist()
            Sc = int(seq[r])
            m = models[r]
            if Sc > D:
                seen["slow_calls"] += 1
                misses = [t for t in row if t >= 0 and t not in m.slot_of]
                if any(pool.row(r, t) is None for t in misses):
                    seen["no_host_row_call"] += 1
                    assert st[r] == O.NO_HOST_ROW and (out[r] == -1).all() and cnt[r] == 0
                    continue
            assert st[r] == 0
            mo, mp = m.call(row, Sc)
            assert out[r].tolist() == mo
            assert cnt[r] == len(mp)
            assert [tuple(x) for x in plan[r, :cnt[r]].tolist()] == \
                [(pool.row(r, t), v) for t, v in mp]
            for t, v in mp:
                dev_ids[r, v] = pool_ids[pool.row(r, t)]
        check_state(f"seed {seed} step {step} call")

        # growth: reserve one more token (usually) and back up position S
        pos = np.full(R, -1, dtype=np.int32)
        rows = np.zeros((R, B), dtype=np.uint8)
        ids = [0] * R
        for r in range(R):
            if models[r] is None:
                continue
            if rng.random() < 0.9 and S[r] + 1 <= cap[r]:
                want = pool.reserve([r], [S[r] + 1])
                assert orc.reserve([r], [S[r] + 1]) == want
                seen["pool_full"] += want == -2
            if S[r] < cap[r]:
                pos[r] = S[r]
                ids[r] = new_id()
                rows[r] = _rows_of_ids([ids[r]])[0]
        bst = orc.backup(0, rows, pos)
        for r in range(R):
            if pos[r] < 0:
                continue
            row = pool.row(r, int(pos[r]))
            if row is None:
                seen["no_host_row_backup"] += 1
                assert bst[r] == O.NO_HOST_ROW
                continue
            assert bst[r] == 0
            pool_ids[row] = ids[r]
            if pos[r] < D:
                dev_ids[r, pos[r]] = ids[r]
                models[r].backup(int(pos[r]))
            S[r] += 1
        check_state(f"seed {seed} step {step} backup")

        # finished requests leave and give their blocks back
        for r in range(R):
            if models[r] is not None and (S[r] >= cap[r] or rng.random() < 0.08):
                pool.release([r])
                assert orc.release([r]) == 0
                models[r] = None
                seen["releases"] += 1
        check_state(f"seed {seed} step {step} release")
    return seen


def pin_random_paged_programs(lib_path=None):
    total = {}
    for seed in range(4):
        for key, v in run_random_paged_program(seed, lib_path).items():
            total[key] = total.get(key, 0) + v
    # every case the programs are meant to reach occurred
    assert all(v > 0 for v in total.values()), total


PAGED_PINS = [pin_paged_pool_rounds_down, pin_reserve_worked_example,
              pin_prefill_needs_the_newest_rows,
              pin_paged_in_request_order_equals_contiguous, pin_random_paged_programs]


@pytest.mark.parametrize("pin", PAGED_PINS, ids=[p.__name__[4:] for p in PAGED_PINS])
def test_paged_pin(pin):
    pin()


def test_paged_layout_rejections():
    with pytest.raises(ValueError):   # budget of 4 rows: not one whole block of 5
        O.Oracle(1, 1, 16, 2, 4, [-1], [10], host_block_tokens=5, ratio=1)


def test_contiguous_oracle_refuses_pool_calls():
    orc = O.Oracle(1, 1, 16, 2, 4, [-1], [10])
    assert orc.reserve([0], [1]) == -1 and orc.release([0]) == -1
