"""Pins of the CPU oracle against things other than itself (CPU only).

- hand-derived golden traces (tests/golden/, worked out from the pages' rules);
- an independently written recency-list LRU model, exhaustively on tiny
  buffers and randomly on small ones;
- invariants after every call of a real workload, closed forms, the
  fast-path identity and plain set arithmetic for the miss count.
"""

import itertools

import numpy as np
import pytest

import oracle as O
from golden_trace import load, names
from lru_model import ListLRU
from hierarchical_sparse_kv_request_gb300 import workload as W


# ----------------------------------------------------------------------------
# golden traces
# ----------------------------------------------------------------------------

def run_trace_on_oracle(name, lib_path=None):
    layout, ops = load(name)
    D, k, cap = layout["D"], layout["k"], layout["cap"]
    orc = O.Oracle(1, 1, 16, k, D, [-1], [cap], track_bytes=True, lib_path=lib_path)
    if layout.get("protect"):
        orc.set_protected_calls(layout["protect"])
    S = None
    resident = None
    for op, a in ops:
        if op == "resident":
            resident = np.array([a["ids"]], dtype=np.int32)
        elif op == "clear":
            orc.status_clear()
        elif op in ("prefill", "backup"):
            if op == "prefill":
                orc.host_rows(0, 0)[:] = np.arange(cap, dtype=np.uint8)[:, None]
                st = orc.prefill([a["S"]])
            else:
                row = np.full((1, 16), (200 + a["pos"]) % 256, dtype=np.uint8)
                st = orc.backup(0, row, [a["pos"]])
            got = {"status": int(st[0]), "word": int(orc.status_word()[0])}
            want = {"status": a["status"], "word": a.get("word", got["word"])}
            if got != want:
                return got, want
        else:
            out, plan, cnt, st = orc.swap_in(0, np.array([a["topk"]]), [a["S"]],
                                             resident, layout.get("bs", 0))
            e = a["expect"]
            s2t, lu, _, _ = orc.state(0)
            got = {"out": out[0].tolist(), "status": int(st[0]),
                   "plan": [tuple(p) for p in plan[0, : cnt[0]].tolist()],
                   "slot2tok": s2t[0].tolist(), "last_used": lu[0].tolist(),
                   "word": int(orc.status_word()[0])}
            want = {"out": e["out"], "status": e["status"], "plan": e["plan"],
                    "slot2tok": e["slot2tok"], "last_used": e["last_used"],
                    "word": e.get("word", got["word"])}
            if got != want:
                return got, want
    return None


@pytest.mark.parametrize("name", names())
def test_golden_trace(name):
    assert run_trace_on_oracle(name) is None


# ----------------------------------------------------------------------------
# brute force against the recency-list model
# ----------------------------------------------------------------------------

def compare_with_model(D, k, seq_lens, programs, lib_path=None, protect=0, counts=None):
    """programs[r] = list of top-k rows for request r (same number of calls).

    Runs all requests in one oracle handle and each in its own ListLRU.
    Returns the first mismatch as a string, or None.  With protect > 0 the
    slots of the last `protect` calls are kept (counts["capacity"] counts
    the calls that failed for lack of victims).
    """
    R = len(programs)
    ncalls = len(programs[0])
    cap = [max(S, 1) for S in seq_lens]
    orc = O.Oracle(R, 1, 16, k, D, [-1], cap, track_bytes=False, lib_path=lib_path)
    if protect:
        orc.set_protected_calls(protect)
    orc.prefill(seq_lens)
    models = [ListLRU(D, S, protect) for S in seq_lens]
    for c in range(ncalls):
        topk = np.array([programs[r][c] for r in range(R)], dtype=np.int32)
        out, plan, cnt, st = orc.swap_in(0, topk, seq_lens)
        s2t, lu, t2s, tick = orc.state(0)
        if (tick != c + 1).any():
            return f"tick {tick} after call {c + 1}"
        for r in range(R):
            mo, mp = models[r].call(programs[r][c], seq_lens[r])
            if models[r].failed:
                if counts is not None:
                    counts["capacity"] = counts.get("capacity", 0) + 1
                if st[r] != O.CAPACITY or (out[r] != -1).any() or cnt[r] != 0:
                    return f"r{r} c{c}: expected CAPACITY, got status {st[r]}"
                continue
            if st[r] != 0:
                return f"r{r} c{c}: status {st[r]}"
            if out[r].tolist() != mo:
                return f"r{r} c{c}: out {out[r].tolist()} != {mo}"
            if [tuple(p) for p in plan[r, : cnt[r]].tolist()] != mp:
                return f"r{r} c{c}: plan {plan[r, :cnt[r]].tolist()} != {mp}"
            if s2t[r].tolist() != models[r].slot2tok():
                return f"r{r} c{c}: slot2tok {s2t[r].tolist()} != {models[r].slot2tok()}"
            # the oracle's stamps must order the slots exactly as the list does
            if seq_lens[r] > D:
                order = sorted(range(D), key=lambda s: (int(lu[r, s]), s))
                if order != models[r].recency:
                    return f"r{r} c{c}: LRU order {order} != {models[r].recency}"
            off = int(orc.host_off[r])
            for t in range(seq_lens[r]):
                want = models[r].slot_of.get(t, -1) if seq_lens[r] > D else \
                    (t if t < seq_lens[r] and seq_lens[r] <= D else -1)
                if seq_lens[r] > D and t2s[off + t] != want:
                    return f"r{r} c{c}: tok2slot[{t}] {t2s[off + t]} != {want}"
    return None


def _exhaustive_programs(S, k, ncalls, reverse_odd=True):
    sets = list(itertools.combinations(range(S), k))
    progs = []
    for seq in itertools.product(sets, repeat=ncalls):
        prog = []
        for i, s in enumerate(seq):
            row = list(s)
            if reverse_odd and i % 2 == 1:
                row = row[::-1]          # output order follows input order
            prog.append(row)
        progs.append(prog)
    return progs


@pytest.mark.parametrize("D,S,k,ncalls", [
    (2, 3, 1, 3), (2, 4, 2, 3), (3, 4, 2, 3), (3, 5, 2, 3), (3, 6, 3, 2),
    (4, 5, 2, 2), (4, 6, 3, 2), (4, 7, 4, 2), (5, 7, 3, 2), (3, 5, 1, 4),
])
def test_exhaustive_vs_list_model(D, S, k, ncalls):
    progs = _exhaustive_programs(S, k, ncalls)
    assert compare_with_model(D, k, [S] * len(progs), progs) is None


def _random_programs(rng, R, D, k, S, ncalls, pad_prob=0.15):
    progs = []
    for _ in range(R):
        prog = []
        for _ in range(ncalls):
            row = rng.choice(S, size=k, replace=False).tolist()
            row = [-1 if rng.random() < pad_prob else t for t in row]
            prog.append(row)
        progs.append(prog)
    return progs


@pytest.mark.parametrize("seed", range(4))
def test_random_vs_list_model(seed):
    rng = np.random.default_rng(1000 + seed)
    D = int(rng.integers(4, 12))
    k = int(rng.integers(1, D + 1))
    lens = [int(rng.integers(k, 3 * D)) for _ in range(64)]
    lens = [max(S, k) for S in lens]
    progs = []
    for S in lens:
        progs += _random_programs(rng, 1, D, k, S, 10)
    assert compare_with_model(D, k, lens, progs) is None


def compare_resident_with_model(D, k, S, bs, programs, tables, lib_path=None):
    """Like compare_with_model, with a resident block table per call."""
    R = len(programs)
    orc = O.Oracle(R, 1, 16, k, D, [-1], [S] * R, track_bytes=False, lib_path=lib_path)
    orc.prefill([S] * R)
    models = [ListLRU(D, S) for _ in range(R)]
    for c in range(len(programs[0])):
        topk = np.array([programs[r][c] for r in range(R)], dtype=np.int32)
        tab = np.array([tables[r][c] for r in range(R)], dtype=np.int32)
        out, plan, cnt, st = orc.swap_in(0, topk, [S] * R, tab, bs)
        s2t, lu, _, _ = orc.state(0)
        for r in range(R):
            res = {t: int(tab[r][t // bs]) * bs + t % bs for t in range(S)
                   if t // bs < tab.shape[1] and tab[r][t // bs] >= 0}
            mo, mp = models[r].call(programs[r][c], S, res)
            if st[r] != 0 or out[r].tolist() != mo or \
                    [tuple(p) for p in plan[r, :cnt[r]].tolist()] != mp or \
                    s2t[r].tolist() != models[r].slot2tok():
                return f"r{r} c{c}: {out[r].tolist()} vs {mo}"
            if S > D:
                order = sorted(range(D), key=lambda s_: (int(lu[r, s_]), s_))
                if order != models[r].recency:
                    return f"r{r} c{c}: LRU order"
    return None


@pytest.mark.parametrize("seed", range(3))
def test_random_resident_tables_vs_list_model(seed, lib_path=None):
    rng = np.random.default_rng(500 + seed)
    D, k, bs = 8, 5, 3
    S = 40 if seed < 2 else 7          # the last seed runs the fast path
    nb = -(-S // bs) - (1 if seed == 1 else 0)   # seed 1: table shorter than S
    R, ncalls = 60, 8
    progs, tabs = [], []
    for _ in range(R):
        progs.append([rng.choice(S, k, replace=False).tolist() for _ in range(ncalls)])
        tabs.append([np.where(rng.random(nb) < 0.3, rng.integers(0, 50, nb), -1).tolist()
                     for _ in range(ncalls)])
    assert compare_resident_with_model(D, k, S, bs, progs, tabs, lib_path) is None


@pytest.mark.parametrize("D,S,k,ncalls,protect", [(4, 7, 2, 3, 2), (5, 8, 2, 3, 2), (4, 6, 3, 2, 1)])
def test_exhaustive_protected_vs_list_model(D, S, k, ncalls, protect):
    counts = {}
    progs = _exhaustive_programs(S, k, ncalls)
    assert compare_with_model(D, k, [S] * len(progs), progs, protect=protect, counts=counts) is None
    assert counts.get("capacity", 0) > 0


def test_random_protected_vs_list_model(lib_path=None):
    """Protection of the last 1-3 calls on random programs with padding."""
    rng = np.random.default_rng(31)
    counts = {}
    for protect in (1, 2, 3):
        D, k, S, R = 10, 4, 30, 80
        progs = _random_programs(rng, R, D, k, S, 12)
        assert compare_with_model(D, k, [S] * R, progs, lib_path, protect, counts) is None
    assert counts.get("capacity", 0) > 0


def test_random_biased_reuse_vs_list_model():
    """Sets that mostly reuse the previous call's tokens (hits + old stamps)."""
    rng = np.random.default_rng(77)
    D, k, S, R, ncalls = 8, 5, 20, 200, 12
    progs = []
    for _ in range(R):
        cur = rng.choice(S, size=k, replace=False)
        prog = [cur.tolist()]
        for _ in range(ncalls - 1):
            keep = rng.choice(cur, size=3, replace=False)
            rest = rng.permutation(np.setdiff1d(np.arange(S), keep))[: k - 3]
            cur = rng.permutation(np.concatenate([keep, rest]))
            prog.append(cur.tolist())
        progs.append(prog)
    assert compare_with_model(D, k, [S] * R, progs) is None


# ----------------------------------------------------------------------------
# invariants on a real workload (tiny config, bytes tracked)
# ----------------------------------------------------------------------------

def check_invariants(orc, w, layer, topk, seq_lens, out, plan, cnt, st, tick,
                     resident_before):
    s2t, lu, t2s, otick = orc.state(layer)
    assert (otick == tick).all()
    D = w.device_buffer_size
    copied = 0
    for r in range(w.num_requests):
        assert st[r] == 0
        S = int(seq_lens[r])
        off = int(orc.host_off[r])
        valid = topk[r][topk[r] >= 0]
        if S <= D:
            # fast-path identity
            assert np.array_equal(out[r], topk[r])
            assert cnt[r] == 0
            continue
        # every selected token is resident at the slot that was emitted
        assert np.array_equal(t2s[off + valid], out[r][topk[r] >= 0])
        # the maps are mutual inverses on their non-negative entries
        filled = np.nonzero(s2t[r] >= 0)[0]
        assert np.array_equal(t2s[off + s2t[r][filled]], filled)
        resident = np.nonzero(t2s[off: off + int(orc.cap[r])] >= 0)[0]
        assert resident.size == filled.size
        # miss count = |top-k \ resident-before| by plain set arithmetic
        m = len(set(valid.tolist()) - resident_before[r])
        assert cnt[r] == m
        # no hit slot is a victim
        hit_tokens = set(valid.tolist()) & resident_before[r]
        victims = set(plan[r, :m, 1].tolist())
        assert not (victims & {int(t2s[off + t]) for t in hit_tokens})
        # stamps never exceed the tick; exactly the selected slots carry it
        assert lu[r].max() <= tick
        assert int((lu[r] == tick).sum()) == valid.size
        # each resident slot's bytes equal its host row
        dev = orc.dev_rows(layer, r)
        host = orc.host_rows(layer, r)
        assert np.array_equal(dev[filled], host[s2t[r][filled]])
        copied += m
    return copied


def pin_invariants_tiny_workload(lib_path=None):
    w = W.make_config(1)
    sched = W.topk_schedule(w)[0]
    orc = O.Oracle.for_workload(w, track_bytes=True, lib_path=lib_path)
    for r in range(w.num_requests):
        W.fill_host_rows(w, 0, r, orc.host_rows(0, r), int(w.seq_lens0[r]))
    orc.prefill(w.seq_lens0)
    total_misses = 0
    for c in range(w.steps):
        s2t, _, t2s, _ = orc.state(0)
        before = [set(np.nonzero(t2s[int(orc.host_off[r]): int(orc.host_off[r] + orc.cap[r])] >= 0)[0].tolist())
                  for r in range(w.num_requests)]
        seq = w.seq_lens_at(c)
        out, plan, cnt, st = orc.swap_in(0, sched[c], seq)
        total_misses += check_invariants(orc, w, 0, sched[c], seq, out, plan, cnt,
                                         st, c + 1, before)
    assert total_misses > 0


def pin_prefill_last_k_is_all_hits(lib_path=None):
    """Closed form: right after prefill, the newest k tokens are all hot."""
    D, k, S = 16, 6, 40
    orc = O.Oracle(1, 1, 16, k, D, [-1], [S], lib_path=lib_path)
    orc.prefill([S])
    topk = np.arange(S - k, S, dtype=np.int32)[::-1].copy()
    out, plan, cnt, st = orc.swap_in(0, topk[None], [S])
    assert cnt[0] == 0 and st[0] == 0
    # slot i holds token S - D + i
    assert np.array_equal(out[0], topk - (S - D))


def pin_repeat_is_all_hits(lib_path=None):
    """Closed form: the same set twice in a row misses nothing the 2nd time."""
    rng = np.random.default_rng(5)
    D, k, S = 32, 12, 200
    orc = O.Oracle(1, 1, 16, k, D, [-1], [S], lib_path=lib_path)
    orc.prefill([S])
    topk = rng.choice(S, k, replace=False).astype(np.int32)
    out1, _, c1, _ = orc.swap_in(0, topk[None], [S])
    out2, _, c2, _ = orc.swap_in(0, rng.permutation(topk)[None], [S])
    assert c2[0] == 0
    s2t, lu, _, tick = orc.state(0)
    assert (tick == 2).all() and int((lu[0] == 2).sum()) == k


def pin_disjoint_sets_closed_form(lib_path=None):
    """Closed form with D = 2k and pairwise-disjoint sets never seen before:
    call 1 evicts prefill slots 0..k-1, call 2 evicts k..2k-1, and from call 3
    on the victims are exactly the slots selected two calls earlier."""
    k = 5
    D = 2 * k
    ncalls = 8
    S = D + k * ncalls + 3
    orc = O.Oracle(1, 1, 16, k, D, [-1], [S], lib_path=lib_path)
    orc.prefill([S])
    # prefill holds the last D tokens; draw sets from [0, S - D), disjoint
    pool = np.random.default_rng(9).permutation(S - D)[: k * ncalls]
    selected = []
    for c in range(ncalls):
        topk = pool[c * k:(c + 1) * k].astype(np.int32)
        out, plan, cnt, st = orc.swap_in(0, topk[None], [S])
        assert cnt[0] == k
        victims = sorted(plan[0, :k, 1].tolist())
        if c == 0:
            assert victims == list(range(k))
        elif c == 1:
            assert victims == list(range(k, 2 * k))
        else:
            assert victims == selected[c - 2]
        selected.append(sorted(out[0].tolist()))


def pin_errors_leave_state_untouched(lib_path=None):
    D, k, S = 8, 4, 20
    orc = O.Oracle(3, 1, 16, k, D, [-1], [S, S, S], lib_path=lib_path)
    orc.prefill([S, S, S])
    before = orc.state(0)
    topk = np.array([[0, 1, 2, 20], [3, 3, 4, 5], [-1, 6, 7, 8]], dtype=np.int32)
    out, plan, cnt, st = orc.swap_in(0, topk, [S, S, S + 5])
    assert st.tolist() == [O.BAD_INDEX, O.DUPLICATE, O.BAD_SEQ_LEN]
    assert (out == -1).all() and (cnt == 0).all()
    after = orc.state(0)
    for a, b in zip(before[:3], after[:3]):
        assert np.array_equal(a, b)
    assert (after[3] == 1).all()


def pin_backup_grows_short_request_into_slow_path(lib_path=None):
    D, k = 6, 3
    S0, steps = 4, 5
    cap = S0 + steps
    orc = O.Oracle(1, 1, 16, k, D, [-1], [cap], lib_path=lib_path)
    rows = np.arange(cap * 16, dtype=np.uint8).reshape(cap, 16)
    orc.host_rows(0, 0)[:S0] = rows[:S0]
    orc.prefill([S0])
    model = ListLRU(D, S0)
    rng = np.random.default_rng(3)
    S = S0
    for c in range(steps):
        topk = rng.choice(S, k, replace=False).astype(np.int32)
        out, plan, cnt, st = orc.swap_in(0, topk[None], [S])
        mo, mp = model.call(topk.tolist(), S)
        assert out[0].tolist() == mo
        assert [tuple(p) for p in plan[0, :cnt[0]].tolist()] == mp
        assert orc.backup(0, rows[S][None], [S])[0] == 0
        model.backup(S)
        S += 1
        s2t = orc.state(0)[0]
        assert s2t[0].tolist() == model.slot2tok()
        dev, host = orc.dev_rows(0, 0), orc.host_rows(0, 0)
        filled = np.nonzero(s2t[0] >= 0)[0]
        assert np.array_equal(dev[filled], host[s2t[0][filled]])
    assert S > D


def pin_replay_copies_plan_rows_to_other_layer(lib_path=None):
    w = W.make_config(4, steps=2, num_requests=2)
    w.top_k, w.device_buffer_size, w.keep = 64, 128, 40
    w.seq_lens0 = np.array([1000, 1500], dtype=np.int32)
    orc = O.Oracle.for_workload(w, track_bytes=True, lib_path=lib_path)
    for l in range(w.num_layers):
        for r in range(w.num_requests):
            W.fill_host_rows(w, l, r, orc.host_rows(l, r), int(w.seq_lens0[r]))
    orc.prefill(w.seq_lens0)
    sched = W.topk_schedule(w)[0]
    for c in range(w.steps):
        out, plan, cnt, st = orc.swap_in(0, sched[c], w.seq_lens0)
        for l in (1, 2, 3):
            orc.replay(plan, cnt, l)
    s2t = orc.state(0)[0]
    for l in range(w.num_layers):
        for r in range(w.num_requests):
            dev, host = orc.dev_rows(l, r), orc.host_rows(l, r)
            assert np.array_equal(dev, host[s2t[r]])
    with pytest.raises(ValueError):
        orc.swap_in(1, sched[0], w.seq_lens0)     # skip layers hold no hot state


def pin_protected_slots_vs_list_model(lib_path=None):
    """The protected mode against the list model: exhaustive tiny programs
    and random ones, with calls failing for lack of victims."""
    counts = {}
    for D, S, k, ncalls, protect in [(4, 7, 2, 3, 2), (4, 6, 3, 2, 1)]:
        progs = _exhaustive_programs(S, k, ncalls)
        assert compare_with_model(D, k, [S] * len(progs), progs, lib_path, protect, counts) is None
    rng = np.random.default_rng(32)
    for protect in (1, 3):
        progs = _random_programs(rng, 40, 10, 4, 30, 10)
        assert compare_with_model(10, 4, [30] * 40, progs, lib_path, protect, counts) is None
    assert counts.get("capacity", 0) > 0


def pin_all_resident_touches_nothing(lib_path=None):
    """Closed form ([Arch] Resident device pages: a resident hit exits before
    the hot-LRU lookup or a host copy): with every block of a request
    resident, each position resolves to its resident row, nothing misses and
    only the tick moves; the same holds on the fast path."""
    rng = np.random.default_rng(8)
    D, k, bs = 16, 8, 4
    lens = [100, 12]                                 # slow path, fast path
    orc = O.Oracle(2, 1, 16, k, D, [-1], lens, lib_path=lib_path)
    orc.prefill(lens)
    s2t0, lu0, t2s0, _ = orc.state(0)
    nb = max(lens) // bs + 1
    ids = rng.permutation(2 * nb).astype(np.int32).reshape(2, nb)
    topk = np.stack([rng.choice(S, k, replace=False) for S in lens]).astype(np.int32)
    out, plan, cnt, st = orc.swap_in(0, topk, lens, ids, bs)
    assert (st == 0).all() and (cnt == 0).all()
    want = (1 << 30) | (ids[np.arange(2)[:, None], topk // bs] * bs + topk % bs)
    assert np.array_equal(out, want)
    s2t, lu, t2s, tick = orc.state(0)
    assert np.array_equal(s2t, s2t0) and np.array_equal(lu, lu0) and np.array_equal(t2s, t2s0)
    assert (tick == 1).all()


def pin_empty_resident_table_is_the_plain_call(lib_path=None):
    """Special case: a resident table with no resident block gives exactly
    the plain swap-in (outputs, plans, statuses and state)."""
    rng = np.random.default_rng(9)
    D, k = 12, 5
    lens = [60, 10, 90]
    a = O.Oracle(3, 1, 16, k, D, [-1], lens, lib_path=lib_path)
    b = O.Oracle(3, 1, 16, k, D, [-1], lens, lib_path=lib_path)
    a.prefill(lens)
    b.prefill(lens)
    empty = np.full((3, 7), -1, dtype=np.int32)
    for c in range(12):
        topk = np.stack([rng.choice(S, k, replace=False) for S in lens]).astype(np.int32)
        ra = a.swap_in(0, topk, lens)
        rb = b.swap_in(0, topk, lens, empty, 3)
        for x, y in zip(ra, rb):
            assert np.array_equal(x, y)
    for x, y in zip(a.state(0), b.state(0)):
        assert np.array_equal(x, y)


def pin_status_word_survives_later_layers_and_backups(lib_path=None):
    """Hand-worked: the status word of a request keeps an error of layer 0
    while layer 1's call and a backup succeed, collects the bits of several
    calls, layers and kinds, and is reset only by a clear ([Arch] Performance
    invariants: no device readback, so an error must stay on the device until
    the caller reads it).  Bit c stands for status code c."""
    D, k, S = 8, 4, 20
    orc = O.Oracle(3, 2, 16, k, D, [-1, -1], [S + 2] * 3, lib_path=lib_path)
    assert orc.prefill([S, S, S]).tolist() == [0, 0, 0]
    assert orc.status_word().tolist() == [0, 0, 0]
    good = np.array([[0, 1, 2, 3], [4, 5, 6, 7], [8, 9, 10, 11]], dtype=np.int32)
    bad = good.copy()
    bad[1, 2] = S                                    # request 1: outside [0, S)
    assert orc.swap_in(0, bad, [S, S, S])[3].tolist() == [0, O.BAD_INDEX, 0]
    assert orc.swap_in(1, good, [S, S, S])[3].tolist() == [0, 0, 0]
    assert orc.status_word().tolist() == [0, 1 << O.BAD_INDEX, 0]
    rows = np.zeros((3, 16), dtype=np.uint8)
    assert orc.backup(1, rows, [S, S, S])[0] == 0       # a good backup changes nothing
    assert orc.status_word().tolist() == [0, 1 << O.BAD_INDEX, 0]
    assert orc.backup(1, rows, [S + 2, -1, S])[0] == O.BAD_POSITION
    dup = good.copy()
    dup[1, 3] = dup[1, 0]                            # request 1: a duplicate on layer 1
    assert orc.swap_in(1, dup, [S, S, S])[3].tolist() == [0, O.DUPLICATE, 0]
    assert orc.status_word().tolist() == [1 << O.BAD_POSITION,
                                          (1 << O.BAD_INDEX) | (1 << O.DUPLICATE), 0]
    assert orc.prefill([-1, -1, S + 3])[2] == O.BAD_SEQ_LEN
    assert orc.status_word().tolist() == [1 << O.BAD_POSITION,
                                          (1 << O.BAD_INDEX) | (1 << O.DUPLICATE),
                                          1 << O.BAD_SEQ_LEN]
    orc.status_clear()
    assert orc.status_word().tolist() == [0, 0, 0]
    assert orc.swap_in(0, good, [S, S, S])[3].tolist() == [0, 0, 0]
    assert orc.status_word().tolist() == [0, 0, 0]


PINS = [pin_invariants_tiny_workload, pin_prefill_last_k_is_all_hits,
        pin_repeat_is_all_hits, pin_disjoint_sets_closed_form,
        pin_errors_leave_state_untouched,
        pin_backup_grows_short_request_into_slow_path,
        pin_replay_copies_plan_rows_to_other_layer, pin_protected_slots_vs_list_model,
        pin_all_resident_touches_nothing, pin_empty_resident_table_is_the_plain_call,
        pin_status_word_survives_later_layers_and_backups]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__[4:] for p in PINS])
def test_pin(pin):
    pin()


def test_layout_rejections():
    with pytest.raises(ValueError):
        O.Oracle(1, 1, 16, 9, 8, [-1], [100])     # top_k > device_buffer_size
    with pytest.raises(ValueError):
        O.Oracle(1, 2, 16, 4, 8, [-1, 1], [100])  # a layer anchored on itself
