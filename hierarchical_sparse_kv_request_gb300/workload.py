"""Seeded synthetic workloads for the HiSparse decode-time swap-in resolver.

This module only *generates inputs*: sequence lengths, per-step top-k index
sets, KV row bytes and backup rows.  It holds none of the resolver's
arithmetic (no hit test, no LRU, no victim choice), so both the CPU oracle
(tests only) and the CUDA path can be fed from it without sharing any of the
method's logic.

Random numbers come from one counter-based generator, splitmix64
(Steele, Lea & Flood, "Fast splittable pseudorandom number generators",
OOPSLA 2014): output i of a stream with key K is mix(K + (i + 1) * 0x9E3779B97F4A7C15).
Integers in [0, n) are drawn as ((u >> 32) * n) >> 32, so draws are exact
integer arithmetic and identical on every machine.

Workload shapes follow the pages' decode setting: the user guide's example
config (top_k 2048, device_buffer_size 6144, host_to_device_ratio 10), its
40K-token random-input benchmark, and MLA-sized KV rows (fp8 e4m3 latent +
fp32 scales + bf16 rope = 656 B, or 576 bf16 values = 1152 B).
"""

from __future__ import annotations

import dataclasses
import os
from typing import Dict, List, Optional

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_MASK32 = np.uint64(0xFFFFFFFF)


def _mix(z: np.ndarray) -> np.ndarray:
    """splitmix64 finaliser on a uint64 array (wrapping arithmetic)."""
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _mix_scalar(x: int) -> int:
    return int(_mix(np.array([x & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64))[0])


def stream_key(seed: int, *ids: int) -> int:
    """Derive an independent stream key from a seed and integer ids."""
    k = _mix_scalar(seed)
    for i in ids:
        k = _mix_scalar(k ^ ((i * 0xD1B54A32D192ED03) & 0xFFFFFFFFFFFFFFFF))
    return k


class Stream:
    """A sequential splitmix64 stream (keyed, counter-based)."""

    def __init__(self, key: int):
        self.key = np.uint64(key & 0xFFFFFFFFFFFFFFFF)
        self.ctr = 0

    def u64(self, n: int) -> np.ndarray:
        idx = np.arange(self.ctr + 1, self.ctr + 1 + n, dtype=np.uint64)
        self.ctr += n
        with np.errstate(over="ignore"):
            return _mix(self.key + idx * _GOLDEN)

    def below(self, n: int, bound) -> np.ndarray:
        """n integers uniform in [0, bound) (bound scalar or array, < 2^32)."""
        u = self.u64(n) >> np.uint64(32)
        b = np.asarray(bound, dtype=np.uint64)
        return ((u * b) >> np.uint64(32)).astype(np.int64)

    def unit(self, n: int) -> np.ndarray:
        """n doubles uniform in [0, 1) with 53 random bits."""
        return (self.u64(n) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


# --------------------------------------------------------------------------
# Workload configurations
# --------------------------------------------------------------------------

@dataclasses.dataclass
class Workload:
    """One synthetic decode workload (shapes of the pages' decode setting)."""

    name: str
    config_no: int
    num_requests: int
    num_layers: int
    anchor_of_layer: List[int]      # -1: layer owns its top-k and hot state
    steps: int                      # decode steps
    substeps: int                   # swap-in calls per decode step (spec verify)
    top_k: int
    device_buffer_size: int
    row_bytes: int
    row_kind: str                   # "bf16" or "mla_fp8"
    host_to_device_ratio: int
    keep: int                       # indices kept from the previous set
    new_mix: str                    # "uniform" or "mixture"
    backup: bool                    # one backup row per request per layer per step
    seq_lens0: np.ndarray           # int32 [R], lengths before step 0
    seed: int
    capacity: Optional[np.ndarray] = None  # explicit host capacity per request

    @property
    def growth(self) -> int:
        return self.steps if self.backup else 0

    @property
    def host_capacity(self) -> np.ndarray:
        """Tokens of host storage per request: the context plus growth."""
        if self.capacity is not None:
            return np.asarray(self.capacity, dtype=np.int64)
        return (self.seq_lens0.astype(np.int64) + self.growth).astype(np.int64)

    def seq_lens_at(self, step: int) -> np.ndarray:
        if self.backup:
            return (self.seq_lens0 + step).astype(np.int32)
        return self.seq_lens0.astype(np.int32)

    @property
    def anchors(self) -> List[int]:
        return [l for l in range(self.num_layers) if self.anchor_of_layer[l] < 0]


def _seed(config_no: int) -> int:
    return 0x48530000 + config_no


def custom(R: int, k: int, D: int, seq_lens, row_bytes: int = 16, layers: int = 1,
           anchor_of_layer: Optional[List[int]] = None, capacity=None, seed: int = 7,
           ratio: int = 1000) -> Workload:
    """A small ad-hoc workload (bf16 rows) for edge-case tests."""
    lens = np.asarray(seq_lens, dtype=np.int32)
    return Workload("custom", 0, R, layers, anchor_of_layer or [-1] * layers, 1, 1, k, D,
                    row_bytes, "bf16", ratio, 0, "uniform", False, lens, seed,
                    None if capacity is None else np.asarray(capacity, dtype=np.int64))


def make_config(config_no: int, *, steps: Optional[int] = None,
                num_requests: Optional[int] = None) -> Workload:
    """The workloads (1-5, and 6: a pipelined 16-layer index-sharing slice);
    ``steps``/``num_requests`` shrink a config for tests."""
    seed = _seed(config_no)
    if config_no == 1:
        # Tiny check: 4 requests, seq_len {400,3000,5000,8000}, k 256, D 512,
        # 576 bf16 values per row, 70% of each set redrawn from the previous.
        R = 4
        w = Workload("tiny", 1, R, 1, [-1], 8, 1, 256, 512, 1152, "bf16", 10,
                     int(round(0.7 * 256)), "uniform", False,
                     np.array([400, 3000, 5000, 8000], dtype=np.int32), seed)
    elif config_no == 2:
        # The guide's decode setting: 32 x 40000 tokens, k 2048, D 6144, ratio
        # 10, 656 B MLA fp8 rows, 80% reuse, new indices from the mixture.
        R = 32
        w = Workload("decode_40k", 2, R, 1, [-1], 64, 1, 2048, 6144, 656,
                     "mla_fp8", 10, int(round(0.8 * 2048)), "mixture", False,
                     np.full(R, 40000, dtype=np.int32), seed)
    elif config_no == 3:
        # Mixed lengths U[2048, 81920], 4 independent layers, 60% reuse,
        # eager backup of one row per request per layer per step.
        R = 128
        st = Stream(stream_key(seed, 0xC3))
        lens = (2048 + st.below(R, 81920 - 2048 + 1)).astype(np.int32)
        w = Workload("mixed_len", 3, R, 4, [-1, -1, -1, -1], 32, 1, 2048, 6144,
                     656, "mla_fp8", 10, int(round(0.6 * 2048)), "mixture", True,
                     lens, seed)
    elif config_no == 4:
        # Shared-index prefetch: 1 anchor + 3 skip layers, 64 x 65536 tokens,
        # 70% reuse.  Ratio 11: 64*65536 tokens exceed 10 x 64 x 6144 slots.
        R = 64
        w = Workload("shared_index", 4, R, 4, [-1, 0, 0, 0], 32, 1, 2048, 6144,
                     656, "mla_fp8", 11, int(round(0.7 * 2048)), "mixture", False,
                     np.full(R, 65536, dtype=np.int32), seed)
    elif config_no == 5:
        # Stress + speculative verify: 256 x 32768, D 4096, bf16 1152 B rows,
        # 3 sub-steps per step at 50% overlap, backup once per decode step.
        R = 256
        w = Workload("spec_verify", 5, R, 1, [-1], 16, 3, 2048, 4096, 1152,
                     "bf16", 10, 1024, "mixture", True,
                     np.full(R, 32768, dtype=np.int32), seed)
    elif config_no == 6:
        # Pipelined index sharing over a 16-layer slice: 4 anchors, each
        # followed by 3 skip layers reusing its top-k, decode_40k shapes.
        R = 32
        anchors = []
        for g in range(4):
            anchors += [-1, 4 * g, 4 * g, 4 * g]
        w = Workload("index_share_16", 6, R, 16, anchors, 32, 1, 2048, 6144, 656,
                     "mla_fp8", 10, int(round(0.8 * 2048)), "mixture", False,
                     np.full(R, 40000, dtype=np.int32), seed)
    else:
        raise ValueError(f"unknown config {config_no}")
    if steps is not None:
        w.steps = steps
    if num_requests is not None and num_requests != w.num_requests:
        w.num_requests = num_requests
        w.seq_lens0 = w.seq_lens0[:num_requests].copy()
    return w


# --------------------------------------------------------------------------
# Top-k index sets
# --------------------------------------------------------------------------

class _ZipfRecency:
    """Inverse-CDF sampler of recency d in [0, S) with P(d) ~ (d+1)^-s."""

    def __init__(self, s: float, max_len: int):
        w = np.power(np.arange(1, max_len + 1, dtype=np.float64), -s)
        self.cum = np.cumsum(w)

    def sample(self, u: np.ndarray, S: int) -> np.ndarray:
        total = self.cum[S - 1]
        d = np.searchsorted(self.cum[:S], u * total, side="right")
        return np.minimum(d, S - 1)


class TopkSource:
    """Per-(layer, request) top-k sequences of distinct token indices.

    Step 0 draws ``top_k`` distinct indices; each later call keeps ``keep``
    of the previous set (a uniform subset) and draws the rest from the
    workload's mixture, rejecting duplicates.  Each set is emitted in a
    random order, as an indexer's score order would be.
    """

    def __init__(self, w: Workload, layer: int, request: int):
        self.w = w
        self.st = Stream(stream_key(w.seed, 0x70, layer, request))
        self.prev: Optional[np.ndarray] = None
        self.zipf: Optional[_ZipfRecency] = None

    def _draw_new(self, n: int, S: int, exclude: np.ndarray) -> np.ndarray:
        taken = np.zeros(S, dtype=bool)
        taken[exclude] = True
        out: List[np.ndarray] = []
        need = n
        while need > 0:
            c = max(2 * need, 64)
            if self.w.new_mix == "uniform":
                cand = self.st.below(c, S)
            else:
                coin = self.st.below(c, 2)
                uni = self.st.below(c, S)
                if self.zipf is None:
                    self.zipf = _ZipfRecency(1.1, int(self.w.host_capacity.max()))
                d = self.zipf.sample(self.st.unit(c), S)
                cand = np.where(coin == 0, uni, S - 1 - d)
            # keep first occurrences, in draw order, of indices not yet taken
            _, first = np.unique(cand, return_index=True)
            first.sort()
            cand = cand[first]
            cand = cand[~taken[cand]][:need]
            taken[cand] = True
            out.append(cand)
            need -= cand.size
        return np.concatenate(out)

    def next(self, S: int) -> np.ndarray:
        k = self.w.top_k
        if S < k:
            raise ValueError("sequence shorter than top_k")
        if self.prev is None:
            cur = self._draw_new(k, S, np.zeros(0, dtype=np.int64))
        else:
            order = np.argsort(self.st.u64(self.prev.size), kind="stable")
            kept = self.prev[order[: self.w.keep]]
            kept = kept[kept < S]
            new = self._draw_new(k - kept.size, S, kept)
            cur = np.concatenate([kept, new])
        perm = np.argsort(self.st.u64(cur.size), kind="stable")
        cur = cur[perm]
        self.prev = cur
        return cur.astype(np.int32)


def _stream_calls(w: Workload, layer: int, r: int) -> np.ndarray:
    """int32 [steps*substeps][k]: the top-k sets of one (layer, request)."""
    calls = w.steps * w.substeps
    src = TopkSource(w, layer, r)
    out = np.empty((calls, w.top_k), dtype=np.int32)
    for c in range(calls):
        out[c] = src.next(int(w.seq_lens_at(c // w.substeps)[r]))
    return out


def _stream_job(args) -> np.ndarray:
    return _stream_calls(*args)


# Schedules with more index draws than this are generated by a pool of
# worker processes (each (layer, request) stream is independent, so the
# result is the same either way).
_PARALLEL_DRAWS = 1 << 22


def topk_schedule(w: Workload, workers: Optional[int] = None) -> Dict[int, np.ndarray]:
    """All top-k inputs: {anchor layer: int32 [steps*substeps][R][k]}.

    Call c of a layer is decode step c // substeps; sets chain across
    sub-steps and decode steps alike.  `workers` > 1 spreads the independent
    (layer, request) streams over that many processes (started with
    "spawn", never forked); None picks a pool for large schedules.
    """
    calls = w.steps * w.substeps
    jobs = [(l, r) for l in w.anchors for r in range(w.num_requests)]
    if workers is None:
        big = len(jobs) * calls * w.top_k > _PARALLEL_DRAWS
        workers = min(16, os.cpu_count() or 1, len(jobs)) if big else 1
    rows = None
    if workers > 1:
        import concurrent.futures as cf
        import multiprocessing as mp
        try:
            with cf.ProcessPoolExecutor(workers, mp_context=mp.get_context("spawn")) as ex:
                rows = list(ex.map(_stream_job, [(w, l, r) for l, r in jobs],
                                   chunksize=max(1, len(jobs) // (4 * workers))))
        except cf.process.BrokenProcessPool:
            rows = None     # e.g. a main script the workers cannot import: go serial
    if rows is None:
        rows = [_stream_calls(w, l, r) for l, r in jobs]
    out = {}
    for l in w.anchors:
        out[l] = np.empty((calls, w.num_requests, w.top_k), dtype=np.int32)
    for (l, r), a in zip(jobs, rows):
        out[l][:, r] = a
    return out


# --------------------------------------------------------------------------
# KV row bytes
# --------------------------------------------------------------------------

def _pool_words(seed: int, n: int, nwords: int) -> np.ndarray:
    """uint64 [n][nwords] of seeded random words."""
    st = Stream(stream_key(seed, 0x50))
    return st.u64(n * nwords).reshape(n, nwords)


def _to_bf16_bits(f: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (round to nearest even), returning uint16 bits."""
    b = np.asarray(f, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return b.astype(np.uint16)


_POOL_ROWS = 4096
_pools: Dict[tuple, np.ndarray] = {}


def _row_pool(w: Workload) -> np.ndarray:
    """uint8 [4096][row_bytes] of random rows in the workload's row format.

    "mla_fp8" (656 B): 512 fp8 e4m3 latent bytes (random, never the NaN
    codes 0x7F/0xFF) + 4 fp32 scales uniform in [2^-8, 1] + 64 bf16 rope
    values uniform in [-1, 1] (rounded to nearest even).  "bf16":
    row_bytes/2 bf16 values uniform in [-1, 1].
    """
    key = (w.seed, w.row_kind, w.row_bytes)
    if key in _pools:
        return _pools[key]
    n, B = _POOL_ROWS, w.row_bytes
    if w.row_kind == "mla_fp8":
        assert B == 656
        words = _pool_words(w.seed, n, 64 + 34)
        latent = words[:, :64].copy().view(np.uint8).reshape(n, 512)
        latent[latent == 0x7F] = 0x7E
        latent[latent == 0xFF] = 0xFE
        u32 = words[:, 64:].copy().view(np.uint32).reshape(n, 68)
        sc = (2.0 ** -8 + (1.0 - 2.0 ** -8) * (u32[:, :4] >> 8) * (2.0 ** -24)).astype(np.float32)
        rope = _to_bf16_bits((u32[:, 4:] >> 8).astype(np.float64) * (2.0 ** -23) - 1.0)
        pool = np.concatenate([latent, sc.view(np.uint8).reshape(n, 16),
                               rope.view(np.uint8).reshape(n, 128)], axis=1)
    elif w.row_kind == "bf16":
        nv = B // 2
        words = _pool_words(w.seed, n, (nv + 1) // 2)
        u32 = words.copy().view(np.uint32).reshape(n, -1)[:, :nv]
        pool = _to_bf16_bits((u32 >> 8).astype(np.float64) * (2.0 ** -23) - 1.0) \
            .view(np.uint8).reshape(n, B)
    else:
        raise ValueError(w.row_kind)
    _pools[key] = np.ascontiguousarray(pool)
    return _pools[key]


def kv_rows(w: Workload, layer: int, request: int, tokens) -> np.ndarray:
    """uint8 [len(tokens)][row_bytes]: the KV rows of these token positions.

    Each row is a random row of the workload's format (drawn from a seeded
    pool by a hash of its coordinates) that also carries its own identity
    in fields whose values stay in the format's ranges, so no two
    (layer, request, token) rows are equal:
      "mla_fp8": the 4 fp32 scales become 0.5 * (1 + f / 2^23) with f =
                 token, request, layer and hash bits (values in [0.5, 1));
      "bf16":    the first 6 values become +-0.5 * (1 + m / 128), carrying
                 8 bits of (token | request << 20 | layer << 36) each.
    """
    tokens = np.atleast_1d(np.asarray(tokens, dtype=np.int64))
    pool = _row_pool(w)
    key = np.uint64(stream_key(w.seed, 0x52, layer, request))
    with np.errstate(over="ignore"):
        hsh = _mix(key + (tokens.astype(np.uint64) + np.uint64(1)) * _GOLDEN)
    rows = pool[(hsh % np.uint64(_POOL_ROWS)).astype(np.int64)]
    n = tokens.size
    if w.row_kind == "mla_fp8":
        f = np.empty((n, 4), dtype=np.uint32)
        f[:, 0] = tokens.astype(np.uint32) & 0x7FFFFF
        f[:, 1] = request & 0x7FFFFF
        f[:, 2] = layer & 0x7FFFFF
        f[:, 3] = (hsh >> np.uint64(41)).astype(np.uint32) & 0x7FFFFF
        bits = (np.uint32(126) << np.uint32(23)) | f          # 0.5 * (1 + f/2^23)
        rows[:, 512:528] = bits.view(np.uint8).reshape(n, 16)
    else:
        ident = (tokens.astype(np.uint64) | (np.uint64(request) << np.uint64(20))
                 | (np.uint64(layer) << np.uint64(36)))
        vals = np.empty((n, 6), dtype=np.uint16)
        for q in range(6):
            byte = ((ident >> np.uint64(8 * q)) & np.uint64(0xFF)).astype(np.uint16)
            vals[:, q] = ((byte >> 7) << 15) | (np.uint16(126) << 7) | (byte & 0x7F)
        rows[:, :12] = vals.view(np.uint8).reshape(n, 12)
    return rows


def fill_host_rows(w: Workload, layer: int, request: int, dst: np.ndarray,
                   upto: int, chunk: int = 8192) -> None:
    """Write rows [0, upto) of (layer, request) into dst ([cap][B] uint8)."""
    for t0 in range(0, upto, chunk):
        t1 = min(upto, t0 + chunk)
        dst[t0:t1] = kv_rows(w, layer, request, np.arange(t0, t1))
