"""CPU oracle of the HiSparse swap-in resolver (TEST INFRASTRUCTURE ONLY).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg import this package.  It wraps ``hisparse_oracle.c`` (plain C, built with
gcc) through ctypes; it shares nothing with the CUDA library.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "hisparse_oracle.c")
_LIB = os.path.join(_HERE, "libhisparse_oracle.so")

OK, BAD_INDEX, DUPLICATE, BAD_SEQ_LEN, BAD_POSITION, BAD_RESIDENT, NO_HOST_ROW = 0, 1, 2, 3, 4, 5, 6
CAPACITY = 7
RESIDENT_FLAG = 1 << 30


def build(force: bool = False, extra_flags: Sequence[str] = ()) -> str:
    """Compile the oracle with gcc; returns the library path."""
    out = _LIB
    if extra_flags:
        tag = "_".join(f.strip("-").replace("=", "_") for f in extra_flags)
        out = os.path.join(_HERE, f"libhisparse_oracle_{tag}.so")
    if force or extra_flags or not os.path.exists(out) or \
            os.path.getmtime(out) < os.path.getmtime(_SRC):
        tmp = out + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-Wall", "-Wextra",
                               "-shared", "-fPIC", *extra_flags, "-o", tmp, _SRC])
        os.replace(tmp, out)
    return out


_libs = {}


def _load(path: Optional[str] = None) -> ctypes.CDLL:
    path = path or build()
    if path in _libs:
        return _libs[path]
    lib = ctypes.CDLL(path)
    P, I, I64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    lib.hso_create.restype = P
    lib.hso_create.argtypes = [I, I, I64, I, I, P, P, I]
    lib.hso_create_paged.restype = P
    lib.hso_create_paged.argtypes = [I, I, I64, I, I, P, P, I, I, I]
    lib.hso_pool_blocks.restype = I
    lib.hso_pool_blocks.argtypes = [P]
    lib.hso_free_blocks.restype = I
    lib.hso_free_blocks.argtypes = [P]
    lib.hso_reserve.argtypes = [P, I, P, P]
    lib.hso_set_protected_calls.argtypes = [P, I]
    lib.hso_release.argtypes = [P, I, P]
    lib.hso_block_table.restype = I
    lib.hso_block_table.argtypes = [P, I, P]
    lib.hso_block_rows.restype = P
    lib.hso_block_rows.argtypes = [P, I, I]
    lib.hso_destroy.argtypes = [P]
    lib.hso_host_row.restype = P
    lib.hso_host_row.argtypes = [P, I, I, I64]
    lib.hso_dev_row.restype = P
    lib.hso_dev_row.argtypes = [P, I, I, I64]
    lib.hso_prefill.argtypes = [P, P, P]
    lib.hso_swap_in.argtypes = [P, I, P, P, P, P, P, P]
    lib.hso_swap_in_resident.argtypes = [P, I, P, P, P, I, I, P, P, P, P]
    lib.hso_replay.argtypes = [P, P, P, I]
    lib.hso_backup.argtypes = [P, I, P, P, P]
    lib.hso_state.argtypes = [P, I, P, P, P, P]
    lib.hso_status_word.argtypes = [P, P]
    lib.hso_status_clear.argtypes = [P]
    lib.hso_total_capacity.restype = I64
    lib.hso_total_capacity.argtypes = [P]
    _libs[path] = lib
    return lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


class Oracle:
    """Numpy-facing wrapper of the C oracle state for one layout.

    host_block_tokens > 0 selects the paged host pool: floor(ratio * R * D /
    host_block_tokens) blocks per layer, handed to requests by reserve()."""

    def __init__(self, num_requests: int, num_layers: int, row_bytes: int,
                 top_k: int, device_buffer_size: int,
                 anchor_of_layer: Sequence[int], host_capacity: Sequence[int],
                 track_bytes: bool = True, lib_path: Optional[str] = None,
                 host_block_tokens: int = 0, ratio: int = 0):
        self.lib = _load(lib_path)
        self.R, self.L, self.B = num_requests, num_layers, row_bytes
        self.k, self.D = top_k, device_buffer_size
        self.anchor = np.ascontiguousarray(anchor_of_layer, dtype=np.int32)
        self.cap = np.ascontiguousarray(host_capacity, dtype=np.int64)
        self.track_bytes = track_bytes
        self.hb = int(host_block_tokens)
        if self.hb > 0:
            self.h = self.lib.hso_create_paged(self.R, self.L, self.B, self.k, self.D,
                                               _ptr(self.anchor), _ptr(self.cap), int(ratio),
                                               self.hb, 1 if track_bytes else 0)
        else:
            self.h = self.lib.hso_create(self.R, self.L, self.B, self.k, self.D,
                                         _ptr(self.anchor), _ptr(self.cap),
                                         1 if track_bytes else 0)
        if not self.h:
            raise ValueError("oracle rejected the layout")
        self.total_cap = int(self.lib.hso_total_capacity(self.h))
        self.host_off = np.concatenate([[0], np.cumsum(self.cap)[:-1]]).astype(np.int64)
        self.pool_blocks = int(self.lib.hso_pool_blocks(self.h))

    @classmethod
    def for_workload(cls, w, track_bytes: bool = True, lib_path: Optional[str] = None,
                     host_block_tokens: int = 0):
        return cls(w.num_requests, w.num_layers, w.row_bytes, w.top_k,
                   w.device_buffer_size, w.anchor_of_layer, w.host_capacity,
                   track_bytes, lib_path, host_block_tokens, w.host_to_device_ratio)

    def close(self):
        if self.h:
            self.lib.hso_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -- bytes ------------------------------------------------------------
    def host_rows(self, layer: int, r: int) -> np.ndarray:
        """Writable view [cap_r][B] of the oracle's host rows of (layer, r)
        (contiguous host regions only)."""
        if self.hb:
            raise RuntimeError("a paged pool has no per-request region; use block_rows")
        p = self.lib.hso_host_row(self.h, layer, r, 0)
        if not p:
            raise RuntimeError("oracle built without byte tracking")
        n = int(self.cap[r]) * self.B
        buf = (ctypes.c_uint8 * n).from_address(p)
        return np.frombuffer(buf, dtype=np.uint8).reshape(int(self.cap[r]), self.B)

    def dev_rows(self, layer: int, r: int) -> np.ndarray:
        """View [D][B] of the oracle's device buffer of (layer, r)."""
        p = self.lib.hso_dev_row(self.h, layer, r, 0)
        if not p:
            raise RuntimeError("oracle built without byte tracking")
        n = self.D * self.B
        buf = (ctypes.c_uint8 * n).from_address(p)
        return np.frombuffer(buf, dtype=np.uint8).reshape(self.D, self.B)

    def block_rows(self, layer: int, block: int) -> np.ndarray:
        """Writable view [hb][B] of host block `block` of a layer's paged pool."""
        p = self.lib.hso_block_rows(self.h, layer, block)
        if not p:
            raise RuntimeError("no such block, or byte tracking off")
        n = self.hb * self.B
        buf = (ctypes.c_uint8 * n).from_address(p)
        return np.frombuffer(buf, dtype=np.uint8).reshape(self.hb, self.B)

    def set_protected_calls(self, calls: int) -> None:
        """Slots selected by each request's last `calls` calls are not victims."""
        if self.lib.hso_set_protected_calls(self.h, calls) != 0:
            raise ValueError("negative count")

    # -- paged host pool ----------------------------------------------------
    def reserve(self, requests, num_tokens) -> int:
        """0, -1 (bad argument) or -2 (pool exhausted); nothing changes on error."""
        q = np.ascontiguousarray(requests, dtype=np.int32)
        n = np.ascontiguousarray(num_tokens, dtype=np.int64)
        assert q.shape == n.shape
        return int(self.lib.hso_reserve(self.h, q.size, _ptr(q), _ptr(n)))

    def release(self, requests) -> int:
        q = np.ascontiguousarray(requests, dtype=np.int32)
        return int(self.lib.hso_release(self.h, q.size, _ptr(q)))

    def block_table(self, r: int) -> np.ndarray:
        n = int(self.lib.hso_block_table(self.h, r, None))
        if n < 0:
            raise ValueError("no paged pool, or bad request")
        ids = np.empty(max(n, 1), dtype=np.int32)
        self.lib.hso_block_table(self.h, r, _ptr(ids))
        return ids[:n].copy()

    def free_blocks(self) -> int:
        return int(self.lib.hso_free_blocks(self.h))

    # -- calls ------------------------------------------------------------
    def prefill(self, seq_lens) -> np.ndarray:
        """Restart requests (S = -1 leaves one alone); returns the status
        array (entries of skipped requests are 0)."""
        s = np.ascontiguousarray(seq_lens, dtype=np.int32)
        st = np.zeros(self.R, dtype=np.int32)
        self.lib.hso_prefill(self.h, _ptr(s), _ptr(st))
        return st

    def swap_in(self, layer: int, topk, seq_lens, resident_blocks=None, block_size: int = 0):
        """Returns (out [R][k], plan [R][k][2], count [R], status [R]).
        resident_blocks: optional int32 [R][max_blocks] resident block table."""
        t = np.ascontiguousarray(topk, dtype=np.int32).reshape(self.R, self.k)
        s = np.ascontiguousarray(seq_lens, dtype=np.int32)
        out = np.full((self.R, self.k), -7, dtype=np.int32)
        plan = np.full((self.R, self.k, 2), -7, dtype=np.int32)
        cnt = np.zeros(self.R, dtype=np.int32)
        st = np.zeros(self.R, dtype=np.int32)
        if resident_blocks is None:
            rc = self.lib.hso_swap_in(self.h, layer, _ptr(t), _ptr(s), _ptr(out),
                                      _ptr(plan), _ptr(cnt), _ptr(st))
        else:
            rb = np.ascontiguousarray(resident_blocks, dtype=np.int32).reshape(self.R, -1)
            rc = self.lib.hso_swap_in_resident(self.h, layer, _ptr(t), _ptr(s), _ptr(rb),
                                               rb.shape[1], block_size, _ptr(out), _ptr(plan),
                                               _ptr(cnt), _ptr(st))
        if rc != 0:
            raise ValueError("layer holds no hot state")
        return out, plan, cnt, st

    def replay(self, plan, count, layer: int) -> None:
        p = np.ascontiguousarray(plan, dtype=np.int32)
        c = np.ascontiguousarray(count, dtype=np.int32)
        if self.lib.hso_replay(self.h, _ptr(p), _ptr(c), layer) != 0:
            raise ValueError("bad layer")

    def backup(self, layer: int, rows, positions) -> np.ndarray:
        rw = np.ascontiguousarray(rows, dtype=np.uint8).reshape(self.R, self.B)
        pos = np.ascontiguousarray(positions, dtype=np.int32)
        st = np.zeros(self.R, dtype=np.int32)
        if self.lib.hso_backup(self.h, layer, _ptr(rw), _ptr(pos), _ptr(st)) != 0:
            raise ValueError("bad layer")
        return st

    def status_word(self) -> np.ndarray:
        """int32 [R]: per request, the OR of (1 << code) over every error
        code a call returned for it since creation or the last clear."""
        words = np.empty(self.R, dtype=np.int32)
        self.lib.hso_status_word(self.h, _ptr(words))
        return words

    def status_clear(self) -> None:
        self.lib.hso_status_clear(self.h)

    def state(self, layer: int):
        """(slot2tok [R][D], last_used [R][D], tok2slot [total_cap], ticks [R])."""
        s2t = np.empty((self.R, self.D), dtype=np.int32)
        lu = np.empty((self.R, self.D), dtype=np.uint32)
        t2s = np.empty(max(self.total_cap, 1), dtype=np.int32)
        ticks = np.empty(self.R, dtype=np.uint32)
        if self.lib.hso_state(self.h, layer, _ptr(s2t), _ptr(lu), _ptr(t2s), _ptr(ticks)) != 0:
            raise ValueError("layer holds no hot state")
        return s2t, lu, t2s[: self.total_cap], ticks
