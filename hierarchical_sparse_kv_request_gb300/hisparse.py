"""Thin ctypes binding of libhisparse.so (include/hisparse.h).

Argument marshalling only: every step of the swap-in path runs in the CUDA
library.  Device arrays may be passed as torch CUDA tensors or raw integer
addresses; streams as torch streams, raw ``cudaStream_t`` integers or None
(torch's current stream).  There is no CPU fallback: if the library is not
built, loading it raises.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libhisparse.so")

OK = 0
ERR_INVALID_ARG, ERR_LAYOUT, ERR_CAPACITY, ERR_LAYER = -1, -2, -3, -4
ERR_CUDA, ERR_NO_MEMORY, ERR_UNSUPPORTED, ERR_ALIGNMENT = -5, -6, -7, -8
STATUS_OK, STATUS_BAD_INDEX, STATUS_DUPLICATE, STATUS_BAD_SEQ_LEN, STATUS_BAD_POSITION = 0, 1, 2, 3, 4
STATUS_BAD_RESIDENT, STATUS_NO_HOST_ROW, STATUS_CAPACITY, STATUS_COPY_TIMEOUT = 5, 6, 7, 8


def STATUS_BIT(code: int) -> int:
    """The bit a status code sets in a request's status word."""
    return 1 << code


RESIDENT_FLAG = 1 << 30
COPY_FUSED, COPY_SPLIT, COPY_AUTO = 1, 2, 3
NOALLOC_SCRATCH_BYTES = 8 << 20   # HISPARSE_NOALLOC_SCRATCH_BYTES


class HiSparseError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {error_string(code)} ({code})")
        self.code = code


class Layout(ctypes.Structure):
    _fields_ = [("num_requests", ctypes.c_int32), ("num_layers", ctypes.c_int32),
                ("row_bytes", ctypes.c_int64), ("top_k", ctypes.c_int32),
                ("device_buffer_size", ctypes.c_int32),
                ("host_to_device_ratio", ctypes.c_int32),
                ("swap_in_block_size", ctypes.c_int32),
                ("anchor_of_layer", ctypes.c_void_p), ("host_capacity", ctypes.c_void_p)]


class Plan(ctypes.Structure):
    _fields_ = [("rows", ctypes.c_void_p), ("counts", ctypes.c_void_p)]


_lib: Optional[ctypes.CDLL] = None


def load_library(path: Optional[str] = None) -> ctypes.CDLL:
    """Load libhisparse.so (built in-tree by ``__graft_entry__.build()``)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"{p} is missing: build the CUDA library first "
                           "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(p)
    P, I32, I64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    sig = {
        "hisparse_create": [P, P],
        "hisparse_create_paged": [P, I32, P],
        "hisparse_host_reserve": [P, I32, P, P, P],
        "hisparse_host_release": [P, I32, P, P],
        "hisparse_host_block_table": [P, I32, P, I32, P],
        "hisparse_host_pool_info": [P, P, P, P],
        "hisparse_host_block_rows": [P, I32, I32, P],
        "hisparse_destroy": [P],
        "hisparse_host_rows": [P, I32, I32, P],
        "hisparse_device_buffer": [P, I32, P],
        "hisparse_prefill": [P, P, P],
        "hisparse_swap_in": [P, I32, P, P, P, P, P],
        "hisparse_swap_in_noalloc": [P, I32, P, P, P, P],
        "hisparse_swap_in_resident": [P, I32, P, P, P, I32, I32, P, P, P],
        "hisparse_replay_plan": [P, P, I32, I32, P],
        "hisparse_replay_plan_layers": [P, P, P, I32, I32, P],
        "hisparse_backup": [P, I32, P, P, P],
        "hisparse_backup_layers": [P, P, I32, P, P, P],
        "hisparse_status": [P, P],
        "hisparse_status_clear": [P, P],
        "hisparse_read_state": [P, I32, P, P, P, P, P, P],
        "hisparse_write_state": [P, I32, P, P, P, I32, P],
        "hisparse_set_copy_mode": [P, I32],
        "hisparse_set_protected_calls": [P, I32],
        "hisparse_set_stage_rows": [P, I32],
        "hisparse_set_programmatic_launch": [P, I32],
        "hisparse_set_copy_ctas": [P, I32],
        "hisparse_get_copy_ctas": [P, P],
        "hisparse_check_guards": [P, P],
        "hisparse_version": [],
        "hisparse_synthetic_compute": [P, I64, I32, I32, P],
        "hisparse_link_probe": [P, P, I64, I32, P],
        "hisparse_link_gather": [P, I64, P, I64, P, I32, P],
    }
    for name, args in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = ctypes.c_int
    lib.hisparse_error_string.argtypes = [ctypes.c_int]
    lib.hisparse_error_string.restype = ctypes.c_char_p
    if path is None:
        _lib = lib
    return lib


def error_string(code: int) -> str:
    try:
        return load_library().hisparse_error_string(code).decode()
    except RuntimeError:
        return "unknown"


def _addr(x) -> Optional[int]:
    """Device/host address of a torch tensor, numpy array or raw integer."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if isinstance(x, np.ndarray):
        return x.ctypes.data
    return x.data_ptr()


def _stream(s) -> Optional[int]:
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(rc: int, what: str) -> None:
    if rc != OK:
        raise HiSparseError(rc, what)


class HiSparse:
    """One handle of the swap-in resolver (see include/hisparse.h).

    host_block_tokens > 0 creates a paged host pool (hisparse_create_paged):
    host_capacity then only bounds each request's length, and rows come from
    blocks that host_reserve hands out."""

    def __init__(self, num_requests: int, num_layers: int, row_bytes: int, top_k: int,
                 device_buffer_size: int, host_to_device_ratio: int,
                 host_capacity: Sequence[int], anchor_of_layer: Optional[Sequence[int]] = None,
                 swap_in_block_size: int = 960, host_block_tokens: int = 0):
        self.lib = load_library()
        self.R, self.L, self.B = num_requests, num_layers, row_bytes
        self.k, self.D = top_k, device_buffer_size
        self.cap = np.ascontiguousarray(host_capacity, dtype=np.int64)
        self.anchor = np.ascontiguousarray(
            anchor_of_layer if anchor_of_layer is not None else [-1] * num_layers, dtype=np.int32)
        self.total_cap = int(self.cap.sum())
        lay = Layout(num_requests, num_layers, row_bytes, top_k, device_buffer_size,
                     host_to_device_ratio, swap_in_block_size,
                     self.anchor.ctypes.data, self.cap.ctypes.data)
        h = ctypes.c_void_p()
        self.hb = int(host_block_tokens)
        if self.hb:
            _check(self.lib.hisparse_create_paged(ctypes.byref(lay), self.hb, ctypes.byref(h)),
                   "hisparse_create_paged")
        else:
            _check(self.lib.hisparse_create(ctypes.byref(lay), ctypes.byref(h)), "hisparse_create")
        self.h = h

    @classmethod
    def for_workload(cls, w, host_block_tokens: int = 0) -> "HiSparse":
        return cls(w.num_requests, w.num_layers, w.row_bytes, w.top_k, w.device_buffer_size,
                   w.host_to_device_ratio, w.host_capacity, w.anchor_of_layer,
                   host_block_tokens=host_block_tokens)

    def close(self) -> None:
        if getattr(self, "h", None) and self.h.value:
            self.lib.hisparse_destroy(self.h)
            self.h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -- storage ------------------------------------------------------------
    def host_rows_ptr(self, layer: int, request: int) -> int:
        p = ctypes.c_void_p()
        _check(self.lib.hisparse_host_rows(self.h, layer, request, ctypes.byref(p)),
               "hisparse_host_rows")
        return p.value

    def host_rows(self, layer: int, request: int) -> np.ndarray:
        """Writable numpy view [host_capacity[request]][B] of pinned host rows."""
        n = int(self.cap[request]) * self.B
        buf = (ctypes.c_uint8 * n).from_address(self.host_rows_ptr(layer, request))
        return np.frombuffer(buf, dtype=np.uint8).reshape(int(self.cap[request]), self.B)

    # -- paged host pool ----------------------------------------------------
    def host_reserve(self, requests, num_tokens, stream=None) -> None:
        """Grow the block tables so request requests[i] covers tokens
        [0, num_tokens[i]); raises HiSparseError (code ERR_CAPACITY when the
        pool is short, nothing reserved)."""
        q = np.ascontiguousarray(requests, dtype=np.int32)
        n = np.ascontiguousarray(num_tokens, dtype=np.int64)
        if q.shape != n.shape:
            raise ValueError("requests and num_tokens differ in length")
        _check(self.lib.hisparse_host_reserve(self.h, q.size, q.ctypes.data, n.ctypes.data,
                                              _stream(stream)), "hisparse_host_reserve")

    def host_release(self, requests, stream=None) -> None:
        q = np.ascontiguousarray(requests, dtype=np.int32)
        _check(self.lib.hisparse_host_release(self.h, q.size, q.ctypes.data, _stream(stream)),
               "hisparse_host_release")

    def host_block_table(self, request: int) -> np.ndarray:
        cnt = ctypes.c_int32()
        _check(self.lib.hisparse_host_block_table(self.h, request, None, 0, ctypes.byref(cnt)),
               "hisparse_host_block_table")
        ids = np.empty(max(cnt.value, 1), dtype=np.int32)
        _check(self.lib.hisparse_host_block_table(self.h, request, ids.ctypes.data, cnt.value,
                                                  ctypes.byref(cnt)), "hisparse_host_block_table")
        return ids[: cnt.value].copy()

    def host_pool_info(self):
        """(host_block_tokens, pool_blocks, free_blocks)."""
        v = [ctypes.c_int32() for _ in range(3)]
        _check(self.lib.hisparse_host_pool_info(self.h, *[ctypes.byref(x) for x in v]),
               "hisparse_host_pool_info")
        return tuple(x.value for x in v)

    def host_block_rows(self, layer: int, block: int) -> np.ndarray:
        """Writable numpy view [host_block_tokens][B] of a pinned pool block."""
        p = ctypes.c_void_p()
        _check(self.lib.hisparse_host_block_rows(self.h, layer, block, ctypes.byref(p)),
               "hisparse_host_block_rows")
        buf = (ctypes.c_uint8 * (self.hb * self.B)).from_address(p.value)
        return np.frombuffer(buf, dtype=np.uint8).reshape(self.hb, self.B)

    def write_host_rows(self, layer: int, request: int, t0: int, rows: np.ndarray) -> None:
        """Copy rows ([n][B] uint8) into the pinned host rows of tokens
        [t0, t0 + n) of (layer, request): the request's region, or, with a
        paged pool, the blocks its table names (which must be reserved)."""
        n = rows.shape[0]
        if not self.hb:
            self.host_rows(layer, request)[t0:t0 + n] = rows
            return
        hb = self.hb
        table = self.host_block_table(request)
        t1 = t0 + n
        if n and (t1 - 1) // hb >= table.size:
            raise ValueError("rows beyond the request's reserved host blocks")
        for b in range(t0 // hb, (t1 + hb - 1) // hb):
            a, e = max(b * hb, t0), min((b + 1) * hb, t1)
            self.host_block_rows(layer, int(table[b]))[a - b * hb:e - b * hb] = rows[a - t0:e - t0]

    def device_buffer_ptr(self, layer: int) -> int:
        p = ctypes.c_void_p()
        _check(self.lib.hisparse_device_buffer(self.h, layer, ctypes.byref(p)),
               "hisparse_device_buffer")
        return p.value

    def device_buffer(self, layer: int):
        """torch uint8 CUDA tensor [R][D][B] aliasing the layer's hot buffer."""
        import torch

        class _View:
            __cuda_array_interface__ = {
                "shape": (self.R, self.D, self.B), "typestr": "|u1",
                "data": (self.device_buffer_ptr(layer), False), "version": 3,
                "strides": None}
        return torch.as_tensor(_View(), device="cuda")

    def status_ptr(self) -> int:
        p = ctypes.c_void_p()
        _check(self.lib.hisparse_status(self.h, ctypes.byref(p)), "hisparse_status")
        return p.value

    def status_clear(self, stream=None) -> None:
        """hisparse_status_clear: zero every request's status word (stream-ordered)."""
        _check(self.lib.hisparse_status_clear(self.h, _stream(stream)), "hisparse_status_clear")

    def status(self):
        """torch int32 CUDA tensor [R] aliasing the status words: bit
        STATUS_BIT(code) of entry r is set for every error code request r met
        since the handle was created or the words were last cleared."""
        import torch

        class _View:
            __cuda_array_interface__ = {
                "shape": (self.R,), "typestr": "<i4", "data": (self.status_ptr(), False),
                "version": 3, "strides": None}
        return torch.as_tensor(_View(), device="cuda")

    # -- decode path --------------------------------------------------------
    def prefill(self, seq_lens, stream=None) -> None:
        _check(self.lib.hisparse_prefill(self.h, _addr(seq_lens), _stream(stream)),
               "hisparse_prefill")

    def swap_in(self, layer: int, topk, seq_lens, out_slot_ids, plan_rows=None,
                plan_counts=None, stream=None) -> None:
        plan = None
        if plan_rows is not None or plan_counts is not None:
            plan = ctypes.byref(Plan(_addr(plan_rows), _addr(plan_counts)))
        _check(self.lib.hisparse_swap_in(self.h, layer, _addr(topk), _addr(seq_lens),
                                         _addr(out_slot_ids), plan, _stream(stream)),
               "hisparse_swap_in")

    def swap_in_resident(self, layer: int, topk, seq_lens, resident_blocks, block_size: int,
                         out_slot_ids, plan_rows=None, plan_counts=None, stream=None) -> None:
        """hisparse_swap_in_resident; resident_blocks is a [R][max_blocks]
        int32 device tensor of resident page ids (-1 = not resident)."""
        plan = None
        if plan_rows is not None or plan_counts is not None:
            plan = ctypes.byref(Plan(_addr(plan_rows), _addr(plan_counts)))
        max_blocks = int(resident_blocks.shape[1])
        _check(self.lib.hisparse_swap_in_resident(self.h, layer, _addr(topk), _addr(seq_lens),
                                                  _addr(resident_blocks), max_blocks, block_size,
                                                  _addr(out_slot_ids), plan, _stream(stream)),
               "hisparse_swap_in_resident")

    def swap_in_noalloc(self, layer: int, topk, seq_lens, out_slot_ids, stream=None) -> None:
        """hisparse_swap_in_noalloc: the split-copy swap-in whose internal
        miss plan lives in the library's fixed per-GPU array, so the call
        causes no device allocation (for callers that may not allocate)."""
        _check(self.lib.hisparse_swap_in_noalloc(self.h, layer, _addr(topk), _addr(seq_lens),
                                                 _addr(out_slot_ids), _stream(stream)),
               "hisparse_swap_in_noalloc")

    def replay_plan(self, plan_rows, plan_counts, layer: int, num_ctas: int = 0,
                    stream=None) -> None:
        plan = Plan(_addr(plan_rows), _addr(plan_counts))
        _check(self.lib.hisparse_replay_plan(self.h, ctypes.byref(plan), layer, num_ctas,
                                             _stream(stream)), "hisparse_replay_plan")

    def replay_plan_layers(self, plan_rows, plan_counts, layers, num_ctas: int = 0,
                           stream=None) -> None:
        plan = Plan(_addr(plan_rows), _addr(plan_counts))
        lay = np.ascontiguousarray(layers, dtype=np.int32)
        _check(self.lib.hisparse_replay_plan_layers(self.h, ctypes.byref(plan), lay.ctypes.data,
                                                    len(lay), num_ctas, _stream(stream)),
               "hisparse_replay_plan_layers")

    def backup(self, layer: int, rows, positions, stream=None) -> None:
        _check(self.lib.hisparse_backup(self.h, layer, _addr(rows), _addr(positions),
                                        _stream(stream)), "hisparse_backup")

    def backup_layers(self, layers, rows, positions, stream=None) -> None:
        """hisparse_backup_layers: rows is a [len(layers)][R][B] uint8 device tensor."""
        lay = np.ascontiguousarray(layers, dtype=np.int32)
        _check(self.lib.hisparse_backup_layers(self.h, lay.ctypes.data, len(lay), _addr(rows),
                                               _addr(positions), _stream(stream)),
               "hisparse_backup_layers")

    def write_state(self, layer: int, slot2tok, last_used, ticks, rebuild_rows: bool = True,
                    stream=None) -> None:
        """hisparse_write_state from numpy arrays (slot2tok [R][D] int32,
        last_used [R][D] uint32, ticks [R] uint32)."""
        s2t = np.ascontiguousarray(slot2tok, dtype=np.int32).reshape(self.R, self.D)
        lu = np.ascontiguousarray(last_used, dtype=np.uint32).reshape(self.R, self.D)
        tk = np.ascontiguousarray(ticks, dtype=np.uint32).reshape(self.R)
        _check(self.lib.hisparse_write_state(self.h, layer, s2t.ctypes.data, lu.ctypes.data,
                                             tk.ctypes.data, 1 if rebuild_rows else 0,
                                             _stream(stream)), "hisparse_write_state")

    def check_guards(self) -> int:
        """Overwritten guard bands (handle created with HISPARSE_DEBUG_GUARDS=1)."""
        n = ctypes.c_int32()
        _check(self.lib.hisparse_check_guards(self.h, ctypes.byref(n)), "hisparse_check_guards")
        return n.value

    def set_protected_calls(self, calls: int) -> None:
        """Keep the hot rows of each request's last `calls` calls (0: off)."""
        _check(self.lib.hisparse_set_protected_calls(self.h, calls),
               "hisparse_set_protected_calls")

    def set_stage_rows(self, rows: int) -> None:
        """Miss rows per request the fused copy stages through shared memory
        with the bulk-copy engine (0: none, the default; -1: as many as fit)."""
        _check(self.lib.hisparse_set_stage_rows(self.h, rows), "hisparse_set_stage_rows")

    def set_copy_ctas(self, ctas: int) -> None:
        """CTAs per request of a fused-copy swap-in: 1 resolves and copies in
        one CTA; 2-4 form a cluster whose rank 0 resolves and whose other
        CTAs copy (hisparse_set_copy_ctas)."""
        _check(self.lib.hisparse_set_copy_ctas(self.h, ctas), "hisparse_set_copy_ctas")

    def copy_ctas(self) -> int:
        """CTAs per request that fused-copy swap-ins use now."""
        v = ctypes.c_int32(0)
        _check(self.lib.hisparse_get_copy_ctas(self.h, ctypes.byref(v)), "hisparse_get_copy_ctas")
        return int(v.value)

    def set_programmatic_launch(self, on: bool) -> None:
        """Launch swap-ins and backups with a programmatic dependency on the
        stream's previous kernel (off by default)."""
        _check(self.lib.hisparse_set_programmatic_launch(self.h, 1 if on else 0),
               "hisparse_set_programmatic_launch")

    def set_copy_mode(self, mode: int) -> None:
        _check(self.lib.hisparse_set_copy_mode(self.h, mode), "hisparse_set_copy_mode")

    def read_state(self, layer: int, stream=None):
        """(slot2tok [R][D], last_used [R][D], tok2slot [total_cap], lru [R][D], ticks [R])."""
        s2t = np.empty((self.R, self.D), dtype=np.int32)
        lu = np.empty((self.R, self.D), dtype=np.uint32)
        t2s = np.empty(self.total_cap, dtype=np.int32)
        lru = np.empty((self.R, self.D), dtype=np.int32)
        ticks = np.empty(self.R, dtype=np.uint32)
        _check(self.lib.hisparse_read_state(self.h, layer, s2t.ctypes.data, lu.ctypes.data,
                                            t2s.ctypes.data, lru.ctypes.data, ticks.ctypes.data,
                                            _stream(stream)), "hisparse_read_state")
        return s2t, lu, t2s, lru, ticks


# -- measurement kernels (include/hisparse_measure.h) -----------------------

def synthetic_compute(buf, passes: int, ctas_per_sm: int = 2, stream=None) -> None:
    """The memory-bound bf16 stand-in compute over torch tensor `buf`."""
    lib = load_library()
    _check(lib.hisparse_synthetic_compute(_addr(buf), buf.numel() * buf.element_size(), passes,
                                          ctas_per_sm, _stream(stream)),
           "hisparse_synthetic_compute")


def link_gather(src, row_bytes: int, rows, dst, num_ctas: int = 0, stream=None) -> None:
    """hisparse_link_gather: dst row i <- src row rows[i] (rows: device int64
    tensor, every entry in range -- the kernel does not check)."""
    lib = load_library()
    _check(lib.hisparse_link_gather(_addr(src), row_bytes, _addr(rows), int(rows.numel()),
                                    _addr(dst), num_ctas, _stream(stream)),
           "hisparse_link_gather")


def link_probe(src, dst, nbytes: int, num_ctas: int = 0, stream=None) -> None:
    lib = load_library()
    _check(lib.hisparse_link_probe(_addr(src), _addr(dst), nbytes, num_ctas, _stream(stream)),
           "hisparse_link_probe")
