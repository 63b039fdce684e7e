"""The C ABI library loads and exports every declared entry point; its
host-side checks return the documented codes (CPU only, no GPU calls)."""

import ctypes
import glob
import os
import re

import numpy as np
import pytest

from hierarchical_sparse_kv_request_gb300 import build as B
from hierarchical_sparse_kv_request_gb300 import hisparse as H

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    B.build_library()
    return H.load_library()


def declared_functions():
    names = set()
    for hdr in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(hdr).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"\b(hisparse_\w+)\s*\(", text))
    return sorted(names)


def test_headers_declare_the_entry_points():
    names = declared_functions()
    for n in ["hisparse_create", "hisparse_swap_in", "hisparse_replay_plan", "hisparse_backup",
              "hisparse_prefill", "hisparse_destroy", "hisparse_link_probe"]:
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_version_and_error_strings(lib):
    assert lib.hisparse_version() == 201
    for code in range(0, -9, -1):
        assert lib.hisparse_error_string(code) not in (None, b"unknown error")
    assert lib.hisparse_error_string(-99) == b"unknown error"


def _create(lib, R=2, L=1, B_=16, k=8, D=16, ratio=10, caps=(50, 50), anchors=None):
    caps = np.ascontiguousarray(caps, dtype=np.int64)
    anc = None if anchors is None else np.ascontiguousarray(anchors, dtype=np.int32)
    lay = H.Layout(R, L, B_, k, D, ratio, 960, None if anc is None else anc.ctypes.data,
                   caps.ctypes.data)
    h = ctypes.c_void_p(1234)
    rc = lib.hisparse_create(ctypes.byref(lay), ctypes.byref(h))
    return rc, h


@pytest.mark.parametrize("kw,code", [
    (dict(k=17, D=16), H.ERR_LAYOUT),                     # top_k > device_buffer_size
    (dict(B_=24), H.ERR_LAYOUT),                          # row_bytes not a multiple of 16
    (dict(B_=0), H.ERR_LAYOUT),
    (dict(R=0, caps=()), H.ERR_LAYOUT),
    (dict(ratio=0), H.ERR_LAYOUT),
    (dict(caps=(200, 200), ratio=10), H.ERR_CAPACITY),   # 400 > 10 * 2 * 16
    (dict(caps=(-1, 5)), H.ERR_LAYOUT),
    (dict(caps=(0, 0)), H.ERR_LAYOUT),
    (dict(L=2, anchors=(0, 0)), H.ERR_LAYOUT),            # a layer anchored on itself
    (dict(L=3, anchors=(-1, 0, 1)), H.ERR_LAYOUT),        # an anchor that owns no state
    (dict(L=2, anchors=(1, 0)), H.ERR_LAYOUT),            # no layer owns state
    (dict(L=2, anchors=(-1, 5)), H.ERR_LAYOUT),
    (dict(k=9000, D=9000, caps=(1, 1), ratio=1), H.ERR_UNSUPPORTED),
    (dict(D=40000, caps=(1, 1)), H.ERR_UNSUPPORTED),
    (dict(caps=((1 << 20) + 1, 1), ratio=100000), H.ERR_UNSUPPORTED),
])
def test_create_rejects_bad_layouts_before_any_gpu_work(lib, kw, code):
    rc, h = _create(lib, **kw)
    assert rc == code
    assert h.value is None                      # *out cleared on error


def _create_paged(lib, hb, R=2, D=16, ratio=10, caps=(500, 500)):
    caps = np.ascontiguousarray(caps, dtype=np.int64)
    lay = H.Layout(R, 1, 16, 8, D, ratio, 960, None, caps.ctypes.data)
    h = ctypes.c_void_p(1234)
    rc = lib.hisparse_create_paged(ctypes.byref(lay), hb, ctypes.byref(h))
    return rc, h


@pytest.mark.parametrize("kw,code", [
    (dict(hb=0), H.ERR_LAYOUT),
    (dict(hb=-4), H.ERR_LAYOUT),
    (dict(hb=64, ratio=1), H.ERR_CAPACITY),               # 1 * 2 * 16 rows: no whole block of 64
    (dict(hb=(1 << 16) + 1), H.ERR_UNSUPPORTED),
    (dict(hb=16, ratio=0), H.ERR_LAYOUT),
    (dict(hb=4, caps=((1 << 20) + 1, 1)), H.ERR_UNSUPPORTED),
])
def test_create_paged_rejects_bad_layouts_before_any_gpu_work(lib, kw, code):
    rc, h = _create_paged(lib, **kw)
    assert rc == code
    assert h.value is None


def test_null_arguments(lib):
    h = ctypes.c_void_p()
    assert lib.hisparse_create(None, ctypes.byref(h)) == H.ERR_INVALID_ARG
    assert lib.hisparse_create(None, None) == H.ERR_INVALID_ARG
    assert lib.hisparse_destroy(None) == H.OK
    assert lib.hisparse_swap_in(None, 0, None, None, None, None, None) == H.ERR_INVALID_ARG
    assert lib.hisparse_replay_plan(None, None, 0, 0, None) == H.ERR_INVALID_ARG
    assert lib.hisparse_backup(None, 0, None, None, None) == H.ERR_INVALID_ARG
    assert lib.hisparse_prefill(None, None, None) == H.ERR_INVALID_ARG
    assert lib.hisparse_status(None, None) == H.ERR_INVALID_ARG
    assert lib.hisparse_read_state(None, 0, None, None, None, None, None, None) == H.ERR_INVALID_ARG
    assert lib.hisparse_set_copy_mode(None, 1) == H.ERR_INVALID_ARG
    assert lib.hisparse_set_protected_calls(None, 1) == H.ERR_INVALID_ARG
    assert lib.hisparse_set_stage_rows(None, 1) == H.ERR_INVALID_ARG
    assert lib.hisparse_set_programmatic_launch(None, 1) == H.ERR_INVALID_ARG
    assert lib.hisparse_status_clear(None, None) == H.ERR_INVALID_ARG
    assert lib.hisparse_backup_layers(None, None, 1, None, None, None) == H.ERR_INVALID_ARG
    assert lib.hisparse_write_state(None, 0, None, None, None, 1, None) == H.ERR_INVALID_ARG
    assert lib.hisparse_check_guards(None, None) == H.ERR_INVALID_ARG
    assert lib.hisparse_link_probe(None, None, 16, 0, None) == H.ERR_INVALID_ARG
    assert lib.hisparse_link_gather(None, 16, None, 1, None, 0, None) == H.ERR_INVALID_ARG
    assert lib.hisparse_synthetic_compute(None, 0, 1, 1, None) == H.ERR_INVALID_ARG
    assert lib.hisparse_create_paged(None, 16, ctypes.byref(h)) == H.ERR_INVALID_ARG
    assert lib.hisparse_create_paged(None, 16, None) == H.ERR_INVALID_ARG
    assert lib.hisparse_host_reserve(None, 0, None, None, None) == H.ERR_INVALID_ARG
    assert lib.hisparse_host_release(None, 0, None, None) == H.ERR_INVALID_ARG
    assert lib.hisparse_host_block_table(None, 0, None, 0, None) == H.ERR_INVALID_ARG
    assert lib.hisparse_host_pool_info(None, None, None, None) == H.ERR_INVALID_ARG
    assert lib.hisparse_host_block_rows(None, 0, 0, None) == H.ERR_INVALID_ARG


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError):
        H.load_library(str(tmp_path / "libhisparse.so"))


def test_binding_constants_match_the_header():
    """The Python binding's return codes, status codes, copy modes and sizes
    are the values include/hisparse.h defines."""
    text = open(os.path.join(ROOT, "include", "hisparse.h")).read()
    defs = {}
    for name, val in re.findall(r"#define\s+HISPARSE_(\w+)\s+(\([^)]*\)|-?\w+)", text):
        v = val.strip("()")
        if "<<" in v:
            a, b = v.split("<<")
            defs[name] = int(a) << int(b)
        else:
            try:
                defs[name] = int(v, 0)
            except ValueError:
                pass
    pairs = {"OK": H.OK, "ERR_INVALID_ARG": H.ERR_INVALID_ARG, "ERR_LAYOUT": H.ERR_LAYOUT,
             "ERR_CAPACITY": H.ERR_CAPACITY, "ERR_LAYER": H.ERR_LAYER, "ERR_CUDA": H.ERR_CUDA,
             "ERR_NO_MEMORY": H.ERR_NO_MEMORY, "ERR_UNSUPPORTED": H.ERR_UNSUPPORTED,
             "ERR_ALIGNMENT": H.ERR_ALIGNMENT,
             "STATUS_OK": H.STATUS_OK, "STATUS_BAD_INDEX": H.STATUS_BAD_INDEX,
             "STATUS_DUPLICATE": H.STATUS_DUPLICATE, "STATUS_BAD_SEQ_LEN": H.STATUS_BAD_SEQ_LEN,
             "STATUS_BAD_POSITION": H.STATUS_BAD_POSITION,
             "STATUS_BAD_RESIDENT": H.STATUS_BAD_RESIDENT,
             "STATUS_NO_HOST_ROW": H.STATUS_NO_HOST_ROW, "STATUS_CAPACITY": H.STATUS_CAPACITY,
             "STATUS_COPY_TIMEOUT": H.STATUS_COPY_TIMEOUT,
             "RESIDENT_FLAG": H.RESIDENT_FLAG, "COPY_FUSED": H.COPY_FUSED,
             "COPY_SPLIT": H.COPY_SPLIT, "COPY_AUTO": H.COPY_AUTO,
             "NOALLOC_SCRATCH_BYTES": H.NOALLOC_SCRATCH_BYTES}
    for name, value in pairs.items():
        assert defs.get(name) == value, (name, defs.get(name), value)


def test_create_refuses_a_chunk_count_beyond_32_bits(lib):
    """top_k x row_bytes / 16 above 2^31 - 1 is refused before any GPU work
    (k 8192 with 4 MB rows on a single request would fit in HBM)."""
    rc, h = _create(lib, R=1, L=1, B_=4 << 20, k=8192, D=8192, ratio=10, caps=(8192,))
    assert rc == H.ERR_UNSUPPORTED
