"""The measurement kernels move the right bytes: the row gather (both its
mappings: 64-byte-aligned spans for rows under 1 KB, consecutive chunks for
longer rows, from bases at every 16-byte offset within 64 bytes) and the
sequential link probe, against numpy copies of the same pinned buffers."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from hierarchical_sparse_kv_request_gb300 import hisparse as H

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("row_bytes", [16, 48, 656, 1008, 1024, 1152])
@pytest.mark.parametrize("base_off", [0, 16, 32, 48])
def test_link_gather_rows(row_bytes, base_off):
    rng = np.random.default_rng(row_bytes * 7 + base_off)
    nrows_pool = 3000
    pool = torch.empty(nrows_pool * row_bytes + 64, dtype=torch.uint8, pin_memory=True)
    host = pool.numpy()
    host[:] = rng.integers(0, 256, host.size, dtype=np.uint8)
    base = pool.data_ptr() + base_off
    assert base % 16 == 0
    src = host[base_off: base_off + nrows_pool * row_bytes].reshape(nrows_pool, row_bytes)
    for n, ctas in [(1, 0), (37, 1), (1000, 3), (2500, 0)]:
        rows = rng.choice(nrows_pool, n, replace=False).astype(np.int64)
        rows_d = torch.from_numpy(rows).cuda()
        dst = torch.full((n * row_bytes + 32,), 0xA5, dtype=torch.uint8, device="cuda")
        H.link_gather(base, row_bytes, rows_d, dst, num_ctas=ctas)
        torch.cuda.synchronize()
        got = dst.cpu().numpy()
        assert np.array_equal(got[:n * row_bytes].reshape(n, row_bytes), src[rows]), (n, ctas)
        assert (got[n * row_bytes:] == 0xA5).all(), "wrote past the last row"


def test_link_probe_copies_bytes():
    rng = np.random.default_rng(3)
    nbytes = (5 << 20) + 48
    src = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    src.numpy()[:] = rng.integers(0, 256, nbytes, dtype=np.uint8)
    dst = torch.full((nbytes + 16,), 7, dtype=torch.uint8, device="cuda")
    H.link_probe(src, dst, nbytes)
    torch.cuda.synchronize()
    got = dst.cpu().numpy()
    assert np.array_equal(got[:nbytes], src.numpy())
    assert (got[nbytes:] == 7).all()
