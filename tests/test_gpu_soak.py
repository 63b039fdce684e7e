"""A long run: 600 decode calls of decode_40k-shaped requests (k 2048,
D 6144, 656 B rows, the workload's top-k process) with eager backups growing
every request, all in one process and one handle.  Every call's outputs are
compared with the oracle; the hot state and sampled device rows every 50
calls, and every device row at the end."""

import pytest
import torch

from harness import Pair, assert_call_equal, assert_device_rows, assert_state_equal
from hierarchical_sparse_kv_request_gb300 import workload as W

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

CALLS = 600


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def test_six_hundred_calls_with_growth():
    w = W.make_config(2, steps=CALLS, num_requests=6)
    w.backup = True                       # one new row per request per call
    sched = W.topk_schedule(w)[0]
    p = Pair(w, track_bytes=False)
    for c in range(CALLS):
        g, o = p.swap_in(0, sched[c])
        assert_call_equal(g, o, f"call {c}")
        if c % 50 == 49:
            s2t = assert_state_equal(p, 0, f"call {c}")
            assert_device_rows(p, 0, s2t, sample=64, seed=c, ctx=f"call {c}")
        st = p.backup(0, p.seq.copy())    # rows of position S, then S + 1
        assert (st == 0).all()
        p.advance()
    s2t = assert_state_equal(p, 0, "end")
    assert_device_rows(p, 0, s2t, ctx="end")
    assert (p.seq == w.seq_lens0 + CALLS).all()
    p.close()
