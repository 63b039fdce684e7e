"""Multi-rank host logic of bench.py on CPU: two gloo ranks.

The swap-in path shards by request with no exchange step, so N GPUs run N
independent replicas; the only cross-rank work is timing: the job's time is
the slowest rank's, and the job's throughput counts every rank's rows.
"""

import os
import socket
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, q):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    from hierarchical_sparse_kv_request_gb300 import workload as W

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = bench.dist_env()
        my_time = 1.0 + rank          # rank 1 is the slower one
        job_time = bench.max_over_ranks(my_time, "cpu")
        value = bench.job_throughput(1000.0, ws, job_time)
        # each rank's replica draws its own top-k sets
        w = W.make_config(1)
        w.seed = bench.replica_seed(w.seed, rank)
        first = W.topk_schedule(w)[0][0, 1]
        q.put((rank, ws, r, job_time, value, first.tolist()))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_time_and_throughput():
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, ws0, rr0, t0, v0, f0), (r1, ws1, rr1, t1, v1, f1) = res
    assert (ws0, ws1, rr0, rr1) == (2, 2, 0, 1)
    assert t0 == t1 == 2.0                 # the slowest rank's time
    assert v0 == v1 == 1000.0 * 2 / 2.0    # all ranks' rows over the job time
    assert f0 != f1                        # independent replicas


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_throughput(100.0, 1, 2.0) == 50.0
    assert bench.replica_seed(7, 0) == 7
