"""N > 1 host path of bench.py on CPU: two gloo ranks, each with its own batch
(weak scaling, no data-path collective); the timing is the max over ranks and
the throughput counts every rank's tokens."""
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist

    import bench
    import workloads
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, lr, w = bench.dist_env()
    assert (r, lr, w) == (rank, rank, world)
    # each rank draws its own decode batch (seed offset by rank), as bench.py does
    wl = workloads.decode_heavy(seed=1 + 1000 * rank, num_requests=8, values=False)
    tokens = wl.layout.num_tokens
    ms = 10.0 + 5.0 * rank                       # pretend per-rank step time
    bench.barrier(world)
    ms_max = bench.max_over_ranks(ms, world, "cpu")
    tot = bench.sum_over_ranks(tokens, world, "cpu")
    q.put((rank, ms_max, tot, int(wl.layout.kv_len.sum())))
    dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_like_bench():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert all(r[1] == 15.0 for r in res)            # max over ranks
    assert all(r[2] == 16 for r in res)              # 8 decode tokens per rank, summed
    assert res[0][3] != res[1][3]                    # ranks run different batches
