"""N > 1 host paths on CPU with two gloo ranks: bench.py's aggregation (each
rank its own batch, weak scaling, max of the times, sum of the tokens), and one
batch split by pps_partition whose parts, computed on their own ranks, give
exactly the whole batch's output."""
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


def _shard_worker(rank, world, port, q):
    """One rank of a sharded batch: pps_partition assigns the requests, the rank
    computes its part (the fp64 oracle stands in for the GPU), and rank 0
    gathers every rank's rows over gloo -- a test-only gather; the path itself
    needs no collective because every output row belongs to one rank."""
    import sys
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import numpy as np
    import torch
    import torch.distributed as dist

    import paged_prefix_shared_gb300 as pps
    import workloads
    from oracle_run import oracle_steps
    dist.init_process_group("gloo", rank=rank, world_size=world)
    wl = workloads.radix_sharing(groups=3, root=32, branch=16, pairs=2, tail_lo=1, tail_hi=20,
                                 num_q_heads=8, num_kv_heads=2, head_dim=32, page_size=16,
                                 keep_segments=True)
    L = wl.layout
    part, load = pps.partition(L.q_indptr, L.kv_len, L.page_indptr, L.page_indices,
                               L.page_size, world)
    mine = [r for r in range(L.num_requests) if part[r] == rank]
    sub = workloads.sub_workload(wl, 0, mine)
    out, _ = oracle_steps(sub)
    rows = np.zeros((L.num_tokens, L.num_q_heads, L.head_dim))
    for i, r in enumerate(mine):
        a, b = int(L.q_indptr[r]), int(L.q_indptr[r + 1])
        sa, sb = int(sub.layout.q_indptr[i]), int(sub.layout.q_indptr[i + 1])
        rows[a:b] = out[0][sa:sb]
    t = torch.from_numpy(rows)
    dist.all_reduce(t)                               # each row is non-zero on one rank only
    if rank == 0:
        whole, _ = oracle_steps(wl)
        q.put((bool(np.array_equal(t.numpy(), whole[0])), [int(x) for x in load],
               sorted(set(part.tolist()))))
    dist.destroy_process_group()


def test_partitioned_batch_over_two_ranks_matches_the_whole_batch():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_shard_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    same, load, parts = q.get(timeout=180)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert same and parts == [0, 1] and min(load) > 0
