"""Pins for the reference batch partition (oracle/partition.py):
subtrees are never split (brute force over shared pages), every request is
placed, the loads add up, the largest-first greedy bound holds
(max load <= mean load + largest subtree), and a worked example."""
from __future__ import annotations

import numpy as np
import pytest

import workloads
from oracle import partition as op


def _shares_a_page(L, a, b):
    pa = set(L.page_indices[L.page_indptr[a]:L.page_indptr[a] + int(L.cached_len[a]) // L.page_size].tolist())
    pb = set(L.page_indices[L.page_indptr[b]:L.page_indptr[b] + int(L.cached_len[b]) // L.page_size].tolist())
    return bool(pa & pb)


@pytest.mark.parametrize("parts", [1, 2, 3, 8])
@pytest.mark.parametrize("name,kw", [
    ("radix_sharing", dict(groups=5, root=64, branch=32, pairs=2, tail_lo=1, tail_hi=80)),
    ("mixed_budget", dict(budget=300, prefill_q=100, prefill_cached=40, num_verify=5, mu=4.0,
                          sigma=1.0, clip_lo=1, clip_hi=600)),
    ("tiny_mixed", dict()),
])
def test_partition_properties(name, kw, parts):
    L = workloads.make(name, values=False, **kw).layout
    part, load = op.partition(L.q_indptr, L.kv_len, L.page_indptr, L.page_indices, L.page_size,
                              parts)
    R = L.num_requests
    assert len(part) == R and all(0 <= p < parts for p in part)
    for a in range(R):
        for b in range(a + 1, R):
            if _shares_a_page(L, a, b):
                assert part[a] == part[b], "a radix subtree was split"
    w = [max(1, int(L.q_len[r])) * int(L.kv_len[r]) for r in range(R)]
    assert sum(load) == sum(w)
    for p in range(parts):
        assert load[p] == sum(w[r] for r in range(R) if part[r] == p)
    # greedy bound: the part that got the last item was the least loaded then
    biggest = max(sum(w[r] for r in range(R) if part[r] == part[x] and _shares_a_page(L, r, x))
                  if L.cached_len[x] >= L.page_size else w[x] for x in range(R))
    assert max(load) <= sum(load) / parts + biggest


def test_worked_example():
    # 4 requests, P = 2: r0 and r1 share first page 7 (subtree work 1*10 + 1*10 = 20),
    # r2 alone with first page 8 (work 3*5 = 15), r3 alone with first page 9 (work 1*4 = 4)
    q_indptr = [0, 1, 2, 5, 6]
    kv_len = [10, 10, 5, 4]
    page_indptr = [0, 5, 10, 13, 15]
    page_indices = [7, 1, 2, 3, 4, 7, 1, 5, 6, 8, 10, 11, 12, 9, 13]
    part, load = op.partition(q_indptr, kv_len, page_indptr, page_indices, 2, 2)
    assert part == [0, 0, 1, 1] and load == [20, 19]
