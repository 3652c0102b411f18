"""The library's host prefix cache (pps_cache_*, C++) against the reference
radix cache in oracle/, operation by operation, CPU only.

Both are driven by the same seeded trace (requests that share prompt
prefixes, decode extensions, finishes with and without insertion, a pool small
enough to force evictions and full-cache failures).  After every call the
results (request id, reused length, copy-on-write triple, failure), every
active request's page list, the free-page count and the whole tree (page,
parent page, chunk, last use, hits of every node) must be identical.
"""
from __future__ import annotations

import time

import numpy as np
import pytest

from oracle import radix_cache as rc


def _oracle_tree(o):
    out = []
    for n in o.nodes.values():
        parent = o.nodes[n["parent"]]["page"] if n["parent"] >= 0 else -1
        out.append((n["page"], parent, tuple(n["chunk"]), n["last"], n["hits"]))
    return sorted(out)


def _run_both(pps, seed, n_ops, num_pages, P, policy, vocab=50, n_prompts=5):
    rng = np.random.default_rng(seed)
    o = rc.RadixCacheOracle(num_pages, P, policy)
    c = pps.Cache(num_pages, P, pps.CACHE_LRU if policy == "lru" else pps.CACHE_LFU)
    prompts = [list(rng.integers(0, vocab, size=rng.integers(1, 4 * P))) for _ in range(n_prompts)]
    active = []
    fails = 0
    for step in range(n_ops):
        op = rng.random()
        if op < 0.45 or not active:
            base = prompts[rng.integers(len(prompts))]
            cut = int(rng.integers(0, len(base) + 1))
            toks = base[:cut] + list(rng.integers(0, vocab, size=rng.integers(1, 2 * P)))
            try:
                want = o.begin(toks)
            except rc.CacheFull:
                want = "full"
            try:
                got = c.begin(toks)
            except pps.CacheFull:
                got = "full"
            assert got == want, (step, got, want)
            if want != "full":
                active.append(want[0])
            else:
                fails += 1
        elif op < 0.75:
            rid = active[rng.integers(len(active))]
            toks = list(rng.integers(0, vocab, size=rng.integers(1, P + 2)))
            try:
                want = o.extend(rid, toks)
            except rc.CacheFull:
                want = "full"
            try:
                got = c.extend(rid, toks)
            except pps.CacheFull:
                got = "full"
            assert got == want, (step, got, want)
        else:
            rid = active.pop(rng.integers(len(active)))
            ins = bool(rng.random() < 0.9)
            o.finish(rid, insert=ins)
            c.finish(rid, insert=ins)
        for rid in active:
            assert list(c.pages(rid)) == o.pages(rid), step
        st = c.stats()
        assert st["free_pages"] == o.num_free()
        assert st["tree_nodes"] == len(o.nodes)
        assert st["evictions"] == len(o.evictions)
        assert sorted(c.dump()) == _oracle_tree(o), step
    return o, fails


@pytest.mark.parametrize("policy", ["lru", "lfu"])
@pytest.mark.parametrize("seed", range(8))
def test_cache_matches_reference_call_by_call(pps, seed, policy):
    o, fails = _run_both(pps, seed, 400, num_pages=24, P=4, policy=policy)
    assert o.evictions


def test_cache_page_size_16_and_full_failures(pps):
    o, fails = _run_both(pps, 99, 300, num_pages=12, P=16, policy="lru", vocab=5, n_prompts=3)
    assert fails > 0 and o.evictions


def test_cache_rejects_bad_arguments(pps):
    with pytest.raises(pps.PPSError):
        pps.Cache(0, 16)
    with pytest.raises(pps.PPSError):
        pps.Cache(8, 16, policy=7)
    c = pps.Cache(8, 16)
    with pytest.raises(pps.PPSError):
        c.begin([])
    with pytest.raises(pps.PPSError):
        c.finish(12345)


def test_cache_is_fast_on_a_serving_trace(pps):
    """10k requests over 200 shared system prompts (2k-token prompts, P=16):
    begin + finish for all of them in well under a second."""
    rng = np.random.default_rng(3)
    prompts = [rng.integers(0, 32000, size=int(rng.integers(256, 2048))).astype(np.int32)
               for _ in range(200)]
    c = pps.Cache(200_000, 16)
    reqs = []
    for i in range(10_000):
        base = prompts[int(rng.integers(len(prompts)))]
        reqs.append(np.concatenate([base, rng.integers(0, 32000, size=int(rng.integers(16, 256)))
                                    ]).astype(np.int32))
    t0 = time.perf_counter()
    for toks in reqs:
        rid, cached, copy = c.begin(toks)
        c.finish(rid)
    dt = time.perf_counter() - t0
    st = c.stats()
    assert st["reused_tokens"] > 0.7 * st["begun_tokens"]
    assert dt < 5.0, dt


def test_batch_calls_equal_single_calls(pps):
    rng = np.random.default_rng(7)
    a, b = pps.Cache(64, 4), pps.Cache(64, 4)
    prompts = [list(rng.integers(0, 9, size=12)) for _ in range(3)]
    rids = []
    for k in range(6):
        toks = prompts[k % 3] + list(rng.integers(0, 9, size=3))
        ra, rb = a.begin(toks), b.begin(toks)
        assert ra == rb
        rids.append(ra[0])
    for step in range(5):
        lens = rng.integers(0, 3, size=len(rids))
        indptr = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        toks = rng.integers(0, 9, size=int(indptr[-1])).astype(np.int32)
        first_b = b.extend_batch(rids, indptr, toks)
        first_a = [a.extend(r, toks[indptr[i]:indptr[i + 1]]) for i, r in enumerate(rids)]
        assert list(first_b) == first_a
        assert sorted(a.dump()) == sorted(b.dump()) and a.stats() == b.stats()
    order = rids[::-1]
    kv, ip, px = b.tables(order)
    for i, r in enumerate(order):
        assert list(px[ip[i]:ip[i + 1]]) == list(b.pages(r))
        assert len(b.pages(r)) == -(-int(kv[i]) // 4)      # pages cover exactly kv_len tokens


def test_extend_batch_stops_at_the_first_failure(pps):
    c = pps.Cache(3, 4)
    r0, _, _ = c.begin([1, 2, 3, 4])                 # one page
    r1, _, _ = c.begin([5, 6, 7, 8])                 # one page
    with pytest.raises(pps.CacheFull):               # r0 takes the last page, r1 finds none
        c.extend_batch([r0, r1], np.array([0, 1, 2], np.int32), np.array([9, 9], np.int32))
    kv, ip, px = c.tables([r0, r1])
    assert list(kv) == [5, 4] and c.stats()["free_pages"] == 0
