"""Pins for the reference radix cache (oracle/radix_cache.py), each against
something other than the oracle itself:

* K/V semantics under copy-on-write and eviction (the property the XY-Serve
  review's assumption list asks of block table + radix tree): a simulated pool
  that stores token ids is written exactly as a serving loop would (copy-on-
  write slots, then the step's new tokens); after every call, every active
  request reads its own tokens back through its page list and every tree node
  still holds its chunk;
* page accounting: every page is free, or held by tree nodes and active
  requests exactly as often as they list it; no two siblings hold equal chunks;
* best reuse: the reused length equals the longest prefix any cached sequence
  shares with the request (brute force over all root-to-node sequences), capped
  at n - 1;
* eviction order: a hand-worked trace where LRU and LFU must evict different
  pages;
* planted mistakes: each textual mutation of the oracle fails one of these.
"""
from __future__ import annotations

import os
import types

import numpy as np
import pytest

from oracle import radix_cache as rc


class Sim:
    """Drives a cache like a serving loop and keeps a token-id 'pool'."""

    def __init__(self, cache):
        self.c = cache
        self.pool = {}

    def _write(self, pages, start, tokens):
        P = self.c.P
        for k, t in enumerate(tokens):
            p = start + k
            self.pool.setdefault(pages[p // P], [None] * P)[p % P] = t

    def begin(self, tokens):
        rid, cached, copy = self.c.begin(tokens)
        if copy is not None:
            src, dst, n = copy
            s = self.pool.setdefault(src, [None] * self.c.P)
            d = self.pool.setdefault(dst, [None] * self.c.P)
            d[:n] = s[:n]
        self._write(self.c.pages(rid), cached, list(tokens)[cached:])
        return rid, cached, copy

    def extend(self, rid, tokens):
        n0 = self.c.extend(rid, tokens)
        self._write(self.c.pages(rid), n0, tokens)

    def check(self):
        c, P = self.c, self.c.P
        for rid, req in c.requests.items():
            got = [self.pool[req["pages"][p // P]][p % P] for p in range(len(req["tokens"]))]
            assert got == req["tokens"], f"request {rid} reads other tokens"
        for n in c.nodes.values():
            assert self.pool[n["page"]][:len(n["chunk"])] == list(n["chunk"])
        held = [0] * c.num_pages
        for n in c.nodes.values():
            held[n["page"]] += 1
        for req in c.requests.values():
            for p in req["pages"]:
                held[p] += 1
        assert held == c.holders
        kids = {}
        for i, n in c.nodes.items():
            assert len(n["chunk"]) <= P
            key = (n["parent"], n["chunk"])
            assert key not in kids, "two siblings hold the same chunk"
            kids[key] = i
            if len(n["chunk"]) < P:
                assert not any(m["parent"] == i for m in c.nodes.values()), "partial page with children"


def _trace(seed, n_ops, num_pages, P, policy):
    rng = np.random.default_rng(seed)
    sim = Sim(rc.RadixCacheOracle(num_pages, P, policy))
    prompts = [list(rng.integers(0, 50, size=rng.integers(1, 4 * P))) for _ in range(5)]
    active = []
    for _ in range(n_ops):
        op = rng.random()
        if op < 0.45 or not active:
            base = prompts[rng.integers(len(prompts))]
            cut = int(rng.integers(0, len(base) + 1))
            toks = base[:cut] + list(rng.integers(0, 50, size=rng.integers(1, 2 * P)))
            before = [(s, p) for s, p in sim.c.node_sequences()]
            try:
                rid, cached, copy = sim.begin(toks)
            except rc.CacheFull:
                sim.check()
                continue
            best = max([min(len(toks) - 1, rc._lcp(s, toks)) for s, _ in before] + [0])
            assert cached == best
            active.append(rid)
        elif op < 0.75:
            rid = active[rng.integers(len(active))]
            try:
                sim.extend(rid, list(rng.integers(0, 50, size=rng.integers(1, P + 2))))
            except rc.CacheFull:
                pass
        else:
            rid = active.pop(rng.integers(len(active)))
            sim.c.finish(rid, insert=bool(rng.random() < 0.9))
        sim.check()
    return sim


@pytest.mark.parametrize("policy", ["lru", "lfu"])
@pytest.mark.parametrize("seed", range(6))
def test_kv_semantics_and_accounting_under_cow_and_eviction(seed, policy):
    sim = _trace(seed, 300, num_pages=24, P=4, policy=policy)
    assert sim.c.evictions, "the trace should force evictions"


def test_reuse_is_token_wise_with_copy_on_write():
    c = rc.RadixCacheOracle(8, 4)
    sim = Sim(c)
    a, cached, copy = sim.begin([1, 2, 3, 4, 5, 6])
    assert cached == 0 and copy is None and c.pages(a) == [0, 1]
    c.finish(a)
    b, cached, copy = sim.begin([1, 2, 3, 4, 5, 9, 9])
    # page 0 (1,2,3,4) is shared; token 5 of page 1 is copied into a new page
    assert cached == 5 and copy == (1, 2, 1) and c.pages(b) == [0, 2]
    sim.check()
    d, cached, copy = sim.begin([1, 2, 3, 4])
    assert cached == 3 and copy == (0, 3, 3)          # at most n - 1 reused
    sim.check()


def _eviction_trace(policy):
    """Three one-page documents A, B, C fill a 4-page pool with a live
    request holding one page; A is reused twice (hits 2), B once, and B is the
    most recently used.  A new request then needs a page."""
    c = rc.RadixCacheOracle(4, 4, policy)
    sim = Sim(c)
    for doc in ([1, 1, 1], [2, 2, 2], [3, 3, 3]):
        r, _, _ = sim.begin(doc)
        c.finish(r)
    for doc in ([1, 1, 1, 7], [1, 1, 1, 8], [2, 2, 2, 9]):
        r, cached, copy = sim.begin(doc)    # 3 tokens copied from the doc's page
        assert cached == 3
        c.finish(r, insert=False)
    live, _, _ = sim.begin([5, 5])          # holds page 3
    assert c.pages(live) == [3]
    r, _, _ = sim.begin([6, 6])
    sim.check()
    return c.evictions


def test_lru_and_lfu_evict_what_their_rule_says():
    # C was used only when inserted, A and B later: LRU evicts C (page 2);
    # hits A 2, B 1, C 0: LFU evicts C too.
    assert _eviction_trace("lru") == [2]
    assert _eviction_trace("lfu") == [2]
    # make C recently used but rarely: reuse C once more, then A and B are
    # older; LRU now evicts A (page 0, last use earliest), LFU evicts C (hits 1 < 2).
    for policy, want in (("lru", 0), ("lfu", 2)):
        c = rc.RadixCacheOracle(4, 4, policy)
        sim = Sim(c)
        for doc in ([1, 1, 1], [2, 2, 2], [3, 3, 3]):
            r, _, _ = sim.begin(doc)
            c.finish(r)
        for doc in ([1, 1, 1, 7], [1, 1, 1, 8], [2, 2, 2, 9], [2, 2, 2, 9], [3, 3, 3, 4]):
            r, _, _ = sim.begin(doc)
            c.finish(r, insert=False)
        live, _, _ = sim.begin([5, 5])
        sim.begin([6, 6])
        assert c.evictions == [want], (policy, c.evictions)


def test_full_cache_fails_cleanly():
    c = rc.RadixCacheOracle(2, 4)
    sim = Sim(c)
    a, _, _ = sim.begin(list(range(8)))          # both pages, held by a live request
    with pytest.raises(rc.CacheFull):
        sim.begin([9, 9])
    assert c.holders == [1, 1] and len(c.requests) == 1
    c.finish(a, insert=False)
    assert c.num_free() == 2


MUTATIONS = {
    "lru_uses_hits": ('return (n["last"], n["page"])', 'return (n["hits"], n["last"], n["page"])'),
    "cow_one_slot_short": ('copy = (src, pages[0], partial[1])', 'copy = (src, pages[0], partial[1] - 1)'),
    "no_dedupe": ('same = [c for c in self._children(node) if self.nodes[c]["chunk"] == chunk]',
                  'same = []'),
    "reuse_all_tokens": ("limit = n - 1", "limit = n"),
    "path_not_released": ('        for c in req["path"]:\n            self.holders[self.nodes[c]["page"]] -= 1\n',
                          "        pass\n"),
    "evict_held_leaf": ("if self.holders[n[\"page\"]] == 1:", "if self.holders[n[\"page\"]] >= 1:"),
}


def _mutant(name):
    src_path = os.path.join(os.path.dirname(rc.__file__), "radix_cache.py")
    src = open(src_path).read()
    old, new = MUTATIONS[name]
    assert src.count(old) == 1, name
    mod = types.ModuleType("radix_mutant_" + name)
    exec(compile(src.replace(old, new), src_path, "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name", list(MUTATIONS))
def test_planted_mistake_is_caught(name, monkeypatch):
    mod = _mutant(name)
    monkeypatch.setattr(rc, "RadixCacheOracle", mod.RadixCacheOracle)
    monkeypatch.setattr(rc, "CacheFull", mod.CacheFull)
    caught = False
    try:
        test_lru_and_lfu_evict_what_their_rule_says()
        test_reuse_is_token_wise_with_copy_on_write()
        for seed in range(4):
            for policy in ("lru", "lfu"):
                _trace(seed, 300, 24, 4, policy)
    except (AssertionError, KeyError, IndexError, TypeError, ValueError):
        caught = True
    assert caught, f"mutation {name} slipped past the pins"
