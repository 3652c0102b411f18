"""The serving-step runtime (pps_engine_*, C++) against the reference cache and
scheduler in oracle/ composed by hand, CPU only.

A seeded trace admits requests that share prompt prefixes (copy-on-write
included), runs schedule/commit steps with decode and 3-token verify entries,
and retires requests with and without insertion, in a pool small enough that
admissions fail and some generation entries find no page.  The reference side
is the plain composition the engine stands for: SchedulerOracle.step picks the
batch; a prefill entry starts at (tokens cached at admission + prompt tokens
already scheduled); a generation entry's tokens go to RadixCacheOracle.extend,
and one that finds the cache full is left out of the step.  Every batch, every
table the engine writes, the cache statistics and the whole tree must match.
"""
from __future__ import annotations

import numpy as np
import pytest

from oracle import radix_cache as rc
from oracle.scheduler import SchedulerOracle
from test_radix_cache import _oracle_tree


def _reference_commit(o, progress, batch, gen_tokens):
    """The tables of the entries kept, computed from the reference cache."""
    rows, g = [], 0
    for r, k, pre in batch:
        if pre:
            first = progress[r][0] + progress[r][1]
            progress[r][1] += k
        else:
            toks = list(gen_tokens[g:g + k])
            g += k
            try:
                first = o.extend(r, toks)
            except rc.CacheFull:
                continue
        rows.append((r, first, k, o.pages(r)))
    return rows


@pytest.mark.parametrize("seed,budget,reserved,policy",
                         [(0, 48, 8, "lru"), (1, 20, 4, "lfu"), (2, 64, 0, "lru"),
                          (3, 33, 10, "lfu"), (4, 12, 3, "lru")])
def test_engine_matches_cache_and_scheduler_composed(pps, seed, budget, reserved, policy):
    P, num_pages, vocab = 4, 40, 30
    rng = np.random.default_rng(seed)
    eng = pps.Engine(num_pages, P, budget, reserved,
                     pps.CACHE_LRU if policy == "lru" else pps.CACHE_LFU)
    o = rc.RadixCacheOracle(num_pages, P, policy)
    s = SchedulerOracle(budget, reserved)
    progress = {}                   # request -> [cached at admission, prompt tokens scheduled]
    prompts = [list(rng.integers(0, vocab, size=int(rng.integers(3, 6 * P)))) for _ in range(4)]
    produced = {}
    kept = dropped = admitted = 0
    for step in range(150):
        for _ in range(int(rng.integers(0, 3))):
            base = prompts[int(rng.integers(len(prompts)))]
            toks = base[:int(rng.integers(0, len(base) + 1))] + \
                list(rng.integers(0, vocab, size=int(rng.integers(1, 3 * P))))
            k = int(rng.choice([1, 3]))
            try:
                want = o.begin(toks)
            except rc.CacheFull:
                want = "full"
            try:
                got = eng.add(toks, k)
            except pps.CacheFull:
                got = "full"
            assert got == want, (step, got, want)
            if want != "full":
                s.add(want[0], len(toks) - want[1], k)
                progress[want[0]] = [want[1], 0]
                produced[want[0]] = 0
                admitted += 1
        want_batch = s.step()
        req, tok, pre = eng.schedule()
        got_batch = list(zip(req.tolist(), tok.tolist(), [bool(x) for x in pre.tolist()]))
        assert got_batch == want_batch, step
        n_gen = sum(k for _, k, p in want_batch if not p)
        gen = rng.integers(0, vocab, size=n_gen).astype(np.int32)
        rows = _reference_commit(o, progress, want_batch, gen)
        rq, qi, cl, kl, pi, px = eng.commit(gen)
        assert rq.tolist() == [r for r, _, _, _ in rows], step
        assert qi.tolist() == [0] + np.cumsum([k for _, _, k, _ in rows]).tolist()
        assert cl.tolist() == [f for _, f, _, _ in rows]
        assert kl.tolist() == [f + k for _, f, k, _ in rows]
        assert pi.tolist() == [0] + np.cumsum([len(p) for *_, p in rows]).tolist()
        assert px.tolist() == [x for *_, p in rows for x in p]
        kept += len(rows)
        dropped += len(want_batch) - len(rows)
        gen_rows = {r for r, k, p in want_batch if not p}
        for r, _, _, _ in rows:
            if r in gen_rows:
                produced[r] += 1
        # retire some requests that have generated a few steps
        for r in list(progress):
            if produced[r] >= 4 and rng.random() < 0.5:
                ins = bool(rng.random() < 0.8)
                s.remove(r)
                o.finish(r, insert=ins)
                eng.finish(r, ins)
                del progress[r], produced[r]
        st = eng.stats()
        assert st["free_pages"] == o.num_free(), step
        assert st["tree_nodes"] == len(o.nodes)
        assert st["evictions"] == len(o.evictions)
        pr, _, gr = eng.counts()
        assert pr == len(s.prefill) and gr == len(s.gen)
        c = pps.Cache.__new__(pps.Cache)          # a non-owning view for the tree dump
        c._h, c.page_size = eng._cache, P
        assert sorted(c.dump()) == _oracle_tree(o), step
        c._h = None
    assert admitted > 10 and kept > 100
    assert dropped > 0                         # some generation entries found no page


def test_engine_rejects_calls_out_of_order(pps):
    eng = pps.Engine(16, 4, budget=16, reserved=2)
    with pytest.raises(pps.PPSError):
        eng.commit(np.zeros(0, np.int32))         # nothing scheduled
    rid, cached, copy = eng.add([1, 2, 3, 4, 5], gen_tokens=1)
    assert (rid, cached, copy) == (0, 0, None)
    req, tok, pre = eng.schedule()
    assert req.tolist() == [0] and tok.tolist() == [5] and pre.tolist() == [1]
    with pytest.raises(pps.PPSError):
        eng.add([1, 2], gen_tokens=1)             # a batch is pending
    with pytest.raises(pps.PPSError):
        eng.finish(rid)
    with pytest.raises(pps.PPSError):
        eng.schedule()
    rq, qi, cl, kl, pi, px = eng.commit(np.zeros(0, np.int32))
    assert rq.tolist() == [0] and cl.tolist() == [0] and kl.tolist() == [5]
    assert px.tolist() == eng.pages(0).tolist()
    with pytest.raises(pps.PPSError):
        eng.finish(7)                             # unknown request
    with pytest.raises(pps.PPSError):
        eng.add([1, 2], gen_tokens=0)
    eng.finish(rid)
    assert eng.counts() == (0, 0, 0)


def test_engine_grows_its_page_buffer(pps):
    """A batch whose tables exceed the binding's page buffer: the library
    reports the bound and changes nothing until the retry succeeds."""
    P = 16
    n_req, plen = 40, 200 * P
    eng = pps.Engine(n_req * 210, P, budget=n_req * plen, reserved=0)
    for i in range(n_req):
        eng.add(list(range(i * 100000, i * 100000 + plen)), gen_tokens=2)
    eng._px = np.zeros(8, np.int32)
    req, tok, pre = eng.schedule()
    assert len(req) == n_req and pre.all()
    rq, qi, cl, kl, pi, px = eng.commit(np.zeros(0, np.int32))
    assert int(pi[-1]) == n_req * 200 and len(px) == n_req * 200
    req, tok, pre = eng.schedule()                # every request now generates
    assert (tok == 2).all() and not pre.any()
    rq, qi, cl, kl, pi, px = eng.commit(np.arange(2 * n_req, dtype=np.int32))
    assert (cl == plen).all() and (kl == plen + 2).all()
    assert int(pi[-1]) == n_req * 201
