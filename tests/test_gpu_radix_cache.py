"""GPU: the prefix cache's page lists drive the attention path end to end.

A serving trace runs through pps_cache_* on the host.  Every step applies the
cache's copy-on-write copies with pps_copy_slots, appends the step's new K/V
rows with pps_kv_append at the positions the cache says are not yet cached,
and attends with pps_attn_plan / pps_attn_run over the cache's page lists.
The K/V row of position p of a request depends only on (token at p, p), so a
prefix shared by two requests has the same K/V in both, as in a real model.
Expected outputs come from the fp64 oracle run on each request's K/V rows laid
out contiguously (its own identity page table): no cache, no shared pages.  A
wrong page, a missing copy or a page reused while still needed shows up as a
mismatch; unwritten pool slots hold NaN.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
from gpu_run import errors

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS = 2e-2, 2e-3
Hq, Hkv, D, P = 8, 2, 64, 16
VOCAB = 40


@pytest.fixture(scope="module", autouse=True)
def _lib(pps):
    assert torch.cuda.is_available()
    return pps


def _tables(seed=0, max_pos=512):
    g = torch.Generator().manual_seed(seed)
    tok_k = torch.randn((VOCAB, Hkv, D), generator=g)
    pos_k = torch.randn((max_pos, Hkv, D), generator=g)
    tok_v = torch.randn((VOCAB, Hkv, D), generator=g)
    pos_v = torch.randn((max_pos, Hkv, D), generator=g)
    return tok_k, pos_k, tok_v, pos_v


def _kv(tabs, tokens, positions):
    tok_k, pos_k, tok_v, pos_v = tabs
    t = torch.as_tensor(tokens, dtype=torch.long)
    p = torch.as_tensor(positions, dtype=torch.long)
    return ((tok_k[t] + pos_k[p]).to(torch.bfloat16), (tok_v[t] + pos_v[p]).to(torch.bfloat16))


def _reference(q_rows, tokens, n_cached, tabs):
    """fp64 oracle on the request's contiguous K/V (identity page table)."""
    n = len(tokens)
    k, v = _kv(tabs, tokens, range(n))
    npg = -(-n // P)
    pk = torch.full((npg, Hkv, P, D), float("nan"), dtype=torch.bfloat16)
    pv = pk.clone()
    for p in range(n):
        pk[p // P, :, p % P] = k[p]
        pv[p // P, :, p % P] = v[p]
    m = q_rows.shape[0]
    return oracle.paged_attention(q_rows, pk, pv, np.array([0, m]), np.array([n]),
                                  np.array([0, npg]), np.arange(npg), P, 1 / math.sqrt(D), Hkv)


@pytest.mark.parametrize("policy", [0, 1])
def test_cache_driven_steps_match_the_oracle(pps, policy):
    rng = np.random.default_rng(11 + policy)
    tabs = _tables(policy)
    num_pages = 40
    cache = pps.Cache(num_pages, P, policy)
    pool_k = torch.full((num_pages, Hkv, P, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    pool_v = torch.full_like(pool_k, float("nan"))
    prompts = [list(rng.integers(0, VOCAB, size=int(rng.integers(20, 90)))) for _ in range(4)]
    active = {}                       # rid -> tokens
    pps.get_device_error(clear=True)
    checked = 0
    for step in range(12):
        # new requests (prefill), decode of some active ones, finishes
        new, grow = [], []
        for _ in range(int(rng.integers(1, 4))):
            base = prompts[int(rng.integers(len(prompts)))]
            toks = base[:int(rng.integers(1, len(base) + 1))] + \
                list(rng.integers(0, VOCAB, size=int(rng.integers(1, 30))))
            try:
                rid, cached, copy = cache.begin(toks)
            except pps.CacheFull:
                continue
            if copy is not None:
                # enqueued at once, in call order: a later call may hand the
                # source page out again
                c3 = torch.tensor([copy], dtype=torch.int32, device="cuda")
                pps.copy_slots(pool_k, pool_v, c3[:, 0].contiguous(), c3[:, 1].contiguous(),
                               c3[:, 2].contiguous())
            active[rid] = list(toks)
            new.append((rid, cached, copy))
        for rid in list(active):
            if rid in [x[0] for x in new] or rng.random() < 0.4:
                continue
            t = int(rng.integers(0, VOCAB))
            try:
                first = cache.extend(rid, [t])
            except pps.CacheFull:
                continue
            active[rid].append(t)
            grow.append((rid, first))
        batch = [(rid, cached) for rid, cached, _ in new] + grow
        if not batch:
            continue
        # CSR tables of the step
        q_len = [len(active[rid]) - c for rid, c in batch]
        q_indptr = np.concatenate([[0], np.cumsum(q_len)]).astype(np.int32)
        kv_len = np.array([len(active[rid]) for rid, _ in batch], np.int32)
        cached = np.array([c for _, c in batch], np.int32)
        plists = [cache.pages(rid) for rid, _ in batch]
        page_indptr = np.concatenate([[0], np.cumsum([len(p) for p in plists])]).astype(np.int32)
        page_indices = np.concatenate(plists).astype(np.int32)
        ks, vs = [], []
        for (rid, c), ql in zip(batch, q_len):
            k, v = _kv(tabs, active[rid][c:], range(c, c + ql))
            ks.append(k)
            vs.append(v)
        T = int(q_indptr[-1])
        dev = lambda a: torch.as_tensor(a, dtype=torch.int32, device="cuda")
        pps.kv_append(pool_k, pool_v, torch.cat(ks).cuda(), torch.cat(vs).cuda(), dev(q_indptr),
                      dev(cached), dev(page_indptr), dev(page_indices))
        q = torch.randn((T, Hq, D), generator=torch.Generator().manual_seed(step)).to(torch.bfloat16)
        plan = pps.attn_plan(q_indptr, kv_len, page_indptr, page_indices, Hq, Hkv, D, P, num_pages)
        ws = torch.empty(max(plan.workspace_bytes, 256), dtype=torch.uint8, device="cuda")
        out = torch.full((T, Hq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
        pps.attn_run(plan, q.cuda(), pool_k, pool_v, out, ws)
        torch.cuda.synchronize()
        assert pps.get_device_error(clear=True) == 0
        for r, (rid, c) in enumerate(batch):
            a, b = int(q_indptr[r]), int(q_indptr[r + 1])
            ref = _reference(q[a:b], active[rid], c, tabs)
            mx, mean = errors(out[a:b], ref)
            assert mx <= MAX_ABS and mean <= MEAN_ABS, (step, rid, mx, mean)
            checked += 1
        # finish some
        for rid in list(active):
            if rng.random() < 0.35:
                cache.finish(rid, insert=rng.random() < 0.9)
                del active[rid]
    st = cache.stats()
    assert checked > 10 and st["reused_tokens"] > 0 and st["evictions"] > 0, st


def test_copy_slots_is_bit_exact_and_checks_ids(pps):
    g = torch.Generator().manual_seed(5)
    pk = torch.randn((6, Hkv, P, D), generator=g).to(torch.bfloat16).cuda()
    pv = torch.randn((6, Hkv, P, D), generator=g).to(torch.bfloat16).cuda()
    want_k, want_v = pk.clone(), pv.clone()
    src, dst, n = [0, 3, 5], [1, 4, 2], [5, 16, 1]
    for s_, d_, n_ in zip(src, dst, n):
        want_k[d_, :, :n_] = want_k[s_, :, :n_]
        want_v[d_, :, :n_] = want_v[s_, :, :n_]
    dev = lambda a: torch.tensor(a, dtype=torch.int32, device="cuda")
    pps.get_device_error(clear=True)
    pps.copy_slots(pk, pv, dev(src), dev(dst), dev(n))
    torch.cuda.synchronize()
    assert torch.equal(pk.view(torch.int16), want_k.view(torch.int16))
    assert torch.equal(pv.view(torch.int16), want_v.view(torch.int16))
    assert pps.get_device_error(clear=True) == 0
    before = pk.clone()
    pps.copy_slots(pk, pv, dev([0]), dev([99]), dev([3]))      # destination out of range
    torch.cuda.synchronize()
    assert pps.get_device_error(clear=True) == 5                # PPS_DEV_ERR_COPY_ARGUMENT
    assert torch.equal(pk.view(torch.int16), before.view(torch.int16))


@pytest.mark.parametrize("budget,reserved", [(96, 16), (40, 8)])
def test_scheduler_and_cache_drive_chunked_steps(pps, budget, reserved):
    """The engine loop: the token-wise scheduler picks each step's tokens
    (whole generation steps, including 3-token verify drafts, then chunks of
    pending prompts within the budget), the prefix cache holds the pages
    (copy-on-write at admission), and every scheduled token's output is
    checked against the oracle on the request's contiguous K/V."""
    rng = np.random.default_rng(21)
    tabs = _tables(3, max_pos=1024)
    num_pages = 96
    cache = pps.Cache(num_pages, P)
    sched = pps.Scheduler(budget, reserved)
    pool_k = torch.full((num_pages, Hkv, P, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    pool_v = torch.full_like(pool_k, float("nan"))
    prompts = [list(rng.integers(0, VOCAB, size=int(rng.integers(30, 120)))) for _ in range(3)]
    state = {}                      # rid -> dict(tokens, cached0, done, gen_k, produced, goal)
    pps.get_device_error(clear=True)
    checked = 0
    for step in range(40):
        for _ in range(int(rng.integers(0, 3))):
            if len(state) >= 6:
                break
            base = prompts[int(rng.integers(len(prompts)))]
            toks = base[:int(rng.integers(1, len(base) + 1))] + \
                list(rng.integers(0, VOCAB, size=int(rng.integers(1, 70))))
            try:
                rid, cached, copy = cache.begin(toks)
            except pps.CacheFull:
                continue
            if copy is not None:
                c3 = torch.tensor([copy], dtype=torch.int32, device="cuda")
                pps.copy_slots(pool_k, pool_v, c3[:, 0].contiguous(), c3[:, 1].contiguous(),
                               c3[:, 2].contiguous())
            k = int(rng.choice([1, 3]))
            sched.add(rid, len(toks) - cached, k)
            state[rid] = dict(tokens=list(toks), cached0=cached, done=0, gen_k=k, produced=0,
                              goal=int(rng.integers(2, 12)))
        req, tok, pre = sched.step()
        if len(req) == 0:
            continue
        batch = []                  # (rid, first position, tokens this step)
        for r, k, p in zip(req.tolist(), tok.tolist(), pre.tolist()):
            s = state[r]
            if p:
                first = s["cached0"] + s["done"]
                s["done"] += k
            else:
                new = list(rng.integers(0, VOCAB, size=k))
                try:
                    first = cache.extend(r, new)
                except pps.CacheFull:
                    continue
                s["tokens"] += new
                s["produced"] += k
            batch.append((r, first, k))
        if not batch:
            continue
        q_len = [k for _, _, k in batch]
        q_indptr = np.concatenate([[0], np.cumsum(q_len)]).astype(np.int32)
        cached = np.array([f for _, f, _ in batch], np.int32)
        kv_len = cached + np.array(q_len, np.int32)
        plists = [cache.pages(r) for r, _, _ in batch]
        page_indptr = np.concatenate([[0], np.cumsum([len(p) for p in plists])]).astype(np.int32)
        page_indices = np.concatenate(plists).astype(np.int32)
        ks, vs = [], []
        for (r, f, k) in batch:
            kk, vv = _kv(tabs, state[r]["tokens"][f:f + k], range(f, f + k))
            ks.append(kk)
            vs.append(vv)
        T = int(q_indptr[-1])
        dev = lambda a: torch.as_tensor(a, dtype=torch.int32, device="cuda")
        pps.kv_append(pool_k, pool_v, torch.cat(ks).cuda(), torch.cat(vs).cuda(), dev(q_indptr),
                      dev(cached), dev(page_indptr), dev(page_indices))
        q = torch.randn((T, Hq, D), generator=torch.Generator().manual_seed(100 + step)) \
            .to(torch.bfloat16)
        plan = pps.attn_plan(q_indptr, kv_len, page_indptr, page_indices, Hq, Hkv, D, P, num_pages)
        ws = torch.empty(max(plan.workspace_bytes, 256), dtype=torch.uint8, device="cuda")
        out = torch.full((T, Hq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
        pps.attn_run(plan, q.cuda(), pool_k, pool_v, out, ws)
        torch.cuda.synchronize()
        assert pps.get_device_error(clear=True) == 0
        for i, (r, f, k) in enumerate(batch):
            a, b = int(q_indptr[i]), int(q_indptr[i + 1])
            ref = _reference(q[a:b], state[r]["tokens"][:f + k], f, tabs)
            mx, mean = errors(out[a:b], ref)
            assert mx <= MAX_ABS and mean <= MEAN_ABS, (step, r, mx, mean)
            checked += 1
        for r in list(state):
            s = state[r]
            if s["done"] == len(s["tokens"]) - s["cached0"] - s["produced"] and \
                    s["produced"] >= s["goal"]:
                sched.remove(r)
                cache.finish(r)
                del state[r]
    assert checked > 20


def test_engine_drives_chunked_steps(pps):
    """The same loop through the native serving-step runtime: pps_engine_add
    admits, pps_engine_schedule picks the batch, pps_engine_commit appends the
    generated tokens and hands back the tables that kv_append and attn_plan
    take; every scheduled token's output is checked against the oracle."""
    rng = np.random.default_rng(22)
    tabs = _tables(4, max_pos=1024)
    num_pages = 80
    eng = pps.Engine(num_pages, P, budget=72, reserved=12)
    pool_k = torch.full((num_pages, Hkv, P, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    pool_v = torch.full_like(pool_k, float("nan"))
    prompts = [list(rng.integers(0, VOCAB, size=int(rng.integers(30, 120)))) for _ in range(3)]
    tokens, goal, produced = {}, {}, {}
    pps.get_device_error(clear=True)
    dev = lambda a: torch.as_tensor(np.asarray(a), dtype=torch.int32, device="cuda")
    checked = 0
    for step in range(40):
        for _ in range(int(rng.integers(0, 3))):
            if len(tokens) >= 6:
                break
            base = prompts[int(rng.integers(len(prompts)))]
            toks = base[:int(rng.integers(1, len(base) + 1))] + \
                list(rng.integers(0, VOCAB, size=int(rng.integers(1, 70))))
            try:
                rid, cached, copy = eng.add(toks, int(rng.choice([1, 3])))
            except pps.CacheFull:
                continue
            if copy is not None:
                pps.copy_slots(pool_k, pool_v, dev([copy[0]]), dev([copy[1]]), dev([copy[2]]))
            tokens[rid], goal[rid], produced[rid] = list(toks), int(rng.integers(2, 12)), 0
        req, tok, pre = eng.schedule()
        gen = {int(r): int(k) for r, k, p in zip(req, tok, pre) if not p}
        new = {r: list(rng.integers(0, VOCAB, size=k)) for r, k in gen.items()}
        flat = np.array([t for r in req.tolist() if r in new for t in new[r]], np.int32)
        rq, qi, cl, kl, pi, px = [a.copy() for a in eng.commit(flat)]
        for r in rq.tolist():
            if r in new:
                tokens[r] += new[r]
                produced[r] += 1
        if len(rq) == 0:
            continue
        ks, vs = [], []
        for r, f, e in zip(rq.tolist(), cl.tolist(), kl.tolist()):
            kk, vv = _kv(tabs, tokens[r][f:e], range(f, e))
            ks.append(kk)
            vs.append(vv)
        T = int(qi[-1])
        pps.kv_append(pool_k, pool_v, torch.cat(ks).cuda(), torch.cat(vs).cuda(), dev(qi),
                      dev(cl), dev(pi), dev(px))
        q = torch.randn((T, Hq, D), generator=torch.Generator().manual_seed(200 + step)) \
            .to(torch.bfloat16)
        plan = pps.attn_plan(qi, kl, pi, px, Hq, Hkv, D, P, num_pages)
        ws = torch.empty(max(plan.workspace_bytes, 256), dtype=torch.uint8, device="cuda")
        out = torch.full((T, Hq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
        pps.attn_run(plan, q.cuda(), pool_k, pool_v, out, ws)
        torch.cuda.synchronize()
        assert pps.get_device_error(clear=True) == 0
        for i, (r, f, e) in enumerate(zip(rq.tolist(), cl.tolist(), kl.tolist())):
            a, b = int(qi[i]), int(qi[i + 1])
            ref = _reference(q[a:b], tokens[r][:e], f, tabs)
            mx, mean = errors(out[a:b], ref)
            assert mx <= MAX_ABS and mean <= MEAN_ABS, (step, r, mx, mean)
            checked += 1
        for r in list(tokens):
            if produced[r] >= goal[r]:
                eng.finish(r)
                del tokens[r], goal[r], produced[r]
    assert checked > 20
