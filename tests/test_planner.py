"""Host planner (pps_attn_plan) checks, CPU only.

Coverage is the planner's correctness contract: across all tasks, every
(new token, kv head, KV position the token may see) is read exactly once and
nothing else is read; the page ids a task reads for a token are that token's
own request's page ids (group tasks read one member's list for all members);
tokens read by more than one task get partial slots and a merge list, tokens
read once are written directly.
"""
import time

import numpy as np
import pytest

import workloads


def _plan(pps, L, **kw):
    return pps.attn_plan(L.q_indptr, L.kv_len, L.page_indptr, L.page_indices, L.num_q_heads,
                         L.num_kv_heads, L.head_dim, L.page_size, L.num_pages, **kw)


def check_plan(pps, L, plan):
    rows = plan.array("rows")
    pages = plan.array("pages")
    tasks = np.concatenate([plan.array("bw_tasks"), plan.array("mma_tasks")])
    R, T, Hkv, P = L.num_requests, L.num_tokens, L.num_kv_heads, L.page_size
    req_of = np.searchsorted(L.q_indptr, np.arange(T), side="right") - 1
    cover = {t: np.zeros((Hkv, int(L.kv_len[req_of[t]])), np.int32) for t in range(T)}
    per_token_tasks = {t: [] for t in range(T)}
    for (row_off, n_tok, h, page_off, b, e, causal, pid) in tasks:
        assert 0 <= h < Hkv and b < e
        for i in range(n_tok):
            t = int(rows[row_off + i])
            r = int(req_of[t])
            lim = min(e, causal + i + 1)
            assert lim > b, "a task row that sees nothing"
            cover[t][h, b:lim] += 1
            own = L.page_indices[L.page_indptr[r]:L.page_indptr[r + 1]]
            pos = np.arange(b, lim)
            assert np.array_equal(pages[page_off + pos // P], own[pos // P])
            per_token_tasks[t].append((h, pid, i))
    for t in range(T):
        r = int(req_of[t])
        j = t - int(L.q_indptr[r])
        vis = int(L.cached_len[r]) + j + 1
        assert (cover[t][:, :vis] == 1).all(), f"token {t} not covered exactly once"
        assert (cover[t][:, vis:] == 0).all(), f"token {t} reads beyond its causal limit"
    # partials / merge bookkeeping
    m_tok = plan.array("merge_tokens")
    m_ptr = plan.array("merge_indptr")
    m_pid = plan.array("merge_pids")
    merged = {int(t): set(m_pid[m_ptr[k]:m_ptr[k + 1]].tolist()) for k, t in enumerate(m_tok)}
    info = plan.info()
    for t in range(T):
        lst = per_token_tasks[t]
        per_head = len(lst) // Hkv
        assert len(lst) == per_head * Hkv
        if per_head == 1:
            assert all(pid == -1 for _, pid, _ in lst) and t not in merged
        else:
            assert all(pid >= 0 for _, pid, _ in lst)
            pids = {pid + i for _, pid, i in lst}
            assert merged[t] == pids and len(pids) == per_head
            assert all(0 <= p < info["num_partials"] for p in pids)
    # work-sorted (descending) inside each kernel class; key-tile tables in
    # per-CTA ranges, each descending in 128-key tiles (+ 2 per task)
    G = L.num_q_heads // Hkv
    off = plan.array("tt_cta")
    for name, rows_eff in (("bw_tasks", None), ("mma_tasks", 128)):
        tk = plan.array(name)
        if not len(tk):
            continue
        if name == "bw_tasks" and len(off):
            w = -(-(tk[:, 5] - tk[:, 4]) // 128) + 2
            for b in range(len(off) - 1):
                assert (np.diff(w[off[b]:off[b + 1]]) <= 0).all()
        else:
            w = (tk[:, 1] * G if rows_eff is None else rows_eff) * (tk[:, 5] - tk[:, 4])
            assert (np.diff(w) <= 0).all()
    return info


SMALL = dict(num_q_heads=8, num_kv_heads=2, head_dim=64, page_size=16, values=False)


@pytest.mark.parametrize("flags", [0, 1, 2])
@pytest.mark.parametrize("name,kw", [
    ("tiny_mixed", dict(values=False)),
    ("decode_heavy", dict(num_requests=5, kv_lo=1, kv_hi=700, **SMALL)),
    ("radix_sharing", dict(groups=3, root=64, branch=32, pairs=2, tail_lo=1, tail_hi=80, **SMALL)),
    ("mixed_budget", dict(budget=200, prefill_q=100, prefill_cached=40, num_verify=5,
                          mu=4.0, sigma=1.0, clip_lo=1, clip_hi=600, **SMALL)),
    ("long_prefill", dict(num_requests=2, chunk=300, num_chunks=3, **SMALL)),
])
def test_plan_covers_every_visible_key_once(pps, name, kw, flags):
    wl = workloads.make(name, **kw)
    for st in wl.steps:
        plan = _plan(pps, st.layout, flags=flags, num_sms=4)
        check_plan(pps, st.layout, plan)


TT = dict(num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16, values=False)


@pytest.mark.parametrize("num_sms", [1, 3, 152])
@pytest.mark.parametrize("name,kw", [
    ("decode_heavy", dict(num_requests=9, kv_lo=1, kv_hi=900, **TT)),
    ("radix_sharing", dict(groups=2, root=128, branch=32, pairs=2, tail_lo=1, tail_hi=200, **TT)),
    ("mixed_budget", dict(budget=300, prefill_q=150, prefill_cached=40, num_verify=5,
                          mu=4.0, sigma=1.0, clip_lo=1, clip_hi=900, **TT)),
    ("tree_verify", dict(num_requests=4, tree_size=8, kv_lo=1, kv_hi=700, **TT)),
])
def test_key_tile_plans_cover_every_visible_key_once(pps, name, kw, num_sms):
    """The same coverage checks on plans whose small-row tasks run on the
    key-tile kernel (head_dim 128): per-CTA ranges instead of one order."""
    wl = workloads.make(name, **kw)
    for st in wl.steps:
        plan = _plan(pps, st.layout, num_sms=num_sms, tree_parent=st.layout.tree_parent)
        assert plan.info()["small_rows_on_tensor"] == 1
        check_plan(pps, st.layout, plan)
        assert len(plan.array("tt_cta")) == min(num_sms, plan.info()["num_bw_tasks"]) + 1


@pytest.mark.parametrize("chunk", [16, 48, 128])
def test_forced_small_chunks_still_cover(pps, chunk):
    wl = workloads.make("mixed_budget", budget=120, prefill_q=40, prefill_cached=33, num_verify=4,
                        mu=4.0, sigma=1.0, clip_lo=1, clip_hi=500, **SMALL)
    plan = _plan(pps, wl.layout, bw_chunk_tokens=chunk, mma_chunk_tokens=128)
    info = check_plan(pps, wl.layout, plan)
    assert info["num_partials"] > 0


def test_groups_detected(pps):
    plan = _plan(pps, workloads.tiny_mixed(values=False).layout)
    assert plan.info()["num_groups"] == 1      # the 2-page prefix shared by all four requests
    wl = workloads.radix_sharing(groups=3, root=64, branch=32, pairs=2, tail_lo=1, tail_hi=80,
                                 **SMALL)
    info = _plan(pps, wl.layout).info()
    assert info["num_groups"] == 3 * (1 + 2)   # per subtree: the root and two pair branches
    assert _plan(pps, wl.layout, flags=pps.PLAN_NO_GROUPS).info()["num_groups"] == 0
    # shared pages are read once per group: bytes read < bytes read without groups
    a = _plan(pps, wl.layout).info()["kv_bytes_read"]
    b = _plan(pps, wl.layout, flags=pps.PLAN_NO_GROUPS).info()["kv_bytes_read"]
    assert a < b


def test_wide_prefill_rows_read_shared_pages_in_their_own_tiles(pps):
    """A request whose rows fill more than half a tensor-core tile stays out of
    the shared-prefix grouping (a group would only add fp32 partials to tiles
    it already fills); narrower requests on the same pages still group.  Four
    requests share a 4-page prefix at G = 4: two decode rows, a 32-token chunk
    (128 rows: grouped) and a 33-token chunk (132 rows: alone).  CUDA-core-only
    plans group all four."""
    reqs = [([0], 20, [1]), ([0], 30, [1]), ([0], 40, [32]), ([0], 50, [33])]
    L = workloads.build_workload("wide", num_q_heads=32, num_kv_heads=8, head_dim=128,
                                 page_size=16, shared_lens=[64], requests=reqs, seed=3,
                                 values=False).layout
    for flags, members in ((0, [0, 1, 2]), (pps.PLAN_CUDA_CORES_ONLY, [0, 1, 2, 3])):
        plan = _plan(pps, L, flags=flags)
        check_plan(pps, L, plan)
        assert plan.info()["num_groups"] == 1
        rows = plan.array("rows")
        tasks = np.concatenate([plan.array("bw_tasks"), plan.array("mma_tasks")])
        grp = tasks[(tasks[:, 6] == pps.NO_CAUSAL) & (tasks[:, 4] == 0) & (tasks[:, 5] == 64)]
        toks = {int(t) for rec in grp for t in rows[rec[0]:rec[0] + rec[1]]}
        want = {t for r in members for t in range(int(L.q_indptr[r]), int(L.q_indptr[r + 1]))}
        assert toks == want
        if 3 not in members:                   # request 3 reads the prefix itself
            own = tasks[(tasks[:, 6] != pps.NO_CAUSAL) & (tasks[:, 3] == L.page_indptr[3])]
            assert own.size and own[:, 4].min() == 0


def test_unique_bytes_of_full_radix_workload(pps):
    L = workloads.radix_sharing(values=False).layout
    info = _plan(pps, L).info()
    tok_bytes = 2 * 8 * 128 * 2
    # 8 roots of 2048 + 32 branches of 512 + private tails (+1 new token each)
    tails = int((L.kv_len - 2048 - 512).sum())
    assert info["kv_bytes_unique"] == (8 * 2048 + 32 * 512 + tails) * tok_bytes
    if info["num_mma_tasks"] or info["small_rows_on_tensor"]:
        # a root group of 8 decode rows x G=4 runs as one 32-row key-tile task
        # (or one 128-row tile): every shared page read once
        assert info["kv_bytes_read"] == info["kv_bytes_unique"]
        assert info["num_mma_tasks"] == 0 and info["num_bw_tasks"] > 0
    else:
        # CUDA cores only: a root group of 8 decode rows x G=4 needs two 16-row tiles
        assert info["kv_bytes_read"] == info["kv_bytes_unique"] + 8 * 2048 * tok_bytes


def test_small_row_routing(pps):
    """Tasks of up to 32 rows go to the key-tile tensor kernel (head_dim 128,
    no draft tree); the CUDA-core kernel takes them under the flag, with head_dim
    64, or in draft-tree batches."""
    wl = workloads.radix_sharing(values=False)
    L = wl.layout
    on = _plan(pps, L).info()
    off = _plan(pps, L, flags=pps.PLAN_SMALL_ROWS_CUDA_CORES).info()
    assert on["small_rows_on_tensor"] == 1 and off["small_rows_on_tensor"] == 0
    assert on["num_mma_tasks"] == 0 and off["num_mma_tasks"] > 0   # 32-row roots move over
    assert _plan(pps, workloads.tiny_mixed(values=False).layout).info()["small_rows_on_tensor"] == 0


def test_plan_is_deterministic(pps):
    L = workloads.radix_sharing(groups=2, root=64, branch=32, pairs=2, tail_lo=1, tail_hi=80,
                                **SMALL).layout
    a, b = _plan(pps, L), _plan(pps, L)
    for name in ("bw_tasks", "mma_tasks", "rows", "merge_tokens", "merge_pids"):
        assert np.array_equal(a.array(name), b.array(name))


def test_zero_length_requests_contribute_no_rows(pps):
    q_indptr = np.array([0, 0, 3, 3], np.int32)
    kv_len = np.array([10, 7, 0], np.int32)
    page_indptr = np.array([0, 1, 2, 2], np.int32)
    plan = pps.attn_plan(q_indptr, kv_len, page_indptr, np.array([0, 1], np.int32), 8, 2, 64, 16, 2)
    rows = plan.array("rows")
    assert set(rows.tolist()) == {0, 1, 2}


@pytest.mark.parametrize("name", ["decode_heavy", "mixed_budget", "long_prefill", "radix_sharing"])
def test_full_size_plans_fast(pps, name):
    wl = workloads.make(name, values=False)
    for st in wl.steps:
        t0 = time.perf_counter()
        plan = _plan(pps, st.layout)
        dt = time.perf_counter() - t0
        info = plan.info()
        assert info["workspace_bytes"] > 0
        assert dt < 3.0, f"planning {name} took {dt:.3f}s"


# --- draft trees -------------------------------------------------------------

def _lookback(parent):
    """Expected lookback words: bit k set when the key k positions before the
    token is visible (its ancestor-or-self among the draft, or cached)."""
    anc = []
    words = []
    for j, a in enumerate(parent):
        anc.append({j} | (anc[a] if a >= 0 else set()))
        w = 0
        for k in range(64):
            if k > j or (j - k) in anc[j]:
                w |= 1 << k
        words.append(w)
    return words


def _tree_layout(n_tree=3, seed=0):
    wl = workloads.tree_verify(num_requests=n_tree, tree_size=20, kv_lo=1, kv_hi=300, **SMALL)
    L = wl.steps[0].layout
    return L


def test_tree_masks_in_the_plan(pps):
    L = _tree_layout()
    plan = _plan(pps, L, tree_parent=L.tree_parent)
    info = plan.info()
    assert info["num_tree_requests"] == L.num_requests
    words = plan.array("tree_mask").view(np.uint64)
    assert len(words) == L.num_tokens
    for r in range(L.num_requests):
        a, b = int(L.q_indptr[r]), int(L.q_indptr[r + 1])
        assert [int(x) for x in words[a:b]] == _lookback(L.tree_parent[a:b].tolist())
    check_plan(pps, L, plan)          # causal coverage is unchanged; masks apply in-kernel


def test_chain_parents_make_no_tree(pps):
    L = _tree_layout()
    chain = np.concatenate([workloads.chain_parents(int(q)) for q in L.q_len])
    plan = _plan(pps, L, tree_parent=chain)
    assert plan.info()["num_tree_requests"] == 0
    assert len(plan.array("tree_mask")) == 0
    ref = _plan(pps, L)
    for name in ("bw_tasks", "mma_tasks", "rows", "merge_pids"):
        assert np.array_equal(plan.array(name), ref.array(name))


def test_tree_flops_count_only_visible_pairs(pps):
    L = _tree_layout()
    plan = _plan(pps, L, tree_parent=L.tree_parent)
    pairs = 0                       # cached keys plus the ancestor-or-self set

    for r in range(L.num_requests):
        a, b = int(L.q_indptr[r]), int(L.q_indptr[r + 1])
        par = L.tree_parent[a:b].tolist()
        anc = []
        for j, p in enumerate(par):
            anc.append({j} | (anc[p] if p >= 0 else set()))
            pairs += int(L.cached_len[r]) + len(anc[j])
    expect = pairs * L.num_q_heads * 4.0 * L.head_dim
    assert plan.info()["flops_total"] == pytest.approx(expect, rel=1e-12)


@pytest.mark.parametrize("bad,code", [
    ([-1, 1], "invalid argument"),      # a token cannot be its own parent
    ([0, -1], "invalid argument"),      # token 0 has no earlier token
    ([-1, -2], "invalid argument"),
])
def test_tree_parent_validation(pps, bad, code):
    with pytest.raises(pps.PPSError, match=code):
        pps.attn_plan([0, 2], [10], [0, 1], [0], 8, 2, 64, 16, 1, tree_parent=bad)


def test_tree_size_limit(pps):
    q = pps.TREE_MAX_TOKENS + 1
    star = [-1] * q
    with pytest.raises(pps.PPSError, match="unsupported"):
        pps.attn_plan([0, q], [q + 5], [0, 5], list(range(5)), 8, 2, 64, 16, 5, tree_parent=star)
    # a chain of the same length is plain causal and has no limit
    plan = pps.attn_plan([0, q], [q + 5], [0, 5], list(range(5)), 8, 2, 64, 16, 5,
                         tree_parent=list(range(-1, q - 1)))
    assert plan.info()["num_tree_requests"] == 0


def test_key_tile_splits_are_even_whole_tiles(pps):
    """Adaptive chunking for key-tile tasks: a span within a quarter over the
    chunk stays whole; longer spans split into pieces of whole 128-key tiles
    that differ by at most one tile; no piece is a one-tile remainder unless
    its span is that short."""
    for L in (workloads.radix_sharing(values=False).layout,
              workloads.decode_heavy(values=False).layout):
        plan = _plan(pps, L)
        assert plan.info()["small_rows_on_tensor"] == 1
        t = plan.array("bw_tasks")
        Hkv = L.num_kv_heads
        heads0 = t[t[:, 2] == 0]                       # one record per task set
        by_span = {}
        for rec in heads0:
            by_span.setdefault((int(rec[0]), int(rec[6])), []).append(rec)
        for pieces in by_span.values():
            pieces.sort(key=lambda r: r[4])
            lens = [int(r[5] - r[4]) for r in pieces]
            for r in pieces[:-1]:
                assert (r[5] - r[4]) % 128 == 0       # whole tiles before the last piece
            if len(pieces) > 1:
                assert max(lens[:-1]) - min(lens[:-1]) <= 128
                assert lens[-1] > 128 or sum(lens) <= 2 * 128
    # the radix roots (2048 keys) stay whole: 8 subtrees x 8 kv heads of 16 tiles
    t = _plan(pps, workloads.radix_sharing(values=False).layout).array("bw_tasks")
    assert int(((t[:, 5] - t[:, 4]) == 2048).sum()) == 64


@pytest.mark.parametrize("num_sms", [152, 37, 5])
def test_key_tile_ranges_are_filled_least_loaded(pps, num_sms):
    """Key-tile plans give each persistent CTA a contiguous range of the task
    table (TT_CTA offsets), filled longest task first onto the CTA with the
    least work (whole 128-key tiles + 2 per task): every range is non-empty
    and in descending work order, and the most loaded CTA exceeds the least
    loaded by at most one task's work (the list-scheduling bound: the last
    task placed on the fullest CTA went to the least loaded CTA of its time)."""
    for L in (workloads.radix_sharing(values=False).layout,
              workloads.decode_heavy(values=False).layout,
              workloads.decode_heavy(num_requests=3, values=False).layout):
        plan = _plan(pps, L, num_sms=num_sms)
        assert plan.info()["small_rows_on_tensor"] == 1
        t = plan.array("bw_tasks")
        off = plan.array("tt_cta")
        C = min(len(t), num_sms)
        assert len(off) == C + 1 and off[0] == 0 and off[-1] == len(t)
        assert (np.diff(off) >= 1).all()
        work = -(-(t[:, 5] - t[:, 4]) // 128) + 2
        load = np.array([work[off[b]:off[b + 1]].sum() for b in range(C)])
        for b in range(C):
            assert (np.diff(work[off[b]:off[b + 1]]) <= 0).all()
        assert load.max() - load.min() <= work.max()
        assert load.sum() == work.sum()
    # the radix batch: the snake order this replaced left one CTA 35 tiles
    # (30.3 on average); balancing tiles + 2 per task leaves at most 32
    t = _plan(pps, workloads.radix_sharing(values=False).layout).array("bw_tasks")
    off = _plan(pps, workloads.radix_sharing(values=False).layout).array("tt_cta")
    tiles = -(-(t[:, 5] - t[:, 4]) // 128)
    per = np.array([tiles[off[b]:off[b + 1]].sum() for b in range(len(off) - 1)])
    assert per.max() <= 32


def test_plans_without_the_key_tile_kernel_have_no_ranges(pps):
    L = workloads.decode_heavy(num_requests=6, **SMALL).layout       # head_dim 64
    plan = _plan(pps, L)
    assert plan.info()["small_rows_on_tensor"] == 0 and len(plan.array("tt_cta")) == 0
    L = workloads.decode_heavy(num_requests=6, values=False).layout
    plan = _plan(pps, L, flags=pps.PLAN_SMALL_ROWS_CUDA_CORES)
    assert plan.info()["small_rows_on_tensor"] == 0 and len(plan.array("tt_cta")) == 0
