"""Pins for the fp64 oracle: each checks it against something other than itself.

* brute force: the softmax definition as plain Python loops over the unpaged
  K/V rows the generator drew before paging (no page table involved);
* closed forms: zero keys (uniform weights), constant values, a single
  visible key, a dominant key, and a worked two-key case from tests/golden;
* invariances the pages state: page order does not matter, a shared prefix
  gives what a private copy gives (radix sharing keeps K/V semantics), and
  splitting the keys then merging by log-sum-exp gives plain softmax
  (online-softmax equivalence);
* batch composition: a request's rows do not depend on the other requests;
* draft trees: a token's output equals that of the last token of a plain
  causal request made of its root-to-node path; a chain tree is the causal
  mask; brute force with each token's key list built bottom-up;
* planted mistakes: textual mutations of the oracle (a dropped scale, a
  shifted causal limit, a transposed head mapping, a wrong page slot, a
  missing max-subtraction guard) each make one of these pins fail.
"""
from __future__ import annotations

import json
import math
import os
import types

import numpy as np
import pytest
import torch

import oracle
import workloads
from oracle_run import oracle_steps

HERE = os.path.dirname(os.path.abspath(__file__))


def small_workloads():
    """Down-scaled copies of the five workloads (same structure, tiny sizes)."""
    kw = dict(num_q_heads=8, num_kv_heads=2, head_dim=32, page_size=16, keep_segments=True)
    return {
        "tiny_mixed": workloads.tiny_mixed(),
        "decode_heavy": workloads.decode_heavy(num_requests=3, kv_lo=20, kv_hi=50, **kw),
        "radix_sharing": workloads.radix_sharing(groups=2, root=32, branch=16, pairs=2,
                                                 tail_lo=3, tail_hi=20, **kw),
        "mixed_budget": workloads.mixed_budget(budget=30, prefill_q=8, prefill_cached=16,
                                               num_verify=2, verify_lo=2, verify_hi=4, mu=3.0,
                                               sigma=0.5, clip_lo=16, clip_hi=40, **kw),
        "long_prefill": workloads.long_prefill(num_requests=2, chunk=8, num_chunks=3, **kw),
        "tree_verify": workloads.tree_verify(num_requests=3, tree_size=12, kv_lo=5, kv_hi=40,
                                             **kw),
    }


SMALL = None


def _small():
    global SMALL
    if SMALL is None:
        SMALL = small_workloads()
    return SMALL


@pytest.mark.parametrize("name", list(workloads.WORKLOADS))
def test_bruteforce_on_unpaged_copies(name):
    wl = _small()[name]
    outs, _ = oracle_steps(wl)
    for s, st in enumerate(wl.steps):
        L = st.layout
        for r in range(L.num_requests):
            a, b = int(L.q_indptr[r]), int(L.q_indptr[r + 1])
            if a == b:
                continue
            k, v = workloads.contiguous_kv(wl, r, upto_step=s)
            assert k.shape[0] == int(L.kv_len[r])
            keys = None
            if L.tree_parent is not None:
                keys = _tree_keys(L.tree_parent[a:b], int(L.cached_len[r]))
            bf = np.array(oracle.dense_attention_loops(st.q[a:b], k, v, int(L.cached_len[r]),
                                                       L.sm_scale, L.num_kv_heads, keys=keys))
            np.testing.assert_allclose(outs[s][a:b], bf, rtol=0, atol=1e-12)


def _tree_keys(parent, c):
    """Key positions of each draft token, built bottom-up (a token sees what
    its parent sees plus its own position), independently of the oracle's
    upward walk."""
    keys = []
    for j, a in enumerate(parent):
        base = list(range(c)) if a < 0 else keys[a]
        keys.append(base + [c + j])
    return keys


@pytest.mark.parametrize("name", list(workloads.WORKLOADS))
def test_scatter_places_rows_where_the_page_walk_reads_them(name):
    wl = _small()[name]
    pk, pv = wl.pool_k, wl.pool_v
    for s, st in enumerate(wl.steps):
        L = st.layout
        before_k = pk.clone()
        pk, pv = oracle.reference_scatter(pk, pv, st.k_new, st.v_new, L.q_indptr, L.cached_len,
                                          L.page_indptr, L.page_indices, L.page_size)
        touched = torch.zeros(pk.shape[:1] + pk.shape[2:3], dtype=torch.bool)
        for r in range(L.num_requests):
            k, v = workloads.contiguous_kv(wl, r, upto_step=s)
            gk, gv = oracle.gather_request_kv(pk, pv, r, L.kv_len, L.page_indptr,
                                              L.page_indices, L.page_size)
            assert np.array_equal(gk, k.double().numpy())
            assert np.array_equal(gv, v.double().numpy())
            for p in range(int(L.cached_len[r]), int(L.kv_len[r])):
                touched[int(L.page_indices[L.page_indptr[r] + p // L.page_size]), p % L.page_size] = True
        # Nothing outside the new rows' slots changed (NaN stays NaN bit for bit).
        same = (pk.view(torch.int16) == before_k.view(torch.int16)).all(dim=(1, 3))
        assert bool((same | touched).all())


def _relabel_pages(wl, seed):
    rng = np.random.default_rng(seed)
    perm = rng.permutation(wl.pool_k.shape[0])
    inv = torch.as_tensor(np.argsort(perm))
    pk = wl.pool_k.index_select(0, inv)   # new page perm[p] holds old page p
    pv = wl.pool_v.index_select(0, inv)
    steps = []
    for st in wl.steps:
        L = st.layout
        nl = workloads.Layout(L.num_q_heads, L.num_kv_heads, L.head_dim, L.page_size,
                              L.num_pages, L.q_indptr, L.cached_len, L.kv_len, L.page_indptr,
                              perm[L.page_indices].astype(np.int32))
        steps.append(workloads.Step(nl, st.q, st.k_new, st.v_new))
    return workloads.Workload(wl.name, pk, pv, steps)


@pytest.mark.parametrize("name", ["tiny_mixed", "radix_sharing", "long_prefill"])
def test_page_order_does_not_matter(name):
    wl = _small()[name]
    ref, _ = oracle_steps(wl)
    got, _ = oracle_steps(_relabel_pages(wl, 7))
    for a, b in zip(ref, got):
        assert np.array_equal(a, b)


def _unshare(wl):
    """Give every request private copies of the pages it shares (same values)."""
    L0 = wl.steps[0].layout
    counts = {}
    for p in L0.page_indices.tolist():
        counts[p] = counts.get(p, 0) + 1
    shared = sorted(p for p, c in counts.items() if c > 1)
    assert shared, "workload has no shared pages"
    pk, pv = wl.pool_k, wl.pool_v
    extra_k, extra_v, new_lists = [], [], []
    nxt = pk.shape[0]
    for r in range(L0.num_requests):
        pl = L0.page_indices[L0.page_indptr[r]:L0.page_indptr[r + 1]].copy()
        for i, p in enumerate(pl):
            if counts[int(p)] > 1:
                extra_k.append(pk[int(p)])
                extra_v.append(pv[int(p)])
                pl[i] = nxt
                nxt += 1
        new_lists.append(pl)
    pk = torch.cat([pk, torch.stack(extra_k)])
    pv = torch.cat([pv, torch.stack(extra_v)])
    indptr = np.concatenate([[0], np.cumsum([len(p) for p in new_lists])]).astype(np.int32)
    nl = workloads.Layout(L0.num_q_heads, L0.num_kv_heads, L0.head_dim, L0.page_size, nxt,
                          L0.q_indptr, L0.cached_len, L0.kv_len, indptr,
                          np.concatenate(new_lists).astype(np.int32))
    st = wl.steps[0]
    return workloads.Workload(wl.name, pk, pv, [workloads.Step(nl, st.q, st.k_new, st.v_new)])


@pytest.mark.parametrize("name", ["tiny_mixed", "radix_sharing"])
def test_shared_prefix_equals_private_copy(name):
    wl = _small()[name]
    ref, _ = oracle_steps(wl)
    got, _ = oracle_steps(_unshare(wl))
    assert np.array_equal(ref[0], got[0])


def test_request_alone_equals_request_in_batch():
    wl = _small()["mixed_budget"]
    ref, _ = oracle_steps(wl)
    L = wl.steps[0].layout
    for r in range(L.num_requests):
        sub = workloads.sub_workload(wl, 0, [r])
        got, _ = oracle_steps(sub)
        assert np.array_equal(got[0], ref[0][L.q_indptr[r]:L.q_indptr[r + 1]])


# --- draft trees ------------------------------------------------------------

def _tree_request(parent, n_cached, Hq=4, Hkv=2, d=16, P=4, seed=3):
    wl = workloads.build_workload("tree", num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d,
                                  page_size=P, shared_lens=[], requests=[([], n_cached, [len(parent)])],
                                  seed=seed, keep_segments=True)
    wl.steps[0].layout.tree_parent = np.asarray(parent, np.int32)
    return wl


def _chain_output(q_rows, k, v, P=4):
    """Causal (chain) attention of ``q_rows`` [m, Hq, d] over contiguous K/V
    [n, Hkv, d], run through the paged oracle with a fresh identity page table."""
    n, Hkv, d = k.shape
    npg = -(-n // P)
    pk = torch.full((npg, Hkv, P, d), float("nan"), dtype=torch.bfloat16)
    pv = pk.clone()
    for p in range(n):
        pk[p // P, :, p % P] = k[p]
        pv[p // P, :, p % P] = v[p]
    m = q_rows.shape[0]
    return oracle.paged_attention(q_rows, pk, pv, np.array([0, m]), np.array([n]),
                                  np.array([0, npg]), np.arange(npg), P, 1 / math.sqrt(d), Hkv)


TREES = {
    "random": workloads.draft_tree(np.random.default_rng(11), 14),
    "star": np.full(9, -1, np.int32),                       # every token hangs off the context
    "two_chains": np.array([-1, 0, 1, 2, -1, 4, 5], np.int32),
    "binary": np.array([-1, 0, 0, 1, 1, 2, 2, 3, 3, 4], np.int32),
}


@pytest.mark.parametrize("tree", list(TREES))
def test_tree_node_equals_its_path_as_a_chain(tree):
    """A draft token's output is the output of the last token of a plain
    causal request whose new tokens are the token's root-to-node path."""
    parent = TREES[tree]
    c = 10
    wl = _tree_request(parent, c)
    out, _ = oracle_steps(wl)
    st = wl.steps[0]
    k, v = workloads.contiguous_kv(wl, 0)
    for j in range(len(parent)):
        path = []
        i = j
        while i >= 0:
            path.append(i)
            i = int(parent[i])
        path = path[::-1]
        idx = list(range(c)) + [c + i for i in path]
        ref = _chain_output(st.q[path], k[idx], v[idx])
        np.testing.assert_allclose(out[0][j], ref[-1], rtol=0, atol=1e-12)


def test_chain_tree_is_the_causal_mask():
    wl = _small()["mixed_budget"]
    ref, _ = oracle_steps(wl)
    L = wl.steps[0].layout
    L.tree_parent = np.concatenate([workloads.chain_parents(int(q)) for q in L.q_len])
    try:
        got, _ = oracle_steps(wl)
    finally:
        L.tree_parent = None
    assert np.array_equal(ref[0], got[0])


def test_tree_parent_must_precede_the_token():
    with pytest.raises(ValueError):
        oracle.tree_ancestors([-1, 1])
    with pytest.raises(ValueError):
        oracle.tree_ancestors([0])
    assert oracle.tree_ancestors([-1, 0, 0, 2]) == [{0}, {0, 1}, {0, 2}, {0, 2, 3}]


TREE_MUTATIONS = {
    "parent_only": ("            i = parent[i]\n", "            i = parent[i] if i == j else -1\n"),
    "mask_offset": ("visible[x, c + i] = False", "visible[x, c + i - 1] = False"),
    "tree_ignored": ("        if tree_parent is not None:\n            anc =",
                     "        if False:\n            anc ="),
}


@pytest.mark.parametrize("name", list(TREE_MUTATIONS))
def test_planted_tree_mistake_is_caught(name):
    src_path = os.path.join(os.path.dirname(oracle.__file__), "attention.py")
    src = open(src_path).read()
    old, new = TREE_MUTATIONS[name]
    assert src.count(old) == 1, name
    mod = types.ModuleType("oracle_tree_mutant_" + name)
    exec(compile(src.replace(old, new), src_path, "exec"), mod.__dict__)
    parent = TREES["binary"]
    c = 10
    wl = _tree_request(parent, c)
    st = wl.steps[0]
    L = st.layout
    pk, pv = oracle.reference_scatter(wl.pool_k, wl.pool_v, st.k_new, st.v_new, L.q_indptr,
                                      L.cached_len, L.page_indptr, L.page_indices, L.page_size)
    out = mod.paged_attention(st.q, pk, pv, L.q_indptr, L.kv_len, L.page_indptr, L.page_indices,
                              L.page_size, L.sm_scale, L.num_kv_heads, tree_parent=parent)
    k, v = workloads.contiguous_kv(wl, 0)
    bf = np.array(oracle.dense_attention_loops(st.q, k, v, c, L.sm_scale, L.num_kv_heads,
                                               keys=_tree_keys(parent, c)))
    assert not np.allclose(out, bf, rtol=0, atol=1e-12), f"tree mutation {name} slipped through"


# --- closed forms -----------------------------------------------------------

def _single_request(n_cached, q_len, Hq=4, Hkv=2, d=16, P=4, seed=0):
    return workloads.build_workload("closed", num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d,
                                    page_size=P, shared_lens=[], requests=[([], n_cached, [q_len])],
                                    seed=seed, keep_segments=True)


def _run_single(wl, pool_k=None, pool_v=None, q=None, k_new=None, v_new=None):
    st = wl.steps[0]
    L = st.layout
    pk, pv = oracle.reference_scatter(wl.pool_k if pool_k is None else pool_k,
                                      wl.pool_v if pool_v is None else pool_v,
                                      st.k_new if k_new is None else k_new,
                                      st.v_new if v_new is None else v_new,
                                      L.q_indptr, L.cached_len, L.page_indptr, L.page_indices,
                                      L.page_size)
    return oracle.paged_attention(st.q if q is None else q, pk, pv, L.q_indptr, L.kv_len,
                                  L.page_indptr, L.page_indices, L.page_size, L.sm_scale,
                                  L.num_kv_heads), (pk, pv)


def test_zero_keys_give_the_mean_of_visible_values():
    wl = _single_request(9, 5)
    L = wl.steps[0].layout
    zk = torch.where(torch.isnan(wl.pool_k), wl.pool_k, torch.zeros_like(wl.pool_k))
    out, (pk, pv) = _run_single(wl, pool_k=zk, k_new=torch.zeros_like(wl.steps[0].k_new))
    k, v = workloads.contiguous_kv(wl, 0)
    v = v.double().numpy()
    G = L.num_q_heads // L.num_kv_heads
    for j in range(5):
        for h in range(L.num_q_heads):
            expect = v[: 9 + j + 1, h // G, :].mean(axis=0)
            np.testing.assert_allclose(out[j, h], expect, rtol=0, atol=1e-14)


def test_constant_values_give_that_constant():
    wl = _single_request(11, 3)
    L = wl.steps[0].layout
    const = torch.arange(L.head_dim, dtype=torch.float32).to(torch.bfloat16) / 8
    cv = torch.where(torch.isnan(wl.pool_v), wl.pool_v, const.expand_as(wl.pool_v))
    out, _ = _run_single(wl, pool_v=cv, v_new=const.expand_as(wl.steps[0].v_new).clone())
    np.testing.assert_allclose(out, np.broadcast_to(const.double().numpy(), out.shape),
                               rtol=0, atol=1e-14)


def test_single_visible_key_gives_its_value():
    wl = _single_request(0, 1)
    out, _ = _run_single(wl)
    v = wl.steps[0].v_new.double().numpy()   # [1, Hkv, d]
    G = 2
    for h in range(4):
        assert np.array_equal(out[0, h], v[0, h // G])


def test_dominant_key_takes_all_the_weight():
    wl = _single_request(7, 1, d=16)
    st = wl.steps[0]
    L = st.layout
    q = torch.zeros_like(st.q)
    q[0, :, 0] = 64.0
    kn = st.k_new.clone()
    kn[0, :, :] = 0
    kn[0, :, 0] = 64.0           # logit 64*64/4 = 1024 against O(16) for the rest
    out, _ = _run_single(wl, q=q, k_new=kn)
    v = st.v_new.double().numpy()
    for h in range(4):
        np.testing.assert_allclose(out[0, h], v[0, h // 2], rtol=0, atol=1e-12)


def test_worked_two_key_case():
    with open(os.path.join(HERE, "golden", "two_key_softmax.json")) as f:
        case = json.load(f)
    d = case["head_dim"]
    q = np.zeros((1, 1, d))
    q[0, 0, 0] = case["q0"]
    k = np.zeros((2, 1, d))
    k[1, 0, 0] = case["k1_0"]
    v = np.array(case["v"], dtype=np.float64).reshape(2, 1, d)
    pool_k = k.reshape(1, 2, 1, d).transpose(0, 2, 1, 3)
    pool_v = v.reshape(1, 2, 1, d).transpose(0, 2, 1, 3)
    out = oracle.paged_attention(q, pool_k, pool_v, np.array([0, 1]), np.array([2]),
                                 np.array([0, 1]), np.array([0]), 2, 1 / math.sqrt(d), 1)
    np.testing.assert_allclose(out[0, 0], np.array(case["expected_o"]), rtol=0, atol=1e-12)


# --- online softmax / merge ---------------------------------------------------

def test_split_and_merge_equals_plain_softmax():
    rng = np.random.default_rng(5)
    m, n, d = 6, 97, 32
    q = rng.standard_normal((m, d))
    k = rng.standard_normal((n, d))
    v = rng.standard_normal((n, d))
    vis = np.arange(n)[None, :] <= (n - m + np.arange(m))[:, None]
    full, _ = oracle.attention_partial(q, k, v, vis, 1 / math.sqrt(d))
    # reference written independently: explicit softmax per row
    for i in range(m):
        s = np.array([q[i] @ k[p] / math.sqrt(d) for p in range(n) if vis[i, p]])
        w = np.exp(s - s.max())
        w /= w.sum()
        np.testing.assert_allclose(full[i], w @ v[: len(s)], rtol=0, atol=1e-12)
    for bounds in ([(0, 16), (16, 50), (50, 97)], [(0, 1), (1, 96), (96, 97)], [(0, 97)]):
        got = oracle.split_kv_attention(q, k, v, vis, 1 / math.sqrt(d), bounds)
        np.testing.assert_allclose(got, full, rtol=0, atol=1e-12)


def test_merge_ignores_an_empty_partial():
    rng = np.random.default_rng(6)
    o = rng.standard_normal((3, 8))
    merged, lse = oracle.lse_merge([o, np.zeros((3, 8))], [np.array([0.5, 1.0, -2.0]),
                                                            np.full(3, -np.inf)])
    np.testing.assert_allclose(merged, o, rtol=0, atol=0)
    np.testing.assert_allclose(lse, [0.5, 1.0, -2.0], rtol=0, atol=1e-15)


# --- planted mistakes ---------------------------------------------------------

MUTATIONS = {
    "dropped_scale": ("s = sm_scale * (qb.reshape(-1, d) @ kg.T)", "s = (qb.reshape(-1, d) @ kg.T)"),
    "causal_off_by_one": ("<= (c + jb)[:, None]", "< (c + jb)[:, None]"),
    "head_mapping": ("kg = k[:, g, :]", "kg = k[:, (g + 1) % Hkv, :]"),
    "page_slot": ("slots = pos % P", "slots = (pos + 1) % P"),
    "scatter_position": ("p = int(cached_len[r]) + j", "p = int(cached_len[r]) + j + 1"),
    "values_from_keys": ("vg = v[:, g, :]", "vg = k[:, g, :]"),
}


def _mutant(name):
    src_path = os.path.join(os.path.dirname(oracle.__file__), "attention.py")
    src = open(src_path).read()
    old, new = MUTATIONS[name]
    assert src.count(old) == 1, name
    mod = types.ModuleType("oracle_mutant_" + name)
    exec(compile(src.replace(old, new), src_path, "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name", list(MUTATIONS))
def test_planted_mistake_is_caught(name, monkeypatch):
    mut = _mutant(name)
    wl = _small()["tiny_mixed"]
    st = wl.steps[0]
    L = st.layout
    caught = False
    try:
        pk, pv = mut.reference_scatter(wl.pool_k, wl.pool_v, st.k_new, st.v_new, L.q_indptr,
                                       L.cached_len, L.page_indptr, L.page_indices, L.page_size)
        out = mut.paged_attention(st.q, pk, pv, L.q_indptr, L.kv_len, L.page_indptr,
                                  L.page_indices, L.page_size, L.sm_scale, L.num_kv_heads)
        for r in range(L.num_requests):
            a, b = int(L.q_indptr[r]), int(L.q_indptr[r + 1])
            k, v = workloads.contiguous_kv(wl, r)
            bf = np.array(oracle.dense_attention_loops(st.q[a:b], k, v, int(L.cached_len[r]),
                                                       L.sm_scale, L.num_kv_heads))
            if not np.allclose(out[a:b], bf, rtol=0, atol=1e-12):
                caught = True
    except (IndexError, ValueError):
        caught = True
    assert caught, f"mutation {name} slipped past the brute-force pin"
