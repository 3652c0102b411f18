"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Tolerance, on bf16 outputs: max abs <= 2e-2 and mean abs <= 2e-3 against
fp64.  kv_append is compared bit for bit with the oracle's scatter.  Inputs
come from the seeded generators only; expected values only from ``oracle``.
Every pool slot that holds no row (slots past a request's length, unused
pages) is NaN, so reading one would show up as a NaN output.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_run import errors, run_workload, to_device
from oracle_run import oracle_steps, oracle_tokens

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS = 2e-2, 2e-3

KW = dict(num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16, keep_segments=False)


def small_cases():
    """Sizes the oracle finishes in seconds, spanning several KV blocks, row
    tiles and chunks, with ragged tails."""
    return {
        "tiny_mixed": lambda: workloads.tiny_mixed(),
        "decode_heavy": lambda: workloads.decode_heavy(num_requests=24, kv_lo=1, kv_hi=1500, **KW),
        "radix_sharing": lambda: workloads.radix_sharing(groups=2, root=256, branch=64, pairs=2,
                                                         tail_lo=1, tail_hi=300, **KW),
        "mixed_budget": lambda: workloads.mixed_budget(budget=400, prefill_q=190, prefill_cached=77,
                                                       num_verify=6, mu=5.0, sigma=1.0,
                                                       clip_lo=1, clip_hi=3000, **KW),
        "long_prefill": lambda: workloads.long_prefill(num_requests=2, chunk=300, num_chunks=3,
                                                       **dict(KW, page_size=64)),
        "d64_g8": lambda: workloads.mixed_budget(budget=120, prefill_q=70, prefill_cached=5,
                                                 num_verify=3, mu=4.0, sigma=1.0, clip_lo=1,
                                                 clip_hi=700, num_q_heads=16, num_kv_heads=2,
                                                 head_dim=64, page_size=32),
        "g1_p128": lambda: workloads.mixed_budget(budget=100, prefill_q=40, prefill_cached=200,
                                                  num_verify=3, mu=4.0, sigma=1.0, clip_lo=1,
                                                  clip_hi=700, num_q_heads=4, num_kv_heads=4,
                                                  head_dim=128, page_size=128),
        # prefill chunks written directly by tensor-core tiles at G = 1 and 2:
        # the rows of a lane quad are not one token's heads there, so they take
        # the per-row stores instead of the quad transpose
        "g2_prefill": lambda: workloads.long_prefill(num_requests=2, chunk=200, num_chunks=2,
                                                     num_q_heads=8, num_kv_heads=4, head_dim=128,
                                                     page_size=64),
        "g1_prefill_d64": lambda: workloads.long_prefill(num_requests=2, chunk=150, num_chunks=2,
                                                         num_q_heads=4, num_kv_heads=4,
                                                         head_dim=64, page_size=32),
        # draft trees: 40-token trees (tensor-core tiles of 160 rows), 64-token
        # trees at G = 8 (two tasks per tree), 8-token trees at G = 1 (bandwidth
        # kernel), and trees behind a shared prefix (group tasks + tree tasks)
        "tree_verify": lambda: workloads.tree_verify(num_requests=6, tree_size=40, kv_lo=1,
                                                     kv_hi=1500, **KW),
        "tree_g8_d64": lambda: workloads.tree_verify(num_requests=3, tree_size=64, kv_lo=1,
                                                     kv_hi=700, num_q_heads=16, num_kv_heads=2,
                                                     head_dim=64, page_size=32),
        "tree_g1_bw": lambda: _star_and_chains(),
        # small trees at G = 4 (8 and 5 tokens: 32 and 20 rows, one key-tile task
        # each, masks inside the last KV tile, short contexts too)
        "tree_small_g4": lambda: _small_trees(),
        "tree_shared": lambda: _tree_shared(),
        # KV ends at every kind of place inside a 128-key tile (16- and
        # 64-token pages: one or two page boxes per tile on the key-tile kernel)
        "tile_edges": lambda: _tile_edges(),
        "tile_edges_p64": lambda: _tile_edges(page_size=64),
    }


def _tile_edges(page_size=16):
    """Decode rows and 3-token verify rows whose KV ends 1, 15, 16, 17, 31, 32,
    33, 111, 112, 113, 127 and 128 keys into the last 128-key tile, after 0 to
    2 whole tiles: the number of 16-key PV steps that run and the rows zeroed
    inside the last one take each of their edge values (the slots past every
    end hold NaN)."""
    ends = [1, 15, 16, 17, 31, 32, 33, 111, 112, 113, 127, 128]
    reqs = []
    for i, e in enumerate(ends):
        q = 3 if i % 2 and e >= 3 else 1
        kv = 128 * (i % 3) + e
        reqs.append(([], kv - q, [q]))
    kw = {k: v for k, v in KW.items() if k != "keep_segments"}
    kw["page_size"] = page_size
    return workloads.build_workload("tile_edges", shared_lens=[], requests=reqs, seed=23, **kw)


def _star_and_chains():
    """G = 1, 8-token drafts: every token off the context, two chains, random."""
    wl = workloads.tree_verify(num_requests=5, tree_size=8, kv_lo=1, kv_hi=900, num_q_heads=4,
                               num_kv_heads=4, head_dim=128, page_size=16, seed=8)
    par = wl.steps[0].layout.tree_parent
    par[0:8] = -1
    par[8:16] = [-1, 0, 1, 2, -1, 4, 5, 6]
    return wl


def _small_trees():
    rng = np.random.default_rng(12)
    sizes = [8, 5, 8, 5, 8, 3]
    kv = [1, 40, 130, 700, 1300, 2]
    reqs = [([], int(c), [q]) for c, q in zip(kv, sizes)]
    wl = workloads.build_workload("tree_small", shared_lens=[], requests=reqs, seed=21,
                                  **{k: v for k, v in KW.items() if k != "keep_segments"})
    wl.steps[0].layout.tree_parent = np.concatenate([workloads.draft_tree(rng, q) for q in sizes])
    return wl


def _tree_shared():
    rng = np.random.default_rng(9)
    tails = rng.integers(1, 400, size=6)
    wl = workloads.build_workload("tree_shared", shared_lens=[256], requests=[([0], int(t), [24])
                                                                             for t in tails],
                                  seed=19, **{k: v for k, v in KW.items() if k != "keep_segments"})
    wl.steps[0].layout.tree_parent = np.concatenate([workloads.draft_tree(rng, 24)
                                                     for _ in tails])
    return wl


_CACHE = {}


def _small(name):
    if name not in _CACHE:
        wl = small_cases()[name]()
        _CACHE[name] = (wl, oracle_steps(wl))
    return _CACHE[name]


@pytest.fixture(scope="module", autouse=True)
def _lib(pps):
    assert torch.cuda.is_available()
    return pps


@pytest.mark.parametrize("name", list(small_cases()))
def test_kv_append_bit_exact(name):
    wl, (_, (ok, ov)) = _small(name)
    _, (gk, gv), _ = run_workload(wl)
    assert torch.equal(gk.cpu().view(torch.int16), ok.view(torch.int16))
    assert torch.equal(gv.cpu().view(torch.int16), ov.view(torch.int16))


# 0: default routing (small-row tasks on the key-tile tensor kernel where it
# applies), 1: no shared-prefix groups, 2: CUDA cores only, 4: small-row tasks
# on the CUDA-core kernel with the tensor-core tiles for wide tasks
@pytest.mark.parametrize("flags", [0, 1, 2, 4])
@pytest.mark.parametrize("name", list(small_cases()))
def test_parity_small(pps, name, flags):
    wl, (ref, _) = _small(name)
    pps.get_device_error(clear=True)
    outs, _, plans = run_workload(wl, flags=flags)
    assert pps.get_device_error(clear=True) == 0
    for s, (o, r) in enumerate(zip(outs, ref)):
        assert torch.isfinite(o).all(), f"step {s}: non-finite output (a NaN slot was read?)"
        mx, mean = errors(o, r)
        assert mx <= MAX_ABS and mean <= MEAN_ABS, (s, mx, mean, plans[s].info())


@pytest.mark.parametrize("num_sms", [1, 3])
@pytest.mark.parametrize("name", ["decode_heavy", "radix_sharing", "mixed_budget", "tree_small_g4",
                                  "tile_edges", "tile_edges_p64"])
def test_parity_few_ctas(pps, name, num_sms):
    """Plans for 1 and 3 persistent CTAs: every CTA runs a long range of tasks
    back to back (query-row and output double buffers, QK across task ends,
    deferred outputs), against the oracle."""
    wl, (ref, _) = _small(name)
    pps.get_device_error(clear=True)
    outs, _, plans = run_workload(wl, num_sms=num_sms)
    assert pps.get_device_error(clear=True) == 0
    for s, (o, r) in enumerate(zip(outs, ref)):
        assert torch.isfinite(o).all(), s
        mx, mean = errors(o, r)
        assert mx <= MAX_ABS and mean <= MEAN_ABS, (s, mx, mean, plans[s].info())


@pytest.mark.parametrize("flags", [0, 4])
@pytest.mark.parametrize("chunk", [512, 2048])
def test_parity_long_tasks(pps, chunk, flags):
    """Tasks of hundreds of sub-blocks or tiles per CTA (consumer warps drift
    apart; the key-tile ring wraps many times)."""
    wl = workloads.decode_heavy(num_requests=16, kv_lo=3000, kv_hi=6000, seed=5, **KW)
    ref, _ = oracle_steps(wl)
    pps.get_device_error(clear=True)
    outs, _, plans = run_workload(wl, bw_chunk_tokens=chunk, num_sms=4, flags=flags)
    assert pps.get_device_error(clear=True) == 0
    mx, mean = errors(outs[0], ref[0])
    assert mx <= MAX_ABS and mean <= MEAN_ABS, (mx, mean)


@pytest.mark.parametrize("flags", [0, 4])
@pytest.mark.parametrize("name", ["decode_heavy", "radix_sharing", "mixed_budget", "tree_small_g4",
                                  "long_prefill", "tree_verify"])
def test_parity_wide_scores(pps, name, flags):
    """Query rows scaled by 32 (exact in bf16): scores spread over hundreds of
    log2 units, so first tiles fall outside the one-pass window (exact maxima),
    references rise mid-task (O rescaled in TMEM), and softmax rows are sharply
    peaked.  On the tensor-core tiles (long_prefill, tree_verify) masked tiles
    whose one-pass check fails fall back to the two-pass path over the -inf
    they were given."""
    wl = small_cases()[name]()
    for st in wl.steps:
        st.q = (st.q.float() * 32.0).to(torch.bfloat16)
    ref, _ = oracle_steps(wl)
    pps.get_device_error(clear=True)
    outs, _, plans = run_workload(wl, flags=flags)
    assert pps.get_device_error(clear=True) == 0
    for s, (o, r) in enumerate(zip(outs, ref)):
        assert torch.isfinite(o).all()
        mx, mean = errors(o, r)
        assert mx <= MAX_ABS and mean <= MEAN_ABS, (s, mx, mean)


@pytest.mark.parametrize("chunk", [16, 64, 200])
def test_parity_forced_split(chunk):
    wl, (ref, _) = _small("mixed_budget")
    outs, _, _ = run_workload(wl, bw_chunk_tokens=chunk, mma_chunk_tokens=128)
    mx, mean = errors(outs[0], ref[0])
    assert mx <= MAX_ABS and mean <= MEAN_ABS


def test_page_order_is_bit_invariant():
    wl, _ = _small("radix_sharing")
    rng = np.random.default_rng(11)
    perm = rng.permutation(wl.pool_k.shape[0])
    inv = torch.as_tensor(np.argsort(perm))
    steps = []
    for st in wl.steps:
        L = st.layout
        nl = workloads.Layout(L.num_q_heads, L.num_kv_heads, L.head_dim, L.page_size, L.num_pages,
                              L.q_indptr, L.cached_len, L.kv_len, L.page_indptr,
                              perm[L.page_indices].astype(np.int32))
        steps.append(workloads.Step(nl, st.q, st.k_new, st.v_new))
    wl2 = workloads.Workload(wl.name, wl.pool_k.index_select(0, inv), wl.pool_v.index_select(0, inv),
                             steps)
    a, _, _ = run_workload(wl)
    b, _, _ = run_workload(wl2)
    assert torch.equal(a[0].view(torch.int16), b[0].view(torch.int16))


def test_empty_and_degenerate_rows():
    # request 0: no new tokens; request 1: a single token with nothing cached
    # (output = its own V row); request 2: 3 new tokens on a 1-token cache.
    wl = workloads.build_workload("edge", num_q_heads=8, num_kv_heads=2, head_dim=64, page_size=16,
                                  shared_lens=[], requests=[([], 5, [0]), ([], 0, [1]),
                                                            ([], 1, [3])], seed=9)
    ref, _ = oracle_steps(wl)
    outs, _, _ = run_workload(wl)
    mx, mean = errors(outs[0], ref[0])
    assert mx <= MAX_ABS and mean <= MEAN_ABS
    v = wl.steps[0].v_new.double().numpy()
    np.testing.assert_allclose(outs[0][0].double().cpu().numpy(),
                               np.repeat(v[0], 4, axis=0), atol=1e-2)


def test_empty_batch():
    wl = workloads.build_workload("empty", num_q_heads=8, num_kv_heads=2, head_dim=64, page_size=16,
                                  shared_lens=[], requests=[([], 5, [0])], seed=9)
    outs, _, plans = run_workload(wl)
    assert outs[0].numel() == 0 and plans[0].info()["num_bw_tasks"] == 0


def test_kv_append_flags_bad_page_id_on_device(pps):
    wl = workloads.tiny_mixed()
    pk, pv, steps = to_device(wl)
    st = steps[0]
    bad = st["tabs"]["page_indices"].clone()
    bad[:] = 10_000                                  # every page id out of range
    before = pk.clone()
    pps.get_device_error(clear=True)
    pps.kv_append(pk, pv, st["k_new"], st["v_new"], st["tabs"]["q_indptr"],
                  st["tabs"]["cached_len"], st["tabs"]["page_indptr"], bad)
    torch.cuda.synchronize()
    assert pps.get_device_error(clear=True) == 1     # PPS_DEV_ERR_APPEND_PAGE_ID
    assert torch.equal(pk.view(torch.int16), before.view(torch.int16))
    # the context is still usable
    outs, _, _ = run_workload(wl)
    assert torch.isfinite(outs[0]).all()


def test_stream_error_words_keep_each_batch_errors_apart(pps):
    """Two batches on two streams, each stream with its own registered error
    word: the bad page id in one stream's append tables shows in that stream's
    word only; the other stream's word and the device's word stay 0."""
    wl = workloads.tiny_mixed()
    pk_a, pv_a, steps_a = to_device(wl)
    pk_b, pv_b, steps_b = to_device(wl)
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    wa = torch.zeros(1, dtype=torch.int32, device="cuda")
    wb = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    pps.get_device_error(clear=True)
    pps.set_stream_error_word(wa, stream=sa)
    pps.set_stream_error_word(wb, stream=sb)
    try:
        a, b = steps_a[0], steps_b[0]
        bad = a["tabs"]["page_indices"].clone()
        bad[:] = 10_000                              # every page id out of range
        torch.cuda.synchronize()
        with torch.cuda.stream(sa):
            pps.kv_append(pk_a, pv_a, a["k_new"], a["v_new"], a["tabs"]["q_indptr"],
                          a["tabs"]["cached_len"], a["tabs"]["page_indptr"], bad, stream=sa)
        with torch.cuda.stream(sb):
            pps.kv_append(pk_b, pv_b, b["k_new"], b["v_new"], b["tabs"]["q_indptr"],
                          b["tabs"]["cached_len"], b["tabs"]["page_indptr"],
                          b["tabs"]["page_indices"], stream=sb)
            L = b["layout"]
            plan = pps.attn_plan(L.q_indptr, L.kv_len, L.page_indptr, L.page_indices,
                                 L.num_q_heads, L.num_kv_heads, L.head_dim, L.page_size,
                                 pk_b.shape[0])
            ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
            out = torch.full_like(b["q"], float("nan"))
            pps.attn_run(plan, b["q"], pk_b, pv_b, out, ws, stream=sb)
        assert pps.get_stream_error(stream=sa, clear=False) == 1   # PPS_DEV_ERR_APPEND_PAGE_ID
        assert pps.get_stream_error(stream=sb, clear=False) == 0
        torch.cuda.synchronize()
        assert int(wa.item()) == 1 and int(wb.item()) == 0
        assert pps.get_device_error(clear=True) == 0
        assert torch.isfinite(out).all()
        # clearing through the call resets the caller's word
        assert pps.get_stream_error(stream=sa, clear=True) == 1
        torch.cuda.synchronize()
        assert int(wa.item()) == 0
    finally:
        pps.set_stream_error_word(None, stream=sa)
        pps.set_stream_error_word(None, stream=sb)
    # without a registration the stream reports the device's word again
    assert pps.get_stream_error(stream=sa) == 0


def test_run_rejects_small_workspace(pps):
    wl = workloads.tiny_mixed()
    pk, pv, steps = to_device(wl)
    L = steps[0]["layout"]
    plan = pps.attn_plan(L.q_indptr, L.kv_len, L.page_indptr, L.page_indices, 8, 2, 64, 16, 64)
    ws = torch.empty(plan.workspace_bytes - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(pps.PPSError, match="workspace"):
        pps.attn_run(plan, steps[0]["q"], pk, pv, torch.empty_like(steps[0]["q"]), ws)


# --- full sizes, sampled rows ------------------------------------------------

FULL = ["tiny_mixed", "decode_heavy", "radix_sharing", "mixed_budget", "long_prefill",
        "tree_verify"]


def _sample_tokens(L, n, seed):
    T = L.num_tokens
    rng = np.random.default_rng(seed)
    pick = set(rng.choice(T, size=min(n, T), replace=False).tolist())
    pick |= {0, T - 1}
    # every request's last token (the longest causal row)
    pick |= set((L.q_indptr[1:] - 1)[L.q_len > 0][:8].tolist())
    return np.array(sorted(pick))


@pytest.mark.parametrize("name", FULL)
def test_parity_full_size_sampled(pps, name):
    if name == "long_prefill" and not pps_has_mma(pps):
        pytest.skip("long prefill at full size needs the tensor-core path")
    wl = workloads.make(name, device="cuda")
    pps.get_device_error(clear=True)
    outs, _, plans = run_workload(wl)
    assert pps.get_device_error(clear=True) == 0     # no bounded wait ran out
    for s, st in enumerate(wl.steps):
        L = st.layout
        assert torch.isfinite(outs[s]).all()
        toks = _sample_tokens(L, 24, 100 + s) if name != "tiny_mixed" else np.arange(L.num_tokens)
        ref = oracle_tokens(wl, s, toks)
        mx, mean = errors(outs[s][torch.as_tensor(toks, device="cuda")], ref)
        assert mx <= MAX_ABS and mean <= MEAN_ABS, (name, s, mx, mean)
    del wl, outs
    torch.cuda.empty_cache()


def pps_has_mma(pps):
    L = workloads.tiny_mixed(values=False).layout
    plan = pps.attn_plan(L.q_indptr, L.kv_len, L.page_indptr, L.page_indices, 8, 2, 64, 16, 64)
    return plan.info()["num_mma_tasks"] > 0


def test_bounded_wait_reports_timeout_and_context_survives(pps):
    pps.get_device_error(clear=True)
    pps.selftest_wait_timeout(20_000_000)            # 20 ms; nothing ever arrives
    torch.cuda.synchronize()
    assert pps.get_device_error(clear=True) == 4     # PPS_DEV_ERR_WAIT_TIMEOUT
    outs, _, _ = run_workload(workloads.tiny_mixed())
    assert torch.isfinite(outs[0]).all()
    assert pps.get_device_error(clear=True) == 0
