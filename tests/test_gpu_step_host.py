"""GPU: the one-call steps -- pps_attn_step_host (host rows and tables in, host
output out) and pps_attn_step (device rows, host tables) -- against the
device-side calls (pps_kv_append + pps_attn_plan + pps_attn_run) on the same
batch: the same kernels and plan, so the output rows and the pool must match
bit for bit (the device path is checked against the oracle in test_gpu_parity)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from gpu_run import run_workload, to_device
from test_gpu_parity import small_cases

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(pps):
    assert torch.cuda.is_available()
    return pps


@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("name", ["decode_heavy", "radix_sharing", "mixed_budget", "tree_small_g4",
                                  "d64_g8"])
def test_step_host_matches_device_calls(pps, name, pinned):
    wl = small_cases()[name]()
    dev_in = to_device(wl)
    outs, (pk, pv), _ = run_workload(wl, device_inputs=dev_in)
    pk2, pv2 = wl.pool_k.to("cuda", copy=True), wl.pool_v.to("cuda", copy=True)
    for s, st in enumerate(wl.steps):
        L = st.layout
        host = lambda t: t.cpu().contiguous().pin_memory() if pinned else t.cpu().contiguous()
        q, k, v = host(st.q), host(st.k_new), host(st.v_new)
        out = torch.full(tuple(st.q.shape), float("nan"), dtype=torch.bfloat16)
        out = out.pin_memory() if pinned else out
        pps.get_device_error(clear=True)
        pps.attn_step_host(pk2, pv2, q, k, v, L.q_indptr, L.kv_len, L.page_indptr, L.page_indices,
                           out, tree_parent=L.tree_parent)
        torch.cuda.synchronize()
        assert pps.get_device_error(clear=True) == 0
        assert torch.equal(out.view(torch.int16), outs[s].cpu().view(torch.int16)), s
    assert torch.equal(pk2.view(torch.int16), pk.view(torch.int16))
    assert torch.equal(pv2.view(torch.int16), pv.view(torch.int16))


@pytest.mark.parametrize("name", ["decode_heavy", "radix_sharing", "mixed_budget", "tree_small_g4",
                                  "d64_g8", "long_prefill"])
def test_step_device_matches_device_calls(pps, name):
    wl = small_cases()[name]()
    dev_in = to_device(wl)
    outs, (pk, pv), _ = run_workload(wl, device_inputs=dev_in)
    pk2, pv2 = wl.pool_k.to("cuda", copy=True), wl.pool_v.to("cuda", copy=True)
    nk = pps.NUM_KERNEL_CLASSES
    for s, st in enumerate(dev_in[2]):
        L = st["layout"]
        out = torch.full_like(st["q"], float("nan"))
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * nk)]
        pps.get_device_error(clear=True)
        pps.attn_step(pk2, pv2, st["q"], st["k_new"], st["v_new"], L.q_indptr, L.kv_len,
                      L.page_indptr, L.page_indices, out, tree_parent=L.tree_parent,
                      events=ev if s == 0 else None)
        torch.cuda.synchronize()
        assert pps.get_device_error(clear=True) == 0
        assert torch.equal(out.view(torch.int16), outs[s].view(torch.int16)), s
        if s == 0:
            assert all(ev[2 * c].elapsed_time(ev[2 * c + 1]) >= 0 for c in range(nk))
    assert torch.equal(pk2.view(torch.int16), pk.view(torch.int16))
    assert torch.equal(pv2.view(torch.int16), pv.view(torch.int16))


def test_step_host_scratch_checks(pps):
    wl = small_cases()["decode_heavy"]()
    st = wl.steps[0]
    L = st.layout
    pk, pv = wl.pool_k.to("cuda", copy=True), wl.pool_v.to("cuda", copy=True)
    before = pk.clone()
    out = torch.empty(tuple(st.q.shape), dtype=torch.bfloat16)
    tiny = torch.empty(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(pps.PPSError, match="workspace"):
        pps.attn_step_host(pk, pv, st.q.cpu(), st.k_new.cpu(), st.v_new.cpu(), L.q_indptr,
                           L.kv_len, L.page_indptr, L.page_indices, out, scratch=tiny)
    torch.cuda.synchronize()
    assert torch.equal(pk.view(torch.int16), before.view(torch.int16))   # nothing enqueued
    with pytest.raises(pps.PPSError):
        pps.attn_step_host(pk, pv, st.q.cuda(), st.k_new.cpu(), st.v_new.cpu(), L.q_indptr,
                           L.kv_len, L.page_indptr, L.page_indices, out)


def _host_rows(st):
    pin = lambda t: t.cpu().contiguous().pin_memory()
    out = torch.full(tuple(st.q.shape), float("nan"), dtype=torch.bfloat16).pin_memory()
    return pin(st.q), pin(st.k_new), pin(st.v_new), out


def test_step_host_back_to_back_one_scratch(pps):
    """Six chunked-prefill steps enqueued with no synchronization between them,
    one scratch: the input rows of step n+2 go into the slot step n's kernels
    read, so every output is right only if that copy waited for them."""
    import workloads
    wl = workloads.long_prefill(num_requests=2, chunk=300, num_chunks=6, num_q_heads=32,
                                num_kv_heads=8, head_dim=128, page_size=64, keep_segments=False)
    dev_in = to_device(wl)
    outs, (pk, pv), _ = run_workload(wl, device_inputs=dev_in)
    pk2, pv2 = wl.pool_k.to("cuda", copy=True), wl.pool_v.to("cuda", copy=True)
    rows = [_host_rows(st) for st in wl.steps]
    scratch = torch.empty(128 << 20, dtype=torch.uint8, device="cuda")
    pps.get_device_error(clear=True)
    for st, (q, k, v, out) in zip(wl.steps, rows):
        L = st.layout
        pps.attn_step_host(pk2, pv2, q, k, v, L.q_indptr, L.kv_len, L.page_indptr, L.page_indices,
                           out, scratch=scratch)
    torch.cuda.synchronize()
    assert pps.get_device_error(clear=True) == 0
    for s, (_, _, _, out) in enumerate(rows):
        assert torch.equal(out.view(torch.int16), outs[s].cpu().view(torch.int16)), s
    assert torch.equal(pk2.view(torch.int16), pk.view(torch.int16))
    assert torch.equal(pv2.view(torch.int16), pv.view(torch.int16))


def test_step_host_two_streams(pps):
    """Two independent batches (own pool, scratch and stream) with their steps
    interleaved call by call: each stream's results match its batch's device
    calls, whatever the other stream does meanwhile."""
    import workloads
    mk = lambda seed: workloads.long_prefill(num_requests=2, chunk=200, num_chunks=4,
                                             num_q_heads=32, num_kv_heads=8, head_dim=128,
                                             page_size=16, keep_segments=False, seed=seed)
    wls = [mk(11), mk(12)]
    refs, pools, rows, scratches, streams = [], [], [], [], []
    for wl in wls:
        outs, _, _ = run_workload(wl, device_inputs=to_device(wl))
        refs.append(outs)
        pools.append((wl.pool_k.to("cuda", copy=True), wl.pool_v.to("cuda", copy=True)))
        rows.append([_host_rows(st) for st in wl.steps])
        scratches.append(torch.empty(128 << 20, dtype=torch.uint8, device="cuda"))
        streams.append(torch.cuda.Stream())
    torch.cuda.synchronize()
    pps.get_device_error(clear=True)
    for s in range(len(wls[0].steps)):
        for b, wl in enumerate(wls):
            L = wl.steps[s].layout
            q, k, v, out = rows[b][s]
            pps.attn_step_host(*pools[b], q, k, v, L.q_indptr, L.kv_len, L.page_indptr,
                               L.page_indices, out, scratch=scratches[b], stream=streams[b])
    torch.cuda.synchronize()
    assert pps.get_device_error(clear=True) == 0
    for b in range(2):
        for s, (_, _, _, out) in enumerate(rows[b]):
            assert torch.equal(out.view(torch.int16), refs[b][s].cpu().view(torch.int16)), (b, s)


def test_step_with_large_task_table(pps):
    """4096 decode rows: a task table over 1 MB, which the step calls upload
    apart from the step's tables (smaller ones ride in the same copy).  The
    device-row and host-row steps must match the separate calls bit for bit."""
    import workloads
    wl = workloads.decode_heavy(num_requests=4096, kv_lo=16, kv_hi=80, num_q_heads=32,
                                num_kv_heads=8, head_dim=128, page_size=16, keep_segments=False)
    L = wl.steps[0].layout
    plan = pps.attn_plan(L.q_indptr, L.kv_len, L.page_indptr, L.page_indices, L.num_q_heads,
                         L.num_kv_heads, L.head_dim, L.page_size, L.num_pages)
    assert plan.info()["table_bytes"] > 1 << 20
    dev_in = to_device(wl)
    outs, (pk, pv), _ = run_workload(wl, device_inputs=dev_in)
    st = dev_in[2][0]
    for host in (False, True):
        pk2, pv2 = wl.pool_k.to("cuda", copy=True), wl.pool_v.to("cuda", copy=True)
        pps.get_device_error(clear=True)
        if host:
            q, k, v, out = _host_rows(wl.steps[0])
            pps.attn_step_host(pk2, pv2, q, k, v, L.q_indptr, L.kv_len, L.page_indptr,
                               L.page_indices, out)
        else:
            out = torch.full_like(st["q"], float("nan"))
            pps.attn_step(pk2, pv2, st["q"], st["k_new"], st["v_new"], L.q_indptr, L.kv_len,
                          L.page_indptr, L.page_indices, out)
        torch.cuda.synchronize()
        assert pps.get_device_error(clear=True) == 0
        assert torch.equal(out.cpu().view(torch.int16), outs[0].cpu().view(torch.int16)), host
        assert torch.equal(pk2.view(torch.int16), pk.view(torch.int16))
        assert torch.equal(pv2.view(torch.int16), pv.view(torch.int16))


@pytest.mark.parametrize("locked", [True, False])
def test_step_host_split_output_copy(pps, locked):
    """Host-row prefill steps whose output (over 16 MB, several requests, only
    tensor-core tasks, no groups, no partials) goes back in two parts when the
    output is page-locked: the first requests' rows leave after a tensor-core
    launch over just their tasks, the rest after the second (pageable output:
    one copy after one launch).  Outputs and pool must match the separate
    calls bit for bit, steps enqueued back to back."""
    import workloads
    wl = workloads.long_prefill(num_requests=4, chunk=640, num_chunks=3, num_q_heads=32,
                                num_kv_heads=8, head_dim=128, page_size=64, keep_segments=False)
    for st in wl.steps:
        L = st.layout
        assert st.q.numel() * 2 >= 16 << 20
        info = pps.attn_plan(L.q_indptr, L.kv_len, L.page_indptr, L.page_indices, L.num_q_heads,
                             L.num_kv_heads, L.head_dim, L.page_size, L.num_pages).info()
        assert info["num_bw_tasks"] == 0 and info["num_merge_tokens"] == 0
        assert info["num_groups"] == 0
    dev_in = to_device(wl)
    outs, (pk, pv), _ = run_workload(wl, device_inputs=dev_in)
    pk2, pv2 = wl.pool_k.to("cuda", copy=True), wl.pool_v.to("cuda", copy=True)
    rows = [_host_rows(st) for st in wl.steps]
    if not locked:
        rows = [(q, k, v, torch.full(tuple(o.shape), float("nan"), dtype=torch.bfloat16))
                for q, k, v, o in rows]
    scratch = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    pps.get_device_error(clear=True)
    for st, (q, k, v, out) in zip(wl.steps, rows):
        L = st.layout
        pps.attn_step_host(pk2, pv2, q, k, v, L.q_indptr, L.kv_len, L.page_indptr, L.page_indices,
                           out, scratch=scratch)
    torch.cuda.synchronize()
    assert pps.get_device_error(clear=True) == 0
    for s, (_, _, _, out) in enumerate(rows):
        assert torch.equal(out.view(torch.int16), outs[s].cpu().view(torch.int16)), s
    assert torch.equal(pk2.view(torch.int16), pk.view(torch.int16))
    assert torch.equal(pv2.view(torch.int16), pv.view(torch.int16))


def test_step_host_many_scratch_buffers(pps):
    """The library keeps copy streams and slot events for up to 32 scratch
    buffers and retires the least recently used one (after the work it fences)
    when another comes: 40 steps, each with a scratch of its own, all kept
    alive so every address is new, give the separate calls' output each time."""
    wl = small_cases()["decode_heavy"]()
    st = wl.steps[0]
    L = st.layout
    dev_in = to_device(wl)
    outs, _, _ = run_workload(wl, device_inputs=dev_in)
    q, k, v, _ = _host_rows(st)
    keep = []
    for i in range(40):
        pk, pv = wl.pool_k.to("cuda", copy=True), wl.pool_v.to("cuda", copy=True)
        out = torch.full(tuple(st.q.shape), float("nan"), dtype=torch.bfloat16).pin_memory()
        scratch = torch.empty(8 << 20, dtype=torch.uint8, device="cuda")
        keep.append((pk, pv, out, scratch))
        pps.attn_step_host(pk, pv, q, k, v, L.q_indptr, L.kv_len, L.page_indptr,
                           L.page_indices, out, scratch=scratch)
    torch.cuda.synchronize()
    assert pps.get_device_error(clear=True) == 0
    for i, (_, _, out, _) in enumerate(keep):
        assert torch.equal(out.view(torch.int16), outs[0].cpu().view(torch.int16)), i
