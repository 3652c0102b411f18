"""pps_attn_run_noalloc: the attention entry point for callers that cannot
allocate device memory (it uses the library's fixed scratch array instead of a
caller workspace).  Its output must match pps_attn_run's on the same plan and
inputs, on two calls in a row (the array keeps the previous call's contents),
and plans larger than the array must be refused.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""
import numpy as np
import pytest
import torch

import workloads
from gpu_run import errors, to_device

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS = 2e-2, 2e-3


def _prepare(pps, wl):
    pk, pv, steps = to_device(wl)
    st = steps[0]
    L, t = st["layout"], st["tabs"]
    pps.kv_append(pk, pv, st["k_new"], st["v_new"], t["q_indptr"], t["cached_len"],
                  t["page_indptr"], t["page_indices"])
    plan = pps.attn_plan(L.q_indptr, L.kv_len, L.page_indptr, L.page_indices, L.num_q_heads,
                         L.num_kv_heads, L.head_dim, L.page_size, pk.shape[0])
    return pk, pv, st["q"], plan


@pytest.mark.parametrize("make", [
    lambda: workloads.radix_sharing(groups=2, root=256, branch=64, pairs=2, tail_lo=1,
                                    tail_hi=300, num_q_heads=32, num_kv_heads=8, head_dim=128,
                                    page_size=16),
    lambda: workloads.mixed_budget(budget=300, prefill_q=150, prefill_cached=40, num_verify=5,
                                   mu=5.0, sigma=1.0, clip_lo=1, clip_hi=3000, num_q_heads=32,
                                   num_kv_heads=8, head_dim=128, page_size=16),
    lambda: workloads.tiny_mixed(),
], ids=["radix", "mixed", "tiny"])
def test_noalloc_matches_workspace_entry_point(pps, make):
    wl = make()
    pk, pv, q, plan = _prepare(pps, wl)
    assert plan.workspace_bytes <= pps.NOALLOC_SCRATCH_BYTES
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    ref = torch.full_like(q, float("nan"))
    pps.attn_run(plan, q, pk, pv, ref, ws)
    torch.cuda.synchronize()
    ref64 = ref.double().cpu().numpy()
    for call in range(2):
        out = torch.full_like(q, float("nan"))
        pps.attn_run_noalloc(plan, q, pk, pv, out)
        torch.cuda.synchronize()
        assert torch.isfinite(out).all(), f"call {call}"
        mx, mean = errors(out, ref64)
        assert mx <= MAX_ABS and mean <= MEAN_ABS, (call, mx, mean)
    assert pps.get_device_error(clear=True) == 0


def test_noalloc_rejects_plans_larger_than_its_scratch(pps):
    # The full mixed-budget layout split into 128-token tasks needs over 1 GiB
    # of partials: far above the cap.
    L = workloads.mixed_budget(values=False).layout
    plan = pps.attn_plan(L.q_indptr, L.kv_len, L.page_indptr, L.page_indices, L.num_q_heads,
                         L.num_kv_heads, L.head_dim, L.page_size, L.num_pages,
                         bw_chunk_tokens=128)
    assert plan.workspace_bytes > pps.NOALLOC_SCRATCH_BYTES
    dummy = torch.zeros((1, 1, 16, 128), dtype=torch.bfloat16, device="cuda")
    q = torch.zeros((L.num_tokens, 32, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(pps.PPSError, match="scratch"):
        pps.attn_run_noalloc(plan, q, dummy, dummy, torch.empty_like(q))
