"""pps_attn_run_noalloc: the attention entry point for callers that cannot
allocate device memory (it uses the library's fixed scratch array instead of a
caller workspace).  The same plan through the same kernels must give output
bit-identical to pps_attn_run's, on two calls in a row, also when the array
still holds another plan's task table and partials; plans larger than the
array must be refused.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""
import os
import re

import pytest
import torch

import workloads
from gpu_run import to_device

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _prepare(pps, wl, **plan_kw):
    pk, pv, steps = to_device(wl)
    st = steps[0]
    L, t = st["layout"], st["tabs"]
    pps.kv_append(pk, pv, st["k_new"], st["v_new"], t["q_indptr"], t["cached_len"],
                  t["page_indptr"], t["page_indices"])
    plan = pps.attn_plan(L.q_indptr, L.kv_len, L.page_indptr, L.page_indices, L.num_q_heads,
                         L.num_kv_heads, L.head_dim, L.page_size, pk.shape[0], **plan_kw)
    return pk, pv, st["q"], plan


def _bits(t):
    return t.view(torch.int16)


def test_scratch_size_matches_the_header(pps):
    """The binding's constant is the header's PPS_NOALLOC_SCRATCH_BYTES."""
    src = open(os.path.join(ROOT, "include", "pps.h")).read()
    m = re.search(r"#define\s+PPS_NOALLOC_SCRATCH_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)", src)
    assert m, "PPS_NOALLOC_SCRATCH_BYTES not found in pps.h"
    assert pps.NOALLOC_SCRATCH_BYTES == int(m.group(1)) << int(m.group(2))


def _radix():
    return workloads.radix_sharing(groups=2, root=256, branch=64, pairs=2, tail_lo=1,
                                   tail_hi=300, num_q_heads=32, num_kv_heads=8, head_dim=128,
                                   page_size=16)


def _mixed():
    return workloads.mixed_budget(budget=300, prefill_q=150, prefill_cached=40, num_verify=5,
                                  mu=5.0, sigma=1.0, clip_lo=1, clip_hi=3000, num_q_heads=32,
                                  num_kv_heads=8, head_dim=128, page_size=16)


@pytest.mark.gpu
@pytest.mark.parametrize("make", [_radix, _mixed, workloads.tiny_mixed],
                         ids=["radix", "mixed", "tiny"])
def test_noalloc_matches_workspace_entry_point(pps, make):
    # First fill the shared array with a different plan's table and partials
    # (the mixed batch split into 64-token pieces: many partial rows), so the
    # plan under test starts on stale contents.
    opk, opv, oq, other = _prepare(pps, _mixed(), bw_chunk_tokens=64)
    assert other.info()["num_partials"] > 0
    assert other.workspace_bytes <= pps.NOALLOC_SCRATCH_BYTES
    pps.attn_run_noalloc(other, oq, opk, opv, torch.empty_like(oq))
    torch.cuda.synchronize()

    pk, pv, q, plan = _prepare(pps, make())
    assert plan.workspace_bytes <= pps.NOALLOC_SCRATCH_BYTES
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    ref = torch.full_like(q, float("nan"))
    pps.attn_run(plan, q, pk, pv, ref, ws)
    torch.cuda.synchronize()
    assert torch.isfinite(ref).all()
    for call in range(2):
        out = torch.full_like(q, float("nan"))
        pps.attn_run_noalloc(plan, q, pk, pv, out)
        torch.cuda.synchronize()
        assert torch.isfinite(out).all(), f"call {call}"
        # same plan, same kernels, same inputs: the same bits
        assert torch.equal(_bits(out), _bits(ref)), f"call {call}"
    assert pps.get_device_error(clear=True) == 0


@pytest.mark.gpu
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
