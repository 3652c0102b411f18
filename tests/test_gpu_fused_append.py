"""GPU: the append fused into the first attention kernel of a step
(PPS_PLAN_FUSED_APPEND) against the separate kv_append launch, on the same
batches: the same copy and the same attention kernels, so the pool must come
out bit for bit as the oracle's scatter writes it and the output rows must be
bit-identical to the unfused step's (which test_gpu_parity checks against the
oracle).  Plans whose first kernel cannot carry the append (the CUDA-core
kernel for head_dim 64) fall back to the separate launch with the same
results."""
from __future__ import annotations

import pytest
import torch

import oracle
from gpu_run import to_device
from test_gpu_parity import small_cases

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["decode_heavy", "radix_sharing", "mixed_budget", "long_prefill",
                                  "tree_verify", "tree_small_g4", "tile_edges", "tiny_mixed",
                                  "d64_g8"])
def test_fused_append_matches_separate_launch(pps, name):
    wl = small_cases()[name]()
    _, _, steps = to_device(wl)
    pk_a, pv_a = wl.pool_k.to("cuda", copy=True), wl.pool_v.to("cuda", copy=True)
    pk_b, pv_b = wl.pool_k.to("cuda", copy=True), wl.pool_v.to("cuda", copy=True)
    ok, ov = wl.pool_k, wl.pool_v
    pps.get_device_error(clear=True)
    for s, st in enumerate(steps):
        L = st["layout"]
        out_a = torch.full_like(st["q"], float("nan"))
        out_b = torch.full_like(st["q"], float("nan"))
        args = (st["q"], st["k_new"], st["v_new"], L.q_indptr, L.kv_len, L.page_indptr,
                L.page_indices)
        pps.attn_step(pk_a, pv_a, *args, out_a, tree_parent=L.tree_parent)
        pps.attn_step(pk_b, pv_b, *args, out_b, tree_parent=L.tree_parent,
                      flags=pps.PLAN_FUSED_APPEND)
        torch.cuda.synchronize()
        assert pps.get_device_error(clear=True) == 0, s
        assert torch.equal(out_b.view(torch.int16), out_a.view(torch.int16)), s
        ok, ov = oracle.reference_scatter(ok, ov, wl.steps[s].k_new, wl.steps[s].v_new,
                                          L.q_indptr, L.cached_len, L.page_indptr,
                                          L.page_indices, L.page_size)
        assert torch.equal(pk_b.cpu().view(torch.int16), ok.view(torch.int16)), s
        assert torch.equal(pv_b.cpu().view(torch.int16), ov.view(torch.int16)), s
    assert torch.equal(pk_a.view(torch.int16), pk_b.view(torch.int16))

