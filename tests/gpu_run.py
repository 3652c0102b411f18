"""Drive a workload through the CUDA library (test and bench helper).

Only the binding of libpps.so is used to compute; PyTorch allocates memory,
copies the generator's inputs to the device and compares results.
"""
from __future__ import annotations

import numpy as np
import torch

import paged_prefix_shared_gb300 as pps


def to_device(wl, device="cuda"):
    """Device copies of a workload's pools and per-step tensors."""
    # Always a copy: kv_append writes into it, and the generator's pool must
    # stay as drawn for the oracle.
    pk = wl.pool_k.to(device, copy=True).contiguous()
    pv = wl.pool_v.to(device, copy=True).contiguous()
    steps = []
    for st in wl.steps:
        L = st.layout
        tabs = {n: torch.as_tensor(getattr(L, n), dtype=torch.int32, device=device)
                for n in ("q_indptr", "cached_len", "kv_len", "page_indptr", "page_indices")}
        steps.append(dict(layout=L, q=st.q.to(device).contiguous(),
                          k_new=st.k_new.to(device).contiguous(),
                          v_new=st.v_new.to(device).contiguous(), tabs=tabs))
    return pk, pv, steps


def run_workload(wl, flags=0, device_inputs=None, keep_outputs=True, **plan_kw):
    """kv_append + attn_plan + attn_run for every step; returns (outputs, pools, plans)."""
    pk, pv, steps = device_inputs if device_inputs is not None else to_device(wl)
    outs, plans = [], []
    for st in steps:
        L = st["layout"]
        t = st["tabs"]
        pps.kv_append(pk, pv, st["k_new"], st["v_new"], t["q_indptr"], t["cached_len"],
                      t["page_indptr"], t["page_indices"])
        plan = pps.attn_plan(L.q_indptr, L.kv_len, L.page_indptr, L.page_indices, L.num_q_heads,
                             L.num_kv_heads, L.head_dim, L.page_size, pk.shape[0], flags=flags,
                             tree_parent=L.tree_parent, **plan_kw)
        ws = torch.empty(max(plan.workspace_bytes, 256), dtype=torch.uint8, device=pk.device)
        out = torch.full_like(st["q"], float("nan"))
        pps.attn_run(plan, st["q"], pk, pv, out, ws)
        outs.append(out if keep_outputs else None)
        plans.append(plan)
    torch.cuda.synchronize()
    return outs, (pk, pv), plans


def errors(got, ref):
    """(max abs, mean abs) of a bf16 GPU result against an fp64 reference."""
    g = got.double().cpu().numpy() if isinstance(got, torch.Tensor) else np.asarray(got)
    d = np.abs(g - ref)
    return float(np.nanmax(d)) if d.size else 0.0, float(d.mean()) if d.size else 0.0
