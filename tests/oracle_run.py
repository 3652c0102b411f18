"""Test helpers that drive the fp64 oracle over a whole workload (all steps).

Only ``oracle`` is called here; the CUDA library is never imported.
"""
from __future__ import annotations

import numpy as np

import oracle


def oracle_steps(wl, pool_k=None, pool_v=None, upto=None):
    """Run every step of ``wl`` through the oracle: append the step's new rows
    with ``reference_scatter`` and then attend.  Returns (list of fp64
    outputs per step, final pools)."""
    pk = wl.pool_k if pool_k is None else pool_k
    pv = wl.pool_v if pool_v is None else pool_v
    outs = []
    last = len(wl.steps) if upto is None else upto + 1
    for st in wl.steps[:last]:
        L = st.layout
        pk, pv = oracle.reference_scatter(pk, pv, st.k_new, st.v_new, L.q_indptr, L.cached_len,
                                          L.page_indptr, L.page_indices, L.page_size)
        outs.append(oracle.paged_attention(st.q, pk, pv, L.q_indptr, L.kv_len, L.page_indptr,
                                           L.page_indices, L.page_size, L.sm_scale,
                                           L.num_kv_heads, tree_parent=L.tree_parent))
    return outs, (pk, pv)


def oracle_tokens(wl, step, tokens):
    """fp64 oracle output for selected new tokens of one step, computed on a
    compact copy of just the requests those tokens belong to (so it works on
    workloads far larger than the host could attend in full).  Returns
    [len(tokens), Hq, d]."""
    L = wl.steps[step].layout
    tokens = np.asarray(tokens, dtype=np.int64)
    req_of = np.searchsorted(L.q_indptr, tokens, side="right") - 1
    reqs = sorted(set(int(r) for r in req_of))
    import workloads
    sub = workloads.sub_workload(wl, step, reqs)
    outs, _ = oracle_steps_selected(sub, step, reqs, L, tokens, req_of)
    return outs


def oracle_steps_selected(sub, step, reqs, L, tokens, req_of):
    pk, pv = sub.pool_k, sub.pool_v
    for s, st in enumerate(sub.steps):
        SL = st.layout
        pk, pv = oracle.reference_scatter(pk, pv, st.k_new, st.v_new, SL.q_indptr, SL.cached_len,
                                          SL.page_indptr, SL.page_indices, SL.page_size)
    SL = sub.steps[step].layout
    pos = {r: i for i, r in enumerate(reqs)}
    sub_tok = [int(SL.q_indptr[pos[int(r)]]) + int(t - L.q_indptr[r]) for t, r in zip(tokens, req_of)]
    out = oracle.paged_attention(sub.steps[step].q, pk, pv, SL.q_indptr, SL.kv_len, SL.page_indptr,
                                 SL.page_indices, SL.page_size, SL.sm_scale, SL.num_kv_heads,
                                 tokens=sub_tok, tree_parent=SL.tree_parent)
    return out, (pk, pv)
