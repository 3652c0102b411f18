"""fp64 oracle (test infrastructure only; see the package docstring).

Sources, cited by page title and section:

* XY-Serve review -- "Tackling the Dynamicity in a Production LLM Serving
  System with SOTA Optimizations via Hybrid Prefill/Decode/Verify Scheduling
  on Efficient Meta-kernels" (pith.science/paper/ABCKJ6RF):
  - "Core claim": one attention meta-kernel computes matmul-softmax-matmul
    for prefill, decode and verify tokens of one token-budgeted batch, over a
    PagedAttention-style block cache with prefix caching and chunked prefill.
  - "Assumptions & free parameters": online softmax with rescaling gives the
    same result as plain softmax (so KV may be split and merged); the block
    table plus radix tree with copy-on-write keeps K/V semantics; padded
    score entries must not affect the output.
  - Figs. 7, 8, 11, 15 (token-wise K/V reuse, speculative verify, mask-aware
    computation, chunked prefill over earlier chunks' pages).
* SGLang review -- "SGLang: Efficient Execution of Structured Language Model
  Programs" (pith.science/p/2312.07104), "Core claim": RadixAttention reuses
  the KV cache of shared prompt prefixes across requests.

Readings where the pages are silent or garbled (each also listed in the
design notes):

* Padded / out-of-range score entries get probability 0 (logit -inf).  The
  assumption list has padded scores zeroed ahead of the softmax; taken
  literally a zero logit still carries weight exp(0), so the only reading
  that keeps padding from changing the result is exclusion.
* New token j of a request sits at absolute position c_r + j and sees every
  cached position and new positions 0..j (linear causal chain; verify rows
  use the same mask).
* GQA: query head h reads kv head h // G.
* scale = 1 / sqrt(head_dim).
* Tree verify (attentionhub.org listing, the Medusa entry: several candidate
  continuations verified in one step with tree-based attention; XY-Serve
  review, Fig. 8: tree-based speculative algorithms organise their
  predictions as a tree): the draft tokens of a request are
  given in an order where every token's parent comes before it, each with a
  parent index (-1: it hangs directly off the cached context).  Token j sees
  every cached position and the new positions of its ancestors and itself,
  and nothing else of the draft.  A chain (parent j - 1) is the causal mask.
"""
from __future__ import annotations

import math

import numpy as np


def _f64(x):
    """bf16 torch tensors or numpy arrays -> float64 numpy (exact)."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.float64)


def _copy(x):
    return x.clone() if hasattr(x, "clone") else np.array(x, copy=True)


def reference_scatter(pool_k, pool_v, k_new, v_new, q_indptr, cached_len,
                      page_indptr, page_indices, page_size):
    """Append the new rows to the paged pool (the definition of ``kv_append``).

    New token j of request r lands at logical position p = c_r + j, i.e. in
    physical page ``page_indices[page_indptr[r] + p // P]``, slot ``p % P``
    (block-table paging, XY-Serve review "Assumptions": PagedAttention block
    table; chunked-prefill and decode rows are appended the same way).
    Returns new arrays; the inputs are not modified.  Works on any dtype
    (bf16 bit patterns are copied unchanged).
    """
    pk, pv = _copy(pool_k), _copy(pool_v)
    kn, vn = k_new, v_new
    P = int(page_size)
    R = len(cached_len)
    for r in range(R):
        for j in range(int(q_indptr[r + 1]) - int(q_indptr[r])):
            p = int(cached_len[r]) + j
            page = int(page_indices[int(page_indptr[r]) + p // P])
            t = int(q_indptr[r]) + j
            pk[page, :, p % P, :] = kn[t]
            pv[page, :, p % P, :] = vn[t]
    return pk, pv


def gather_request_kv(pool_k, pool_v, r, kv_len, page_indptr, page_indices, page_size):
    """Logical K and V rows [n_r, Hkv, d] of request r, read by walking its
    page list: position p is slot p % P of page page_indices[page_indptr[r] + p // P]."""
    P = int(page_size)
    n = int(kv_len[r])
    pos = np.arange(n)
    pages = np.asarray(page_indices)[int(page_indptr[r]) + pos // P].astype(np.int64)
    slots = pos % P
    if not isinstance(pool_k, np.ndarray):  # torch tensor: index with torch
        import torch
        pages_t = torch.as_tensor(pages, device=pool_k.device)
        slots_t = torch.as_tensor(slots, device=pool_k.device)
        return _f64(pool_k[pages_t, :, slots_t, :]), _f64(pool_v[pages_t, :, slots_t, :])
    return _f64(pool_k[pages, :, slots, :]), _f64(pool_v[pages, :, slots, :])


def tree_ancestors(parent):
    """Ancestor-or-self sets of the draft tokens of one request.

    ``parent[j]`` is the index (within the request's new tokens) of token j's
    parent, or -1 when token j hangs off the cached context; parents come
    before their children.  Returns a list of sets, walking each token's
    parent links up to the context."""
    parent = [int(x) for x in parent]
    for j, a in enumerate(parent):
        if not -1 <= a < j:
            raise ValueError(f"token {j}: parent {a} is not an earlier token or -1")
    out = []
    for j in range(len(parent)):
        seen = set()
        i = j
        while i >= 0:
            seen.add(i)
            i = parent[i]
        out.append(seen)
    return out


def paged_attention(q, pool_k, pool_v, q_indptr, kv_len, page_indptr, page_indices,
                    page_size, sm_scale, num_kv_heads, tokens=None, block_bytes=128 << 20,
                    tree_parent=None):
    """Exact causal GQA attention of every new token over its request's paged KV.

    ``q`` [T, Hq, d]; pools [num_pages, Hkv, P, d] holding every row the step
    attends to (cached rows and this step's new rows already appended).
    Returns float64 [T, Hq, d]; if ``tokens`` (indices into T) is given, only
    those rows are computed and returned as [len(tokens), Hq, d].

    Per request and kv head the G query heads' rows are stacked, scores are
    computed with one fp64 matmul per block of query rows (blocked so a score
    block stays under ``block_bytes``), masked causally (new token j sees
    positions <= c_r + j; XY-Serve review, Figs. 8 and 15), max-subtracted,
    exponentiated, normalised and multiplied by V.

    ``tree_parent`` (optional, [T]): per new token its parent's index within
    the request's new tokens, or -1.  New position c_r + i is then visible to
    token j only when i is j or one of its ancestors (``tree_ancestors``);
    cached positions stay visible.  Omitted, every request is a chain.
    """
    qf = q
    T = int(q_indptr[-1])
    Hq = qf.shape[1]
    d = qf.shape[2]
    Hkv = int(num_kv_heads)
    G = Hq // Hkv
    R = len(kv_len)
    want = None
    if tokens is not None:
        want = {int(t): i for i, t in enumerate(tokens)}
        out = np.zeros((len(tokens), Hq, d))
    else:
        out = np.zeros((T, Hq, d))
    for r in range(R):
        t0, t1 = int(q_indptr[r]), int(q_indptr[r + 1])
        if t1 == t0:
            continue
        js = np.arange(t1 - t0)
        if want is not None:
            js = np.array([j for j in js if (t0 + j) in want], dtype=np.int64)
            if js.size == 0:
                continue
        n = int(kv_len[r])
        c = n - (t1 - t0)
        anc = None
        if tree_parent is not None:
            anc = tree_ancestors(np.asarray(tree_parent)[t0:t1])
        k, v = gather_request_kv(pool_k, pool_v, r, kv_len, page_indptr, page_indices, page_size)
        qr = _f64(qf[t0 + js] if want is None else qf[[t0 + int(j) for j in js]])  # [m, Hq, d]
        rows_per_block = max(1, int(block_bytes // (8 * G * max(n, 1))))
        for g in range(Hkv):
            kg = k[:, g, :]            # [n, d]
            vg = v[:, g, :]
            for b0 in range(0, len(js), rows_per_block):
                jb = js[b0:b0 + rows_per_block]
                qb = qr[b0:b0 + rows_per_block, g * G:(g + 1) * G, :]   # [m, G, d]
                s = sm_scale * (qb.reshape(-1, d) @ kg.T)               # [m*G, n]
                s = s.reshape(len(jb), G, n)
                visible = np.arange(n)[None, :] <= (c + jb)[:, None]    # [m, n]
                if anc is not None:
                    for x, j in enumerate(jb):
                        for i in range(int(j)):
                            if i not in anc[int(j)]:
                                visible[x, c + i] = False
                s = np.where(visible[:, None, :], s, -np.inf)
                s = s - s.max(axis=-1, keepdims=True)
                p = np.exp(s)
                p = p / p.sum(axis=-1, keepdims=True)
                o = (p.reshape(-1, n) @ vg).reshape(len(jb), G, d)
                if want is None:
                    out[t0 + jb, g * G:(g + 1) * G, :] = o
                else:
                    idx = [want[t0 + int(j)] for j in jb]
                    out[idx, g * G:(g + 1) * G, :] = o
    return out


def dense_attention_loops(q_rows, k, v, cached_len, sm_scale, num_kv_heads, keys=None):
    """Brute force, unvectorised: the definition written as plain loops over
    unpaged (contiguous) K/V of one request.

    ``q_rows`` [q, Hq, d], ``k``/``v`` [n, Hkv, d] with n = cached_len + q.
    ``keys`` (optional): per row, the list of key positions it attends to;
    default every position up to cached_len + j.
    Returns a nested list [q][Hq][d] of Python floats.
    """
    q_rows = _f64(q_rows).tolist()
    k = _f64(k).tolist()
    v = _f64(v).tolist()
    Hq = len(q_rows[0]) if q_rows else 0
    G = Hq // int(num_kv_heads)
    out = []
    for j, qj in enumerate(q_rows):
        seen = list(range(cached_len + j + 1)) if keys is None else list(keys[j])
        row = []
        for h in range(Hq):
            g = h // G
            logits = []
            for p in seen:
                acc = 0.0
                for x, y in zip(qj[h], k[p][g]):
                    acc += x * y
                logits.append(acc * sm_scale)
            m = max(logits)
            w = [math.exp(a - m) for a in logits]
            z = sum(w)
            o = [0.0] * len(qj[h])
            for i, p in enumerate(seen):
                for e in range(len(o)):
                    o[e] += w[i] * v[p][g][e]
            row.append([x / z for x in o])
        out.append(row)
    return out


def attention_partial(q_rows, k, v, visible, sm_scale):
    """Softmax attention of rows ``q_rows`` [m, d] over keys ``k``/``v`` [n, d]
    restricted to ``visible`` [m, n] (bool).  Returns the normalised output
    [m, d] and the natural-log sum-exp [m] of the visible logits (-inf for a
    row that sees nothing).  This is one chunk of the split the
    online-softmax assumption allows (XY-Serve review, "Assumptions")."""
    q_rows, k, v = _f64(q_rows), _f64(k), _f64(v)
    s = sm_scale * (q_rows @ k.T)
    s = np.where(visible, s, -np.inf)
    m = s.max(axis=-1, keepdims=True)
    safe = np.where(np.isfinite(m), m, 0.0)
    p = np.exp(s - safe)
    z = p.sum(axis=-1, keepdims=True)
    o = np.where(z > 0, (p @ v) / np.where(z > 0, z, 1.0), 0.0)
    lse = np.where(z[:, 0] > 0, safe[:, 0] + np.log(np.where(z[:, 0] > 0, z[:, 0], 1.0)), -np.inf)
    return o, lse


def lse_merge(outs, lses):
    """Merge partial attention results over disjoint key sets.

    With M = max_i lse_i, the merged output is sum_i e^{lse_i - M} o_i /
    sum_i e^{lse_i - M} (each o_i already normalised by its own sum).  This is
    the split-and-merge that the online-softmax equivalence permits
    (XY-Serve review, "Assumptions"; Flash-Decoding in its reference list)."""
    outs = [np.asarray(o, dtype=np.float64) for o in outs]
    lses = np.stack([np.asarray(l, dtype=np.float64) for l in lses])   # [k, m]
    M = lses.max(axis=0)
    w = np.exp(lses - M[None, :])
    num = sum(w[i][:, None] * outs[i] for i in range(len(outs)))
    return num / w.sum(axis=0)[:, None], M + np.log(w.sum(axis=0))


def split_kv_attention(q_rows, k, v, visible, sm_scale, bounds):
    """Attention computed chunk by chunk over the key ranges ``bounds``
    (a list of [a, b) covering [0, n)) and merged with ``lse_merge``."""
    outs, lses = [], []
    for a, b in bounds:
        o, l = attention_partial(q_rows, k[a:b], v[a:b], visible[:, a:b], sm_scale)
        outs.append(o)
        lses.append(l)
    return lse_merge(outs, lses)[0]
