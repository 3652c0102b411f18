"""Reference partition of one batch over N GPUs (test infrastructure only).

Sources: XY-Serve review, "What carries the argument" (tiles sorted by
computational area and handed out so every core gets a fair share); SGLang
review, "Core claim" (requests sharing a prefix reuse its KV).  With one GPU
per part, read-once reuse of a shared prefix survives only if every request
of a radix subtree lands on the same GPU, and nothing then has to be
exchanged between GPUs.

Rules (plain reading; the library follows the same):
* A request with at least one whole cached page belongs to the subtree named
  by its first cached page id (shared prefixes always start at page 0, so
  requests that share any cached page share the first one); a request
  without a whole cached page is a subtree of its own.
* Work of a request: max(1, new tokens) x KV length (rows x keys, the area
  the planner sorts tiles by); work of a subtree: the sum over its requests.
* Subtrees are taken by work, largest first (ties: the lowest request id in
  the subtree), each going to the part with the least work so far (ties: the
  lowest part).
"""
from __future__ import annotations


def partition(q_indptr, kv_len, page_indptr, page_indices, page_size, num_parts):
    """Part index of every request, and the work of every part."""
    R = len(kv_len)
    subtree = {}
    order = []
    for r in range(R):
        q = int(q_indptr[r + 1]) - int(q_indptr[r])
        cached = int(kv_len[r]) - q
        if cached >= page_size:
            key = ("page", int(page_indices[int(page_indptr[r])]))
        else:
            key = ("alone", r)
        if key not in subtree:
            subtree[key] = []
            order.append(key)
        subtree[key].append(r)
    work = {k: sum(max(1, int(q_indptr[r + 1]) - int(q_indptr[r])) * int(kv_len[r])
                   for r in subtree[k]) for k in order}
    keys = sorted(order, key=lambda k: (-work[k], min(subtree[k])))
    load = [0] * num_parts
    part = [0] * R
    for k in keys:
        p = min(range(num_parts), key=lambda i: (load[i], i))
        load[p] += work[k]
        for r in subtree[k]:
            part[r] = p
    return part, load
