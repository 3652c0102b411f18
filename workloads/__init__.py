"""Seeded synthetic inputs for paged, prefix-shared, mixed-batch attention.

This module is the one piece shared by the fp64 oracle's tests and the CUDA
path's tests and benchmark.  It holds none of the attention arithmetic: it
draws a layout (per-request lengths, which requests share which cached
segments, which physical pages hold each segment) and bf16 values, and puts
every cached segment's rows into its pool pages.  Everything the method
computes (appending new rows, gathering through the page table, softmax,
merging) lives elsewhere, once in the oracle and once in the kernels.

Recipe (the pages publish no workload; these stand in for the ShareGPT and
nightly prefill-/decode-heavy serving benchmarks the XY-Serve review names
under "What would settle it"):

* Layout draws use ``numpy.random.default_rng(seed)`` (PCG64).
* Values are float32 N(0, 1) draws from ``torch.Generator(device).manual_seed(seed)``
  rounded to bf16 (round-to-nearest-even), drawn in a fixed order: K then V
  of every cached segment (a segment shared by several requests is drawn
  once), then per step the new K, the new V and the queries.
* Pool layout ``[num_pages, num_kv_heads, page_size, head_dim]`` (all slots of
  one page and one kv head contiguous).  Every slot that does not hold a
  cached row (new-token slots before they are appended, slots past a
  request's length, unused pages) holds NaN, so a kernel that reads one
  shows it in its output.
* Physical pages are a random permutation of the pool's page ids, taken in
  segment order.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

__all__ = [
    "Layout", "Step", "Workload", "build_workload", "tiny_mixed", "decode_heavy",
    "radix_sharing", "mixed_budget", "long_prefill", "WORKLOADS", "make",
    "contiguous_kv", "sub_workload", "draft_tree", "chain_parents", "tree_verify", "cache_trace",
]


@dataclass
class Layout:
    """Per-step batch metadata (host int32 arrays, CSR page table)."""
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    num_pages: int
    q_indptr: np.ndarray      # [R+1] new-token offsets
    cached_len: np.ndarray    # [R]   tokens cached before this step
    kv_len: np.ndarray        # [R]   cached + new
    page_indptr: np.ndarray   # [R+1]
    page_indices: np.ndarray  # [nnz] physical page ids, in logical order
    # [T] per new token: index of its parent among the request's new tokens, or
    # -1 (hangs off the cached context); None = every request is a chain.
    tree_parent: np.ndarray | None = None

    @property
    def num_requests(self) -> int:
        return int(self.q_len.shape[0])

    @property
    def q_len(self) -> np.ndarray:
        return np.diff(self.q_indptr).astype(np.int32)

    @property
    def num_tokens(self) -> int:
        return int(self.q_indptr[-1])

    @property
    def sm_scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)


@dataclass
class Step:
    layout: Layout
    q: torch.Tensor      # [T, Hq, d] bf16
    k_new: torch.Tensor  # [T, Hkv, d] bf16
    v_new: torch.Tensor  # [T, Hkv, d] bf16


@dataclass
class Workload:
    name: str
    pool_k: torch.Tensor  # [num_pages, Hkv, P, d] bf16, before the first step
    pool_v: torch.Tensor
    steps: list
    # Kept only when requested (small workloads): per-segment cached rows and,
    # per request, the ids of its segments in logical order.
    seg_k: list | None = None
    seg_v: list | None = None
    req_segments: list | None = None
    shared_segments: list = field(default_factory=list)  # ids of segments used by >1 request

    @property
    def layout(self) -> Layout:
        return self.steps[-1].layout


def _round_bf16(x: torch.Tensor) -> torch.Tensor:
    return x.to(torch.bfloat16)


def build_workload(name, *, num_q_heads, num_kv_heads, head_dim, page_size,
                   shared_lens, requests, seed, num_pages=None, pool_factor=1.25,
                   device="cpu", keep_segments=False, values=True):
    """Draw one workload.

    ``shared_lens[i]`` is the length (a multiple of ``page_size``) of shared
    cached segment ``i``.  ``requests`` is a list of
    ``(shared_path, private_cached, q_lens)``: the shared segment ids the
    request's cache starts with, in order, then the length of its private
    cached tail, then its new-token count at each step (one entry per step).
    The private tail's pages also hold the request's new tokens.  With
    ``values=False`` only the layouts are drawn (tensors are None).
    """
    P = page_size
    rng = np.random.default_rng(seed)
    for L in shared_lens:
        if L % P:
            raise ValueError("shared segments must be whole pages")
    n_steps = len(requests[0][2])
    if any(len(r[2]) != n_steps for r in requests):
        raise ValueError("every request needs one q_len per step")

    # Segment list: shared ones first, then one private segment per request.
    seg_cached = list(shared_lens)
    seg_npages = [L // P for L in shared_lens]
    req_segments = []
    for path, priv, qs in requests:
        sid = len(seg_cached)
        tot = priv + sum(qs)
        seg_cached.append(priv)
        seg_npages.append(-(-tot // P))
        req_segments.append(list(path) + [sid])
    needed = sum(seg_npages)
    if num_pages is None:
        num_pages = int(math.ceil(pool_factor * needed))
    if needed > num_pages:
        raise ValueError("pool too small")
    perm = rng.permutation(num_pages).astype(np.int32)
    seg_pages, off = [], 0
    for n in seg_npages:
        seg_pages.append(perm[off:off + n])
        off += n

    Hkv, Hq, d = num_kv_heads, num_q_heads, head_dim
    if not values:
        return _layouts_only(name, requests, shared_lens, seg_pages, req_segments, n_steps,
                             Hq, Hkv, d, P, num_pages)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    nan = float("nan")
    pool_k = torch.full((num_pages, Hkv, P, d), nan, dtype=torch.bfloat16, device=device)
    pool_v = torch.full_like(pool_k, nan)
    seg_k, seg_v = [], []
    for sid, L in enumerate(seg_cached):
        kk = _round_bf16(torch.randn((L, Hkv, d), generator=gen, device=device))
        vv = _round_bf16(torch.randn((L, Hkv, d), generator=gen, device=device))
        if keep_segments:
            seg_k.append(kk)
            seg_v.append(vv)
        if L == 0:
            continue
        npg = -(-L // P)
        pages = torch.as_tensor(seg_pages[sid][:npg], dtype=torch.long, device=device)
        for src, dst in ((kk, pool_k), (vv, pool_v)):
            pad = torch.full((npg * P, Hkv, d), nan, dtype=torch.bfloat16, device=device)
            pad[:L] = src
            dst.index_copy_(0, pages, pad.view(npg, P, Hkv, d).permute(0, 2, 1, 3).contiguous())
        del kk, vv

    steps = []
    q_done = [0] * len(requests)
    for s in range(n_steps):
        q_len = np.array([r[2][s] for r in requests], dtype=np.int64)
        cached = np.array([sum(shared_lens[i] for i in r[0]) + r[1] + q_done[j]
                           for j, r in enumerate(requests)], dtype=np.int64)
        kv_len = cached + q_len
        q_indptr = np.concatenate([[0], np.cumsum(q_len)]).astype(np.int32)
        plists = []
        for j, segs in enumerate(req_segments):
            full = np.concatenate([seg_pages[i] for i in segs])
            plists.append(full[: -(-int(kv_len[j]) // P)])
        page_indptr = np.concatenate([[0], np.cumsum([len(p) for p in plists])]).astype(np.int32)
        page_indices = (np.concatenate(plists) if plists else np.zeros(0)).astype(np.int32)
        T = int(q_indptr[-1])
        k_new = _round_bf16(torch.randn((T, Hkv, d), generator=gen, device=device))
        v_new = _round_bf16(torch.randn((T, Hkv, d), generator=gen, device=device))
        q = _round_bf16(torch.randn((T, Hq, d), generator=gen, device=device))
        lay = Layout(Hq, Hkv, d, P, num_pages, q_indptr, cached.astype(np.int32),
                     kv_len.astype(np.int32), page_indptr, page_indices)
        steps.append(Step(lay, q, k_new, v_new))
        for j in range(len(requests)):
            q_done[j] += int(q_len[j])

    use = {}
    for segs in req_segments:
        for i in segs:
            use[i] = use.get(i, 0) + 1
    shared = sorted(i for i, c in use.items() if c > 1)
    return Workload(name, pool_k, pool_v, steps,
                    seg_k if keep_segments else None,
                    seg_v if keep_segments else None,
                    req_segments, shared)


def _layouts_only(name, requests, shared_lens, seg_pages, req_segments, n_steps, Hq, Hkv, d, P,
                  num_pages):
    steps = []
    q_done = [0] * len(requests)
    for s in range(n_steps):
        q_len = np.array([r[2][s] for r in requests], dtype=np.int64)
        cached = np.array([sum(shared_lens[i] for i in r[0]) + r[1] + q_done[j]
                           for j, r in enumerate(requests)], dtype=np.int64)
        kv_len = cached + q_len
        q_indptr = np.concatenate([[0], np.cumsum(q_len)]).astype(np.int32)
        plists = [np.concatenate([seg_pages[i] for i in segs])[: -(-int(kv_len[j]) // P)]
                  for j, segs in enumerate(req_segments)]
        page_indptr = np.concatenate([[0], np.cumsum([len(p) for p in plists])]).astype(np.int32)
        page_indices = (np.concatenate(plists) if plists else np.zeros(0)).astype(np.int32)
        steps.append(Step(Layout(Hq, Hkv, d, P, num_pages, q_indptr, cached.astype(np.int32),
                                 kv_len.astype(np.int32), page_indptr, page_indices),
                          None, None, None))
        for j in range(len(requests)):
            q_done[j] += int(q_len[j])
    return Workload(name, None, None, steps, None, None, req_segments, [])


def contiguous_kv(wl: Workload, r: int, upto_step: int | None = None):
    """Request ``r``'s K and V rows in logical order ([n, Hkv, d] each), built
    from the drawn segments and new rows without any page table (needs
    ``keep_segments=True``).  Covers everything up to and including step
    ``upto_step`` (default: the last)."""
    if wl.seg_k is None:
        raise ValueError("workload was built without keep_segments")
    s_last = len(wl.steps) - 1 if upto_step is None else upto_step
    ks = [wl.seg_k[i] for i in wl.req_segments[r]]
    vs = [wl.seg_v[i] for i in wl.req_segments[r]]
    for s in range(s_last + 1):
        lay = wl.steps[s].layout
        a, b = int(lay.q_indptr[r]), int(lay.q_indptr[r + 1])
        ks.append(wl.steps[s].k_new[a:b])
        vs.append(wl.steps[s].v_new[a:b])
    return torch.cat(ks, 0), torch.cat(vs, 0)


# ---------------------------------------------------------------------------
# The five synthetic workloads (full sizes are the defaults).


def tiny_mixed(seed=0, device="cpu", keep_segments=True, values=True):
    """4 requests, 8/2 heads, d=64, P=16; cached {37,64,100,129} all starting
    with one shared 32-token (2-page) prefix; new tokens {1 decode, 1 decode,
    4 verify, 16 prefill chunk}; 64-page pool in random page order."""
    cached = [37, 64, 100, 129]
    qs = [1, 1, 4, 16]
    reqs = [([0], c - 32, [q]) for c, q in zip(cached, qs)]
    return build_workload("tiny_mixed", num_q_heads=8, num_kv_heads=2, head_dim=64,
                          page_size=16, shared_lens=[32], requests=reqs, seed=seed,
                          num_pages=64, device=device, keep_segments=keep_segments, values=values)


def decode_heavy(seed=1, device="cpu", num_requests=256, kv_lo=512, kv_hi=4096,
                 num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16,
                 keep_segments=False, values=True):
    """Decode rows only (q_len 1), cached length uniform in [kv_lo, kv_hi],
    no sharing, pages scattered over a pool 1.25x the pages needed."""
    rng = np.random.default_rng(seed)
    kv = rng.integers(kv_lo, kv_hi + 1, size=num_requests)
    reqs = [([], int(c), [1]) for c in kv]
    return build_workload("decode_heavy", num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
                          head_dim=head_dim, page_size=page_size, shared_lens=[],
                          requests=reqs, seed=seed + 1000, device=device,
                          keep_segments=keep_segments, values=values)


def radix_sharing(seed=2, device="cpu", groups=8, root=2048, branch=512, pairs=4,
                  tail_lo=64, tail_hi=1024, num_q_heads=32, num_kv_heads=8,
                  head_dim=128, page_size=16, keep_segments=False, values=True):
    """Decode rows in ``groups`` radix subtrees: each subtree has one root
    segment shared by ``2*pairs`` requests and ``pairs`` branch segments each
    shared by two of them, then a private tail uniform in [tail_lo, tail_hi]."""
    rng = np.random.default_rng(seed)
    tails = rng.integers(tail_lo, tail_hi + 1, size=groups * 2 * pairs)
    shared_lens, reqs = [], []
    for g in range(groups):
        rid = len(shared_lens)
        shared_lens.append(root)
        for b in range(pairs):
            bid = len(shared_lens)
            shared_lens.append(branch)
            for m in range(2):
                reqs.append(([rid, bid], int(tails[(g * pairs + b) * 2 + m]), [1]))
    return build_workload("radix_sharing", num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
                          head_dim=head_dim, page_size=page_size, shared_lens=shared_lens,
                          requests=reqs, seed=seed + 1000, device=device,
                          keep_segments=keep_segments, values=values)


def mixed_budget(seed=3, device="cpu", budget=8192, prefill_q=2048, prefill_cached=1024,
                 num_verify=24, verify_lo=4, verify_hi=8, mu=7.0, sigma=1.0,
                 clip_lo=16, clip_hi=16384, num_q_heads=32, num_kv_heads=8,
                 head_dim=128, page_size=16, keep_segments=False, values=True):
    """One prefill chunk, ``num_verify`` speculative-verify rows, and the rest
    of the token budget as decode rows; verify/decode cached lengths are
    round(lognormal(mu, sigma)) clipped to [clip_lo, clip_hi]."""
    rng = np.random.default_rng(seed)
    vq = rng.integers(verify_lo, verify_hi + 1, size=num_verify)
    n_dec = budget - prefill_q - int(vq.sum())
    if n_dec < 0:
        raise ValueError("budget too small")
    cached = np.clip(np.rint(rng.lognormal(mu, sigma, size=num_verify + n_dec)),
                     clip_lo, clip_hi).astype(np.int64)
    reqs = [([], prefill_cached, [prefill_q])]
    reqs += [([], int(cached[i]), [int(vq[i])]) for i in range(num_verify)]
    reqs += [([], int(cached[num_verify + i]), [1]) for i in range(n_dec)]
    return build_workload("mixed_budget", num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
                          head_dim=head_dim, page_size=page_size, shared_lens=[],
                          requests=reqs, seed=seed + 1000, device=device,
                          keep_segments=keep_segments, values=values)


def long_prefill(seed=4, device="cpu", num_requests=4, chunk=8192, num_chunks=4,
                 num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=64,
                 keep_segments=False, values=True):
    """``num_requests`` prompts prefilled as ``num_chunks`` causal chunks of
    ``chunk`` tokens; chunk c attends to every earlier chunk's pages."""
    reqs = [([], 0, [chunk] * num_chunks) for _ in range(num_requests)]
    return build_workload("long_prefill", num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
                          head_dim=head_dim, page_size=page_size, shared_lens=[],
                          requests=reqs, seed=seed + 1000, device=device,
                          keep_segments=keep_segments, values=values)


def chain_parents(n: int) -> np.ndarray:
    """Parents of a linear chain of n draft tokens (token j's parent is j - 1)."""
    return np.arange(-1, n - 1, dtype=np.int32)


def draft_tree(rng: np.random.Generator, n: int) -> np.ndarray:
    """A random draft tree of n tokens in parent-before-child order: token 0
    hangs off the cached context, token j >= 1 picks its parent uniformly
    among tokens 0..j-1 (a random recursive tree: branching near the root,
    depth about ln n, the shape of top-k token trees)."""
    par = np.full(n, -1, dtype=np.int32)
    for j in range(1, n):
        par[j] = rng.integers(0, j)
    return par


def tree_verify(seed=5, device="cpu", num_requests=128, tree_size=64, kv_lo=512, kv_hi=4096,
                num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16,
                keep_segments=False, values=True):
    """Speculative tree verification: every request verifies a ``tree_size``
    token draft tree (``draft_tree``) on top of a cached context of uniform
    length in [kv_lo, kv_hi]; no sharing, scattered pages."""
    rng = np.random.default_rng(seed)
    kv = rng.integers(kv_lo, kv_hi + 1, size=num_requests)
    parents = np.concatenate([draft_tree(rng, tree_size) for _ in range(num_requests)])
    reqs = [([], int(c), [tree_size]) for c in kv]
    wl = build_workload("tree_verify", num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
                        head_dim=head_dim, page_size=page_size, shared_lens=[],
                        requests=reqs, seed=seed + 1000, device=device,
                        keep_segments=keep_segments, values=values)
    wl.steps[0].layout.tree_parent = parents
    return wl


def cache_trace(seed=6, num_prompts=32, prompt_lo=1024, prompt_hi=4096, suffix_lo=32,
                suffix_hi=256, out_lo=16, out_hi=128, num_requests=4096, vocab=32000,
                doc_frac=0.0, doc_lo=2048, doc_hi=8192):
    """A serving trace for the prefix cache: ``num_prompts`` shared system
    prompts (lengths uniform in [prompt_lo, prompt_hi]); each request is one
    of them (uniform) followed by a private user suffix (uniform in
    [suffix_lo, suffix_hi] tokens) and then generates ``out`` tokens (uniform
    in [out_lo, out_hi]), one per decode step.  With probability
    ``doc_frac`` a request also carries a private document (uniform in
    [doc_lo, doc_hi] tokens) between prompt and suffix.  Token ids uniform in
    [0, vocab).  Returns (prompts, requests) with requests a list of
    (prompt index, input token ids, output token ids) as int32 arrays."""
    rng = np.random.default_rng(seed)
    prompts = [rng.integers(0, vocab, size=int(rng.integers(prompt_lo, prompt_hi + 1)))
               .astype(np.int32) for _ in range(num_prompts)]
    reqs = []
    for _ in range(num_requests):
        k = int(rng.integers(num_prompts))
        suffix = rng.integers(0, vocab, size=int(rng.integers(suffix_lo, suffix_hi + 1)))
        out = rng.integers(0, vocab, size=int(rng.integers(out_lo, out_hi + 1)))
        if doc_frac > 0 and rng.random() < doc_frac:
            doc = rng.integers(0, vocab, size=int(rng.integers(doc_lo, doc_hi + 1)))
            suffix = np.concatenate([doc, suffix])
        reqs.append((k, np.concatenate([prompts[k], suffix]).astype(np.int32),
                     out.astype(np.int32)))
    return prompts, reqs


WORKLOADS = {
    "tiny_mixed": tiny_mixed,
    "decode_heavy": decode_heavy,
    "radix_sharing": radix_sharing,
    "mixed_budget": mixed_budget,
    "long_prefill": long_prefill,
    "tree_verify": tree_verify,
}


def make(name, **kw) -> Workload:
    return WORKLOADS[name](**kw)


def sub_workload(wl: Workload, step: int, requests, device="cpu"):
    """Copy the inputs of a subset of requests at one step into a compact
    host workload (pages renumbered densely, new rows and queries sliced).

    The pool pages are taken from ``wl.pool_k``/``pool_v`` as drawn (before
    any step's new rows are appended), plus the new rows of all steps up to
    and including ``step`` so a caller can append them in order.  Used to run
    the oracle on a sample of a workload too large for the host."""
    requests = list(requests)
    pages = []
    for r in requests:
        lay = wl.steps[step].layout
        pages.append(lay.page_indices[lay.page_indptr[r]:lay.page_indptr[r + 1]])
    uniq = np.unique(np.concatenate(pages)) if pages else np.zeros(0, np.int32)
    remap = {int(p): i for i, p in enumerate(uniq)}
    idx = torch.as_tensor(uniq, dtype=torch.long, device=wl.pool_k.device)
    pool_k = wl.pool_k.index_select(0, idx).to(device)
    pool_v = wl.pool_v.index_select(0, idx).to(device)
    steps = []
    for s in range(step + 1):
        lay = wl.steps[s].layout
        q_len = np.array([lay.q_indptr[r + 1] - lay.q_indptr[r] for r in requests], np.int64)
        q_indptr = np.concatenate([[0], np.cumsum(q_len)]).astype(np.int32)
        plists = [np.array([remap[int(p)] for p in
                            lay.page_indices[lay.page_indptr[r]:lay.page_indptr[r + 1]]], np.int32)
                  for r in requests]
        page_indptr = np.concatenate([[0], np.cumsum([len(p) for p in plists])]).astype(np.int32)
        page_indices = (np.concatenate(plists) if plists else np.zeros(0)).astype(np.int32)
        sel = [torch.arange(int(lay.q_indptr[r]), int(lay.q_indptr[r + 1])) for r in requests]
        sel = torch.cat(sel) if sel else torch.zeros(0, dtype=torch.long)
        sel = sel.to(wl.steps[s].q.device)
        tp = None
        if lay.tree_parent is not None:
            tp = np.concatenate([lay.tree_parent[lay.q_indptr[r]:lay.q_indptr[r + 1]]
                                 for r in requests] or [np.zeros(0, np.int32)]).astype(np.int32)
        nl = Layout(lay.num_q_heads, lay.num_kv_heads, lay.head_dim, lay.page_size, len(uniq),
                    q_indptr, lay.cached_len[requests].astype(np.int32),
                    lay.kv_len[requests].astype(np.int32), page_indptr, page_indices, tp)
        steps.append(Step(nl, wl.steps[s].q.index_select(0, sel).to(device),
                          wl.steps[s].k_new.index_select(0, sel).to(device),
                          wl.steps[s].v_new.index_select(0, sel).to(device)))
    return Workload(wl.name + "_sample", pool_k, pool_v, steps)
