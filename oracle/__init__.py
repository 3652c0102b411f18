"""fp64 CPU oracle for paged, prefix-shared, mixed-batch attention.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
execute this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` use it.  It shares no code with the CUDA
library (no kernels, headers, helpers or tables) and never takes an input or
an expected value from it.

What it computes (``attention.paged_attention``), for every request r, new
token j and query head h (kv head g = h // G, G = Hq / Hkv):

    o[r, j, h] = sum_{p <= c_r + j} softmax_p(scale * q[r, j, h] . k[r, p, g]) v[r, p, g]

with c_r the request's cached length and k[r, p, g] read through the paged
block table.  With a draft tree (``tree_parent``) the new positions a token
sees are restricted to its ancestors and itself.

``radix_cache.RadixCacheOracle`` is the reference for the host prefix cache
that produces those page tables (token-wise reuse with copy-on-write, page
allocation, LRU/LFU eviction); ``tests/test_radix_cache_oracle.py`` pins it.
``scheduler.SchedulerOracle`` is the reference token-wise budget scheduler and
``gemm.linear`` the definition of the projection GEMM; each has its own pins.  Every function is pinned by ``tests/test_oracle_pins.py``
against something other than itself (brute force on unpaged copies, closed
forms, invariances); none is "parity unpinned".
"""
from .attention import (  # noqa: F401
    reference_scatter, gather_request_kv, paged_attention, dense_attention_loops,
    attention_partial, lse_merge, split_kv_attention, tree_ancestors,
)
