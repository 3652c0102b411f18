"""The library's batch partition (pps_partition, C++) against the reference
partition in oracle/, on seeded layouts (CPU only)."""
from __future__ import annotations

import numpy as np
import pytest

import workloads
from oracle import partition as op


@pytest.mark.parametrize("parts", [1, 2, 5, 8])
@pytest.mark.parametrize("name,kw", [
    ("radix_sharing", dict(groups=6, root=64, branch=32, pairs=3, tail_lo=1, tail_hi=80)),
    ("mixed_budget", dict(budget=500, prefill_q=100, prefill_cached=40, num_verify=5, mu=4.0,
                          sigma=1.0, clip_lo=1, clip_hi=600)),
    ("decode_heavy", dict(num_requests=50)),
    ("tiny_mixed", dict()),
])
def test_partition_matches_reference(pps, name, kw, parts):
    L = workloads.make(name, values=False, **kw).layout
    want_part, want_load = op.partition(L.q_indptr, L.kv_len, L.page_indptr, L.page_indices,
                                        L.page_size, parts)
    part, load = pps.partition(L.q_indptr, L.kv_len, L.page_indptr, L.page_indices,
                               L.page_size, parts)
    assert part.tolist() == want_part and load.tolist() == want_load


def test_partition_of_the_full_radix_batch_is_balanced(pps):
    L = workloads.radix_sharing(values=False).layout
    part, load = pps.partition(L.q_indptr, L.kv_len, L.page_indptr, L.page_indices,
                               L.page_size, 8)
    assert len(set(part.tolist())) == 8
    assert max(load) / min(load) < 1.5            # 8 subtrees of similar size over 8 GPUs
