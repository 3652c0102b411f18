"""Pins for the projection GEMM's fp64 reference (oracle/gemm.py):
brute-force loops, identity and one-hot weights (closed forms), and the
virtual-padding property the pages state (zero rows/columns added around the
real data change no real output)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from oracle import gemm


def _bf16(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g).to(torch.bfloat16)


@pytest.mark.parametrize("m,n,k", [(1, 1, 1), (3, 5, 7), (13, 8, 64), (0, 4, 8)])
def test_matches_brute_force_loops(m, n, k):
    a, w = _bf16((m, k), 1), _bf16((n, k), 2)
    np.testing.assert_allclose(gemm.linear(a, w), gemm.linear_loops(a, w).reshape(m, n),
                               rtol=0, atol=1e-12)


def test_identity_and_one_hot_weights():
    a = _bf16((9, 16), 3)
    np.testing.assert_array_equal(gemm.linear(a, torch.eye(16).to(torch.bfloat16)),
                                  a.double().numpy())
    w = torch.zeros((4, 16), dtype=torch.bfloat16)
    w[0, 3] = 1
    w[1, 0] = 2
    w[3, 15] = -0.5
    c = gemm.linear(a, w)
    ad = a.double().numpy()
    np.testing.assert_array_equal(c[:, 0], ad[:, 3])
    np.testing.assert_array_equal(c[:, 1], 2 * ad[:, 0])
    np.testing.assert_array_equal(c[:, 2], 0 * ad[:, 0])
    np.testing.assert_array_equal(c[:, 3], -0.5 * ad[:, 15])


def test_padding_changes_no_real_output():
    a, w = _bf16((37, 40), 4), _bf16((24, 40), 5)
    ref = gemm.linear(a, w)
    ap = torch.zeros((128, 64), dtype=torch.bfloat16)
    ap[:37, :40] = a
    wp = torch.zeros((256, 64), dtype=torch.bfloat16)
    wp[:24, :40] = w
    got = gemm.linear(ap, wp)
    np.testing.assert_allclose(got[:37, :24], ref, rtol=0, atol=1e-12)
    assert not got[37:].any() and not got[:, 24:].any()


MUTATIONS = {
    "transposed_weight": ("return _f64(a) @ _f64(w).T", "return _f64(a) @ _f64(w)[:, ::-1].T"),
    "dropped_last_k": ("return _f64(a) @ _f64(w).T", "return _f64(a)[:, :-1] @ _f64(w)[:, :-1].T"),
}


@pytest.mark.parametrize("name", list(MUTATIONS))
def test_planted_mistake_is_caught(name):
    import os
    import types
    src_path = os.path.join(os.path.dirname(gemm.__file__), "gemm.py")
    src = open(src_path).read()
    old, new = MUTATIONS[name]
    assert src.count(old) == 1
    mod = types.ModuleType("gemm_mutant")
    mod.__dict__["__package__"] = "oracle"
    exec(compile(src.replace(old, new), src_path, "exec"), mod.__dict__)
    a, w = _bf16((5, 8), 6), _bf16((3, 8), 7)
    assert not np.allclose(mod.linear(a, w), gemm.linear_loops(a, w), rtol=0, atol=1e-12)
