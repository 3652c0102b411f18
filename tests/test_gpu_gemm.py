"""GPU: the virtual-padded projection GEMM (pps_gemm_bf16) against the fp64
oracle (oracle.gemm.linear).

Tolerance, from the arithmetic: products of bf16 values are exact in fp32, the
fp32 sum over K adds error far below the output rounding, and the output is
rounded once to bf16 (at most 2^-9 relative).  The test allows
|got - ref| <= 2^-8 |ref| + 1e-3 elementwise.  Shapes cover ragged M (the
virtual padding), N and K tails, tiny and full sizes (sampled rows)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from oracle import gemm as og

pytestmark = pytest.mark.gpu


def _inputs(M, N, K, seed):
    g = torch.Generator().manual_seed(seed)
    a = torch.randn((M, K), generator=g).to(torch.bfloat16)
    w = (torch.randn((N, K), generator=g) / K ** 0.5).to(torch.bfloat16)
    return a, w


def _check(got, ref):
    g = got.double().cpu().numpy()
    assert np.isfinite(g).all()
    err = np.abs(g - ref)
    bound = 2.0 ** -8 * np.abs(ref) + 1e-3
    assert (err <= bound).all(), (float(err.max()), float((err - bound).max()))


@pytest.mark.parametrize("M,N,K", [(1, 8, 8), (127, 256, 64), (128, 256, 128), (129, 264, 72),
                                   (300, 520, 200), (5, 1024, 4096), (4101, 1024, 512),
                                   # around a CTA pair's 256 x 256 tile and its 128-deep K block
                                   (255, 256, 128), (256, 512, 192), (257, 520, 136),
                                   (513, 8, 256), (384, 768, 4224)])
def test_gemm_matches_oracle(pps, M, N, K):
    a, w = _inputs(M, N, K, M + N + K)
    c = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    pps.get_device_error(clear=True)
    pps.gemm_bf16(a.cuda(), w.cuda(), c)
    torch.cuda.synchronize()
    assert pps.get_device_error(clear=True) == 0
    _check(c, og.linear(a, w))


def test_gemm_projection_sizes_sampled_rows(pps):
    """The mixed batch's projections: 8192 + 37 tokens, hidden 4096, QKV 6144
    outputs and O 4096 outputs; 96 sampled rows checked (all columns)."""
    M, K = 8229, 4096
    rng = np.random.default_rng(3)
    rows = np.unique(np.concatenate([rng.choice(M, 94, replace=False), [0, M - 1]]))
    for N in (6144, 4096):
        a, w = _inputs(M, N, K, N)
        c = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        pps.gemm_bf16(a.cuda(), w.cuda(), c)
        torch.cuda.synchronize()
        _check(c[torch.as_tensor(rows, device="cuda")], og.linear(a[rows], w))


def test_gemm_writes_only_real_rows(pps):
    M, N, K = 130, 256, 64
    a, w = _inputs(M, N, K, 9)
    buf = torch.full((M + 126, N), 7.0, dtype=torch.bfloat16, device="cuda")
    pps.gemm_bf16(a.cuda(), w.cuda(), buf[:M])
    torch.cuda.synchronize()
    assert (buf[M:] == 7.0).all()                       # rows past M of the last tile untouched


def test_gemm_argument_checks(pps):
    a = torch.zeros((4, 8), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((12, 8), dtype=torch.bfloat16, device="cuda")
    c = torch.zeros((4, 12), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(pps.PPSError):
        pps.gemm_bf16(a, w, c)                          # N = 12 not a multiple of 8
    pps.gemm_bf16(a[:0], w[:8], c[:0, :8])              # M = 0: nothing to do
