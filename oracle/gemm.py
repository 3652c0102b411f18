"""fp64 reference for the virtual-padded projection GEMM (test infrastructure only).

Source: XY-Serve review, "Tackling the Dynamicity in a Production LLM Serving
System ..." (pith.science/paper/ABCKJ6RF), "Core claim": GEMM becomes
SmoothGEMM, which keeps fixed-shape kernel efficiency for arbitrary shapes by
padding virtually in on-chip buffers and reading/writing only real data;
"Assumptions & free parameters": padded entries must not affect the output.

What it computes is the plain definition of a linear layer over a token
batch: C[m, n] = sum_k A[m, k] W[n, k] (A: token rows [M, K], W: weight rows
[N, K], both bf16, taken exactly), in fp64.  Virtual padding changes nothing
in this definition: padded rows or columns are zeros that are never written.
"""
from __future__ import annotations

import numpy as np

from .attention import _f64


def linear(a, w):
    """C = A W^T in fp64 ([M, K] x [N, K] -> [M, N])."""
    return _f64(a) @ _f64(w).T


def linear_loops(a, w):
    """The same sum written as plain loops (tiny sizes only)."""
    a = _f64(a).tolist()
    w = _f64(w).tolist()
    out = []
    for row in a:
        out.append([sum(x * y for x, y in zip(row, wr)) for wr in w])
    return np.array(out, dtype=np.float64).reshape(len(a), len(w))
