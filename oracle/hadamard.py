"""Blockwise Hadamard rotation with explicit matrices (oracle; test use only).

The pages rotate activations blockwise with a Walsh-Hadamard transform and sign
vectors: a 128-point transform scaled by 0.088388347648 = 1/sqrt(128)
(sparkinfer PR #90 "moe: integrate EXL3 Trellis into the fused W4A16 API",
review of kernel.py: _had128_quad), applied as H -> svh -> activation -> suh ->
H in the FC1 epilogue and undone after FC2 (same review: _run_activation and
W4A16TopKSumKernel must apply the same H128). Block sizes other than 128 (64
for the intermediate axis of the odd-geometry layer; 1 = identity) come from
the workload definitions.

Reading: H_b is the Sylvester-ordered Hadamard matrix H[i][j] =
(-1)^popcount(i & j), scaled by 1/sqrt(b), built here as an explicit b x b
matrix and applied to consecutive blocks of b entries. It is symmetric and
orthogonal, so the same matrix undoes itself.
"""
from __future__ import annotations

import numpy as np


def sylvester(n: int) -> np.ndarray:
    """Unnormalised Hadamard matrix of order n (a power of two), float64."""
    assert n >= 1 and (n & (n - 1)) == 0, n
    i = np.arange(n)[:, None]
    j = np.arange(n)[None, :]
    parity = np.zeros((n, n), dtype=np.int64)
    v = i & j
    while np.any(v):
        parity ^= v & 1
        v = v >> 1
    return np.where(parity == 1, -1.0, 1.0)


def rotation_matrix(b: int) -> np.ndarray:
    """H_b / sqrt(b)."""
    return sylvester(b) / np.sqrt(float(b))


def rotate(x: np.ndarray, b: int) -> np.ndarray:
    """Apply H_b/sqrt(b) to every consecutive block of b entries of the last axis."""
    x = np.asarray(x, dtype=np.float64)
    if b == 1:
        return x.copy()
    n = x.shape[-1]
    assert n % b == 0, (n, b)
    m = rotation_matrix(b)
    blocks = x.reshape(*x.shape[:-1], n // b, b)
    return (blocks @ m.T).reshape(x.shape)
