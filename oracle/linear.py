"""Dense trellis-coded linear layer in float64 (oracle; test use only).

The same bitshift-trellis weights, scales and Hadamard-and-sign rotations as
one projection of the MoE layer, with no routing: the dense trellis path of
sparkinfer PR #90 "moe: integrate EXL3 Trellis into the fused W4A16 API"
(review of kernel.py: run_trellis256_dense converts the input to fp16,
rotates it, runs the fp16 GEMM and rotates the output; review of
tests/gemm/test_trellis_linear.py). For W~ [N, K], scale s [N], input signs
suh [K] and output signs svh [N]:

  1. x~ = Hblk_in(suh (.) x), rounded to fp16 (the contraction operand)
  2. y  = s (.) (W~ x~)
  3. out = svh (.) Hblk_out(y)

Readings: the pages keep an fp16 GEMM output buffer; here y stays float64
(the CUDA path keeps it in fp32) and out is returned in float64. The input
signs are a vector over K, the output signs over N, as for the layer's FC2.
"""
from __future__ import annotations

import numpy as np

from . import hadamard, trellis
from .layer import bf16_to_f64, fp16_to_f64


def linear_weights(lin) -> np.ndarray:
    """Dense float64 W~ [N, K] decoded from the tiles."""
    tiles = np.asarray(lin.payload, dtype=np.int16).reshape(lin.N // 16, lin.K // 16, 16 * lin.bits)
    return trellis.decode_matrix(tiles, int(lin.bits)).astype(np.float64)


def linear_apply(lin, x: np.ndarray, act_round: bool = True, w: np.ndarray = None) -> np.ndarray:
    """Steps 1-3 on float64 inputs x [T, K]; returns float64 [T, N]."""
    w = linear_weights(lin) if w is None else w
    xt = hadamard.rotate(x * fp16_to_f64(lin.suh)[None, :], lin.rot_in)
    if act_round:
        xt = xt.astype(np.float16).astype(np.float64)
    y = (xt @ w.T) * fp16_to_f64(lin.scale)[None, :]
    return hadamard.rotate(y, lin.rot_out) * fp16_to_f64(lin.svh)[None, :]


def linear_forward(lin, x_bits: np.ndarray, act_round: bool = True) -> np.ndarray:
    """The layer on bf16 activations [T, K] (bit patterns)."""
    return linear_apply(lin, bf16_to_f64(x_bits), act_round)
