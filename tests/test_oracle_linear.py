"""Pins for the oracle's dense trellis linear layer (CPU only)."""
import dataclasses

import numpy as np
import pytest

from oracle import hadamard, linear as olinear, trellis
from trellis_quantized_moe_route_gb300 import synth


def _ones_fp16(n):
    return np.full(n, 0x3C00, dtype=np.uint16)


@pytest.mark.parametrize("bits", [2, 4, 6])
def test_identity_rotations_equal_scalar_decoded_matmul(bits):
    """Rotation blocks 1, unit scales and signs: the layer is x @ W~^T, with W~
    built weight by weight from the scalar state and codebook definitions
    (weight j of tile (tn, tk) at row 16 tn + j / 16, column 16 tk + j % 16)."""
    lin = synth.make_linear(32, 48, bits=bits, rot_in=1, rot_out=1, seed=8)
    lin = dataclasses.replace(lin, scale=_ones_fp16(32), suh=_ones_fp16(48), svh=_ones_fp16(32))
    tiles = np.asarray(lin.payload, dtype=np.int16).reshape(2, 3, 16 * bits)
    w = np.zeros((32, 48))
    for tn in range(2):
        for tk in range(3):
            states = trellis.tile_states_scalar(tiles[tn, tk], bits)
            for j in range(256):
                w[16 * tn + j // 16, 16 * tk + j % 16] = trellis.codebook_scalar(states[j])
    x = synth.make_linear_tokens(lin, 3, seed=2)
    xv = synth.bf16_to_f64(x)
    out = olinear.linear_forward(lin, x, act_round=False)
    np.testing.assert_allclose(out, xv @ w.T, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("rot_in,rot_out", [(128, 128), (64, 128), (128, 64), (1, 64)])
def test_streaming_form_equals_reconstructed_dense_matrix(rot_in, rot_out):
    """out = x @ M^T with M = D_svh Hblk_out^T diag(s) W~ Hblk_in D_suh built
    as explicit matrices (the Sylvester blocks are symmetric); N != K so a
    transposed operand cannot pass."""
    N, K = 256, 384
    lin = synth.make_linear(N, K, bits=3, rot_in=rot_in, rot_out=rot_out, seed=11)
    w = olinear.linear_weights(lin)

    def blockdiag(n, b):
        m = np.zeros((n, n))
        r = hadamard.rotation_matrix(b)
        for i in range(0, n, b):
            m[i:i + b, i:i + b] = r
        return m

    f16 = lambda u: np.asarray(u, dtype=np.uint16).view(np.float16).astype(np.float64)
    m = np.diag(f16(lin.svh)) @ blockdiag(N, rot_out) @ np.diag(f16(lin.scale)) @ w @ blockdiag(K, rot_in) @ np.diag(f16(lin.suh))
    xv = synth.bf16_to_f64(synth.make_linear_tokens(lin, 6, seed=3))
    got = olinear.linear_apply(lin, xv, act_round=False, w=w)
    ref = xv @ m.T
    assert np.max(np.abs(got - ref)) <= 1e-12 * np.max(np.abs(ref))


def test_fp16_operand_rounding_is_the_only_rounding():
    """With fp16-exact rotated inputs the rounded and unrounded forms agree
    exactly, and otherwise they differ by at most the fp16 rounding of x~
    propagated through the (norm-preserving) rotations."""
    lin = synth.make_linear(128, 128, bits=4, rot_in=128, rot_out=128, seed=4)
    w = olinear.linear_weights(lin)
    xv = synth.bf16_to_f64(synth.make_linear_tokens(lin, 4, seed=9))
    a = olinear.linear_apply(lin, xv, act_round=True, w=w)
    b = olinear.linear_apply(lin, xv, act_round=False, w=w)
    xt = hadamard.rotate(xv * lin.suh.view(np.float16).astype(np.float64)[None, :], 128)
    dx = np.abs(xt.astype(np.float16).astype(np.float64) - xt)
    bound = np.linalg.norm(dx, axis=1) * np.linalg.norm(w, 2) * 0.03 + 1e-15
    assert np.all(np.linalg.norm(a - b, axis=1) <= bound)
    assert np.any(a != b)
