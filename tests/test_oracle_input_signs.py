"""Pins for the oracle's separate gate / up input sign layouts (CPU only):
gate_suh and up_suh of one row (shared by the experts) or one row per
expert, as the pages' preparation accepts."""
import dataclasses

import numpy as np
import pytest

from oracle import hadamard, layer as olayer, route
from trellis_quantized_moe_route_gb300 import synth


def _cfg(**kw):
    base = dict(name="s", E=4, H=128, I=64, topk=2, T=6, bits=(3, 4), rot_block_h=64, rot_block_i=32,
                mode="w4a16", logits="normal", seed=13)
    base.update(kw)
    return synth.LayerConfig(**base)


@pytest.mark.parametrize("rows", [1, 4])
@pytest.mark.parametrize("mode", ["w4a16", "w4a8"])
def test_equal_signs_reproduce_the_shared_layout_bitwise(rows, mode):
    """gate_suh = up_suh = in_suh (one row, or the same row per expert) is the
    shared layout: same float64 result bit for bit (rotation and operand
    rounding act row by row)."""
    cfg = _cfg()
    L = synth.make_layer(cfg)
    x, lg = synth.make_tokens(cfg)
    ids, w = route.route_topk_softmax(lg, cfg.topk)
    ref = olayer.layer_forward(L, x, ids, w, mode=mode)
    s = np.tile(L.in_suh[None, :], (rows, 1))
    got = olayer.layer_forward(dataclasses.replace(L, gate_suh=s, up_suh=s.copy()), x, ids, w, mode=mode)
    assert np.array_equal(got, ref)


def _blockdiag(n, b):
    m = np.zeros((n, n))
    r = hadamard.rotation_matrix(b)
    for i in range(0, n, b):
        m[i:i + b, i:i + b] = r
    return m


@pytest.mark.parametrize("rows", [1, 4])
def test_streaming_form_equals_dense_matrices_per_expert(rows):
    """With distinct random gate and up signs, the oracle's streaming form
    (rotations applied blockwise, one x~ per route) equals the layer built
    from explicit matrices per expert: gate rows see
    diag(s1g) W1g Hblk_H diag(gsuh_e), up rows diag(s1u) W1u Hblk_H diag(usuh_e).
    A gate/up swap, a shared row used for all experts or the wrong expert's
    row changes the result far beyond the tolerance."""
    cfg = _cfg()
    L = synth.with_input_signs(synth.make_layer(cfg), rows, seed=5)
    assert not np.array_equal(L.gate_suh, L.up_suh)
    x, lg = synth.make_tokens(cfg)
    ids, w = route.route_topk_softmax(lg, cfg.topk)
    got = olayer.layer_forward(L, x, ids, w, mode="w4a16", act_round=False)

    f16 = lambda u: np.asarray(u, dtype=np.uint16).view(np.float16).astype(np.float64)
    H, I = cfg.H, cfg.I
    HH, HI = _blockdiag(H, cfg.rot_block_h), _blockdiag(I, cfg.rot_block_i)
    xv = synth.bf16_to_f64(x)
    out = np.zeros((cfg.T, H))
    for t in range(cfg.T):
        for j in range(cfg.topk):
            e = int(ids[t, j])
            w1 = olayer.expert_weights(L, 1, e)
            w2 = olayer.expert_weights(L, 2, e)
            s1, s2 = f16(L.fc1_scale[e]), f16(L.fc2_scale[e])
            rot = f16(L.rot_tab[e])
            r = e if rows > 1 else 0
            a_g = np.diag(s1[:I]) @ w1[:I] @ HH @ np.diag(f16(L.gate_suh[r]))
            a_u = np.diag(s1[I:]) @ w1[I:] @ HH @ np.diag(f16(L.up_suh[r]))
            g = np.diag(rot[:I]) @ HI @ a_g @ xv[t]
            u = np.diag(rot[I:2 * I]) @ HI @ a_u @ xv[t]
            z = HI @ np.diag(rot[2 * I:]) @ (g / (1.0 + np.exp(-g)) * u)
            y = np.diag(f16(L.out_svh[e])) @ HH @ np.diag(s2) @ w2 @ z
            out[t] += w[t, j] * y
    assert np.max(np.abs(got - out)) <= 1e-12 * np.max(np.abs(out))
