"""Pins for the oracle's TrellisMX-style layer (CPU only): E4M3 trellis
weights with one UE8M0 scale per 32 weights along the contraction axis, and
the 512-point hidden-side rotation (flashinfer PR #69 "b12x fused MoE:
TrellisMX (procedural NPK) source format with an in-tree P8 runtime",
Description: K2 to K4 trellis streams decoded to E4M3 inside the MMA, one
UE8M0 scale per 32 weights, a coupled H512/H128 boundary)."""
import dataclasses

import numpy as np
import pytest

from oracle import hadamard, layer as olayer, mxfp8, route
from trellis_quantized_moe_route_gb300 import synth


def _mx_cfg(**kw):
    base = dict(name="mx", E=4, H=512, I=64, topk=2, T=5, bits=(2, 3, 4), rot_block_h=512, rot_block_i=64,
                mode="w4a8", logits="normal", seed=23, mx=True)
    base.update(kw)
    return synth.LayerConfig(**base)


def test_hand_built_scales_on_the_all_zero_stream():
    """An all-zero payload decodes every weight to cb(0) = 1.84375, whose E4M3
    rounding is 1.875; a scale byte u makes the block's 32 weights exactly
    1.875 * 2^(u - 127): u = 125 -> 0.46875, 127 -> 1.875, 130 -> 15."""
    cfg = _mx_cfg(E=1, H=64, I=32, topk=1, bits=(4,), rot_block_h=1, rot_block_i=1)
    L = synth.make_layer(cfg)
    L = dataclasses.replace(L, fc1_payload=np.zeros_like(L.fc1_payload), fc2_payload=np.zeros_like(L.fc2_payload))
    u1 = np.full((1, 64, 2), 127, dtype=np.uint8)
    u1[0, 3, 0] = 125
    u1[0, 40, 1] = 130
    u2 = np.full((1, 64, 1), 126, dtype=np.uint8)
    L = dataclasses.replace(L, fc1_wscale=u1, fc2_wscale=u2)
    for mode in ("w4a16", "w4a8"):
        w1 = olayer.expert_weights(L, 1, 0, mode)
        want = np.full((64, 64), 1.875)
        want[3, :32] = 0.46875
        want[40, 32:] = 15.0
        assert np.array_equal(w1, want)
        assert np.array_equal(olayer.expert_weights(L, 2, 0, mode), np.full((64, 32), 0.9375))


def test_scale_byte_moves_exactly_its_block():
    cfg = _mx_cfg()
    L = synth.make_layer(cfg)
    base = olayer.expert_weights(L, 1, 2)
    u = L.fc1_wscale.copy()
    u[2, 17, 5] += 1
    w = olayer.expert_weights(dataclasses.replace(L, fc1_wscale=u), 1, 2)
    changed = np.zeros_like(base, dtype=bool)
    changed[17, 160:192] = True
    assert np.array_equal(w[changed], 2.0 * base[changed])
    assert np.array_equal(w[~changed], base[~changed])


def test_mx_weights_are_e4m3_times_power_of_two_in_both_modes():
    cfg = _mx_cfg()
    L = synth.make_layer(cfg)
    plain = dataclasses.replace(L, fc1_wscale=None, fc2_wscale=None)
    for e in range(cfg.E):
        q = olayer.expert_weights(plain, 1, e, "w4a8")          # E4M3 of the codebook values
        u = L.fc1_wscale[e].astype(np.int64) - 127
        want = q * np.exp2(np.repeat(u, 32, axis=1))
        assert np.array_equal(olayer.expert_weights(L, 1, e, "w4a16"), want)
        assert np.array_equal(olayer.expert_weights(L, 1, e, "w4a8"), want)


def test_512_rotation_is_h4_across_h128_blocks():
    """Sylvester order: H_512 = H_4 (x) H_128, i.e. a 128-point transform of
    each quarter followed by a 4-point transform across the quarters (the
    coupled boundary), scaled 1/sqrt(512)."""
    x = synth.Stream(3, 3).normal(3 * 1024).reshape(3, 1024)
    got = hadamard.rotate(x, 512)
    blocks = x.reshape(3, 2, 4, 128)
    inner = blocks @ hadamard.sylvester(128).T                   # H128 on each quarter
    outer = np.einsum("ij,bqjk->bqik", hadamard.sylvester(4), inner)  # H4 across the quarters
    want = outer.reshape(3, 1024) / np.sqrt(512.0)
    assert np.allclose(got, want, rtol=1e-13, atol=1e-13)
    assert np.allclose(hadamard.rotate(got, 512), x, rtol=1e-13, atol=1e-13)


def _block_diag(n, b):
    return np.eye(n) if b == 1 else np.kron(np.eye(n // b), hadamard.sylvester(b) / np.sqrt(b))


@pytest.mark.parametrize("mode", ["w4a16", "w4a8"])
def test_streaming_equals_dense_with_512_blocks_and_scales(mode):
    """The layer with 512-point hidden rotations and MX weights equals the
    dense FFN built from explicit full-size block-diagonal matrices and the
    scaled E4M3 weights (activation rounding off)."""
    cfg = _mx_cfg(mode=mode)
    L = synth.make_layer(cfg)
    x, lg = synth.make_tokens(cfg)
    ids, w = route.route_topk_softmax(lg, cfg.topk)
    out = olayer.layer_forward(L, x, ids, w, mode=mode, act_round=False)
    H, I = cfg.H, cfg.I
    HH, HI = _block_diag(H, 512), _block_diag(I, cfg.rot_block_i)
    D = lambda v: np.diag(v.view(np.float16).astype(np.float64))
    xv = synth.bf16_to_f64(x)
    ref = np.zeros((cfg.T, H))
    for t in range(cfg.T):
        for j in range(cfg.topk):
            e = int(ids[t, j])
            w1, w2 = olayer.expert_weights(L, 1, e, mode), olayer.expert_weights(L, 2, e, mode)
            s1, s2, rot = L.fc1_scale[e], L.fc2_scale[e], L.rot_tab[e]
            Wg = D(rot[:I]) @ HI @ D(s1[:I]) @ w1[:I] @ HH @ D(L.in_suh)
            Wu = D(rot[I:2 * I]) @ HI @ D(s1[I:]) @ w1[I:] @ HH @ D(L.in_suh)
            Wd = D(L.out_svh[e]) @ HH @ D(s2) @ w2 @ HI @ D(rot[2 * I:])
            g, u = Wg @ xv[t], Wu @ xv[t]
            ref[t] += w[t, j] * (Wd @ (g / (1 + np.exp(-g)) * u))
    assert np.abs(out - ref).max() <= 1e-12 * np.abs(ref).max()


def test_trellismx_workload_shapes():
    cfg = synth.CONFIGS["trellismx"]
    L = synth.make_layer(cfg)
    assert cfg.rot_block_h == 512 and set(np.unique(L.bits)) <= {2, 3, 4}
    assert L.fc1_wscale.shape == (cfg.E, 2 * cfg.I, cfg.H // 32)
    assert L.fc2_wscale.shape == (cfg.E, cfg.H, cfg.I // 32)
    assert 124 <= L.fc1_wscale.min() and L.fc1_wscale.max() <= 130
