"""Pins for the oracle's whole-layer forward (CPU only)."""
import dataclasses

import numpy as np
import pytest

from oracle import hadamard, layer as olayer, mxfp8, route, trellis
from trellis_quantized_moe_route_gb300 import synth

TINY = synth.CONFIGS["tiny"]


def _small_cfg(**kw):
    base = dict(name="t", E=6, H=128, I=64, topk=2, T=5, bits=(2, 3, 4),
                rot_block_h=64, rot_block_i=32, mode="w4a16", logits="normal", seed=21)
    base.update(kw)
    return synth.LayerConfig(**base)


def _ones_fp16(shape):
    return np.full(shape, 0x3C00, dtype=np.uint16)


def test_identity_rotation_top1_equals_dense_swiglu():
    """Rotation blocks 1, all signs +1, top-1 with weight 1: the layer is the
    plain SwiGLU FFN  s2 * W2 (SiLU(s1g * W1g x) * (s1u * W1u x))."""
    cfg = _small_cfg(rot_block_h=1, rot_block_i=1, topk=1)
    L = synth.make_layer(cfg)
    L.in_suh = _ones_fp16(L.in_suh.shape)
    L.rot_tab = _ones_fp16(L.rot_tab.shape)
    L.out_svh = _ones_fp16(L.out_svh.shape)
    x, lg = synth.make_tokens(cfg)
    ids, _ = route.route_topk_softmax(lg, 1)
    w = np.ones((cfg.T, 1))
    out = olayer.layer_forward(L, x, ids, w, act_round=False)
    xv = synth.bf16_to_f64(x)
    I = cfg.I
    for t in range(cfg.T):
        e = int(ids[t, 0])
        w1 = trellis.decode_matrix(trellis.expert_payload(L.fc1_payload, 2 * I, cfg.H, L.bits, e), int(L.bits[e])).astype(np.float64)
        w2 = trellis.decode_matrix(trellis.expert_payload(L.fc2_payload, cfg.H, I, L.bits, e), int(L.bits[e])).astype(np.float64)
        s1 = L.fc1_scale[e].view(np.float16).astype(np.float64)
        s2 = L.fc2_scale[e].view(np.float16).astype(np.float64)
        gate = s1[:I] * (w1[:I] @ xv[t])
        up = s1[I:] * (w1[I:] @ xv[t])
        silu = gate / (1.0 + np.exp(-gate))
        ref = s2 * (w2 @ (silu * up))
        assert np.allclose(out[t], ref, rtol=1e-12, atol=1e-12)


def _block_diag(n, b):
    if b == 1:
        return np.eye(n)
    return np.kron(np.eye(n // b), hadamard.sylvester(b) / np.sqrt(b))


@pytest.mark.parametrize("mode", ["w4a16"])
def test_streaming_equals_reconstructed_dense(mode):
    """The streaming form equals a dense FFN with W = D(svh) H D(s) W~ H D(suh)
    built from explicit full-size block-diagonal matrices."""
    cfg = _small_cfg()
    L = synth.make_layer(cfg)
    x, lg = synth.make_tokens(cfg)
    ids, w = route.route_topk_softmax(lg, cfg.topk)
    out = olayer.layer_forward(L, x, ids, w, mode=mode, act_round=False)
    H, I = cfg.H, cfg.I
    HH = _block_diag(H, cfg.rot_block_h)
    HI = _block_diag(I, cfg.rot_block_i)
    D = lambda v: np.diag(v.view(np.float16).astype(np.float64))
    suh = D(L.in_suh)
    xv = synth.bf16_to_f64(x)
    ref = np.zeros((cfg.T, H))
    for t in range(cfg.T):
        for j in range(cfg.topk):
            e = int(ids[t, j])
            w1 = olayer.expert_weights(L, 1, e)
            w2 = olayer.expert_weights(L, 2, e)
            s1 = L.fc1_scale[e]
            s2 = L.fc2_scale[e]
            rot = L.rot_tab[e]
            Wg = D(rot[:I]) @ HI @ D(s1[:I]) @ w1[:I] @ HH @ suh
            Wu = D(rot[I:2 * I]) @ HI @ D(s1[I:]) @ w1[I:] @ HH @ suh
            Wd = D(L.out_svh[e]) @ HH @ D(s2) @ w2 @ HI @ D(rot[2 * I:])
            g, u = Wg @ xv[t], Wu @ xv[t]
            ref[t] += w[t, j] * (Wd @ (g / (1 + np.exp(-g)) * u))
    scale = np.abs(ref).max()
    assert np.abs(out - ref).max() <= 1e-12 * scale


@pytest.mark.parametrize("mode", ["w4a16", "w4a8"])
def test_token_permutation_equivariance_bitwise(mode):
    cfg = _small_cfg(T=7)
    L = synth.make_layer(cfg)
    x, lg = synth.make_tokens(cfg)
    ids, w = route.route_topk_softmax(lg, cfg.topk)
    out = olayer.layer_forward(L, x, ids, w, mode=mode)
    perm = synth.permutation(synth.Stream(5, 5), cfg.T)
    out_p = olayer.layer_forward(L, x[perm], ids[perm], w[perm], mode=mode)
    assert np.array_equal(out_p, out[perm])


def test_route_weights_are_linear_and_zero_weight_drops_expert():
    cfg = _small_cfg()
    L = synth.make_layer(cfg)
    x, lg = synth.make_tokens(cfg)
    ids, w = route.route_topk_softmax(lg, cfg.topk)
    out = olayer.layer_forward(L, x, ids, w)
    w2 = w.copy()
    w2[:, 1] = 0.0
    out0 = olayer.layer_forward(L, x, ids, w2)
    out1 = olayer.layer_forward(L, x, ids[:, :1], w[:, :1])
    assert np.allclose(out0, out1, rtol=1e-13, atol=1e-13)
    assert np.allclose(olayer.layer_forward(L, x, ids, 2 * w), 2 * out, rtol=1e-13, atol=1e-13)


def test_token_subset_matches_full_batch():
    cfg = _small_cfg(T=6)
    L = synth.make_layer(cfg)
    x, lg = synth.make_tokens(cfg)
    ids, w = route.route_topk_softmax(lg, cfg.topk)
    full = olayer.layer_forward(L, x, ids, w)
    sub = olayer.layer_forward(L, x, ids, w, tokens=[4, 1])
    assert np.allclose(sub, full[[4, 1]], rtol=1e-13, atol=1e-13)


def test_w4a8_close_to_unquantised_and_uses_e4m3_weights():
    cfg = _small_cfg(T=6)
    L = synth.make_layer(cfg)
    x, lg = synth.make_tokens(cfg)
    ids, w = route.route_topk_softmax(lg, cfg.topk)
    exact = olayer.layer_forward(L, x, ids, w, mode="w4a16", act_round=False)
    q8 = olayer.layer_forward(L, x, ids, w, mode="w4a8")
    q16 = olayer.layer_forward(L, x, ids, w, mode="w4a16")
    rms = np.sqrt((exact ** 2).mean(axis=1, keepdims=True))
    err8 = np.abs(q8 - exact) / rms
    err16 = np.abs(q16 - exact) / rms
    assert 1e-3 < err8.max() < 0.25       # E4M3 carries 3 mantissa bits
    assert err16.max() < 5e-3             # fp16 operands only
    # every W4A8 weight is an E4M3 value
    w1 = olayer.expert_weights(L, 1, 0, "w4a8")
    assert np.array_equal(mxfp8.e4m3_round(w1), w1)
    # the all-zero stream decodes to cb(0) = 1.84375 -> E4M3 1.875 (code 0x3F)
    assert mxfp8.e4m3_encode(np.array([1.84375]))[0] == 0x3F


def test_tiny_config_end_to_end_is_finite_and_scaled():
    L = synth.make_layer(TINY)
    x, lg = synth.make_tokens(TINY)
    ids, w = route.route_topk_softmax(lg, TINY.topk)
    out = olayer.layer_forward(L, x, ids, w)
    assert out.shape == (TINY.T, TINY.H) and np.all(np.isfinite(out))
    assert 1e-4 < np.sqrt((out ** 2).mean()) < 10.0
