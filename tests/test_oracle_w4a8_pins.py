"""Pins for the oracle's W4A8 activation quantisation (CPU only).

In W4A8 mode the FC1 input x~ and the FC2 input z~ are MXFP8: E4M3 codes with
one UE8M0 exponent per 32 consecutive values along the contraction axis
(b12x PR #129 "feat(moe): serve canonical Fruit QSRT atoms", Hot path: the
payload is expanded directly into E4M3 MMA operands and the FC1 input is
quantised to MXFP8; flashinfer PR #69 "b12x fused MoE: TrellisMX ...",
Description and Evidence, precision notes: one UE8M0 byte per 32 values, the
exponent from the exact FP32 bits of amax / 448).

The expected outputs are worked out by hand in ``golden/w4a8_layer_cases.txt``
for a layer whose every weight is the same E4M3 value, so that each output is
a closed form of the quantised x~ and z~. Dropping either quantisation step,
taking the 32-blocks along the token axis, or rounding the block exponent the
other way changes them.
"""
import os

import numpy as np

from oracle import layer as olayer
from trellis_quantized_moe_route_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "w4a8_layer_cases.txt")
E, H, I = 2, 64, 32


def _cases():
    out = {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            head, runs = line.split(":")
            name, k, S, y = head.split()
            vals = []
            for r in runs.split():
                v, n = r.split("*")
                vals += [float(v)] * int(n)
            assert len(vals) == H, name
            out[name] = dict(x=np.asarray(vals), k=int(k), S=float(S), y=float(y))
    return out


def _layer():
    """All-zero K=4 payload (every weight cb(0)), identity rotations, unit
    scales and signs."""
    one = np.uint16(0x3C00)
    words1 = (2 * I // 16) * (H // 16) * 16 * 4
    words2 = (H // 16) * (I // 16) * 16 * 4
    return synth.Layer(
        E=E, H=H, I=I, topk=1, rot_block_h=1, rot_block_i=1,
        bits=np.full(E, 4, dtype=np.uint8),
        fc1_payload=np.zeros(E * words1, dtype=np.int16),
        fc2_payload=np.zeros(E * words2, dtype=np.int16),
        fc1_scale=np.full((E, 2 * I), one, dtype=np.uint16),
        fc2_scale=np.full((E, H), one, dtype=np.uint16),
        in_suh=np.full(H, one, dtype=np.uint16),
        rot_tab=np.full((E, 3 * I), one, dtype=np.uint16),
        out_svh=np.full((E, H), one, dtype=np.uint16),
    )


def _token(c, k=None):
    k = c["k"] if k is None else k
    x = c["x"] * 2.0 ** -k
    bits = synth.bf16_bits(x)
    assert np.array_equal(synth.bf16_to_f64(bits), x), "fixture values must be bf16-exact"
    return bits


def _run(tokens, experts=None, mode="w4a8", act_round=True):
    L = _layer()
    x = np.stack(tokens)
    T = x.shape[0]
    ids = np.zeros((T, 1), dtype=np.int32) if experts is None else np.asarray(experts, dtype=np.int32)[:, None]
    w = np.ones((T, 1), dtype=np.float64)
    return olayer.layer_forward(L, x, ids, w, mode=mode, act_round=act_round)


def test_decoded_weight_is_e4m3_of_cb0():
    L = _layer()
    w1 = olayer.expert_weights(L, 1, 0, "w4a8")
    w2 = olayer.expert_weights(L, 2, 1, "w4a8")
    assert np.all(w1 == 1.875) and np.all(w2 == 1.875)
    assert np.all(olayer.expert_weights(L, 1, 0, "w4a16") == 1.84375)


def test_hand_derived_outputs():
    cases = _cases()
    names = sorted(cases)
    out = _run([_token(cases[n]) for n in names], experts=[i % E for i in range(len(names))])
    for i, n in enumerate(names):
        assert np.all(out[i] == cases[n]["y"]), (n, out[i][:4], cases[n]["y"])


def test_unrounded_form_is_the_plain_closed_form():
    """With the activation rounding switched off, the same layer gives
    y = 1.875 * 32 * g^2 with g = 1.875 * S_raw, S_raw the plain sum of the
    token (every intermediate here is exact in float64); S_raw equals the
    golden S exactly where the token's blocks need no rounding."""
    cases = _cases()
    for n, c in cases.items():
        if c["S"] == 0:
            continue
        S_raw = float(np.sum(c["x"])) * 2.0 ** -c["k"]
        y_raw = _run([_token(c)], act_round=False)[0, 0]
        assert y_raw == 60.0 * (1.875 * S_raw) ** 2
        if n in ("L", "s"):
            assert c["S"] == S_raw      # blocks whose values are E4M3 x 2^e already
        else:
            assert c["S"] != S_raw      # the fixture's x~ rounding is not a no-op


def test_z_step_and_x_step_both_matter():
    c = _cases()["A"]
    y = _run([_token(c)])[0, 0]
    g = 1.875 * c["S"]
    assert y == c["y"]
    assert y != 60.0 * g * g                                   # z~ rounding is applied
    assert g != 1.875 * float(np.sum(c["x"]))                  # x~ rounding is applied
    # X: the rounding of x~ moves the output to another z~ bucket
    x = _cases()["X"]
    assert _run([_token(x)])[0, 0] == x["y"]
    assert _run([_token(x)], act_round=False)[0, 0] != x["y"]


def test_blocks_run_along_the_contraction_axis():
    """32 tokens in one call mixing very large (L), ordinary (s, A at several
    powers of two) and all-zero tokens: each output is its own token's closed
    form. Blocks taken across tokens would put s's 3.0 in a block with L's
    2^20 and flush it to zero."""
    cases = _cases()
    tokens, expect = [], []
    for t in range(32):
        kind = ("L", "s", "A", "Z")[t % 4]
        k = (t // 4) % 5 if kind == "A" else 0
        tokens.append(_token(cases[kind], k=k))
        expect.append(cases[kind]["y"] / 4.0 ** k)
    out = _run(tokens, experts=[t % E for t in range(32)])
    for t in range(32):
        assert np.all(out[t] == expect[t]), (t, out[t][0], expect[t])


def test_perturbation_inside_a_bucket_moves_nothing():
    """A block's largest element moved within its E4M3 bucket (450 -> 452)
    leaves the output unchanged; moved across the power of two (450 -> 900)
    it raises the block exponent and gives the hand-computed output."""
    cases = _cases()
    a, b, c = (_run([_token(cases[n])])[0, 0] for n in "ABC")
    assert a == b == cases["A"]["y"]
    assert c == cases["C"]["y"]
