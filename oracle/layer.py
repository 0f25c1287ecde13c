"""The trellis-coded MoE layer in float64 (oracle; test use only).

Steps, in the order the pages give them (b12x PR #129 "feat(moe): serve
canonical Fruit QSRT atoms", Hot path; sparkinfer PR #90 "moe: integrate EXL3
Trellis into the fused W4A16 API", review of kernel.py: _run_activation,
W4A16TopKSumKernel; review of trellis_w4a8.py on page #129: down_svh applied in
the top-k sum):

  1. x~ = Hblk_H(suh (.) x)                        input rotation
  2. y1 = s1 (.) (W1~ x~)          per route        FC1, gate rows 0..I-1, up rows I..2I-1
     (with separate gate / up input signs, shared or per expert, the gate
     rows see x~_g = Hblk_H(gate_suh_e (.) x) and the up rows x~_u)
  3. g = svh_g (.) Hblk_I(y1_gate), u = svh_u (.) Hblk_I(y1_up)
     a = SiLU(g) * u,  z~ = Hblk_I(suh_d (.) a)     activation epilogue
  4. y2 = s2 (.) (W2~ z~)                           FC2
  5. y_t = sum_j w_{t,j} * (svh_d (.) Hblk_H(y2_{t,j}))   unrotate + top-k combine

TrellisMX-style weights (a layer with UE8M0 weight scales; see
expert_weights) keep the same steps; their hidden-side rotation blocks may be
512 wide (H4 (x) H128 in Sylvester order, the "coupled H512/H128 boundary").

Modes:
  * "w4a16": weights are the fp16 codebook values; x~ and z~ are rounded to
    fp16 (the operands of an FP16 x FP16 -> FP32 contraction). Reading: the
    pages run full rotation in fp16 (sparkinfer PR #90, review of host.py:
    fp16 intermediate caches under full rotation).
  * "w4a8": weights are rounded to E4M3; x~ and z~ are rounded to fp32 and
    quantised to MXFP8 along the contraction axis (b12x PR #129, Hot path: W4A8
    expands the payload directly into E4M3 MMA operands and the FC1 input is
    quantised to MXFP8).
  * ``act_round=False`` skips the activation rounding of either mode.

Everything else is float64 with numpy's matmul as the contraction primitive.
"""
from __future__ import annotations

import numpy as np

from . import hadamard, mxfp8, trellis


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def fp16_to_f64(bits: np.ndarray) -> np.ndarray:
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def weight_scales(layer, proj: int, e: int):
    """The UE8M0 weight scale bytes of expert e's projection ([rows, cols/32]),
    or None for a layer without them (TrellisMX-style weights only)."""
    ws = getattr(layer, "fc1_wscale" if proj == 1 else "fc2_wscale", None)
    return None if ws is None else np.asarray(ws)[e]


def expert_weights(layer, proj: int, e: int, mode: str = "w4a16") -> np.ndarray:
    """Dense float64 weights of expert e: proj 1 -> [2I, H], proj 2 -> [H, I].

    Plain trellis weights are the fp16 codebook values (W4A16), rounded to
    E4M3 in W4A8. TrellisMX-style weights (the layer carries fc1_wscale /
    fc2_wscale) decode to E4M3 in both modes and carry one UE8M0 scale per
    32 consecutive weights of a row along the contraction axis (flashinfer PR
    #69 "b12x fused MoE: TrellisMX ...", Description: trellis streams of K2
    to K4 bits that decode to E4M3, one UE8M0 scale per 32 weights):
    w = E4M3(cb(s)) * 2^(u - 127)."""
    rows, cols = (2 * layer.I, layer.H) if proj == 1 else (layer.H, layer.I)
    payload = layer.fc1_payload if proj == 1 else layer.fc2_payload
    tiles = trellis.expert_payload(payload, rows, cols, layer.bits, e)
    w = trellis.decode_matrix(tiles, int(layer.bits[e])).astype(np.float64)
    u = weight_scales(layer, proj, e)
    if mode == "w4a8" or u is not None:
        w = mxfp8.e4m3_round(w)
    if u is not None:
        u = np.asarray(u, dtype=np.int64).reshape(rows, cols // 32)
        w = w * np.exp2(np.repeat(u - 127, 32, axis=1).astype(np.float64))
    return w


def rotate_input(layer, x_bits: np.ndarray, suh: np.ndarray = None) -> np.ndarray:
    """Step 1 in float64: [T, H] (suh: fp16 bits [H], default the shared in_suh)."""
    x = bf16_to_f64(x_bits)
    suh = layer.in_suh if suh is None else suh
    return hadamard.rotate(x * fp16_to_f64(suh)[None, :], layer.rot_block_h)


def input_signs(layer, e: int):
    """The (gate, up) input sign vectors of expert e (fp16 bits [H] each):
    the separate gate_suh / up_suh rows when the layer has them (one row
    shared by the experts, or one per expert; b12x PR #129, review of
    trellis_w4a8.py: gate_suh and up_suh of shape (1, H) or (num_experts, H)),
    else the shared in_suh for both."""
    g = getattr(layer, "gate_suh", None)
    u = getattr(layer, "up_suh", None)
    if g is None and u is None:
        return layer.in_suh, layer.in_suh
    g = np.asarray(g).reshape(-1, layer.H)
    u = np.asarray(u).reshape(-1, layer.H)
    return g[e if g.shape[0] > 1 else 0], u[e if u.shape[0] > 1 else 0]


def round_operand(v: np.ndarray, mode: str, act_round: bool = True) -> np.ndarray:
    """Activation operand rounding of the mode (fp16, or fp32 -> MXFP8)."""
    if not act_round:
        return v
    if mode == "w4a16":
        return v.astype(np.float16).astype(np.float64)
    return mxfp8.quantize_mxfp8(v.astype(np.float32))[2]


def expert_ffn(layer, e: int, xq: np.ndarray, mode: str, act_round: bool = True,
               w1: np.ndarray = None, w2: np.ndarray = None, xq_up: np.ndarray = None) -> np.ndarray:
    """Steps 2-5 (before the route weight) for the rows xq [n, H] routed to e
    (xq_up: the up rows' own operand when the gate and up input signs
    differ; default xq). Returns svh_d (.) Hblk_H(y2) as [n, H]."""
    I = layer.I
    if w1 is None:
        w1 = expert_weights(layer, 1, e, mode)
    if w2 is None:
        w2 = expert_weights(layer, 2, e, mode)
    s1 = fp16_to_f64(layer.fc1_scale[e])
    s2 = fp16_to_f64(layer.fc2_scale[e])
    rot = fp16_to_f64(layer.rot_tab[e])
    svh_g, svh_u, suh_d = rot[:I], rot[I:2 * I], rot[2 * I:]
    svh_d = fp16_to_f64(layer.out_svh[e])
    if xq_up is None:
        y1 = s1[None, :] * (xq @ w1.T)
    else:
        y1 = s1[None, :] * np.concatenate([xq @ w1[:I].T, xq_up @ w1[I:].T], axis=1)
    g = svh_g[None, :] * hadamard.rotate(y1[:, :I], layer.rot_block_i)
    u = svh_u[None, :] * hadamard.rotate(y1[:, I:], layer.rot_block_i)
    # SiLU(g) = g / (1 + e^-g); for large negative g, e^-g overflows to inf and
    # the quotient is the correct -0, so the overflow warning is silenced
    with np.errstate(over="ignore"):
        a = g / (1.0 + np.exp(-g)) * u
    z = hadamard.rotate(suh_d[None, :] * a, layer.rot_block_i)
    zq = round_operand(z, mode, act_round)
    y2 = s2[None, :] * (zq @ w2.T)
    return svh_d[None, :] * hadamard.rotate(y2, layer.rot_block_h)


def layer_forward(layer, x_bits: np.ndarray, ids: np.ndarray, w: np.ndarray,
                  mode: str = "w4a16", act_round: bool = True, tokens=None,
                  return_routes: bool = False):
    """Whole layer for tokens ``tokens`` (default: all). Returns float64 [len, H]
    (and, with return_routes, the per-route unrotated FC2 rows [len, k, H])."""
    T = x_bits.shape[0]
    tokens = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    ids = np.asarray(ids)
    w = np.asarray(w, dtype=np.float64)
    k = ids.shape[1]
    separate = getattr(layer, "gate_suh", None) is not None or getattr(layer, "up_suh", None) is not None
    if not separate:
        xq = round_operand(rotate_input(layer, x_bits[tokens]), mode, act_round)
    per_route = np.zeros((len(tokens), k, layer.H), dtype=np.float64)
    sub_ids = ids[tokens]
    for e in np.unique(sub_ids):
        rows, js = np.nonzero(sub_ids == e)
        if not separate:
            per_route[rows, js] = expert_ffn(layer, int(e), xq[rows], mode, act_round)
        else:
            # one rotation per route: the expert's gate and up signs
            sg, su = input_signs(layer, int(e))
            xe = x_bits[tokens][rows]
            xg = round_operand(rotate_input(layer, xe, sg), mode, act_round)
            xu = round_operand(rotate_input(layer, xe, su), mode, act_round)
            per_route[rows, js] = expert_ffn(layer, int(e), xg, mode, act_round, xq_up=xu)
    out = np.zeros((len(tokens), layer.H), dtype=np.float64)
    for j in range(k):                     # fixed per-token order j = 0..k-1
        out += w[tokens, j][:, None] * per_route[:, j]
    return (out, per_route) if return_routes else out
