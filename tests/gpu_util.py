"""Helpers shared by the GPU parity tests (CUDA path vs. oracle)."""
import numpy as np

from oracle import layer as olayer
from oracle import route as oroute
from trellis_quantized_moe_route_gb300 import synth

TOL = {"w4a16": 2e-2, "w4a8": 6e-2}


def rel_row_err(y, ref):
    """max over tokens of max_h |y - ref| / RMS_h(ref)."""
    y = np.asarray(y, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = np.sqrt((ref ** 2).mean(axis=1))
    return float((np.abs(y - ref).max(axis=1) / rms).max())


def torch_mod():
    import torch
    return torch


def upload_tokens(x_bits, logits):
    torch = torch_mod()
    x = torch.from_numpy(np.ascontiguousarray(x_bits.view(np.int16))).cuda()
    lg = torch.from_numpy(np.ascontiguousarray(logits)).cuda()
    return x, lg


def oracle_routes(logits, k):
    return oroute.route_topk_softmax(logits, k)


def small_cfg(**kw):
    base = dict(name="small", E=16, H=256, I=128, topk=4, T=24, bits=(4,), rot_block_h=128,
                rot_block_i=128, mode="w4a16", logits="normal", seed=31)
    base.update(kw)
    return synth.LayerConfig(**base)


def run_and_compare(moe, L, cfg, T, mode, tokens=None, seed=None):
    """GPU forward from device-routed logits vs. the oracle on `tokens`.
    Returns (err, gpu_out, oracle_out)."""
    torch = torch_mod()
    x_bits, logits = synth.make_tokens(cfg, T=T, seed=seed)
    ids, w = oracle_routes(logits, cfg.topk)
    x, lg = upload_tokens(x_bits, logits)
    out = moe.forward_logits(x, lg, mode=mode)
    torch.cuda.synchronize()
    y = out.cpu().numpy()
    sel = np.arange(T) if tokens is None else np.asarray(tokens)
    ref = olayer.layer_forward(L, x_bits, ids, w.astype(np.float32), mode=mode, tokens=sel)
    return rel_row_err(y[sel], ref), y, ref


def block_cover_tokens(ids, E, block=256, extra=()):
    """Tokens whose routes cover every route block of every expert in a route
    map of `block` slots: per block, the routes at its first slot, at the
    slots either side of the 128-route accumulator split (127, 128) and at
    its last valid slot, so every multi-block expert, both accumulators of a
    block and each block's ragged tail are checked. `extra` tokens are added."""
    ids = np.asarray(ids)
    k = ids.shape[1]
    rm = oroute.route_map(ids, E, block)
    ros = np.asarray(rm["route_of_slot"])
    off = np.asarray(rm["offsets"])
    counts = np.asarray(rm["counts"])
    toks = set(int(t) for t in extra)
    for e in range(E):
        n = int(counts[e])
        for b0 in range(0, n, block):
            last = min(n, b0 + block) - 1
            for s in {b0, min(b0 + 127, last), min(b0 + 128, last), last}:
                toks.add(int(ros[off[e] + s]) // k)
    return np.asarray(sorted(toks), dtype=np.int64)
