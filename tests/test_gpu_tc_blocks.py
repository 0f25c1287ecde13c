"""Route-block boundaries against the oracle: experts whose route counts sit
on both sides of 128 and 256 routes. With at most 128 routes per expert on
average the tensor-core kernels use 128-route blocks (one accumulator each;
the 128 / 129 and 256 / 257 counts give one, two and three blocks per
expert); with more they use 256-route blocks, where 129 routes switch a unit
to two accumulators and 257 to a second block (W4A16). The first layer in
W4A8 (872 routes) runs on the decode rows, whose 8-slot route blocks then
hold many blocks per expert."""
import numpy as np
import pytest

from oracle import layer as olayer
from tests.gpu_util import TOL, rel_row_err, small_cfg
from trellis_quantized_moe_route_gb300 import synth

pytestmark = pytest.mark.gpu

COUNTS = {
    "128-route blocks": [257, 256, 129, 128, 1, 37, 60, 4],   # E = 8, top-2: 109 routes per expert
    "256-route blocks": [257, 256, 129, 128],                 # E = 4, top-2: 192.5 routes per expert
}


def _ids_with_counts(counts):
    """Top-2 ids whose per-expert counts are exactly `counts`: the sorted
    label list paired with itself shifted by half (distinct experts per token
    since no expert holds more than half of the routes)."""
    labels = np.repeat(np.arange(len(counts), dtype=np.int32), counts)
    R = labels.size
    assert R % 2 == 0 and max(counts) <= R // 2
    T = R // 2
    ids = np.stack([labels[:T], labels[T:]], axis=1)
    assert np.all(ids[:, 0] != ids[:, 1])
    return ids


@pytest.mark.parametrize("mode,blocks", [("w4a16", "128-route blocks"), ("w4a16", "256-route blocks"),
                                         ("w4a8", "128-route blocks")])
def test_block_boundaries_match_oracle(mode, blocks):
    import torch
    from trellis_quantized_moe_route_gb300.binding import TrellisMoE
    counts = COUNTS[blocks]
    ids = _ids_with_counts(counts)
    T = ids.shape[0]
    cfg = small_cfg(E=len(counts), topk=2, T=T, seed=77)
    L = synth.make_layer(cfg)
    x_bits, _ = synth.make_tokens(cfg, T=T)
    rng = np.random.default_rng(5)
    w = rng.uniform(0.1, 1.0, size=ids.shape).astype(np.float32)
    w /= w.sum(axis=1, keepdims=True)
    moe = TrellisMoE(L, max_tokens=T)
    x = torch.from_numpy(x_bits.view(np.int16)).cuda()
    out = moe.forward(x, torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda(), mode=mode)
    torch.cuda.synchronize()
    assert moe.poll_error() == 0
    sel = np.arange(0, T, 3)          # every third token: all experts appear
    ref = olayer.layer_forward(L, x_bits, ids, w, mode=mode, tokens=sel)
    err = rel_row_err(out.cpu().numpy()[sel], ref)
    assert err < TOL[mode], err
