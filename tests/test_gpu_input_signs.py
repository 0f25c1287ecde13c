"""Separate gate / up input signs on the CUDA path against the oracle (needs
a GPU).

The FC1 gate rows of a route to expert e see x~_g = H_b(gate_suh[e] * x) and
its up rows x~_u = H_b(up_suh[e] * x), with one sign row shared by the experts
or one row per expert (b12x PR #129 "feat(moe): serve canonical Fruit QSRT
atoms", review of trellis_w4a8.py: gate_suh and up_suh of shape (1, H) or
(num_experts, H)). Covered: both layouts, both modes, the decode rows (few
routes per expert; every W4A8 call) and the tensor-core kernels (W4A16 with
many routes per expert: 128-route blocks, one and several blocks per expert,
64-row FC1 blocks), routes from logits and given ids with a dropped id.
"""
import numpy as np
import pytest

from oracle import layer as olayer
from tests.gpu_util import TOL, oracle_routes, rel_row_err, run_and_compare, small_cfg, upload_tokens
from trellis_quantized_moe_route_gb300 import synth

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from trellis_quantized_moe_route_gb300 import binding, build
    build.build()
    binding.load_library()


def _moe(L, max_tokens, **kw):
    from trellis_quantized_moe_route_gb300.binding import TrellisMoE
    return TrellisMoE(L, max_tokens=max_tokens, **kw)


SHAPES = [
    (dict(T=4, E=16, topk=4), ("w4a16", "w4a8")),                               # decode rows
    (dict(T=3, E=32, topk=4, bits=(2, 3, 4), I=320, rot_block_i=64, H=512), ("w4a16", "w4a8")),
    (dict(T=64, E=8, topk=2), ("w4a16", "w4a8")),                               # W4A16: tensor cores
    (dict(T=300, E=4, topk=2), ("w4a16",)),                                     # 150 routes per expert: 2 blocks
    (dict(T=96, E=8, topk=3, bits=(2, 3, 4), I=320, rot_block_i=64, H=512), ("w4a16",)),  # 64-row FC1 blocks
]


@pytest.mark.parametrize("rows", ["shared", "per_expert"])
@pytest.mark.parametrize("kw,modes", SHAPES)
def test_separate_input_signs_match_oracle(kw, modes, rows):
    cfg = small_cfg(**kw)
    L = synth.with_input_signs(synth.make_layer(cfg), 1 if rows == "shared" else cfg.E, seed=11)
    moe = _moe(L, cfg.T)
    for mode in modes:
        err, _, _ = run_and_compare(moe, L, cfg, cfg.T, mode)
        assert err < TOL[mode], (mode, err)
        assert moe.poll_error() == 0
    moe.close()


@pytest.mark.parametrize("mode,kw", [("w4a8", dict(T=6, E=32, topk=4)), ("w4a16", dict(T=64, E=8, topk=2))])
def test_separate_input_signs_given_ids_and_dropped_id(mode, kw):
    cfg = small_cfg(**kw)
    L = synth.with_input_signs(synth.make_layer(cfg), cfg.E, seed=12)
    moe = _moe(L, cfg.T)
    x_bits, logits = synth.make_tokens(cfg)
    ids, w = oracle_routes(logits, cfg.topk)
    bad = ids.copy()
    bad[1, 0] = cfg.E + 3
    x, _ = upload_tokens(x_bits, logits)
    out = moe.forward(x, torch.from_numpy(bad).cuda(), torch.from_numpy(w.astype(np.float32)).cuda(), mode=mode)
    torch.cuda.synchronize()
    assert moe.poll_error() == 1
    w2 = w.astype(np.float32).copy()
    w2[1, 0] = 0.0
    ref = olayer.layer_forward(L, x_bits, np.where(bad >= cfg.E, 0, bad), w2, mode=mode)
    assert rel_row_err(out.cpu().numpy(), ref) < TOL[mode]
    moe.close()


def test_equal_gate_and_up_signs_reproduce_the_shared_layer_bitwise():
    """gate_suh = up_suh = in_suh (one row) computes what the plain layer
    does; on the decode rows, which then do the same arithmetic per value,
    the bits must equal those of the layer without separate signs."""
    for kw, mode in ((dict(T=4, E=16, topk=4), "w4a8"), (dict(T=4, E=16, topk=4), "w4a16")):
        cfg = small_cfg(**kw)
        L = synth.make_layer(cfg)
        Ls = synth.with_input_signs(L, 1)
        Ls = type(L)(**{**Ls.__dict__, "gate_suh": L.in_suh.reshape(1, -1).copy(), "up_suh": L.in_suh.reshape(1, -1).copy()})
        a, b = _moe(L, cfg.T), _moe(Ls, cfg.T)
        x_bits, logits = synth.make_tokens(cfg)
        x, lg = upload_tokens(x_bits, logits)
        ya = a.forward_logits(x, lg, mode=mode).clone()
        yb = b.forward_logits(x, lg, mode=mode).clone()
        torch.cuda.synchronize()
        assert torch.equal(ya, yb), mode
        a.close()
        b.close()
