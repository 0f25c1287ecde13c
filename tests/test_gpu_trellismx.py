"""TrellisMX-style layers on the CUDA path against the oracle (needs a GPU):
E4M3 trellis weights with one UE8M0 scale per 32 weights (K2-K4) and the
coupled H512/H128 boundary -- 512-point rotation blocks on the hidden side,
128 on the intermediate side (flashinfer PR #69 "b12x fused MoE: TrellisMX
(procedural NPK) source format with an in-tree P8 runtime", Description).
Covered: the decode rows in both modes, the tensor-core kernels (W4A16 with
many routes per expert), 512-point blocks with and without the weight
scales, uniform and mixed K, separate gate / up signs, the full-size
workload, and the prepare-time range check of the scales."""
import dataclasses

import numpy as np
import pytest

from oracle import layer as olayer, mxfp8
from tests.gpu_util import TOL, block_cover_tokens, oracle_routes, rel_row_err, run_and_compare, small_cfg, upload_tokens
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
    # decode rows (few routes per expert)
    (dict(T=4, E=16, topk=4, H=512, I=128, bits=(2, 3, 4), rot_block_h=512, mx=True), ("w4a8", "w4a16")),
    (dict(T=3, E=32, topk=4, H=1024, I=256, bits=(4,), rot_block_h=512, mx=True), ("w4a8", "w4a16")),
    (dict(T=4, E=16, topk=4, H=512, I=128, bits=(3,), rot_block_h=128, mx=True), ("w4a8",)),
    (dict(T=4, E=16, topk=4, H=512, I=128, bits=(4,), rot_block_h=512), ("w4a8", "w4a16")),   # 512 blocks alone
    # W4A8 at 16 routes per expert (still the decode rows)
    (dict(T=64, E=8, topk=2, H=512, I=128, bits=(2, 3, 4), rot_block_h=512, mx=True), ("w4a8", "w4a16")),
    # tensor cores: W4A16 with many routes per expert (128- and 256-route blocks)
    (dict(T=300, E=4, topk=2, H=512, I=128, bits=(2, 3, 4), rot_block_h=512, mx=True), ("w4a16",)),
    (dict(T=400, E=4, topk=3, H=1024, I=320, bits=(4,), rot_block_h=512, rot_block_i=64, mx=True), ("w4a16",)),
    (dict(T=300, E=4, topk=2, H=512, I=128, bits=(4,), rot_block_h=512), ("w4a16",)),
]


@pytest.mark.parametrize("kw,modes", SHAPES)
def test_trellismx_layers_match_oracle(kw, modes):
    cfg = small_cfg(**kw)
    L = synth.make_layer(cfg)
    moe = _moe(L, cfg.T)
    for mode in modes:
        err, _, _ = run_and_compare(moe, L, cfg, cfg.T, mode)
        assert err < TOL[mode], (mode, err)
        assert moe.poll_error() == 0
    moe.close()


@pytest.mark.parametrize("rows", [1, "E"])
def test_trellismx_with_separate_input_signs(rows):
    for kw, mode in ((dict(T=4, E=16, topk=4, H=512, I=128, bits=(2, 3, 4), rot_block_h=512, mx=True), "w4a8"),
                     (dict(T=300, E=4, topk=2, H=512, I=128, bits=(2, 3, 4), rot_block_h=512, mx=True), "w4a16")):
        cfg = small_cfg(**kw)
        L = synth.with_input_signs(synth.make_layer(cfg), 1 if rows == 1 else cfg.E, seed=13)
        moe = _moe(L, cfg.T)
        err, _, _ = run_and_compare(moe, L, cfg, cfg.T, mode)
        assert err < TOL[mode], (mode, err)
        moe.close()


@pytest.mark.parametrize("T", [1, 8])
def test_trellismx_workload_decode_full(T):
    cfg = synth.CONFIGS["trellismx"]
    L = synth.make_layer(cfg)
    moe = _moe(L, 8)
    err, _, _ = run_and_compare(moe, L, cfg, T, "w4a8")
    assert err < TOL["w4a8"], err


def test_trellismx_workload_w4a16_prefill_covering_blocks():
    cfg = synth.CONFIGS["trellismx"]
    L = synth.make_layer(cfg)
    T = 512
    moe = _moe(L, T)
    _, logits = synth.make_tokens(cfg, T=T)
    ids, _ = oracle_routes(logits, cfg.topk)
    sel = block_cover_tokens(ids, cfg.E, 256, extra=(0, T - 1))
    err, _, _ = run_and_compare(moe, L, cfg, T, "w4a16", tokens=sel)
    assert err < TOL["w4a16"], err


def test_512_blocks_atomic_setting_takes_the_ordered_combine():
    cfg = small_cfg(T=300, E=4, topk=2, H=512, I=128, bits=(4,), rot_block_h=512, mx=True)
    L = synth.make_layer(cfg)
    x_bits, logits = synth.make_tokens(cfg)
    x, lg = upload_tokens(x_bits, logits)
    a = _moe(L, cfg.T).forward_logits(x, lg, mode="w4a16").clone()
    b = _moe(L, cfg.T, deterministic=False).forward_logits(x, lg, mode="w4a16").clone()
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_rotate_quant_512_blocks():
    cfg = small_cfg(H=1024, rot_block_h=512, T=9)
    L = synth.make_layer(cfg)
    moe = _moe(L, cfg.T)
    x_bits, logits = synth.make_tokens(cfg)
    x, _ = upload_tokens(x_bits, logits)
    ref = olayer.rotate_input(L, x_bits)
    xq, _ = moe.rotate_quant(x, "w4a16")
    got = xq.cpu().numpy().view(np.float16).astype(np.float64)
    ulp = np.maximum(np.abs(np.spacing(ref.astype(np.float16))), np.abs(np.spacing(got.astype(np.float16))))
    assert np.all(np.abs(got - ref) <= ulp.astype(np.float64))
    codes, e8 = (t.cpu().numpy() for t in moe.rotate_quant(x, "w4a8"))
    rc, re8, _ = mxfp8.quantize_mxfp8(ref.astype(np.float32))
    assert np.array_equal(codes, rc) and np.array_equal(e8, re8)


def test_prepare_rejects_scale_exponents_outside_the_exact_range():
    from trellis_quantized_moe_route_gb300.binding import TrellisMoEError
    cfg = small_cfg(T=4, E=4, topk=2, H=256, I=64, rot_block_i=64, mx=True)
    L = synth.make_layer(cfg)
    for bad in (127 + 14, 127 - 16):
        u = L.fc2_wscale.copy()
        u[1, 7, 1] = bad
        with pytest.raises(TrellisMoEError) as ei:
            _moe(dataclasses.replace(L, fc2_wscale=u), 4)
        assert ei.value.status == -2
    u = L.fc1_wscale.copy()
    u[...] = 127 + 13
    u[0, 0, 0] = 127 - 15
    _moe(dataclasses.replace(L, fc1_wscale=u), 4).close()     # both ends of the range are accepted
