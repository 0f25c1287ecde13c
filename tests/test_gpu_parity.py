"""CUDA path vs. oracle, through the C ABI (needs a GB300)."""
import numpy as np
import pytest

from oracle import hadamard, layer as olayer, mxfp8, route as oroute, trellis
from tests.gpu_util import (TOL, block_cover_tokens, oracle_routes, rel_row_err, run_and_compare, small_cfg,
                            upload_tokens)
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


# ---------------------------------------------------------------- decode ---
@pytest.mark.parametrize("K", [2, 3, 4, 5, 6])
@pytest.mark.parametrize("mode", ["w4a16", "w4a8"])
def test_decode_tiles_bit_exact(K, mode):
    cfg = small_cfg(E=3, H=128, I=64, topk=2, rot_block_i=64, bits=(K,), seed=40 + K)
    L = synth.make_layer(cfg)
    moe = _moe(L, 4)
    for proj, rows, cols in ((1, 2 * cfg.I, cfg.H), (2, cfg.H, cfg.I)):
        ntiles = (rows // 16) * (cols // 16)
        got = moe.decode_tiles(proj, 1, 0, ntiles, mode).cpu().numpy()
        payload = L.fc1_payload if proj == 1 else L.fc2_payload
        tiles = trellis.expert_payload(payload, rows, cols, L.bits, 1).reshape(ntiles, 16 * K)
        ref = trellis.decode_tiles_fp16(tiles, K)
        if mode == "w4a16":
            assert np.array_equal(got.view(np.uint16), ref.view(np.uint16))
        else:
            assert np.array_equal(got, mxfp8.e4m3_encode(ref.astype(np.float64)))


def test_decode_tiles_mixed_bits_offsets():
    cfg = synth.CONFIGS["odd"]
    small = small_cfg(E=6, H=256, I=64, rot_block_i=64, bits=(2, 3, 4), seed=3)
    L = synth.make_layer(small)
    moe = _moe(L, 4)
    for e in range(small.E):
        K = int(L.bits[e])
        ntiles = (small.H // 16) * (small.I // 16)
        got = moe.decode_tiles(2, e, 3, 5, "w4a16").cpu().numpy()
        tiles = trellis.expert_payload(L.fc2_payload, small.H, small.I, L.bits, e).reshape(ntiles, 16 * K)
        assert np.array_equal(got.view(np.uint16), trellis.decode_tiles_fp16(tiles[3:8], K).view(np.uint16))
    assert cfg.bits == (2, 3, 4)


# ---------------------------------------------------------------- routing ---
@pytest.mark.parametrize("name,T", [("decode", 64), ("prefill", 300), ("tiny", 4), ("large", 37)])
def test_router_matches_oracle(name, T):
    from trellis_quantized_moe_route_gb300 import binding
    cfg = synth.CONFIGS[name]
    _, logits = synth.make_tokens(cfg, T=T)
    ids_ref, w_ref = oroute.route_topk_softmax(logits, cfg.topk)
    ids, w = binding.route(torch.from_numpy(logits).cuda(), cfg.topk)
    assert np.array_equal(ids.cpu().numpy(), ids_ref)
    assert np.allclose(w.cpu().numpy(), w_ref, rtol=2e-6, atol=1e-7)


def test_router_ties_go_to_lower_id():
    from trellis_quantized_moe_route_gb300 import binding
    lg = np.round(synth.Stream(9, 9).normal(50 * 40).reshape(50, 40)).astype(np.float32)
    ids_ref, _ = oroute.route_topk_softmax(lg, 6)
    ids, _ = binding.route(torch.from_numpy(lg).cuda(), 6)
    assert np.array_equal(ids.cpu().numpy(), ids_ref)


@pytest.mark.parametrize("T,E,k,block", [(4, 8, 2, 8), (8, 128, 8, 8), (2048, 128, 8, 64), (512, 64, 10, 64),
                                         (1, 160, 8, 8), (129, 16, 8, 64), (3000, 256, 3, 16)])
def test_route_map_bit_exact(T, E, k, block):
    cfg = small_cfg(E=E, topk=k, H=128, I=64, rot_block_i=64)
    L = synth.make_layer(cfg, bits=[4] * E)
    moe = _moe(L, T)
    ids = synth.random_ids(100 + T, T, E, k)
    got = moe.route_map(torch.from_numpy(ids).cuda(), block)
    ref = oroute.route_map(ids, E, block)
    n = int(ref["offsets"][-1])
    assert np.array_equal(got["counts"].cpu().numpy(), ref["counts"])
    assert np.array_equal(got["offsets"].cpu().numpy(), ref["offsets"])
    assert np.array_equal(got["route_of_slot"].cpu().numpy()[:n], ref["route_of_slot"])
    assert np.array_equal(got["slot_of_route"].cpu().numpy(), ref["slot_of_route"])


def test_route_map_skewed_single_expert():
    T, E, k = 3000, 32, 1
    cfg = small_cfg(E=E, topk=k, H=128, I=64, rot_block_i=64)
    moe = _moe(synth.make_layer(cfg, bits=[4] * E), T)
    ids = np.full((T, k), 5, dtype=np.int32)
    got = moe.route_map(torch.from_numpy(ids).cuda(), 64)
    ref = oroute.route_map(ids, E, 64)
    n = int(ref["offsets"][-1])
    assert np.array_equal(got["route_of_slot"].cpu().numpy()[:n], ref["route_of_slot"])
    assert np.array_equal(got["offsets"].cpu().numpy(), ref["offsets"])


def test_out_of_range_ids_are_dropped_and_flagged():
    cfg = small_cfg(E=8, topk=2, H=128, I=64, rot_block_i=64, T=4)
    L = synth.make_layer(cfg)
    moe = _moe(L, 4)
    x_bits, logits = synth.make_tokens(cfg)
    ids, w = oracle_routes(logits, 2)
    bad = ids.copy()
    bad[1, 1] = 8
    bad[3, 0] = -1
    x, _ = upload_tokens(x_bits, logits)
    out = moe.forward(x, torch.from_numpy(bad).cuda(), torch.from_numpy(w.astype(np.float32)).cuda(), mode="w4a16")
    assert moe.poll_error() == 1
    assert moe.poll_error() == 0
    w2 = w.copy()
    w2[1, 1] = 0.0
    w2[3, 0] = 0.0
    ref = olayer.layer_forward(L, x_bits, np.where(bad < 0, 0, np.minimum(bad, 7)), w2, mode="w4a16")
    assert rel_row_err(out.cpu().numpy(), ref) < TOL["w4a16"]


# ---------------------------------------------------------- rotate+quant ---
@pytest.mark.parametrize("rot", [1, 64, 128])
def test_rotate_quant_fp16(rot):
    cfg = small_cfg(H=512, rot_block_h=rot, T=33)
    L = synth.make_layer(cfg)
    moe = _moe(L, cfg.T)
    x_bits, logits = synth.make_tokens(cfg)
    x, _ = upload_tokens(x_bits, logits)
    xq, _ = moe.rotate_quant(x, "w4a16")
    got = xq.cpu().numpy().view(np.float16).astype(np.float64)
    ref = olayer.rotate_input(L, x_bits)
    if rot == 1:
        assert np.array_equal(got, ref.astype(np.float16).astype(np.float64))
    else:
        ulp = np.maximum(np.abs(np.spacing(ref.astype(np.float16))), np.abs(np.spacing(got.astype(np.float16))))
        assert np.all(np.abs(got - ref) <= ulp.astype(np.float64))


@pytest.mark.parametrize("rot", [1, 128])
def test_rotate_quant_mxfp8(rot):
    cfg = small_cfg(H=1024, rot_block_h=rot, T=17)
    L = synth.make_layer(cfg)
    moe = _moe(L, cfg.T)
    x_bits, logits = synth.make_tokens(cfg)
    x, _ = upload_tokens(x_bits, logits)
    xq, xs = moe.rotate_quant(x, "w4a8")
    codes, e8 = xq.cpu().numpy(), xs.cpu().numpy()
    ref = olayer.rotate_input(L, x_bits)
    rc, re8, rdeq = mxfp8.quantize_mxfp8(ref.astype(np.float32))
    # the W4A8 rotation runs in fp64 and rounds once to fp32, as the oracle's
    # float64 rotation does: the codes and exponents agree exactly
    assert np.array_equal(codes, rc) and np.array_equal(e8, re8)


# ---------------------------------------------------------------- layer ----
@pytest.mark.parametrize("mode", ["w4a16", "w4a8"])
def test_tiny_config(mode):
    cfg = synth.CONFIGS["tiny"]
    L = synth.make_layer(cfg)
    moe = _moe(L, cfg.T)
    err, _, _ = run_and_compare(moe, L, cfg, cfg.T, mode)
    assert err < TOL[mode], err


@pytest.mark.parametrize("mode", ["w4a16", "w4a8"])
@pytest.mark.parametrize("kw", [
    dict(),                                                     # rot 128/128, K=4
    dict(bits=(2, 3, 4), I=320, rot_block_i=64, H=512),         # odd geometry, mixed K, 64-wide I blocks
    dict(rot_block_h=1, rot_block_i=1),                         # identity rotations
    dict(bits=(5, 6), E=8, topk=3),                             # wider codes
    dict(T=200, E=8, topk=2),                                   # several 64-route blocks per expert
    dict(H=384),                                                # H % 256 == 128: 128-column FC2 blocks
    dict(rot_block_h=64),                                       # 64-wide H blocks: no level across halves
])
def test_small_layers(mode, kw):
    cfg = small_cfg(**kw)
    L = synth.make_layer(cfg)
    moe = _moe(L, cfg.T)
    err, _, _ = run_and_compare(moe, L, cfg, cfg.T, mode)
    assert err < TOL[mode], err


def test_deterministic_repeat_and_poisoned_workspace():
    cfg = small_cfg(T=100, E=8, topk=2)
    L = synth.make_layer(cfg)
    moe = _moe(L, cfg.T)
    x_bits, logits = synth.make_tokens(cfg)
    x, lg = upload_tokens(x_bits, logits)
    a = moe.forward_logits(x, lg, mode="w4a16").clone()
    b = moe.forward_logits(x, lg, mode="w4a16").clone()
    moe.workspace.fill_(0xFF)
    c = moe.forward_logits(x, lg, mode="w4a16").clone()
    torch.cuda.synchronize()
    assert torch.equal(a, b) and torch.equal(a, c)


@pytest.mark.parametrize("mode", ["w4a16", "w4a8"])
def test_token_permutation_equivariance_bitwise(mode):
    cfg = small_cfg(T=50, E=8, topk=3)
    L = synth.make_layer(cfg)
    moe = _moe(L, cfg.T)
    x_bits, logits = synth.make_tokens(cfg)
    perm = synth.permutation(synth.Stream(2, 2), cfg.T)
    x, lg = upload_tokens(x_bits, logits)
    xp, lgp = upload_tokens(x_bits[perm], logits[perm])
    a = moe.forward_logits(x, lg, mode=mode).cpu().numpy()
    b = moe.forward_logits(xp, lgp, mode=mode).cpu().numpy()
    assert np.array_equal(b, a[perm])


def test_atomic_combine_within_tolerance():
    cfg = small_cfg(T=64, E=8, topk=2)
    L = synth.make_layer(cfg)
    moe = _moe(L, cfg.T, deterministic=False)
    err, _, _ = run_and_compare(moe, L, cfg, cfg.T, "w4a16")
    assert err < TOL["w4a16"], err


def test_forward_host_matches_device_call():
    cfg = small_cfg(T=20)
    L = synth.make_layer(cfg)
    moe = _moe(L, cfg.T)
    x_bits, logits = synth.make_tokens(cfg)
    x, lg = upload_tokens(x_bits, logits)
    dev = moe.forward_logits(x, lg, mode="auto").cpu()
    xh = torch.from_numpy(x_bits.view(np.int16).copy()).pin_memory()
    lh = torch.from_numpy(logits.copy()).pin_memory()
    oh = torch.empty((cfg.T, cfg.H), dtype=torch.float32).pin_memory()
    moe.forward_host(xh, lh, oh, mode="auto")
    assert torch.equal(dev, oh)


@pytest.mark.parametrize("T,mode", [(8, "w4a8"), (20, "w4a16")])
def test_forward_host_graph_replay_reads_current_buffers(T, mode):
    """The host-buffer call runs directly on the first use of a buffer set,
    captures a graph on the second and replays it afterwards: every call must
    read the pinned inputs as they are at that call, and a change of the stage
    events (which the captured graph records) must not leave a stale graph."""
    cfg = small_cfg(T=T)
    L = synth.make_layer(cfg)
    moe = _moe(L, cfg.T)
    xh = torch.empty((T, cfg.H), dtype=torch.int16).pin_memory()
    lh = torch.empty((T, cfg.E), dtype=torch.float32).pin_memory()
    oh = torch.empty((T, cfg.H), dtype=torch.float32).pin_memory()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(7)]
    for call, seed in enumerate((5, 6, 7, 6, 8, 9)):
        x_bits, logits = synth.make_tokens(cfg, seed=seed)
        x, lg = upload_tokens(x_bits, logits)
        want = moe.forward_logits(x, lg, mode=mode).cpu()
        xh.copy_(torch.from_numpy(x_bits.view(np.int16).copy()))
        lh.copy_(torch.from_numpy(logits.copy()))
        if call == 4:
            moe.set_stage_events(ev)
        oh.fill_(float("nan"))
        moe.forward_host(xh, lh, oh, mode=mode)
        assert torch.equal(want, oh), call
        if call == 4:
            assert ev[6].query() and ev[0].elapsed_time(ev[6]) > 0
            moe.set_stage_events(None)
    # pageable buffers take the direct path
    x_bits, logits = synth.make_tokens(cfg, seed=10)
    x, lg = upload_tokens(x_bits, logits)
    want = moe.forward_logits(x, lg, mode=mode).cpu()
    xp = torch.from_numpy(x_bits.view(np.int16).copy())
    lp = torch.from_numpy(logits.copy())
    op = torch.empty((T, cfg.H), dtype=torch.float32)
    moe.forward_host(xp, lp, op, mode=mode)
    assert torch.equal(want, op)
    # the atomic combine keeps the staged copies on pinned buffers too
    moa = _moe(L, cfg.T, deterministic=False)
    xh.copy_(xp)
    lh.copy_(lp)
    for _ in range(3):
        oh.fill_(float("nan"))
        moa.forward_host(xh, lh, oh, mode=mode)
        assert torch.allclose(want, oh, rtol=1e-5, atol=1e-5)


def test_auto_mode_switches_at_decode_rows():
    cfg = small_cfg(T=16)
    L = synth.make_layer(cfg)
    moe = _moe(L, cfg.T, decode_max_rows=8)
    x_bits, logits = synth.make_tokens(cfg)
    for T, mode in ((8, "w4a8"), (9, "w4a16")):
        x, lg = upload_tokens(x_bits[:T], logits[:T])
        auto = moe.forward_logits(x, lg, mode="auto").cpu()
        explicit = moe.forward_logits(x, lg, mode=mode).cpu()
        assert torch.equal(auto, explicit)


def test_host_validation_errors():
    from trellis_quantized_moe_route_gb300.binding import TrellisMoEError
    cfg = small_cfg(T=4)
    L = synth.make_layer(cfg)
    moe = _moe(L, 4)
    x_bits, logits = synth.make_tokens(cfg, T=5)
    x, lg = upload_tokens(x_bits, logits)
    with pytest.raises(TrellisMoEError) as ei:
        moe.forward_logits(x, lg)  # T=5 > max_tokens=4
    assert ei.value.status == -1
    with pytest.raises(TrellisMoEError) as ei:
        moe.forward_logits(x[:4], lg[:4], mode=7)
    assert ei.value.status == -1
    ws, nb = moe.workspace, moe.workspace_bytes
    moe.workspace_bytes = 1024
    with pytest.raises(TrellisMoEError) as ei:
        moe.forward_logits(x[:4], lg[:4])
    assert ei.value.status == -3
    moe.workspace_bytes = nb
    moe.workspace = ws[16:]
    moe.workspace_bytes = nb - 16
    with pytest.raises(TrellisMoEError) as ei:
        moe.forward_logits(x[:4], lg[:4])
    assert ei.value.status == -3
    moe.workspace, moe.workspace_bytes = ws, nb
    out = moe.forward_logits(x[:0], lg[:0])
    assert out.shape == (0, cfg.H)


# ----------------------------------------------- the five workloads, full size ---
@pytest.mark.parametrize("T", [1, 2, 4, 8])
def test_decode_config_full(T):
    cfg = synth.CONFIGS["decode"]
    L = synth.make_layer(cfg)
    moe = _moe(L, 8)
    err, _, _ = run_and_compare(moe, L, cfg, T, "w4a8")
    assert err < TOL["w4a8"], err


def _cover(cfg, T, seed=None, extra=(0,)):
    """The workload's tokens that cover every (expert, 256-route block) of the
    tensor-core path, from the oracle's own router and route map."""
    _, logits = synth.make_tokens(cfg, T=T, seed=seed)
    ids, _ = oracle_routes(logits, cfg.topk)
    return block_cover_tokens(ids, cfg.E, 256, extra=tuple(extra) + (T - 1,))


def test_prefill_config_full_covering_blocks():
    cfg = synth.CONFIGS["prefill"]
    L = synth.make_layer(cfg)
    moe = _moe(L, cfg.T)
    sel = _cover(cfg, cfg.T)
    assert len(sel) > 150
    err, _, _ = run_and_compare(moe, L, cfg, cfg.T, "w4a16", tokens=sel)
    assert err < TOL["w4a16"], err


def test_odd_config_full_covering_blocks():
    cfg = synth.CONFIGS["odd"]
    L = synth.make_layer(cfg)
    moe = _moe(L, cfg.T)
    err, _, _ = run_and_compare(moe, L, cfg, cfg.T, "w4a16", tokens=_cover(cfg, cfg.T))
    assert err < TOL["w4a16"], err


def test_large_config_decode_full():
    cfg = synth.CONFIGS["large"]
    L = synth.make_layer(cfg)
    moe = _moe(L, 1)
    err, _, _ = run_and_compare(moe, L, cfg, 1, "w4a8")
    assert err < TOL["w4a8"], err


def test_large_config_prefill_covering_blocks():
    cfg = synth.CONFIGS["large"]
    L = synth.make_layer(cfg)
    moe = _moe(L, cfg.T)
    sel = _cover(cfg, cfg.T)
    assert len(sel) > 160
    err, _, _ = run_and_compare(moe, L, cfg, cfg.T, "w4a16", tokens=sel)
    assert err < TOL["w4a16"], err


# ------------------------------------- decode-rows path (T*topk small) ---
# These shapes keep T*topk below 4*E, where both modes take the decode-rows kernels.
DECODE_SHAPES = [
    dict(T=4, E=16, topk=2, bits=(2, 3, 4), I=320, rot_block_i=64, H=512),   # mixed K, 64-wide I blocks
    dict(T=3, E=32, topk=4),                                                 # K=4, rotation blocks 128
    dict(T=8, E=64, topk=8, bits=(5,), H=512, I=256),                        # generic K=5 decode
    dict(T=2, E=16, topk=3, rot_block_h=1, rot_block_i=1),                   # identity rotations
    dict(T=1, E=8, topk=8, H=1024, I=512),                                   # every expert, one token
    dict(T=120, E=256, topk=8, H=256, I=128),                                # 960 routes: the regime's largest block table
    dict(T=16, E=32, topk=4, H=768, I=320, rot_block_i=64),                  # 512-column items, ragged last ones (768, 320)
]


@pytest.mark.parametrize("mode", ["w4a8", "w4a16"])
@pytest.mark.parametrize("kw", DECODE_SHAPES)
def test_decode_path_layers(mode, kw):
    cfg = small_cfg(**kw)
    assert cfg.T * cfg.topk < 4 * cfg.E
    L = synth.make_layer(cfg)
    moe = _moe(L, cfg.T)
    err, _, _ = run_and_compare(moe, L, cfg, cfg.T, mode)
    assert err < TOL[mode], err


@pytest.mark.parametrize("mode", ["w4a8", "w4a16"])
@pytest.mark.parametrize("kw", DECODE_SHAPES + [dict(name="decode", E=128, H=1024, I=512, topk=8, T=8)])
def test_decode_path_table_and_hash_agree_bitwise(mode, kw):
    """The decode rows expand weights either by the codebook hash (default) or
    by table lookup; the table holds the hash's own values, so the two must
    agree bit for bit (and the table path must meet the oracle too)."""
    cfg = small_cfg(**kw)
    L = synth.make_layer(cfg)
    moe = _moe(L, cfg.T)
    x_bits, logits = synth.make_tokens(cfg)
    x, lg = upload_tokens(x_bits, logits)
    hashed = moe.forward_logits(x, lg, mode=mode).clone()
    moe.set_decode_lut(True)
    lut = moe.forward_logits(x, lg, mode=mode).clone()
    torch.cuda.synchronize()
    assert torch.equal(lut, hashed)
    err, _, _ = run_and_compare(moe, L, cfg, cfg.T, mode)
    assert err < TOL[mode], err
    moe.set_decode_lut(False)
    assert torch.equal(moe.forward_logits(x, lg, mode=mode), hashed)


def _scale_bf16(bits, k):
    """bf16 bit patterns times 2^k (exact: only the exponent changes)."""
    f = (bits.astype(np.uint32) << 16).view(np.float32) * np.float32(2.0 ** k)
    return (f.view(np.uint32) >> 16).astype(np.uint16)


@pytest.mark.parametrize("scales", [(0, -24, 16, 0), (-24, -24, -24, -24), (16, 16, 16, 16)])
def test_decode_path_w4a8_block_exponent_ranges(scales):
    """W4A8 decode rows keep the activations both as E4M3 codes and as
    code * 2^e; blocks whose exponent falls outside [-15, 7] must take the
    scaled path. Tokens scaled by 2^-24 and 2^16 push x~ (and z~) out of that
    range, alone or mixed with ordinary tokens in one route block."""
    cfg = small_cfg(T=4, E=16, topk=4, H=256, I=128)
    assert cfg.T * cfg.topk < 4 * cfg.E
    L = synth.make_layer(cfg)
    moe = _moe(L, cfg.T)
    x_bits, logits = synth.make_tokens(cfg)
    x_bits = np.stack([_scale_bf16(x_bits[t], k) for t, k in enumerate(scales)])
    ids, w = oracle_routes(logits, cfg.topk)
    x, lg = upload_tokens(x_bits, logits)
    out = moe.forward_logits(x, lg, mode="w4a8")
    torch.cuda.synchronize()
    ref = olayer.layer_forward(L, x_bits, ids, w.astype(np.float32), mode="w4a8")
    assert rel_row_err(out.cpu().numpy(), ref) < TOL["w4a8"]


@pytest.mark.parametrize("pattern", [(0, -24, 16, 0), (-24,), (16,)])
def test_w4a8_many_routes_per_expert_block_exponent_ranges(pattern):
    """Explicit W4A8 with T*topk >= 4E (16 routes per expert): W4A8 runs on
    the decode rows at every T*topk <= 1024. Tokens scaled by 2^-24 and 2^16
    push the block exponents of x~ and of z~ (which scales with the square
    of the input) outside [-15, 7], alone or mixed with ordinary tokens."""
    cfg = small_cfg(T=64, E=8, topk=2, H=256, I=128)
    assert cfg.T * cfg.topk >= 4 * cfg.E
    L = synth.make_layer(cfg)
    moe = _moe(L, cfg.T)
    x_bits, logits = synth.make_tokens(cfg)
    x_bits = np.stack([_scale_bf16(x_bits[t], pattern[t % len(pattern)]) for t in range(cfg.T)])
    ids, w = oracle_routes(logits, cfg.topk)
    x, lg = upload_tokens(x_bits, logits)
    out = moe.forward_logits(x, lg, mode="w4a8")
    torch.cuda.synchronize()
    assert np.all(np.isfinite(out.cpu().numpy()))
    ref = olayer.layer_forward(L, x_bits, ids, w.astype(np.float32), mode="w4a8")
    assert rel_row_err(out.cpu().numpy(), ref) < TOL["w4a8"]


def test_w4a8_beyond_decode_rows_is_refused_and_auto_runs_w4a16():
    from trellis_quantized_moe_route_gb300.binding import TrellisMoEError
    cfg = small_cfg(T=300, E=8, topk=4, H=256, I=128)
    L = synth.make_layer(cfg)
    moe = _moe(L, cfg.T, decode_max_rows=cfg.T)
    x_bits, logits = synth.make_tokens(cfg)
    x, lg = upload_tokens(x_bits, logits)
    with pytest.raises(TrellisMoEError) as ei:
        moe.forward_logits(x, lg, mode="w4a8")   # 1200 routes > 1024
    assert ei.value.status == -2
    auto = moe.forward_logits(x, lg, mode="auto").cpu()
    assert torch.equal(auto, moe.forward_logits(x, lg, mode="w4a16").cpu())
    small = moe.forward_logits(x[:256], lg[:256], mode="auto").cpu()   # 1024 routes: W4A8
    assert torch.equal(small, moe.forward_logits(x[:256], lg[:256], mode="w4a8").cpu())


def test_decode_path_deterministic_poisoned_and_atomic():
    cfg = small_cfg(T=6, E=32, topk=4)
    L = synth.make_layer(cfg)
    moe = _moe(L, cfg.T)
    x_bits, logits = synth.make_tokens(cfg)
    x, lg = upload_tokens(x_bits, logits)
    a = moe.forward_logits(x, lg, mode="w4a8").clone()
    moe.workspace.fill_(0xFF)
    b = moe.forward_logits(x, lg, mode="w4a8").clone()
    moe.workspace.fill_(0x7F)
    c = moe.forward_logits(x, lg, mode="w4a8").clone()
    torch.cuda.synchronize()
    assert torch.equal(a, b) and torch.equal(a, c)
    perm = synth.permutation(synth.Stream(4, 4), cfg.T)
    xp, lgp = upload_tokens(x_bits[perm], logits[perm])
    p = moe.forward_logits(xp, lgp, mode="w4a8").cpu().numpy()
    assert np.array_equal(p, a.cpu().numpy()[perm])
    atomic = _moe(L, cfg.T, deterministic=False)
    err, _, _ = run_and_compare(atomic, L, cfg, cfg.T, "w4a8")
    assert err < TOL["w4a8"], err


def test_decode_path_drops_bad_ids():
    cfg = small_cfg(T=3, E=32, topk=4)
    L = synth.make_layer(cfg)
    moe = _moe(L, cfg.T)
    x_bits, logits = synth.make_tokens(cfg)
    ids, w = oracle_routes(logits, cfg.topk)
    bad = ids.copy()
    bad[0, 3] = 40
    bad[2, 0] = -3
    x, _ = upload_tokens(x_bits, logits)
    out = moe.forward(x, torch.from_numpy(bad).cuda(), torch.from_numpy(w.astype(np.float32)).cuda(), mode="w4a8")
    assert moe.poll_error() == 1
    w2 = w.copy()
    w2[0, 3] = 0.0
    w2[2, 0] = 0.0
    ref = olayer.layer_forward(L, x_bits, np.clip(bad, 0, cfg.E - 1), w2, mode="w4a8")
    assert rel_row_err(out.cpu().numpy(), ref) < TOL["w4a8"]


def test_workspace_size_monotonic_in_tokens():
    """A workspace sized for T tokens serves every smaller T, although the
    decode path's scratch exists only for small T."""
    cfg = small_cfg(T=64, E=16, topk=4)
    moe = _moe(synth.make_layer(cfg), 64)
    sizes = [int(moe.lib.trellis_moe_workspace_size(moe.handle, t)) for t in range(0, 65)]
    assert all(a <= b for a, b in zip(sizes, sizes[1:]))
    assert sizes[-1] == moe.workspace_bytes
