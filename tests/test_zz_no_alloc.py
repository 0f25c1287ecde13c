"""The allocation-free route map against the workspace-based one (needs a GPU).

trellis_moe_route_map_static serves callers that cannot allocate device memory
or lend the library a workspace -- hosts that hand the library only inputs and
outputs from their own fixed memory plan, and loops that must stay out of the
allocator after start-up.
It keeps its scratch in a static device array, so its results must equal
those of trellis_moe_route_map (integer work: bit for bit) on every call,
including a second call that finds the first call's leftovers in that array.
"""
import numpy as np
import pytest

from trellis_quantized_moe_route_gb300 import synth

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def _setup():
    if not torch.cuda.is_available():
        pytest.fail("needs a CUDA device")
    from trellis_quantized_moe_route_gb300 import binding, build
    build.build()
    binding.load_library()
    return binding


def test_static_route_map_equals_workspace_route_map_on_two_calls():
    binding = _setup()
    E, k = 64, 8
    cfg = synth.LayerConfig("static", E=E, H=128, I=64, topk=k, T=128, bits=(4,), rot_block_h=128,
                            rot_block_i=64, mode="w4a16", logits="normal", seed=5)
    moe = binding.TrellisMoE(synth.make_layer(cfg), max_tokens=128)
    first = synth.random_ids(501, 128, E, k)          # 1024 routes: the static limit
    second = synth.random_ids(502, 37, E, k)          # fewer routes than the first call left behind
    second[3, 2] = -1                                 # a dropped id
    second[30, 0] = E
    for ids_np, block in ((first, 64), (second, 8)):
        ids = torch.from_numpy(ids_np).cuda()
        ref = moe.route_map(ids, block)
        got = binding.route_map_static(ids, E, block)
        torch.cuda.synchronize()
        n = int(ref["offsets"][-1].item())
        assert torch.equal(got["counts"], ref["counts"])
        assert torch.equal(got["offsets"], ref["offsets"])
        assert torch.equal(got["route_of_slot"][:n], ref["route_of_slot"][:n])
        assert torch.equal(got["slot_of_route"], ref["slot_of_route"])
    moe.close()


def test_static_route_map_rejects_more_routes_than_its_scratch_holds():
    binding = _setup()
    ids = torch.zeros((129, 8), dtype=torch.int32, device="cuda")
    with pytest.raises(binding.TrellisMoEError) as ei:
        binding.route_map_static(ids, 64, 8)
    assert ei.value.status == -2
    assert "1024" in str(ei.value)
