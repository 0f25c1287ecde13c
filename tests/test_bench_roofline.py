"""The benchmark's roofline bookkeeping on CPU: which regime a workload takes,
the algorithmic work its dominant launch is credited with, and the kernels a
step launches (the library's regime rule, restated in bench.py)."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from trellis_quantized_moe_route_gb300 import synth  # noqa: E402

PK = {"hbm_gbs": 8000.0, "bf16_tflops": 2000.0, "source": "test"}


def _stages(fc1, fc2):
    return {"router": 1.0, "route_map": 1.0, "rotate": 1.0, "fc1": fc1, "fc2": fc2, "combine": 1.0, "step": 10.0}


def test_decode_rows_are_credited_with_fc1_bytes():
    cfg = synth.CONFIGS["decode"]
    roof, decode_path, fused = bench.roofline_record(cfg, 8, "w4a8", _stages(25.0, 20.0), 28.0e6, PK, None)
    assert decode_path and not fused
    assert roof["bound"] == "hbm" and roof["unit"] == "GB/s"
    # 28 MB in 25 us = 1120 GB/s, 14% of an 8000 GB/s peak
    assert roof["achieved"] == pytest.approx(1120.0)
    assert roof["frac"] == pytest.approx(0.14)
    assert roof["bytes_per_launch"] == 28_000_000 and roof["traffic"] is None
    assert bench.launches_per_layer_step(8 * cfg.topk, decode_path, fused) == 5


def test_tensor_core_launch_of_fc1_and_fc2_is_credited_with_both_gemms():
    cfg = synth.CONFIGS["prefill"]
    T = cfg.T
    R = T * cfg.topk
    # the one-launch form: the stage after FC1's event is (nearly) empty
    roof, decode_path, fused = bench.roofline_record(cfg, T, "w4a16", _stages(170.0, 2.0), 0.0, PK, (212e6, "p"))
    assert not decode_path and fused
    flops = 2 * R * 2 * cfg.I * cfg.H + 2 * R * cfg.H * cfg.I   # 6 R H I
    assert roof["flops_per_launch"] == flops == 6 * R * cfg.H * cfg.I
    assert roof["achieved"] == pytest.approx(flops / 170e-6 / 1e12, rel=1e-4)
    assert roof["bound"] == "tensor" and "FC1+FC2" in roof["kernel"] and roof["traffic"] == 212e6
    assert bench.launches_per_layer_step(R, decode_path, fused) == 7   # route map: 3 kernels above 1024 routes
    # two launches: FC1 alone
    roof2, _, fused2 = bench.roofline_record(cfg, T, "w4a16", _stages(120.0, 72.0), 0.0, PK, None)
    assert not fused2
    assert roof2["flops_per_launch"] == 2 * R * 2 * cfg.I * cfg.H
    assert bench.launches_per_layer_step(R, False, False) == 8


def test_regime_boundary_matches_the_library_rule():
    cfg = synth.CONFIGS["prefill"]   # E = 128, top-k 8
    # W4A16 with fewer than 4 routes per expert: decode rows
    _, dp, _ = bench.roofline_record(cfg, 63, "w4a16", _stages(10.0, 8.0), 1.0, PK, None)
    assert dp  # 504 routes < 4 E = 512
    _, dp, _ = bench.roofline_record(cfg, 64, "w4a16", _stages(10.0, 8.0), 1.0, PK, None)
    assert not dp  # 512 routes
    # W4A8 up to 1024 routes: decode rows
    _, dp, _ = bench.roofline_record(cfg, 128, "w4a8", _stages(10.0, 8.0), 1.0, PK, None)
    assert dp
    assert bench.launches_per_layer_step(512, False, True) == 5   # route map in one kernel
