"""The C ABI library builds, loads and exports every entry point the public
header declares; host-side argument validation runs without a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "trellis_moe.h")


@pytest.fixture(scope="module")
def lib():
    from trellis_quantized_moe_route_gb300 import binding, build
    build.build()
    return binding.load_library()


def declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"\b(trellis_(?:moe|linear)_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared()
    for must in ("trellis_moe_prepare", "trellis_moe_forward", "trellis_moe_route", "trellis_moe_destroy"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    from trellis_quantized_moe_route_gb300 import binding
    for name in declared():
        assert hasattr(lib, name), name
    assert sorted(binding.EXPORTED) == declared()


def test_host_validation_without_gpu(lib):
    from trellis_quantized_moe_route_gb300 import binding
    P = ctypes.c_void_p
    # router: k outside 1..min(E, 32) is rejected before any CUDA call
    assert lib.trellis_moe_route(P(8), 4, 8, 0, P(8), P(8), None) == -1
    assert b"k=0" in lib.trellis_moe_last_error()
    assert lib.trellis_moe_route(P(8), 4, 300, 2, P(8), P(8), None) == -2
    # prepare without a descriptor
    h = ctypes.c_void_p()
    assert lib.trellis_moe_prepare(None, ctypes.byref(h), None) == -1
    # prepare with unsupported shapes fails before touching the device
    d = binding.LayerDesc()
    d.E, d.H, d.I, d.topk, d.rot_block_h, d.rot_block_i = 8, 100, 64, 2, 128, 64
    assert lib.trellis_moe_prepare(ctypes.byref(d), ctypes.byref(h), None) == -2
    assert b"H=100" in lib.trellis_moe_last_error()
    d.H = 256
    d.rot_block_i = 32
    assert lib.trellis_moe_prepare(ctypes.byref(d), ctypes.byref(h), None) == -2
    d.rot_block_i, d.topk = 64, 9
    assert lib.trellis_moe_prepare(ctypes.byref(d), ctypes.byref(h), None) == -1
    d.topk, d.max_tokens = 2, 4
    bits = (ctypes.c_uint8 * 8)(*([4] * 8))
    d.bits_per_expert = ctypes.cast(bits, ctypes.c_void_p)
    assert lib.trellis_moe_prepare(ctypes.byref(d), ctypes.byref(h), None) == -1   # NULL payload
    assert b"fc1_payload" in lib.trellis_moe_last_error()
    # separate gate / up input signs: both or neither, 1 or E rows
    d.gate_suh = 4096
    assert lib.trellis_moe_prepare(ctypes.byref(d), ctypes.byref(h), None) == -1
    assert b"together" in lib.trellis_moe_last_error()
    d.up_suh, d.input_sign_rows = 8192, 3
    assert lib.trellis_moe_prepare(ctypes.byref(d), ctypes.byref(h), None) == -1
    assert b"input_sign_rows" in lib.trellis_moe_last_error()
    d.gate_suh = d.up_suh = None
    d.input_sign_rows = 0
    assert lib.trellis_moe_set_wait_test(None, 1000, 1) == -1
    # forward on a NULL handle
    assert lib.trellis_moe_forward(None, P(8), P(8), P(8), 1, 0, P(8), P(256), 1 << 20, None) == -1
    assert lib.trellis_moe_set_stage_events(None, None, 0) == -1
    assert lib.trellis_moe_set_decode_lut(None, 1) == -1
    # dense linear: shape checks before any CUDA call, NULL handles
    ld = binding.LinearDesc()
    ld.N, ld.K, ld.bits, ld.rot_in, ld.rot_out, ld.max_tokens = 256, 200, 4, 128, 128, 8
    assert lib.trellis_linear_prepare(ctypes.byref(ld), ctypes.byref(h), None) == -2
    assert b"K=200" in lib.trellis_moe_last_error()
    ld.K, ld.rot_out = 256, 32
    assert lib.trellis_linear_prepare(ctypes.byref(ld), ctypes.byref(h), None) == -2
    ld.rot_out = 64
    assert lib.trellis_linear_prepare(ctypes.byref(ld), ctypes.byref(h), None) == -1   # NULL payload
    assert b"payload" in lib.trellis_moe_last_error()
    assert lib.trellis_linear_forward(None, P(8), 1, P(16), P(256), 1 << 20, None) == -1
    assert lib.trellis_linear_workspace_size(None, 4) == 0
    lib.trellis_linear_destroy(None)
    lib.trellis_moe_destroy(None)

