"""Thin Python binding of ``libtrellis_moe.so`` (the C ABI in include/trellis_moe.h).

Only argument marshalling lives here: PyTorch provides device memory and the
current CUDA stream, ctypes passes raw pointers, and every step of the layer
runs in the library's CUDA kernels. There is no CPU fallback: if the library
is missing or no CUDA device is present, calls raise.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtrellis_moe.so")

MODE_AUTO, MODE_W4A16, MODE_W4A8 = 0, 1, 2
MODES = {"auto": MODE_AUTO, "w4a16": MODE_W4A16, "w4a8": MODE_W4A8}

TM_OK = 0
STATUS = {0: "TM_OK", -1: "TM_EINVAL", -2: "TM_EUNSUPPORTED", -3: "TM_EWORKSPACE", -4: "TM_ECUDA", -5: "TM_EDEVICE"}

# workspace regions (trellis_moe_workspace_region)
REGION_XQ, REGION_XS, REGION_ZQ, REGION_ZS, REGION_ROWS, REGION_SLOT_OF_ROUTE, REGION_ERR = range(7)

EXPORTED = [
    "trellis_moe_prepare", "trellis_moe_workspace_size", "trellis_moe_forward",
    "trellis_moe_forward_logits", "trellis_moe_forward_host", "trellis_moe_route",
    "trellis_moe_route_map", "trellis_moe_rotate_quant", "trellis_moe_decode_tiles",
    "trellis_moe_workspace_region", "trellis_moe_set_stage_events", "trellis_moe_set_decode_lut",
    "trellis_moe_poll_error", "trellis_moe_set_wait_test",
    "trellis_moe_last_error", "trellis_moe_destroy", "trellis_moe_route_map_static",
    "trellis_linear_prepare", "trellis_linear_workspace_size", "trellis_linear_forward",
    "trellis_linear_poll_error", "trellis_linear_destroy",
]


class LayerDesc(ctypes.Structure):
    _fields_ = [
        ("E", ctypes.c_int32), ("H", ctypes.c_int32), ("I", ctypes.c_int32), ("topk", ctypes.c_int32),
        ("rot_block_h", ctypes.c_int32), ("rot_block_i", ctypes.c_int32),
        ("bits_per_expert", ctypes.c_void_p),
        ("fc1_payload", ctypes.c_void_p), ("fc2_payload", ctypes.c_void_p),
        ("fc1_scale", ctypes.c_void_p), ("fc2_scale", ctypes.c_void_p),
        ("in_suh", ctypes.c_void_p), ("rot_tab", ctypes.c_void_p), ("out_svh", ctypes.c_void_p),
        ("max_tokens", ctypes.c_int32), ("decode_max_rows", ctypes.c_int32), ("deterministic", ctypes.c_int32),
        ("gate_suh", ctypes.c_void_p), ("up_suh", ctypes.c_void_p), ("input_sign_rows", ctypes.c_int32),
        ("fc1_wscale", ctypes.c_void_p), ("fc2_wscale", ctypes.c_void_p),
    ]


class LinearDesc(ctypes.Structure):
    """tm_linear_desc (include/trellis_moe.h)."""
    _fields_ = [("N", ctypes.c_int32), ("K", ctypes.c_int32), ("bits", ctypes.c_int32),
                ("rot_in", ctypes.c_int32), ("rot_out", ctypes.c_int32), ("max_tokens", ctypes.c_int32),
                ("payload", ctypes.c_void_p), ("scale", ctypes.c_void_p), ("suh", ctypes.c_void_p),
                ("svh", ctypes.c_void_p)]


class TrellisMoEError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__("%s: %s" % (STATUS.get(status, status), msg))
        self.status = status


_lib: Optional[ctypes.CDLL] = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError("libtrellis_moe.so is not built (%s); run __graft_entry__.build()" % path)
    lib = ctypes.CDLL(path)
    P, I32, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    sig = {
        "trellis_moe_prepare": (I32, [ctypes.POINTER(LayerDesc), ctypes.POINTER(P), ctypes.POINTER(SZ)]),
        "trellis_moe_workspace_size": (SZ, [P, I32]),
        "trellis_moe_forward": (I32, [P, P, P, P, I32, I32, P, P, SZ, P]),
        "trellis_moe_forward_logits": (I32, [P, P, P, I32, I32, P, P, SZ, P]),
        "trellis_moe_forward_host": (I32, [P, P, P, I32, I32, P, P, SZ, P]),
        "trellis_moe_route": (I32, [P, I32, I32, I32, P, P, P]),
        "trellis_moe_route_map": (I32, [P, P, I32, I32, P, P, P, P, P, SZ, P]),
        "trellis_moe_rotate_quant": (I32, [P, P, I32, I32, P, P, P]),
        "trellis_moe_decode_tiles": (I32, [P, I32, I32, I32, I32, I32, P, P]),
        "trellis_moe_workspace_region": (I32, [P, I32, I32, ctypes.POINTER(SZ), ctypes.POINTER(SZ)]),
        "trellis_moe_set_stage_events": (I32, [P, ctypes.POINTER(P), I32]),
        "trellis_moe_set_decode_lut": (I32, [P, I32]),
        "trellis_moe_poll_error": (I32, [P, P, ctypes.POINTER(ctypes.c_uint32), P]),
        "trellis_moe_set_wait_test": (I32, [P, ctypes.c_uint64, I32]),
        "trellis_moe_last_error": (ctypes.c_char_p, []),
        "trellis_moe_destroy": (None, [P]),
        "trellis_moe_route_map_static": (I32, [P, I32, I32, I32, I32, P, P, P, P, P]),
        "trellis_linear_prepare": (I32, [ctypes.POINTER(LinearDesc), ctypes.POINTER(P), ctypes.POINTER(SZ)]),
        "trellis_linear_workspace_size": (SZ, [P, I32]),
        "trellis_linear_forward": (I32, [P, P, I32, P, P, SZ, P]),
        "trellis_linear_poll_error": (I32, [P, P, ctypes.POINTER(ctypes.c_uint32), P]),
        "trellis_linear_destroy": (None, [P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def _check(status: int):
    if status != TM_OK:
        msg = load_library().trellis_moe_last_error().decode()
        raise TrellisMoEError(status, msg)


def _torch():
    import torch
    if not torch.cuda.is_available():
        raise RuntimeError("trellis_moe needs a CUDA device; no CPU fallback exists")
    return torch


def _stream_ptr(stream=None):
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _raw_stream(stream=None) -> int:
    """The CUDA stream handle as an int: the given stream's, else the current
    one's (read without building a Stream object where torch offers that)."""
    if stream is not None:
        return stream.cuda_stream
    torch = _torch()
    raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
    if raw is not None:
        return raw(torch.cuda.current_device())
    return torch.cuda.current_stream().cuda_stream


def _ptr(t) -> ctypes.c_void_p:
    return ctypes.c_void_p(t.data_ptr())


def to_device_u8(arr: np.ndarray):
    """Upload a uint8 numpy array as a uint8 CUDA tensor."""
    torch = _torch()
    return torch.from_numpy(np.ascontiguousarray(np.asarray(arr, dtype=np.uint8))).cuda()


def to_device_u16(arr: np.ndarray):
    """Upload a uint16 / int16 numpy array as an int16 CUDA tensor."""
    torch = _torch()
    a = np.ascontiguousarray(np.asarray(arr).view(np.int16))
    return torch.from_numpy(a).cuda()


def route(logits, k: int, stream=None):
    """Top-k softmax router on device logits float32 [T, E] -> (ids int32, w float32)."""
    torch = _torch()
    lib = load_library()
    T, E = logits.shape
    ids = torch.empty((T, k), dtype=torch.int32, device=logits.device)
    w = torch.empty((T, k), dtype=torch.float32, device=logits.device)
    _check(lib.trellis_moe_route(_ptr(logits), T, E, k, _ptr(ids), _ptr(w), _stream_ptr(stream)))
    return ids, w


def route_map_static(ids, E: int, block: int, stream=None):
    """Route map through trellis_moe_route_map_static: no workspace and no
    allocation inside the library (for callers that cannot provide scratch).
    The result tensors here are allocated by torch, in the caller's code."""
    torch = _torch()
    lib = load_library()
    T, k = int(ids.shape[0]), int(ids.shape[1])
    R = T * k
    dev = ids.device
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    ros = torch.empty(R + E * (block - 1) + 1, dtype=torch.int32, device=dev)
    sor = torch.empty(max(R, 1), dtype=torch.int32, device=dev)
    with torch.cuda.device(dev):
        _check(lib.trellis_moe_route_map_static(_ptr(ids), T, E, k, block, _ptr(counts), _ptr(offsets), _ptr(ros),
                                                _ptr(sor), _stream_ptr(stream)))
    return {"counts": counts, "offsets": offsets, "route_of_slot": ros, "slot_of_route": sor[:R]}


class TrellisMoE:
    """One prepared layer. ``layer`` has the fields of ``synth.Layer`` (numpy,
    fp16 as uint16 bit patterns); its arrays are uploaded once."""

    def __init__(self, layer, max_tokens: int, decode_max_rows: int = 8, deterministic: bool = True):
        torch = _torch()
        self.lib = load_library()
        # the handle, its tables and workspace belong to the device current now
        self.device = torch.device("cuda", torch.cuda.current_device())
        self.E, self.H, self.I, self.topk = int(layer.E), int(layer.H), int(layer.I), int(layer.topk)
        self.bits = np.ascontiguousarray(np.asarray(layer.bits, dtype=np.uint8))
        self.fc1_payload = to_device_u16(layer.fc1_payload)
        self.fc2_payload = to_device_u16(layer.fc2_payload)
        self.fc1_scale = to_device_u16(layer.fc1_scale)
        self.fc2_scale = to_device_u16(layer.fc2_scale)
        self.in_suh = to_device_u16(layer.in_suh)
        self.rot_tab = to_device_u16(layer.rot_tab)
        self.out_svh = to_device_u16(layer.out_svh)
        g, u = getattr(layer, "gate_suh", None), getattr(layer, "up_suh", None)
        if (g is None) != (u is None):
            raise ValueError("gate_suh and up_suh must be given together")
        self.gate_suh = to_device_u16(np.asarray(g).reshape(-1, self.H)) if g is not None else None
        self.up_suh = to_device_u16(np.asarray(u).reshape(-1, self.H)) if u is not None else None
        w1, w2 = getattr(layer, "fc1_wscale", None), getattr(layer, "fc2_wscale", None)
        if (w1 is None) != (w2 is None):
            raise ValueError("fc1_wscale and fc2_wscale must be given together")
        self.fc1_wscale = to_device_u8(w1) if w1 is not None else None
        self.fc2_wscale = to_device_u8(w2) if w2 is not None else None
        d = LayerDesc()
        d.E, d.H, d.I, d.topk = self.E, self.H, self.I, self.topk
        d.rot_block_h, d.rot_block_i = int(layer.rot_block_h), int(layer.rot_block_i)
        d.bits_per_expert = self.bits.ctypes.data
        d.fc1_payload = self.fc1_payload.data_ptr()
        d.fc2_payload = self.fc2_payload.data_ptr()
        d.fc1_scale = self.fc1_scale.data_ptr()
        d.fc2_scale = self.fc2_scale.data_ptr()
        d.in_suh = self.in_suh.data_ptr()
        d.rot_tab = self.rot_tab.data_ptr()
        d.out_svh = self.out_svh.data_ptr()
        d.max_tokens = int(max_tokens)
        d.decode_max_rows = int(decode_max_rows)
        d.deterministic = 1 if deterministic else 0
        if self.gate_suh is not None:
            if self.gate_suh.shape != self.up_suh.shape:
                raise ValueError("gate_suh and up_suh must have the same shape")
            d.gate_suh = self.gate_suh.data_ptr()
            d.up_suh = self.up_suh.data_ptr()
            d.input_sign_rows = int(self.gate_suh.shape[0])
        if self.fc1_wscale is not None:
            d.fc1_wscale = self.fc1_wscale.data_ptr()
            d.fc2_wscale = self.fc2_wscale.data_ptr()
        self.desc = d
        handle = ctypes.c_void_p()
        ws = ctypes.c_size_t()
        _check(self.lib.trellis_moe_prepare(ctypes.byref(d), ctypes.byref(handle), ctypes.byref(ws)))
        self.handle = handle
        self.max_tokens = int(max_tokens)
        self.workspace_bytes = int(ws.value)
        self.workspace = torch.empty(self.workspace_bytes + 256, dtype=torch.uint8, device=self.device)
        off = (-self.workspace.data_ptr()) % 256
        self.workspace = self.workspace[off:off + self.workspace_bytes]

    def close(self):
        if getattr(self, "handle", None):
            self.lib.trellis_moe_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -- full layer -------------------------------------------------------
    def forward(self, x, ids, w, mode="auto", out=None, stream=None):
        """x bf16/int16 [T, H], ids int32 [T, k], w float32 [T, k] -> float32 [T, H]."""
        torch = _torch()
        T = int(x.shape[0])
        if out is None:
            out = torch.empty((T, self.H), dtype=torch.float32, device=self.device)
        _check(self.lib.trellis_moe_forward(self.handle, _ptr(x), _ptr(ids), _ptr(w), T, MODES.get(mode, mode),
                                            _ptr(out), _ptr(self.workspace), self.workspace_bytes,
                                            _stream_ptr(stream)))
        return out

    def forward_logits(self, x, logits, mode="auto", out=None, stream=None):
        torch = _torch()
        T = int(x.shape[0])
        if out is None:
            out = torch.empty((T, self.H), dtype=torch.float32, device=self.device)
        _check(self.lib.trellis_moe_forward_logits(self.handle, _ptr(x), _ptr(logits), T, MODES.get(mode, mode),
                                                   _ptr(out), _ptr(self.workspace), self.workspace_bytes,
                                                   _stream_ptr(stream)))
        return out

    def forward_host(self, x_host, logits_host, out_host, mode="auto", stream=None):
        """Host (pinned CPU tensor) inputs and output; synchronises the stream.
        The per-call marshalling is kept to plain ints: it is part of every
        end-to-end call."""
        fh = self.__dict__.get("_forward_host_fn")
        if fh is None:
            fh = self._forward_host_fn = self.lib.trellis_moe_forward_host
        st = fh(self.handle, x_host.data_ptr(), logits_host.data_ptr(), x_host.shape[0], MODES.get(mode, mode),
                out_host.data_ptr(), self.workspace.data_ptr(), self.workspace_bytes, _raw_stream(stream))
        if st != TM_OK:
            _check(st)
        return out_host

    # -- single steps (parity tests) -------------------------------------
    def route_map(self, ids, block: int, stream=None):
        torch = _torch()
        T = int(ids.shape[0])
        R = T * self.topk
        dev = self.device
        counts = torch.empty(self.E, dtype=torch.int32, device=dev)
        offsets = torch.empty(self.E + 1, dtype=torch.int32, device=dev)
        ros = torch.empty(R + self.E * (block - 1) + 1, dtype=torch.int32, device=dev)
        sor = torch.empty(max(R, 1), dtype=torch.int32, device=dev)
        _check(self.lib.trellis_moe_route_map(self.handle, _ptr(ids), T, block, _ptr(counts), _ptr(offsets),
                                              _ptr(ros), _ptr(sor), _ptr(self.workspace), self.workspace_bytes,
                                              _stream_ptr(stream)))
        return {"counts": counts, "offsets": offsets, "route_of_slot": ros, "slot_of_route": sor[:R]}

    def rotate_quant(self, x, mode, stream=None):
        torch = _torch()
        T = int(x.shape[0])
        m = MODES.get(mode, mode)
        if m == MODE_W4A8:
            xq = torch.empty((T, self.H), dtype=torch.uint8, device=self.device)
            xs = torch.empty((T, self.H // 32), dtype=torch.uint8, device=self.device)
        else:
            xq = torch.empty((T, self.H), dtype=torch.int16, device=self.device)
            xs = torch.empty(1, dtype=torch.uint8, device=self.device)
        _check(self.lib.trellis_moe_rotate_quant(self.handle, _ptr(x), T, m, _ptr(xq), _ptr(xs), _stream_ptr(stream)))
        return xq, (xs if m == MODE_W4A8 else None)

    def decode_tiles(self, proj: int, expert: int, tile0: int, ntiles: int, mode="w4a16", stream=None):
        torch = _torch()
        m = MODES.get(mode, mode)
        dt = torch.uint8 if m == MODE_W4A8 else torch.int16
        dst = torch.empty((ntiles, 256), dtype=dt, device=self.device)
        _check(self.lib.trellis_moe_decode_tiles(self.handle, proj, expert, tile0, ntiles, m, _ptr(dst),
                                                 _stream_ptr(stream)))
        return dst

    def workspace_region(self, T: int, which: int):
        off, nb = ctypes.c_size_t(), ctypes.c_size_t()
        _check(self.lib.trellis_moe_workspace_region(self.handle, T, which, ctypes.byref(off), ctypes.byref(nb)))
        return self.workspace[off.value:off.value + nb.value]

    def set_decode_lut(self, on: bool):
        """Decode-rows expansion by codebook table lookup (True) or by the
        hash (False, the default); see the C header."""
        _check(self.lib.trellis_moe_set_decode_lut(self.handle, 1 if on else 0))

    def set_stage_events(self, events):
        """events: None, or 7 torch.cuda.Event (or None) recorded at the stage
        boundaries of every later forward call (see the C header)."""
        if events is None:
            _check(self.lib.trellis_moe_set_stage_events(self.handle, None, 0))
            return
        assert len(events) == 7
        arr = (ctypes.c_void_p * 7)()
        for i, ev in enumerate(events):
            if ev is not None:
                if not ev.cuda_event:
                    ev.record()     # torch creates the CUDA event lazily
                arr[i] = ev.cuda_event
        _check(self.lib.trellis_moe_set_stage_events(self.handle, arr, 7))

    def set_wait_test(self, wait_limit_ns: int = 0, stall_issuer: bool = False):
        """Limit of the tensor-core kernels' pipeline waits, and the stalled
        issuer used to test that they give up (see the C header)."""
        _check(self.lib.trellis_moe_set_wait_test(self.handle, int(wait_limit_ns), 1 if stall_issuer else 0))

    def poll_error(self, stream=None) -> int:
        flags = ctypes.c_uint32()
        st = self.lib.trellis_moe_poll_error(self.handle, _ptr(self.workspace), ctypes.byref(flags), _stream_ptr(stream))
        if st not in (TM_OK, -5):
            _check(st)
        return int(flags.value)


class TrellisLinear:
    """One prepared dense trellis linear layer. ``lin`` has the fields of
    ``synth.Linear`` (numpy, fp16 as uint16 bit patterns); its arrays are
    uploaded once."""

    def __init__(self, lin, max_tokens: int):
        torch = _torch()
        self.lib = load_library()
        self.N, self.K = int(lin.N), int(lin.K)
        self.payload = to_device_u16(lin.payload)
        self.scale = to_device_u16(lin.scale)
        self.suh = to_device_u16(lin.suh)
        self.svh = to_device_u16(lin.svh)
        d = LinearDesc()
        d.N, d.K, d.bits = self.N, self.K, int(lin.bits)
        d.rot_in, d.rot_out = int(lin.rot_in), int(lin.rot_out)
        d.max_tokens = int(max_tokens)
        d.payload = self.payload.data_ptr()
        d.scale = self.scale.data_ptr()
        d.suh = self.suh.data_ptr()
        d.svh = self.svh.data_ptr()
        self.desc = d
        handle = ctypes.c_void_p()
        ws = ctypes.c_size_t()
        _check(self.lib.trellis_linear_prepare(ctypes.byref(d), ctypes.byref(handle), ctypes.byref(ws)))
        self.handle = handle
        self.workspace_bytes = int(ws.value)
        self.workspace = torch.empty(self.workspace_bytes + 256, dtype=torch.uint8, device="cuda")
        off = (-self.workspace.data_ptr()) % 256
        self.workspace = self.workspace[off:off + self.workspace_bytes]

    def close(self):
        if getattr(self, "handle", None):
            self.lib.trellis_linear_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def forward(self, x, out=None, stream=None):
        """x bf16/int16 [T, K] -> float32 [T, N]."""
        torch = _torch()
        T = int(x.shape[0])
        if out is None:
            out = torch.empty((T, self.N), dtype=torch.float32, device="cuda")
        _check(self.lib.trellis_linear_forward(self.handle, _ptr(x), T, _ptr(out), _ptr(self.workspace),
                                               self.workspace_bytes, _stream_ptr(stream)))
        return out

    def poll_error(self, stream=None) -> int:
        flags = ctypes.c_uint32(0)
        st = self.lib.trellis_linear_poll_error(self.handle, _ptr(self.workspace), ctypes.byref(flags),
                                                _stream_ptr(stream))
        if st not in (TM_OK, -5):
            _check(st)
        return int(flags.value)
