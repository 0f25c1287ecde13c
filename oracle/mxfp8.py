"""E4M3 rounding and MXFP8 block quantisation (oracle; test use only).

MXFP8 here is E4M3 elements with one UE8M0 (E8M0) power-of-two exponent per 32
consecutive values along the contraction axis (flashinfer PR #69 "b12x fused
MoE: TrellisMX (procedural NPK) source format with an in-tree P8 runtime",
Description: one UE8M0 byte per 32 values; Evidence, precision notes: the
exponent comes from the exact FP32 bits of amax / 448 and is clamped to
[-127, 127]).

Readings where the pages leave the step open:
  * The exponent is the ceiling of log2(q), q = fp32(amax / 448) with IEEE
    round-to-nearest-even division, i.e. the smallest e with 2^e >= q. The
    precision note objects to a log2 that rounds quotients just above a power
    of two *down* onto it, which only matters under a ceiling. amax = 0 gives
    e = -127. The stored byte is e + 127.
  * Elements are E4M3 = round-to-nearest-even with saturation to +-448 of
    v * 2^-e (the cvt.rn.satfinite rule); the sign of a value that rounds to
    zero is kept (negative zero is byte 0x80).
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def _e4m3_table() -> np.ndarray:
    """Magnitudes of the non-negative finite E4M3 codes 0..126 (0x7F is NaN)."""
    vals = []
    for c in range(127):
        e, m = c >> 3, c & 7
        vals.append(m * 2.0 ** -9 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7))
    return np.asarray(vals, dtype=np.float64)


E4M3_VALUES = _e4m3_table()


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """Exact float64 value of E4M3 bytes (NaN for 0x7F / 0xFF)."""
    c = np.asarray(codes, dtype=np.uint8)
    mag_code = (c & 0x7F).astype(np.int64)
    mag = np.where(mag_code == 127, np.nan, E4M3_VALUES[np.minimum(mag_code, 126)])
    return np.where(c & 0x80, -mag, mag)


def e4m3_encode(v: np.ndarray) -> np.ndarray:
    """Round to nearest E4M3 (ties to the even code), saturating to 448."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    idx = np.searchsorted(E4M3_VALUES, a, side="left")      # first value >= a
    idx = np.minimum(idx, 126)
    lo = np.maximum(idx - 1, 0)
    d_hi = E4M3_VALUES[idx] - a
    d_lo = a - E4M3_VALUES[lo]
    pick_lo = (d_lo < d_hi) | ((d_lo == d_hi) & (lo % 2 == 0))
    code = np.where(pick_lo & (idx > 0), lo, idx)
    code = np.where(a >= E4M3_MAX, 126, code)                # satfinite
    code = code.astype(np.uint8)
    sign = np.signbit(v)
    out = np.where(sign, code | 0x80, code).astype(np.uint8)
    return np.where(np.isnan(v), np.uint8(0x7F), out).astype(np.uint8)


def e4m3_round(v: np.ndarray) -> np.ndarray:
    """Value of the E4M3 rounding of v."""
    return e4m3_decode(e4m3_encode(v))


def e8m0_exponent(amax: np.ndarray) -> np.ndarray:
    """Block exponent e in [-127, 127] from the block's max |v| (float32 data)."""
    a = np.asarray(amax, dtype=np.float32).astype(np.float64)
    q = (a / E4M3_MAX).astype(np.float32).astype(np.float64)   # fp32 RNE quotient
    frac, ex = np.frexp(q)            # q = frac * 2^ex, frac in [0.5, 1)
    e = np.where(frac == 0.5, ex - 1, ex)                      # ceil(log2 q), exact
    e = np.where(q == 0.0, -127, e)
    return np.clip(e, -127, 127).astype(np.int64)


def quantize_mxfp8(v: np.ndarray):
    """Quantise float32 data [..., n] (n % 32 == 0) in blocks of 32 along the
    last axis. Returns (E4M3 bytes [..., n], E8M0 bytes [..., n/32],
    dequantised float64 values [..., n])."""
    v32 = np.asarray(v, dtype=np.float32)
    n = v32.shape[-1]
    assert n % 32 == 0, n
    blocks = v32.astype(np.float64).reshape(*v32.shape[:-1], n // 32, 32)
    e = e8m0_exponent(np.max(np.abs(blocks), axis=-1))
    scaled = blocks * np.exp2(-e.astype(np.float64))[..., None]   # exact power-of-two scaling
    codes = e4m3_encode(scaled)
    deq = e4m3_decode(codes) * np.exp2(e.astype(np.float64))[..., None]
    return (codes.reshape(v32.shape), (e + 127).astype(np.uint8),
            deq.reshape(v32.shape))
