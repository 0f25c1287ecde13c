"""Seeded synthetic inputs for the trellis-coded MoE layer.

This module only draws random numbers and lays them out in the shapes the
layer takes. It contains none of the layer's arithmetic (no decoding, no
rotation, no routing, no quantisation), so both the CUDA path and the CPU
oracle can take their inputs from it.

Every draw comes from the raw 64-bit output of a PCG64 generator seeded
through ``numpy.random.SeedSequence([seed, stream])``. Both algorithms are
fixed by their published definitions, so the raw words are identical on every
platform and numpy version. Uniform and normal variates are derived from the
raw words here (53-bit uniforms, Box-Muller normals) instead of through
``Generator`` methods, whose streams numpy does not promise to keep stable.

Recipe (the workloads named in ``CONFIGS``):
  * payload: uniform random int16 words, 16*K words per 256-weight tile;
  * per-channel scales: fp16 of U[0.01, 0.03];
  * rotation sign vectors (input suh, gate/up svh, down suh, output svh): +-1 fp16;
  * activations: bf16 of N(0, 1);
  * router logits: N(0, sigma^2), or a Zipf(s) expert preference plus
    Gumbel(0, 1) noise, which makes top-k selection sample experts without
    replacement with probability proportional to rank^-s;
  * TrellisMX-style weight scales: UE8M0 bytes 127 + k, k uniform in [-3, 3].
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import numpy as np

# Stream ids keep every tensor's draw independent of the others and of the
# order in which they are requested.
_S_BITS, _S_FC1, _S_FC2, _S_S1, _S_S2, _S_SUH, _S_ROT, _S_SVH = range(8)
_S_X, _S_LOGITS, _S_PERM, _S_GUMBEL = 100, 101, 102, 103
_S_LIN_W, _S_LIN_S, _S_LIN_SUH, _S_LIN_SVH, _S_LIN_X = 300, 301, 302, 303, 304
_S_GATE_SUH, _S_UP_SUH = 400, 401
_S_WS1, _S_WS2 = 500, 501


@dataclasses.dataclass(frozen=True)
class LayerConfig:
    """Shape of one MoE layer and of the token batch fed to it."""

    name: str
    E: int            # experts
    H: int            # hidden size
    I: int            # intermediate size (per projection half)
    topk: int
    T: int            # tokens in the default batch
    bits: Sequence[int]   # allowed trellis bit-widths K; one value = uniform
    rot_block_h: int
    rot_block_i: int
    mode: str         # "w4a16" or "w4a8"
    logits: str       # "normal" or "zipf"
    logit_sigma: float = 1.0
    zipf_s: float = 1.1
    seed: int = 0
    mx: bool = False   # TrellisMX-style weights: UE8M0 scale bytes per 32 weights


CONFIGS = {
    "tiny": LayerConfig("tiny", E=8, H=256, I=128, topk=2, T=4, bits=(4,),
                        rot_block_h=128, rot_block_i=128, mode="w4a16",
                        logits="normal", logit_sigma=1.0, seed=0),
    "decode": LayerConfig("decode", E=128, H=1024, I=512, topk=8, T=8, bits=(4,),
                          rot_block_h=128, rot_block_i=128, mode="w4a8",
                          logits="normal", logit_sigma=1.5, seed=1),
    "prefill": LayerConfig("prefill", E=128, H=1024, I=512, topk=8, T=2048, bits=(4,),
                           rot_block_h=128, rot_block_i=128, mode="w4a16",
                           logits="zipf", zipf_s=1.1, seed=2),
    "odd": LayerConfig("odd", E=64, H=2560, I=320, topk=10, T=512, bits=(2, 3, 4),
                       rot_block_h=128, rot_block_i=64, mode="w4a16",
                       logits="normal", logit_sigma=1.0, seed=3),
    "large": LayerConfig("large", E=160, H=5120, I=1536, topk=8, T=4096, bits=(4,),
                         rot_block_h=128, rot_block_i=128, mode="w4a16",
                         logits="normal", logit_sigma=1.0, seed=4),
    # TrellisMX-style decode layer: K2-K4 per expert, E4M3 weights with one
    # UE8M0 scale per 32 weights, 512-point hidden-side rotation blocks
    "trellismx": LayerConfig("trellismx", E=64, H=2048, I=512, topk=8, T=8, bits=(2, 3, 4),
                             rot_block_h=512, rot_block_i=128, mode="w4a8",
                             logits="normal", logit_sigma=1.0, seed=5, mx=True),
}


class Stream:
    """Raw PCG64 words for one (seed, stream) pair, with derived variates."""

    def __init__(self, seed: int, stream: int):
        self._bg = np.random.PCG64(np.random.SeedSequence([int(seed), int(stream)]))

    def raw(self, n: int) -> np.ndarray:
        if n == 0:
            return np.zeros(0, dtype=np.uint64)
        return np.asarray(self._bg.random_raw(int(n)), dtype=np.uint64)

    def uniform(self, n: int) -> np.ndarray:
        """Uniform in [0, 1) with 53 random bits."""
        return (self.raw(n) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)

    def normal(self, n: int) -> np.ndarray:
        """Standard normals by the Box-Muller transform (two per uniform pair)."""
        m = (n + 1) // 2
        u1 = 1.0 - self.uniform(m)          # (0, 1]
        u2 = self.uniform(m)
        r = np.sqrt(-2.0 * np.log(u1))
        out = np.empty(2 * m, dtype=np.float64)
        out[0::2] = r * np.cos(2.0 * np.pi * u2)
        out[1::2] = r * np.sin(2.0 * np.pi * u2)
        return out[:n]

    def words16(self, n: int) -> np.ndarray:
        """n uniform random 16-bit words as int16."""
        m = (n + 3) // 4
        return self.raw(m).view(np.uint16)[:n].astype(np.uint16).view(np.int16)

    def below(self, n: int, bound: int) -> np.ndarray:
        """n integers uniform in [0, bound) (multiply-shift on 32 raw bits)."""
        r = self.raw(n) >> np.uint64(32)
        return ((r * np.uint64(bound)) >> np.uint64(32)).astype(np.int64)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float64 data to bfloat16 (via float32, then round-to-nearest-even
    on the float32 bits) and return the 16-bit patterns as uint16."""
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    rounded = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return rounded.astype(np.uint16)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of bfloat16 bit patterns."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def fp16_bits(x: np.ndarray) -> np.ndarray:
    return np.asarray(x, dtype=np.float64).astype(np.float16).view(np.uint16)


def _signs(stream: Stream, n: int) -> np.ndarray:
    b = (stream.raw(n) >> np.uint64(63)).astype(np.float64)
    return fp16_bits(1.0 - 2.0 * b)


@dataclasses.dataclass
class Layer:
    """Host copy of one layer's parameters (fp16 stored as uint16 bit patterns)."""

    E: int
    H: int
    I: int
    topk: int
    rot_block_h: int
    rot_block_i: int
    bits: np.ndarray          # uint8 [E]
    fc1_payload: np.ndarray   # int16, per expert [2I/16][H/16][16*K_e], concatenated
    fc2_payload: np.ndarray   # int16, per expert [H/16][I/16][16*K_e], concatenated
    fc1_scale: np.ndarray     # uint16 (fp16) [E, 2I]
    fc2_scale: np.ndarray     # uint16 (fp16) [E, H]
    in_suh: np.ndarray        # uint16 (fp16) [H]
    rot_tab: np.ndarray       # uint16 (fp16) [E, 3I] = gate svh | up svh | down suh
    out_svh: np.ndarray       # uint16 (fp16) [E, H]
    # optional input sign layouts: separate gate and up signs, each [1, H]
    # (shared by the experts) or [E, H] (per expert); None = in_suh for both
    gate_suh: Optional[np.ndarray] = None
    up_suh: Optional[np.ndarray] = None
    # optional TrellisMX-style weight scales: UE8M0 bytes, one per 32 weights
    # of a row along the contraction axis: [E, 2I, H/32] and [E, H, I/32]
    fc1_wscale: Optional[np.ndarray] = None
    fc2_wscale: Optional[np.ndarray] = None


def make_layer(cfg: LayerConfig, seed: Optional[int] = None,
               bits: Optional[Sequence[int]] = None) -> Layer:
    """Draw one layer's parameters for ``cfg`` (optionally overriding the seed
    or forcing per-expert bit-widths)."""
    seed = cfg.seed if seed is None else seed
    E, H, I = cfg.E, cfg.H, cfg.I
    if bits is None:
        choices = list(cfg.bits)
        if len(choices) == 1:
            kb = np.full(E, choices[0], dtype=np.uint8)
        else:
            idx = Stream(seed, _S_BITS).below(E, len(choices))
            kb = np.asarray([choices[i] for i in idx], dtype=np.uint8)
    else:
        kb = np.asarray(bits, dtype=np.uint8)
        assert kb.shape == (E,)
    tiles1 = (2 * I // 16) * (H // 16)
    tiles2 = (H // 16) * (I // 16)
    n1 = int(sum(tiles1 * 16 * int(k) for k in kb))
    n2 = int(sum(tiles2 * 16 * int(k) for k in kb))
    s_lo, s_hi = 0.01, 0.03
    return Layer(
        E=E, H=H, I=I, topk=cfg.topk,
        rot_block_h=cfg.rot_block_h, rot_block_i=cfg.rot_block_i,
        bits=kb,
        fc1_payload=Stream(seed, _S_FC1).words16(n1),
        fc2_payload=Stream(seed, _S_FC2).words16(n2),
        fc1_scale=fp16_bits(s_lo + (s_hi - s_lo) * Stream(seed, _S_S1).uniform(E * 2 * I)).reshape(E, 2 * I),
        fc2_scale=fp16_bits(s_lo + (s_hi - s_lo) * Stream(seed, _S_S2).uniform(E * H)).reshape(E, H),
        in_suh=_signs(Stream(seed, _S_SUH), H),
        rot_tab=_signs(Stream(seed, _S_ROT), E * 3 * I).reshape(E, 3 * I),
        out_svh=_signs(Stream(seed, _S_SVH), E * H).reshape(E, H),
        fc1_wscale=_ue8m0(Stream(seed, _S_WS1), (E, 2 * I, H // 32)) if cfg.mx else None,
        fc2_wscale=_ue8m0(Stream(seed, _S_WS2), (E, H, I // 32)) if cfg.mx else None,
    )


def _ue8m0(stream: Stream, shape) -> np.ndarray:
    """UE8M0 scale bytes 127 + k with k uniform in [-3, 3]."""
    n = int(np.prod(shape))
    return (124 + stream.below(n, 7)).astype(np.uint8).reshape(shape)


def make_tokens(cfg: LayerConfig, T: Optional[int] = None, seed: Optional[int] = None):
    """Activations (bf16 bit patterns [T, H]) and router logits (float32 [T, E])."""
    seed = cfg.seed if seed is None else seed
    T = cfg.T if T is None else T
    x = bf16_bits(Stream(seed, _S_X).normal(T * cfg.H)).reshape(T, cfg.H)
    if cfg.logits == "normal":
        logits = (cfg.logit_sigma * Stream(seed, _S_LOGITS).normal(T * cfg.E)).astype(np.float32)
    elif cfg.logits == "zipf":
        rank = permutation(Stream(seed, _S_PERM), cfg.E)
        pref = -cfg.zipf_s * np.log(rank.astype(np.float64) + 1.0)
        u = Stream(seed, _S_GUMBEL).uniform(T * cfg.E)
        u = np.minimum(np.maximum(u, 2.0 ** -53), 1.0 - 2.0 ** -53)
        gumbel = -np.log(-np.log(u))
        logits = (pref[None, :] + gumbel.reshape(T, cfg.E)).astype(np.float32).reshape(-1)
    else:
        raise ValueError(cfg.logits)
    return x, logits.reshape(T, cfg.E)


def permutation(stream: Stream, n: int) -> np.ndarray:
    """Fisher-Yates shuffle of 0..n-1 driven by ``stream``."""
    p = np.arange(n, dtype=np.int64)
    draws = stream.raw(max(n - 1, 0))
    for i in range(n - 1, 0, -1):
        j = int((int(draws[n - 1 - i]) >> 32) * (i + 1) >> 32)
        p[i], p[j] = p[j], p[i]
    return p


def random_ids(seed: int, T: int, E: int, k: int) -> np.ndarray:
    """Top-k expert ids without a router: k distinct experts per token, drawn
    uniformly (used for route-map tests that need arbitrary id patterns)."""
    s = Stream(seed, 200)
    out = np.empty((T, k), dtype=np.int32)
    for t in range(T):
        out[t] = permutation(s, E)[:k]
    return out


@dataclasses.dataclass
class Linear:
    """Host copy of one dense trellis-coded linear layer: W~ [N, K] as tiles
    [N/16][K/16][16*bits] int16 words, output scales and signs [N], input
    signs [K] (fp16 stored as uint16 bit patterns)."""

    N: int
    K: int
    bits: int
    rot_in: int
    rot_out: int
    payload: np.ndarray   # int16 [N/16 * K/16 * 16 * bits]
    scale: np.ndarray     # uint16 (fp16) [N]
    suh: np.ndarray       # uint16 (fp16) [K]
    svh: np.ndarray       # uint16 (fp16) [N]


def make_linear(N: int, K: int, bits: int = 4, rot_in: int = 128, rot_out: int = 128, seed: int = 5) -> Linear:
    """Draw a dense trellis linear layer with the layer recipe (uniform payload
    words, fp16 U[0.01, 0.03] scales, +-1 signs)."""
    n = (N // 16) * (K // 16) * 16 * bits
    return Linear(
        N=N, K=K, bits=bits, rot_in=rot_in, rot_out=rot_out,
        payload=Stream(seed, _S_LIN_W).words16(n),
        scale=fp16_bits(0.01 + 0.02 * Stream(seed, _S_LIN_S).uniform(N)),
        suh=_signs(Stream(seed, _S_LIN_SUH), K),
        svh=_signs(Stream(seed, _S_LIN_SVH), N),
    )


def make_linear_tokens(lin: Linear, T: int, seed: int = 5) -> np.ndarray:
    """Activations for a dense linear: bf16 bit patterns of N(0, 1), [T, K]."""
    return bf16_bits(Stream(seed, _S_LIN_X).normal(T * lin.K)).reshape(T, lin.K)


def with_input_signs(layer: Layer, rows: int, seed: int = 9) -> Layer:
    """A copy of ``layer`` with separate gate and up input signs of ``rows``
    rows (1: shared by the experts, E: per expert), drawn as +-1."""
    assert rows in (1, layer.E)
    return dataclasses.replace(
        layer,
        gate_suh=_signs(Stream(seed, _S_GATE_SUH), rows * layer.H).reshape(rows, layer.H),
        up_suh=_signs(Stream(seed, _S_UP_SUH), rows * layer.H).reshape(rows, layer.H),
    )
