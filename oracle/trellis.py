"""Trellis tile decode, written out from its definition (oracle; test use only).

Format facts from the pages:
  * A tile holds 256 weights at K bits each, stored as 16*K int16 words
    (sparkinfer PR #90 "moe: integrate EXL3 Trellis into the fused W4A16 API",
    review of prepare.py: the trellis3_t256 shape check ``prefix + (16*K,)``).
  * The codebook is the procedural "MCG" one, with the multiplier 0xCBAC1FED,
    the mask 0x8fff8fff and a third constant 0x3b603b60 (same page, review of
    intrinsics.py: _TRELLIS_MCG, _TRELLIS_MASK, _TRELLIS_OR).
  * Each weight is addressed by a 16-bit state of a bitshift trellis that wraps
    around the tile (tail-biting).

Readings where the pages are silent (each a free format choice or the plainest
reading of the constants; the CUDA decoder follows the same statement):
  * Stream order: bit p of a tile's stream is bit (15 - p mod 16) of int16 word
    floor(p / 16) -- most significant bit first, words in storage order.
  * State of weight j (0..255): the 16 stream bits p = (j+1)K-16 .. (j+1)K-1,
    taken modulo 256K, first bit most significant. Consecutive states then
    satisfy s_j = ((s_{j-1} << K) | next K bits) & 0xFFFF, and s_0 reaches
    back around the end of the stream.
  * Codebook: x = s * 0xCBAC1FED mod 2^32; y = (x & 0x8fff8fff) XOR 0x3b603b60;
    the two 16-bit halves of y are fp16 numbers and the weight is their sum
    rounded to nearest-even in fp16. The page names the third constant "OR";
    XOR is read here because OR would force four mantissa bits of every half to
    one and collapse the codebook from 10,746 to 1,545 distinct values. The
    sign bits and exponents are the same under both readings.
    PARITY UNPINNED against an outside implementation: the pages print no
    decoded sample, so only hand-computed values of this reading pin it.
  * Placement: weight j of tile (tn, tk) is W[16*tn + j // 16, 16*tk + j % 16]
    (row = output channel, column = input channel); tiles are stored row-tile
    major, [rows/16][cols/16][16*K] words per expert, experts concatenated.
"""
from __future__ import annotations

import concurrent.futures
import os

import numpy as np

MCG_MULT = 0xCBAC1FED
MCG_MASK = 0x8FFF8FFF
MCG_XOR = 0x3B603B60


def codebook_fp16(states: np.ndarray) -> np.ndarray:
    """cb(s) for an array of 16-bit states; returns float16 values."""
    s = np.asarray(states, dtype=np.uint64)
    x = (s * np.uint64(MCG_MULT)) & np.uint64(0xFFFFFFFF)
    y = (x & np.uint64(MCG_MASK)) ^ np.uint64(MCG_XOR)
    lo = (y & np.uint64(0xFFFF)).astype(np.uint16).view(np.float16)
    hi = (y >> np.uint64(16)).astype(np.uint16).view(np.float16)
    # float64 holds the exact sum of two fp16 numbers, so one conversion to
    # float16 is the correctly rounded (nearest-even) fp16 addition.
    return (lo.astype(np.float64) + hi.astype(np.float64)).astype(np.float16)


def codebook_scalar(s: int) -> float:
    """cb(s) for one state, with plain integer arithmetic."""
    x = (int(s) * MCG_MULT) % (1 << 32)
    y = (x & MCG_MASK) ^ MCG_XOR
    lo = np.array([y & 0xFFFF], dtype=np.uint16).view(np.float16)[0]
    hi = np.array([y >> 16], dtype=np.uint16).view(np.float16)[0]
    return float(np.float16(float(lo) + float(hi)))


def stream_bits(words: np.ndarray) -> np.ndarray:
    """Bits of tile streams: words [..., 16K] int16 -> bits [..., 256K] uint8,
    b_p = bit (15 - p mod 16) of word floor(p/16)."""
    w = np.ascontiguousarray(np.asarray(words).astype(np.int16).view(np.uint16))
    be = w.astype(">u2")                       # big-endian bytes: high byte first
    return np.unpackbits(be.view(np.uint8), axis=-1, bitorder="big")


def state_bit_index(K: int) -> np.ndarray:
    """[256, 16] stream positions of the 16 bits of each state, MSB first."""
    n = 256 * K
    j = np.arange(256)[:, None]
    i = np.arange(16)[None, :]
    return ((j + 1) * K - 16 + i) % n


def tile_states(words: np.ndarray, K: int) -> np.ndarray:
    """States s_0..s_255 of tile streams: words [..., 16K] -> uint32 [..., 256]."""
    words = np.asarray(words)
    assert words.shape[-1] == 16 * K, (words.shape, K)
    bits = stream_bits(words)                       # [..., 256K]
    g = bits[..., state_bit_index(K)]               # [..., 256, 16], MSB first
    packed = np.packbits(g, axis=-1, bitorder="big")  # [..., 256, 2] bytes, high first
    return packed.view(">u2")[..., 0].astype(np.uint32)


def tile_states_scalar(words, K: int) -> list:
    """Bit-by-bit statement of the states of one tile (pure Python)."""
    w = [int(v) & 0xFFFF for v in words]
    n = 256 * K
    bit = lambda p: (w[p // 16] >> (15 - p % 16)) & 1
    out = []
    for j in range(256):
        s = 0
        for i in range(16):
            s = (s << 1) | bit(((j + 1) * K - 16 + i) % n)
        out.append(s)
    return out


def tile_states_words(words: np.ndarray, K: int) -> np.ndarray:
    """The same states read as 16-bit windows of 32-bit word pairs: with
    q = (j+1)K-16 mod 256K, w = q // 16 and o = q % 16, the window is the low
    16 bits of ((word[w] << 16 | word[w+1]) >> (16 - o)), words taken
    circularly. Equal to tile_states (tested); used for speed."""
    words = np.asarray(words)
    nw = 16 * K
    assert words.shape[-1] == nw, (words.shape, K)
    u = words.astype(np.int16).view(np.uint16).astype(np.uint32)
    q = ((np.arange(256) + 1) * K - 16) % (256 * K)
    w, o = q // 16, q % 16
    pair = (u[..., w] << np.uint32(16)) | u[..., (w + 1) % nw]
    return (pair >> (16 - o).astype(np.uint32)) & np.uint32(0xFFFF)


def decode_tiles_fp16(words: np.ndarray, K: int) -> np.ndarray:
    """Decoded weights of tiles in weight order j: [..., 16K] -> float16 [..., 256]."""
    return codebook_fp16(tile_states_words(words, K))


def place_tile(w256: np.ndarray) -> np.ndarray:
    """Weight j -> (row j // 16, column j % 16): [..., 256] -> [..., 16, 16]."""
    return np.asarray(w256).reshape(*np.shape(w256)[:-1], 16, 16)


def expert_word_counts(rows: int, cols: int, bits: np.ndarray) -> np.ndarray:
    """Words each expert's [rows x cols] matrix takes in the concatenated payload."""
    return np.asarray([(rows // 16) * (cols // 16) * 16 * int(k) for k in bits], dtype=np.int64)


def expert_payload(payload: np.ndarray, rows: int, cols: int, bits: np.ndarray, e: int) -> np.ndarray:
    """Expert e's words, shaped [rows/16][cols/16][16K]."""
    counts = expert_word_counts(rows, cols, bits)
    start = int(counts[:e].sum())
    K = int(bits[e])
    return np.asarray(payload[start:start + int(counts[e])]).reshape(rows // 16, cols // 16, 16 * K)


def decode_matrix(tiles: np.ndarray, K: int, chunk: int = 16384) -> np.ndarray:
    """Dense float16 [rows, cols] from one expert's tiles [rows/16][cols/16][16K]."""
    tr, tc, nw = tiles.shape
    assert nw == 16 * K
    flat = tiles.reshape(tr * tc, nw)
    out = np.empty((tr * tc, 256), dtype=np.float16)

    def work(a):
        out[a:a + chunk] = decode_tiles_fp16(flat[a:a + chunk], K)

    starts = range(0, tr * tc, chunk)
    if len(starts) > 1:
        with concurrent.futures.ThreadPoolExecutor(min(len(starts), os.cpu_count() or 1)) as ex:
            list(ex.map(work, starts))
    else:
        for a in starts:
            work(a)
    w = out.reshape(tr, tc, 16, 16).transpose(0, 2, 1, 3)
    return np.ascontiguousarray(w.reshape(tr * 16, tc * 16))
