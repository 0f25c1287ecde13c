"""Pins for the oracle's trellis decoder (CPU only)."""
from fractions import Fraction

import numpy as np
import pytest

from oracle import trellis
from tests.conftest import read_golden
from trellis_quantized_moe_route_gb300 import synth


def _half_exact(h: int) -> Fraction:
    """IEEE binary16 value from its fields (normal numbers only)."""
    e, m = (h >> 10) & 31, h & 1023
    assert 0 < e < 31
    v = Fraction(1024 + m, 1024) * Fraction(2) ** (e - 15)
    return -v if h >> 15 else v


def test_codebook_golden_values():
    rows = read_golden("codebook_states.txt")
    assert len(rows) >= 6
    for s_hex, bits_hex, val, exact_sum in rows:
        s, bits = int(s_hex, 16), int(bits_hex, 16)
        x = (s * 0xCBAC1FED) % (1 << 32)
        y = (x & 0x8FFF8FFF) ^ 0x3B603B60
        assert _half_exact(y & 0xFFFF) + _half_exact(y >> 16) == Fraction(exact_sum)
        got = trellis.codebook_fp16(np.array([s]))[0]
        assert int(got.view(np.uint16)) == bits, (s_hex, hex(int(got.view(np.uint16))))
        assert float(got) == float(val)
        assert trellis.codebook_scalar(s) == float(val)


def _half_rne(v: Fraction) -> int:
    """binary16 bits of the nearest-even rounding of a rational in the normal range."""
    if v == 0:
        return 0
    sign = 0x8000 if v < 0 else 0
    a, e = abs(v), 0
    while a >= 2:
        a, e = a / 2, e + 1
    while a < 1:
        a, e = a * 2, e - 1
    m = a * 1024
    fl = m.numerator // m.denominator
    r = m - fl
    if r > Fraction(1, 2) or (r == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    if fl == 2048:
        fl, e = 1024, e + 1
    return sign | ((e + 15) << 10) | (fl - 1024)


def test_codebook_all_states_vs_exact_rounding():
    """Sampled states: the oracle's fp16 sum equals an exact-rational rounding
    of the two halves' sum (independent of numpy's float16)."""
    cb = trellis.codebook_fp16(np.arange(65536)).view(np.uint16)
    rng = np.random.default_rng(5)
    for s in rng.integers(0, 65536, 400).tolist() + [0, 1, 65535, 32768]:
        x = (s * 0xCBAC1FED) % (1 << 32)
        y = (x & 0x8FFF8FFF) ^ 0x3B603B60
        exact = _half_exact(y & 0xFFFF) + _half_exact(y >> 16)
        assert int(cb[s]) == _half_rne(exact), hex(s)


def test_codebook_statistics():
    """Over all 2^16 states: mean ~ 0, std ~ 1.244, max |cb| = 3.949,
    10,746 distinct values, and the sign pattern is symmetric."""
    cb = trellis.codebook_fp16(np.arange(65536)).astype(np.float64)
    assert len(np.unique(cb)) == 10746
    assert abs(cb.mean()) < 0.02
    assert abs(cb.std() - 1.244) < 0.001
    assert abs(np.abs(cb).max() - 3.949) < 0.001
    assert abs(int((cb > 0).sum()) - int((cb < 0).sum())) < 300


def test_codebook_halves_range():
    """Each fp16 half has exponent field 12..15, so |half| in [1/8, 2)."""
    s = np.arange(65536, dtype=np.uint64)
    x = (s * np.uint64(0xCBAC1FED)) & np.uint64(0xFFFFFFFF)
    y = (x & np.uint64(0x8FFF8FFF)) ^ np.uint64(0x3B603B60)
    for half in ((y & np.uint64(0xFFFF)), (y >> np.uint64(16))):
        e = (half >> np.uint64(10)) & np.uint64(31)
        assert e.min() >= 12 and e.max() <= 15


@pytest.mark.parametrize("K", [2, 3, 4, 5, 6])
def test_all_zero_and_all_one_streams(K):
    zeros = np.zeros(16 * K, dtype=np.int16)
    w = trellis.decode_tiles_fp16(zeros, K)
    assert np.all(w.view(np.uint16) == 0x3F60)           # cb(0) = 1.84375
    ones = np.full(16 * K, -1, dtype=np.int16)             # every bit set
    w = trellis.decode_tiles_fp16(ones, K)
    assert np.all(w.view(np.uint16) == 0x3ACD)           # cb(0xFFFF)


def _stream_words(bits, K):
    """int16 words of a hand-built bit list (MSB-first within each word)."""
    assert len(bits) == 256 * K
    words = []
    for i in range(16 * K):
        v = 0
        for b in bits[16 * i:16 * i + 16]:
            v = (v << 1) | b
        words.append(v)
    return np.array(words, dtype=np.uint16).view(np.int16)


@pytest.mark.parametrize("K,j,state", [(4, 5, 0x1234), (3, 7, 0x8000), (2, 200, 0x0001),
                                       (3, 0, 0x00FF), (2, 0, 0xABCD), (4, 255, 0x0002)])
def test_hand_built_window(K, j, state):
    """Place a 16-bit pattern on the stream positions (j+1)K-16 .. (j+1)K-1
    (mod 256K) of an otherwise zero stream; weight j must decode to cb(pattern)
    and a weight whose window does not touch the pattern must decode to cb(0)."""
    n = 256 * K
    bits = [0] * n
    for i in range(16):
        bits[((j + 1) * K - 16 + i) % n] = (state >> (15 - i)) & 1
    words = _stream_words(bits, K)
    st = trellis.tile_states(words, K)
    assert int(st[j]) == state
    assert trellis.tile_states_scalar(words, K)[j] == state
    far = (j + 128) % 256
    assert int(st[far]) == 0
    w = trellis.decode_tiles_fp16(words, K)
    assert float(w[j]) == trellis.codebook_scalar(state)


@pytest.mark.parametrize("K", [2, 3, 4, 5, 6])
def test_vectorised_states_match_bitwise_loop(K):
    words = synth.Stream(11, K).words16(16 * K * 3).reshape(3, 16 * K)
    st = trellis.tile_states(words, K)
    for t in range(3):
        assert st[t].tolist() == trellis.tile_states_scalar(words[t], K)
    many = synth.Stream(14, K).words16(16 * K * 500).reshape(500, 16 * K)
    assert np.array_equal(trellis.tile_states_words(many, K), trellis.tile_states(many, K))


@pytest.mark.parametrize("K", [2, 3, 4, 5, 6])
def test_trellis_recurrence_and_tail_biting(K):
    """s_j = ((s_{j-1} << K) | new K bits) & 0xFFFF, including s_0 from s_255,
    and rotating the stream left by K bits shifts the states by one."""
    words = synth.Stream(12, K).words16(16 * K)
    st = trellis.tile_states(words, K).astype(np.int64)
    bits = trellis.stream_bits(words)
    n = 256 * K
    for j in range(256):
        new = 0
        for i in range(K):
            new = (new << 1) | int(bits[(j * K + i) % n])
        assert st[j] == (((int(st[j - 1]) << K) | new) & 0xFFFF)
    rolled = np.roll(bits, -K)
    w2 = np.packbits(rolled.reshape(16 * K, 16), axis=-1, bitorder="big").view(">u2")[:, 0]
    st2 = trellis.tile_states(w2.astype(np.uint16).view(np.int16), K)
    assert np.array_equal(st2, np.roll(st, -1))


def test_placement_and_matrix_assembly():
    """decode_matrix puts weight j of tile (tn, tk) at (16tn + j//16, 16tk + j%16)."""
    K = 3
    tiles = synth.Stream(13, 0).words16(2 * 3 * 16 * K).reshape(2, 3, 16 * K)
    dense = trellis.decode_matrix(tiles, K)
    assert dense.shape == (32, 48)
    for tn in range(2):
        for tk in range(3):
            w = trellis.decode_tiles_fp16(tiles[tn, tk], K)
            for j in (0, 17, 100, 255):
                assert dense[16 * tn + j // 16, 16 * tk + j % 16] == w[j]


def test_expert_payload_offsets_mixed_bits():
    bits = np.array([2, 4, 3], dtype=np.uint8)
    rows, cols = 32, 16
    counts = trellis.expert_word_counts(rows, cols, bits)
    assert counts.tolist() == [2 * 1 * 32, 2 * 1 * 64, 2 * 1 * 48]
    payload = np.arange(int(counts.sum()), dtype=np.int64).astype(np.int16)
    t = trellis.expert_payload(payload, rows, cols, bits, 2)
    assert t.shape == (2, 1, 48) and int(t[0, 0, 0]) == 64 + 128
