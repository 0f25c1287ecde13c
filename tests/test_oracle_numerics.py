"""Pins for the oracle's MXFP8/E4M3 rounding and Hadamard rotation (CPU only)."""
import numpy as np
import pytest

from oracle import hadamard, mxfp8
from tests.conftest import read_golden


def test_e8m0_golden_cases():
    rows = [r for r in read_golden("mxfp8_cases.txt") if r[0] != "E4M3"]
    assert len(rows) >= 6
    for amax, e in rows:
        got = int(mxfp8.e8m0_exponent(np.array([float(amax)], dtype=np.float32))[0])
        assert got == int(e), (amax, got, e)


def test_e8m0_powers_of_two_and_neighbours():
    for k in range(-20, 21):
        a = np.float32(448.0 * 2.0 ** k)
        assert int(mxfp8.e8m0_exponent(np.array([a]))[0]) == k
        above = np.nextafter(a, np.float32(np.inf))
        # the quotient of the next float up is above 2^k -> next exponent,
        # unless the fp32 division rounds it back onto 2^k
        q = np.float32(np.float64(above) / 448.0)
        expect = k if q == np.float32(2.0 ** k) else k + 1
        assert int(mxfp8.e8m0_exponent(np.array([above]))[0]) == expect


def test_e4m3_golden_cases():
    rows = [r[1:] for r in read_golden("mxfp8_cases.txt") if r[0] == "E4M3"]
    assert len(rows) >= 10
    for v, code in rows:
        got = int(mxfp8.e4m3_encode(np.array([float(v)]))[0])
        assert got == int(code, 16), (v, hex(got), code)


def test_e4m3_round_trip_all_codes():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    vals = mxfp8.e4m3_decode(codes)
    assert np.array_equal(mxfp8.e4m3_encode(vals), codes)
    assert mxfp8.e4m3_decode(np.array([0x7E]))[0] == 448.0
    assert mxfp8.e4m3_decode(np.array([0x01]))[0] == 2.0 ** -9


def test_e4m3_nearest_and_ties_even():
    """Brute force: for random values, the chosen code is a nearest one and,
    on exact ties, the one with the even code."""
    rng = np.random.default_rng(3)
    v = np.concatenate([rng.normal(0, 50, 4000), rng.normal(0, 0.01, 4000)])
    codes = mxfp8.e4m3_encode(v)
    table = mxfp8.E4M3_VALUES
    for x, c in zip(v[:2000], codes[:2000]):
        a = min(abs(x), 448.0)
        d = np.abs(table - a)
        best = np.flatnonzero(d == d.min())
        chosen = int(c) & 0x7F
        assert chosen in best
        if len(best) == 2:
            assert chosen % 2 == 0


def test_mxfp8_block_quantisation_properties():
    rng = np.random.default_rng(4)
    v = (rng.normal(0, 1, (5, 64)) * np.exp2(rng.integers(-10, 10, (5, 1)))).astype(np.float32)
    codes, e8, deq = mxfp8.quantize_mxfp8(v)
    assert codes.shape == v.shape and e8.shape == (5, 2)
    blocks = v.astype(np.float64).reshape(5, 2, 32)
    e = e8.astype(np.int64) - 127
    scaled = np.abs(blocks) * np.exp2(-e)[..., None]
    assert scaled.max() <= 448.0 * (1 + 2 ** -20)
    # the exponent is the smallest that keeps the block within 448
    assert np.all(np.abs(blocks).max(axis=-1) * np.exp2(-(e - 1)) > 448.0 * (1 - 2 ** -20))
    # relative error of each element is bounded by half an E4M3 ulp (2^-4)
    big = np.abs(blocks) * np.exp2(-e)[..., None] >= 2.0 ** -6
    err = np.abs(deq.reshape(5, 2, 32) - blocks)
    assert np.all(err[big] <= np.abs(blocks[big]) * 2.0 ** -4 + 1e-30)
    zero = np.zeros((1, 32), dtype=np.float32)
    c0, e0, d0 = mxfp8.quantize_mxfp8(zero)
    assert int(e0[0, 0]) == 0 and np.all(c0 == 0) and np.all(d0 == 0)


def test_sylvester_small_and_recursion():
    assert np.array_equal(hadamard.sylvester(1), [[1.0]])
    assert np.array_equal(hadamard.sylvester(2), [[1.0, 1.0], [1.0, -1.0]])
    # Sylvester's construction H_2n = [[H, H], [H, -H]]
    for n in (2, 4, 8, 16, 32, 64):
        h = hadamard.sylvester(n)
        assert np.array_equal(hadamard.sylvester(2 * n), np.block([[h, h], [h, -h]]))


@pytest.mark.parametrize("n", [64, 128])
def test_hadamard_orthogonality(n):
    h = hadamard.sylvester(n)
    assert np.array_equal(h @ h.T, n * np.eye(n))
    m = hadamard.rotation_matrix(n)
    assert np.abs(m @ m - np.eye(n)).max() < 1e-15


@pytest.mark.parametrize("b", [1, 64, 128])
def test_rotate_then_unrotate_identity(b):
    rng = np.random.default_rng(1)
    x = rng.normal(0, 1, (3, 256))
    y = hadamard.rotate(x, b)
    assert np.abs(hadamard.rotate(y, b) - x).max() < 1e-13
    assert np.allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1))


def test_rotate_is_blockwise():
    """A basis vector e_i stays inside its own block: the result is row i of H_b/sqrt(b)."""
    b = 128
    x = np.zeros((1, 384))
    x[0, 130] = 1.0
    y = hadamard.rotate(x, b)
    assert np.all(y[0, :128] == 0) and np.all(y[0, 256:] == 0)
    assert np.allclose(y[0, 128:256], hadamard.sylvester(b)[2] / np.sqrt(b), atol=0, rtol=1e-15)
    assert abs(1.0 / np.sqrt(128.0) - 0.088388347648) < 1e-12
