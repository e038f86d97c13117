"""Pins the oracle's trellis decode.

What the pages fix: the code tensor is int16 [IC/16, OC/16, 16K] with one
16x16 weight tile per (IC/16, OC/16) entry, K = last dim / 16 (radiance_escha.py,
process_weights_after_loading), and the trellis is tail-biting (vllm-quantpack
exl3/linear.py, module docstring).  The bit order, window and codebook are this
library's readings (MSB-first words, 16-bit state ending at bit (t+1)K, QTIP
3INST hash); these tests pin the oracle's code to those readings through
closed forms, a big-integer brute force and numpy's own fp16 arithmetic.
"""
import numpy as np
import pytest

import oracle

KS = (1, 2, 3, 4, 5, 8)


def _stream_int(tile):
    """Big-integer view of the tile's stream: word 0's MSB is the top bit."""
    s = 0
    for w in np.asarray(tile, np.int16).view(np.uint16):
        s = (s << 16) | int(w)
    return s


def _state_bigint(tile, K, t):
    """Window [(t+1)K-16, (t+1)K) of the circular stream, via rotation of a big int."""
    n = 256 * K
    s = _stream_int(tile)
    start = ((t + 1) * K - 16) % n
    rot = ((s << start) | (s >> (n - start))) & ((1 << n) - 1) if start else s
    return rot >> (n - 16)


@pytest.mark.parametrize("K", KS)
def test_state_matches_bigint_rotation(K):
    g = np.random.default_rng(K)
    for _ in range(3):
        tile = g.integers(-32768, 32768, 16 * K, dtype=np.int16)
        for t in range(256):
            assert oracle.state(tile, K, t) == _state_bigint(tile, K, t)


@pytest.mark.parametrize("K", KS)
def test_word_aligned_states_are_whole_words(K):
    # when (t+1)K is a multiple of 16 the window is exactly word (t+1)K/16 - 1
    g = np.random.default_rng(100 + K)
    tile = g.integers(-32768, 32768, 16 * K, dtype=np.int16)
    words = tile.view(np.uint16)
    hits = 0
    for t in range(256):
        if ((t + 1) * K) % 16 == 0:
            assert oracle.state(tile, K, t) == int(words[(t + 1) * K // 16 - 1])
            hits += 1
    assert hits == 16 * int(np.gcd(16, K))   # (t+1) runs over multiples of 16/gcd(16,K)


@pytest.mark.parametrize("K", (2, 3, 4))
def test_tail_biting_first_window(K):
    # weight 0's window is the last 16-K bits of the tile followed by its first K bits
    g = np.random.default_rng(200 + K)
    tile = g.integers(-32768, 32768, 16 * K, dtype=np.int16)
    words = tile.view(np.uint16)
    last, first = int(words[-1]), int(words[0])
    expect = ((last & ((1 << (16 - K)) - 1)) << K) | (first >> (16 - K))
    assert oracle.state(tile, K, 0) == expect


@pytest.mark.parametrize("K", (2, 3, 4))
def test_single_bit_tiles(K):
    # a single set stream bit p lights up bit 15-(p-start) of exactly the states
    # whose window [start, start+16) covers p, wrap-around windows included
    n = 256 * K
    for p in list(range(0, n, 7)) + [0, 1, 15, 16, n - 1, n - 16]:
        tile = np.zeros(16 * K, np.uint16)
        tile[p // 16] = 1 << (15 - p % 16)
        tile = tile.view(np.int16)
        covered = 0
        for t in range(256):
            start = (t + 1) * K - 16
            off = (p - start) % n
            expect = (1 << (15 - off)) if off < 16 else 0
            s = oracle.state(tile, K, t)
            assert s == expect, (p, t)
            covered += s != 0
        # every bit sits in floor or ceil of 16/K windows
        assert covered in (16 // K, -(-16 // K))


def test_codebook_table_against_numpy_fp16():
    # the integer hash in plain modular arithmetic; the fp16 reinterpretation,
    # sum and single rounding done by numpy's float16 (an independent fp16 path)
    s = np.arange(65536, dtype=np.uint64)
    z = (s * 89226354 + 64248484) & 0xFFFFFFFF
    z = (z & 0x8FFF8FFF) ^ 0x3B603B60
    lo = (z & 0xFFFF).astype(np.uint16).view(np.float16)
    hi = (z >> 16).astype(np.uint16).view(np.float16)
    ref = (lo + hi).astype(np.float16).view(np.uint16)
    got = oracle.codebook_table()
    assert np.array_equal(got, ref)


def test_codebook_distribution_properties():
    v = oracle.codebook_table().view(np.float16).astype(np.float64)
    assert np.all(np.isfinite(v)) and np.all(np.abs(v) < 4.0)
    # each half lies in +-[1/8, 2): exponent field pinned by the xor to 0b011xx
    assert abs(v.mean()) < 0.01 and 1.1 < v.std() < 1.4
    assert len(np.unique(v)) > 10000


def test_all_zero_and_all_one_tiles():
    for K in (2, 3, 4):
        z = oracle.decode_tile(np.zeros(16 * K, np.int16), K)
        assert np.all(z == oracle.codebook(0))
        o = oracle.decode_tile(np.full(16 * K, -1, np.int16), K)
        assert np.all(o == oracle.codebook(0xFFFF))


@pytest.mark.parametrize("K", (2, 3, 4))
def test_tile_position_in_dense_matrix(K):
    # tile code[a][b] fills W[16a:16a+16, 16b:16b+16] with weight t at (t//16, t%16);
    # nothing else changes
    IC, OC = 64, 96
    g = np.random.default_rng(300 + K)
    base = np.zeros((IC // 16, OC // 16, 16 * K), np.int16)
    W0 = oracle.reconstruct(base, K)
    a, b = 2, 4
    code = base.copy()
    code[a, b] = g.integers(-32768, 32768, 16 * K, dtype=np.int16)
    W = oracle.reconstruct(code, K)
    diff = W != W0
    rows, cols = np.nonzero(diff)
    assert rows.min() >= 16 * a and rows.max() < 16 * a + 16
    assert cols.min() >= 16 * b and cols.max() < 16 * b + 16
    w256 = oracle.decode_tile(code[a, b], K)
    for t in range(256):
        assert W[16 * a + t // 16, 16 * b + t % 16] == w256[t]
    # column-range reconstruction is the same matrix, sliced
    Wc = oracle.reconstruct(code, K, oc0=32, noc=48)
    assert np.array_equal(Wc, W[:, 32:80])


def test_reconstruct_rejects_wrong_k():
    code = np.zeros((2, 2, 32), np.int16)   # 16*K = 32 -> K = 2
    with pytest.raises(AssertionError):
        oracle.reconstruct(code, 3)
