"""Pins of the oracle's Philox4x32-10 and of the two uniform constructions."""
import math

import numpy as np
import pytest

import oracle
from conftest import golden_lines


def test_known_answer_vectors():
    rows = list(golden_lines("philox4x32_10_kat.txt"))
    assert len(rows) == 3
    for row in rows:
        w = [int(x, 16) for x in row]
        out = oracle.philox4x32_10(w[0:4], w[4:6])
        assert [int(x) for x in out] == w[6:10]


def test_accept_uniform_is_open_and_52_bit():
    # u = (2m + 1) 2^-53 with m < 2^52: strictly inside (0, 1) and on that lattice.
    for r in range(200):
        for i in range(8):
            u = oracle.accept_uniform(12345, r, i)
            assert 0.0 < u < 1.0
            k = u * 2.0 ** 53
            assert k == math.floor(k) and int(k) % 2 == 1
            assert (int(k) - 1) // 2 < 2 ** 52


def test_accept_uniform_uses_top_bits_of_words_0_and_1():
    seed, r, i = 0x0123456789ABCDEF, 77, 3
    w = oracle.philox4x32_10([0, i, r, 0], [seed & 0xFFFFFFFF, seed >> 32])
    m52 = ((int(w[0]) << 32) | int(w[1])) >> 12
    assert oracle.accept_uniform(seed, r, i) == (2 * m52 + 1) * 2.0 ** -53


def test_race_uniform_word_layout():
    seed, r, pos = 99, 5, 2
    for j in range(16):
        w = oracle.philox4x32_10([j >> 2, pos, r, 1], [seed, 0])
        U = oracle.race_uniform(seed, r, pos, j)
        assert U == (2 * (int(w[j & 3]) >> 9) + 1) * 2.0 ** -24
        assert 0.0 < U < 1.0


def test_uniformity_chi_square():
    # 10 equal bins, 100k accept uniforms: chi2 (9 dof) below the 1e-3 critical value.
    n = 100_000
    u = np.array([oracle.accept_uniform(7, r, r % 5) for r in range(n)])
    counts = np.histogram(u, bins=10, range=(0, 1))[0]
    chi2 = ((counts - n / 10) ** 2 / (n / 10)).sum()
    assert chi2 < 27.88


def test_bit_balance():
    ws = np.array([oracle.philox4x32_10([c, 1, 2, 3], [4, 5]) for c in range(20000)],
                  dtype=np.uint64).ravel()
    bits = np.array([(ws >> b) & 1 for b in range(32)])
    frac = bits.mean(axis=1)
    # 80000 words per bit: sd 0.0018; 5 sd bound
    assert np.all(np.abs(frac - 0.5) < 0.009)


def test_bf16_decoding_exact():
    assert oracle.bf16_to_double(0x3F80) == 1.0
    assert oracle.bf16_to_double(0xC000) == -2.0
    assert oracle.bf16_to_double(0x3F81) == 1.0 + 2.0 ** -7
    assert oracle.bf16_to_double(0xFF80) == -math.inf
