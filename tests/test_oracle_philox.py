"""Pins of the oracle's counter-based uniforms (Philox4x32-10, Salmon et al. SC'11)."""
import os

import numpy as np
import pytest
from scipy import stats

import oracle


def _kat(golden_dir):
    rows = []
    for line in open(os.path.join(golden_dir, "philox4x32_10_kat.txt"), encoding="utf-8"):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        w = [int(t, 16) for t in line.split()]
        rows.append((w[0:4], w[4:6], w[6:10]))
    return rows


def test_known_answer_vectors(golden_dir):
    kat = _kat(golden_dir)
    assert len(kat) == 3
    for ctr, key, want in kat:
        got = oracle.philox4x32_10(ctr, key)
        assert [int(v) for v in got] == want


def test_uniforms_are_odd_multiples_of_2_pow_minus_24():
    for seed in (0, 1, 2**40 + 7):
        for row in (0, 1, 255):
            for pos in range(4):
                ua, us = oracle.uniforms(seed, row, pos)
                for u in (ua, us):
                    k = u * 2**24
                    assert 0.0 < u < 1.0
                    assert k == int(k) and int(k) % 2 == 1
                    assert np.float32(u) == u  # exact in fp32


def test_uniforms_follow_counter_and_key():
    # U_acc is built from output word 0 and U_smp from word 1 of Philox(row, pos, 0, 0)
    seed = 0x0123456789ABCDEF
    key = [seed & 0xFFFFFFFF, seed >> 32]
    for row, pos in [(0, 0), (7, 3), (1000, 6)]:
        o = oracle.philox4x32_10([row, pos, 0, 0], key)
        ua, us = oracle.uniforms(seed, row, pos)
        assert ua == (2 * (int(o[0]) >> 9) + 1) / 2**24
        assert us == (2 * (int(o[1]) >> 9) + 1) / 2**24


def test_uniformity_chi_square():
    us = np.array([oracle.uniforms(5, r, j)[k] for r in range(4000) for j in range(8)
                   for k in range(2)])
    counts, _ = np.histogram(us, bins=64, range=(0.0, 1.0))
    assert stats.chisquare(counts).pvalue > 1e-3
    # distinct units give distinct draws
    assert len(np.unique(us)) > 0.99 * us.size
