"""Pins for the oracle's Philox4x32-10 stream and uniform/Gumbel mapping."""

import os

import numpy as np
import pytest
from scipy import stats

from oracle.philox import (gumbel, philox4x32_10, philox4x32_10_np, sampler_words,
                           uniform_from_word)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.txt")


def _kat():
    rows = []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        w = [int(v, 16) for v in line.split()]
        rows.append((tuple(w[0:4]), tuple(w[4:6]), tuple(w[6:10])))
    return rows


@pytest.mark.parametrize("ctr,key,expect", _kat())
def test_known_answer_vectors(ctr, key, expect):
    assert philox4x32_10(ctr, key) == expect


def test_vectorised_matches_scalar():
    rng = np.random.default_rng(7)
    c = rng.integers(0, 2**32, (4, 257), dtype=np.uint64)
    k0, k1 = 0x12345678, 0x9ABCDEF0
    out = philox4x32_10_np(c[0], c[1], c[2], c[3], k0, k1)
    for i in range(257):
        ref = philox4x32_10(tuple(int(c[j, i]) for j in range(4)), (k0, k1))
        assert tuple(int(o[i]) for o in out) == ref


def test_stream_layout():
    # token t uses word t & 3 of Philox((t >> 2, row, step, 0), (seed lo, seed hi))
    seed = 0x0123456789ABCDEF
    words = sampler_words(np.arange(12), row=5, step=9, seed=seed)
    for t in range(12):
        block = philox4x32_10((t >> 2, 5, 9, 0), (seed & 0xFFFFFFFF, seed >> 32))
        assert int(words[t]) == block[t & 3]


def test_uniform_mapping_is_exact_and_open():
    r = np.array([0, 1, 511, 512, 0xFFFFFFFF, 0x80000000], dtype=np.uint64)
    u = uniform_from_word(r)
    assert u[0] == 2.0 ** -24 and u[1] == 2.0 ** -24 and u[2] == 2.0 ** -24
    assert u[3] == 3 * 2.0 ** -24
    assert u[4] == 1.0 - 2.0 ** -24
    assert u[5] == 0.5 + 2.0 ** -24
    assert np.all(u.astype(np.float32).astype(np.float64) == u)   # exact in binary32
    assert np.all((u > 0) & (u < 1))


def test_uniformity_and_independence():
    n = 1 << 18
    w = sampler_words(np.arange(n), row=3, step=11, seed=42)
    u = uniform_from_word(w)
    assert stats.kstest(u, "uniform").pvalue > 1e-4
    counts = np.bincount((u * 64).astype(np.int64), minlength=64)
    assert stats.chisquare(counts).pvalue > 1e-4
    # neighbouring lanes of one block and neighbouring rows are uncorrelated
    assert abs(np.corrcoef(u[0::4], u[1::4])[0, 1]) < 0.02
    u2 = uniform_from_word(sampler_words(np.arange(n), row=4, step=11, seed=42))
    assert abs(np.corrcoef(u, u2)[0, 1]) < 0.02


def test_gumbel_distribution():
    u = uniform_from_word(sampler_words(np.arange(1 << 17), row=0, step=0, seed=1))
    g = gumbel(u)
    assert stats.kstest(g, "gumbel_r").pvalue > 1e-4
    assert abs(g.mean() - np.euler_gamma) < 0.02
