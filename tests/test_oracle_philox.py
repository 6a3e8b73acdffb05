"""Pins for the oracle's counter-based randomness (CPU only)."""
import math

import numpy as np
import pytest
from scipy import stats

from oracle import philox


def test_philox_known_answer_vectors(golden):
    rows = golden("philox4x32_10_kat.txt")
    assert len(rows) == 3
    for r in rows:
        vals = [int(x, 16) for x in r]
        out = philox.philox4x32_10(*vals[:6])
        assert [int(x) for x in out] == vals[6:]


def test_philox_vectorised_matches_scalar():
    rng = np.random.default_rng(0)
    c = rng.integers(0, 2 ** 32, size=(4, 64), dtype=np.uint64)
    k = rng.integers(0, 2 ** 32, size=2, dtype=np.uint64)
    vec = philox.philox4x32_10(c[0], c[1], c[2], c[3], k[0], k[1])
    for j in range(64):
        one = philox.philox4x32_10(c[0, j], c[1, j], c[2, j], c[3, j], k[0], k[1])
        assert [int(x[j]) for x in vec] == [int(x) for x in one]


def test_uniform_map_is_open_interval_and_fp32_exact():
    w = np.array([0, 255, 256, 2 ** 31, 2 ** 32 - 1], dtype=np.uint64)
    u = philox.uniform_from_word(w)
    assert np.all(u > 0) and np.all(u < 1)
    assert u[0] == 2.0 ** -24 and u[-1] == 1 - 2.0 ** -24
    assert np.all(u.astype(np.float32).astype(np.float64) == u)


def test_gumbel_uniform_layout():
    """Word (v mod 4) of counter (v >> 2, j, b, 1) under key (seed lo, seed hi)."""
    seed = 0x1234_5678_9ABC_DEF0
    u = philox.gumbel_uniforms(seed, b=3, j=5, V=10)
    for v in range(10):
        words = philox.philox4x32_10(v >> 2, 5, 3, 1, seed & 0xFFFFFFFF, seed >> 32)
        assert u[v] == philox.uniform_from_word(words[v & 3])
    a = philox.accept_uniform(seed, b=3, i=2)
    words = philox.philox4x32_10(0, 2, 3, 0, seed & 0xFFFFFFFF, seed >> 32)
    assert a == philox.uniform_from_word(words[0])


def test_uniforms_are_uniform():
    u = philox.gumbel_uniforms(1234, 0, 0, 200_000)
    counts, _ = np.histogram(u, bins=64, range=(0, 1))
    assert stats.chisquare(counts).pvalue > 1e-3
    assert abs(u.mean() - 0.5) < 0.005
    # distinct (b, j) streams are not the same numbers
    assert not np.array_equal(u[:1000], philox.gumbel_uniforms(1234, 0, 1, 1000))
    assert not np.array_equal(u[:1000], philox.gumbel_uniforms(1234, 1, 0, 1000))
    assert not np.array_equal(u[:1000], philox.gumbel_uniforms(1235, 0, 0, 1000))


def test_gumbel_moments():
    g = philox.gumbel(philox.gumbel_uniforms(99, 2, 3, 400_000))
    assert abs(g.mean() - 0.5772156649) < 0.01            # Euler-Mascheroni constant
    assert abs(g.var() - math.pi ** 2 / 6) < 0.03
    assert g.max() <= -math.log(-math.log(1 - 2.0 ** -24)) + 1e-12


@pytest.mark.parametrize("V", [8, 5])
def test_gumbel_max_samples_the_categorical_law(V):
    """argmax_v(ln w_v + G_v) ~ w / sum(w): checked by chi-squared over many (b)."""
    rng = np.random.default_rng(V)
    w = rng.random(V) + 0.05
    w[1] = 0.0                                        # outside the support: never drawn
    logw = np.where(w > 0, np.log(np.where(w > 0, w, 1)), -np.inf)
    n = 40_000
    draws = np.empty(n, dtype=np.int64)
    for b in range(n):
        g = philox.gumbel(philox.gumbel_uniforms(7, b, 0, V))
        draws[b] = int(np.argmax(logw + g))
    counts = np.bincount(draws, minlength=V)
    assert counts[1] == 0
    keep = w > 0
    expected = n * w[keep] / w.sum()
    assert stats.chisquare(counts[keep], expected).pvalue > 1e-3
