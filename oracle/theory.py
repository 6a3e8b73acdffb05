"""Closed forms for the number of tokens committed per verification round (oracle).

TEST INFRASTRUCTURE ONLY.

With each draft accepted independently with probability a, a round commits
m = n + 1 tokens, n the number of accepted drafts:
  * "Speculative Decoding: Faster Generation Without Changing the Model",
    "Predicting the speedup": E[m] = (1 - a^(k+1)) / (1 - a); worked values
    about 3.36 at a = 0.8, k = 4 and about 2.31 at a = 0.6, k = 4; and the
    wall-clock estimate E[m] / (k c + 1) for a draft step costing c target steps.
  * "Cascade Speculative Drafting for Even Faster LLM Inference",
    "Theoretical Framework: EWIF and Generating Functions", Theorem 4.1:
    phi(x) = 1 + (x - 1)(1 - a^(k+1) x^(k+1)) / (1 - a x), whose coefficient of
    x^i is a^(i-1) - a^i for i = 1..k and a^k for i = k+1, and phi'(1) = E[m].
"""
from __future__ import annotations

import numpy as np


def expected_committed(a: float, k: int) -> float:
    """E[m] = (1 - a^(k+1)) / (1 - a); k + 1 when a = 1."""
    if a == 1.0:
        return float(k + 1)
    return (1.0 - a ** (k + 1)) / (1.0 - a)


def committed_pmf(a: float, k: int) -> np.ndarray:
    """P(m = i) for i = 0..k+1 (index 0 is always 0): the PGF's coefficients."""
    pmf = np.zeros(k + 2)
    for i in range(1, k + 1):
        pmf[i] = a ** (i - 1) - a ** i
    pmf[k + 1] = a ** k
    return pmf


def pgf(a: float, k: int, x: float) -> float:
    """phi(x) in the closed form of Theorem 4.1."""
    return 1.0 + (x - 1.0) * (1.0 - (a * x) ** (k + 1)) / (1.0 - a * x)


def speedup(a: float, k: int, c: float) -> float:
    """Expected tokens per round divided by the round's cost k c + 1."""
    return expected_committed(a, k) / (k * c + 1.0)
