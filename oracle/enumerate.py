"""Exact output distribution of the verification rule on tiny vocabularies (oracle).

TEST INFRASTRUCTURE ONLY.

``verify_sequence`` takes its randomness through two hooks.  Here the hooks
branch instead of sampling: every accept decision splits into accept (weight
min(1, ratio)) and reject (1 - min(1, ratio)), every draw splits into each
support element v (weight w_v / sum w).  Replaying the rule once per branch
sequence, and also summing over the draft tokens x ~ q, gives the exact law of
the committed tokens -- the quantity whose equality with the target's law is
the losslessness claim of "Speculative Decoding: Faster Generation Without
Changing the Model" ("The acceptance rule") and of the other pages.
"""
from __future__ import annotations

import itertools
from collections import defaultdict

import numpy as np

from .verify import verify_sequence


class _Branch(Exception):
    def __init__(self, options):
        self.options = options


class _Replay:
    """Hooks that follow a fixed script of choices and raise at its end."""

    def __init__(self, script):
        self.script = list(script)
        self.pos = 0
        self.prob = 1.0

    def _next(self, options):
        if self.pos < len(self.script):
            choice = self.script[self.pos]
            self.pos += 1
            weight = dict(options)[choice]
            self.prob *= weight
            return choice
        raise _Branch(options)

    def accept(self, i, ratio):
        a = min(1.0, ratio)
        return self._next([(True, a), (False, 1.0 - a)])

    def draw(self, j, logw, kind):
        w = np.exp(np.asarray(logw, dtype=np.float64))
        w = w / w.sum()
        return self._next([(v, float(w[v])) for v in range(w.shape[0]) if w[v] > 0])


def output_law(logp: np.ndarray, logq: np.ndarray, tokens, lenience: float = 1.0):
    """Exact law of the committed-token tuple for fixed draft tokens."""
    law = defaultdict(float)
    stack = [[]]
    while stack:
        script = stack.pop()
        rp = _Replay(script)
        try:
            out, _ = verify_sequence(logp, logq, tokens, rp.accept, rp.draw, lenience=lenience)
        except _Branch as br:
            for choice, weight in br.options:
                if weight > 0:
                    stack.append(script + [choice])
            continue
        law[tuple(out)] += rp.prob
    return law


def full_law(logp: np.ndarray, logq: np.ndarray, lenience: float = 1.0):
    """Exact law of the committed tuple when the drafts themselves are drawn
    x_i ~ q_i independently (context-free rows)."""
    k, V = logq.shape
    q = np.exp(logq)
    law = defaultdict(float)
    for xs in itertools.product(range(V), repeat=k):
        w = float(np.prod([q[i, xs[i]] for i in range(k)]))
        if w == 0.0:
            continue
        for out, pr in output_law(logp, logq, xs, lenience).items():
            law[out] += w * pr
    return law
