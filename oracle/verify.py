"""Batched speculative-decoding verification, restated plainly in fp64 (oracle).

TEST INFRASTRUCTURE ONLY (see the package docstring).

The rule, as "Speculative Decoding: Faster Generation Without Changing the
Model" states it under "The acceptance rule": draft tokens x_1..x_k are examined
left to right; x_i is accepted with probability min(1, p_i(x_i) / q_i(x_i)); at
the first rejection the scan stops and a replacement is drawn from the residual
distribution proportional to max(0, p_i - q_i); if every draft is accepted, one
bonus token is drawn from the target distribution at position k+1.  Under greedy
decoding a draft is accepted iff it equals the target's argmax, and the first
mismatch is replaced by that argmax.  "Cascade Speculative Drafting for Even
Faster LLM Inference" restates the same review step (accept when
q <= p, otherwise reject with probability 1 - p/q; lenience fixed to 1 at the
target), which is the form used below.

Readings where the pages are silent (each also listed in the design notes):
  * p and q are softmax(logits / T) of the given target / draft rows, same T.
  * Accept iff q <= p or u < p/q with u the counter-based uniform of (b, i);
    the q <= p branch also settles p = q = 0 as an accept.
  * Categorical draws use the Gumbel-max form: argmax over the support of
    ln w_v + G(seed, b, j, v), lowest index on ties.  This is exact in law.
  * If the residual is empty in working precision, draw from p_i instead.
  * A decision that floating point makes about an integer (accept or not, which
    index wins) is taken on fp32-rounded quantities -- the precision of the
    CUDA path -- while every value and every margin is fp64.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Callable, List, Optional

import numpy as np

from . import philox

STATUS_OK = 0
STATUS_TOKEN = -3
STATUS_NONFINITE = -4


def decode_logits(arr: np.ndarray, dtype: str) -> np.ndarray:
    """Stored logits to fp64: bf16 bit patterns are widened exactly, fp32 as is."""
    if dtype == "bf16":
        bits = np.asarray(arr, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
        return bits.view(np.float32).astype(np.float64)
    return np.asarray(arr, dtype=np.float32).astype(np.float64)


def log_softmax(logits: np.ndarray, temperature: float):
    """Natural-log probabilities of softmax(x / T) over the last axis, and log Z.

    log Z = m + ln(sum_v exp(z_v - m)), z = x / T, m = max z.
    """
    z = np.asarray(logits, dtype=np.float64) / float(temperature)
    m = np.max(z, axis=-1, keepdims=True)
    lse = m + np.log(np.sum(np.exp(z - m), axis=-1, keepdims=True))
    return z - lse, lse[..., 0]


# ----------------------------------------------------------------------------
# The rule for one sequence, with its two sources of randomness as hooks.
# ----------------------------------------------------------------------------

def verify_sequence(logp: np.ndarray, logq: np.ndarray, tokens, accept: Callable, draw: Callable,
                    lenience: float = 1.0):
    """One sequence of speculative verification.

    logp   (k+1, V) natural-log target probabilities (row k is the bonus row)
    logq   (k, V)   natural-log draft probabilities
    tokens k draft token ids
    accept(i, ratio) -> bool     True with probability min(1, ratio)
    draw(j, logw, kind) -> int   one draw from the law proportional to exp(logw)
                                 (-inf entries excluded); kind names the draw
    lenience l >= 1              "Cascade Speculative Drafting ...", "Asymmetric
                                 lenience": accept when q <= l p, otherwise reject
                                 with probability 1 - l p / q; the residual stays
                                 norm(max(0, p - q)).  l = 1 is the exact rule.

    Returns (committed token list, number of accepted drafts n).
    """
    k = logq.shape[0]
    out: List[int] = []
    for i in range(k):
        x = int(tokens[i])
        p = float(np.exp(logp[i, x]))
        q = float(np.exp(logq[i, x]))
        if q <= lenience * p or accept(i, lenience * p / q):
            out.append(x)
            continue
        # residual max(0, p - q), as a log weight: ln p + ln(1 - q/p) where p > q
        with np.errstate(divide="ignore", invalid="ignore"):
            pos = logp[i] > logq[i]
            logr = np.full(logp.shape[1], -np.inf)
            logr[pos] = logp[i, pos] + np.log1p(-np.exp(logq[i, pos] - logp[i, pos]))
        if np.any(np.isfinite(logr)):
            out.append(int(draw(i, logr, "residual")))
        else:
            out.append(int(draw(i, logp[i], "empty-residual")))
        return out, i
    out.append(int(draw(k, logp[k], "bonus")))
    return out, k


@dataclass
class SequenceTrace:
    """What one sequence's production run observed (for parity bookkeeping)."""
    draw_gap: float = np.inf       # top-1 minus top-2 Gumbel score of the draw
    empty_residual: bool = False


def _gumbel_draw(seed: int, b: int, trace: SequenceTrace):
    def draw(j: int, logw: np.ndarray, kind: str) -> int:
        g = philox.gumbel(philox.gumbel_uniforms(seed, b, j, logw.shape[0]))
        score = logw + g                                   # -inf outside the support
        s32 = score.astype(np.float32)                     # decision precision: fp32
        y = int(np.argmax(s32))                            # first index among equal maxima
        finite = np.sort(score[np.isfinite(score)])
        gap = float(finite[-1] - finite[-2]) if finite.size >= 2 else np.inf
        if kind == "empty-residual":
            trace.empty_residual = True
            gap = 0.0
        trace.draw_gap = gap
        return y
    return draw


def _philox_accept(seed: int, b: int):
    def accept(i: int, ratio: float) -> bool:
        u = philox.accept_uniform(seed, b, i)
        return bool(np.float32(u) < np.float32(ratio))     # decision precision: fp32
    return accept


def position_margins(seed: int, b: int, p_draft, q_draft, n: int, k: int, draw_gap: float,
                     lenience: float = 1.0) -> np.ndarray:
    """Distance of each committed position's decision from its boundary.

    Position i < n: |u_i - min(1, l p/q)| of its accept decision.  Position n:
    the smaller of that distance for the rejecting decision (when n < k) and
    the Gumbel top-1 / top-2 gap of the draw.  A position whose margin is
    below the parity threshold may legitimately come out differently in fp32.
    """
    m = np.empty(n + 1)
    for i in range(min(n + 1, k)):
        ratio = np.inf if q_draft[i] == 0 else lenience * p_draft[i] / q_draft[i]
        m[i] = abs(philox.accept_uniform(seed, b, i) - min(1.0, ratio))
    m[n] = min(m[n], draw_gap) if n < k else draw_gap
    return m


def _bad_rows(x: np.ndarray) -> bool:
    """NaN or +inf anywhere, or a row with no finite entry (no distribution)."""
    return bool(np.any(np.isnan(x)) or np.any(x == np.inf) or np.any(~np.any(np.isfinite(x), axis=-1)))


@dataclass
class StochasticResult:
    out_tokens: np.ndarray      # [B][k+1] int32, -1 after the committed tokens
    n_accepted: np.ndarray      # [B] int32
    p_draft: np.ndarray         # [B][k] p_i(x_i), fp64
    q_draft: np.ndarray         # [B][k] q_i(x_i), fp64
    lse_target: np.ndarray      # [B][k+1] log Z of each target row (of x / T)
    lse_draft: np.ndarray       # [B][k]
    status: np.ndarray          # [B] int32
    margins: list               # per sequence: array of n+1 margins, one per committed position
    empty_residual: np.ndarray  # [B] bool


def verify_stochastic(target, draft, tokens, dtype: str, temperature: float, seed: int,
                      seq_offset: int = 0, lenience: float = 1.0) -> StochasticResult:
    """Stochastic verification of B sequences (oracle).

    target [B][k+1][V], draft [B][k][V] stored logits; tokens [B][k].  Sequence b
    draws the randomness of global sequence index seq_offset + b.  lenience as in
    verify_sequence.
    """
    t = decode_logits(target, dtype)
    d = decode_logits(draft, dtype)
    tokens = np.asarray(tokens, dtype=np.int64)
    B, k1, V = t.shape
    k = k1 - 1
    out = np.full((B, k + 1), -1, dtype=np.int32)
    n_acc = np.zeros(B, dtype=np.int32)
    p_d = np.zeros((B, k))
    q_d = np.zeros((B, k))
    lse_t = np.zeros((B, k + 1))
    lse_d = np.zeros((B, k))
    status = np.zeros(B, dtype=np.int32)
    empty = np.zeros(B, dtype=bool)
    margins = []
    for b in range(B):
        trace = SequenceTrace()
        margins.append(np.zeros(0))
        if np.any(tokens[b] < 0) or np.any(tokens[b] >= V):
            status[b] = STATUS_TOKEN
            continue
        if _bad_rows(t[b, :k]) or _bad_rows(d[b]):
            status[b] = STATUS_NONFINITE
            continue
        with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
            logp, lse_t[b] = log_softmax(t[b], temperature)
            logq, lse_d[b] = log_softmax(d[b], temperature)
        p_d[b] = np.exp(logp[np.arange(k), tokens[b]])
        q_d[b] = np.exp(logq[np.arange(k), tokens[b]])
        gb = seq_offset + b
        seq, n = verify_sequence(logp, logq, tokens[b], _philox_accept(seed, gb),
                                 _gumbel_draw(seed, gb, trace), lenience=lenience)
        if n == k and _bad_rows(t[b, k:k + 1]):
            status[b] = STATUS_NONFINITE
            continue
        out[b, :len(seq)] = seq
        n_acc[b] = n
        empty[b] = trace.empty_residual
        margins[b] = position_margins(seed, gb, p_d[b], q_d[b], n, k, trace.draw_gap, lenience)
    return StochasticResult(out, n_acc, p_d, q_d, lse_t, lse_d, status, margins, empty)


# ----------------------------------------------------------------------------
# Greedy (T = 0) and greedy tree verification.
# ----------------------------------------------------------------------------

def argmax_first(row: np.ndarray) -> int:
    """Index of the largest value, the lowest index among equal maxima."""
    best = 0
    for v in range(1, row.shape[0]):
        if row[v] > row[best]:
            best = v
    return best


def row_argmax(rows: np.ndarray) -> np.ndarray:
    """argmax_first over the last axis (numpy's argmax has the same first-index rule)."""
    return np.argmax(rows, axis=-1).astype(np.int32)


@dataclass
class GreedyResult:
    out_tokens: np.ndarray   # [B][k+1]
    n_accepted: np.ndarray   # [B]
    argmax: np.ndarray       # [B][k+1] target argmax per row
    status: np.ndarray       # [B]


def verify_greedy(target, tokens, dtype: str) -> GreedyResult:
    """Greedy verification: accept while x_i equals the target argmax of row i;
    the first mismatch is replaced by that argmax; all accepted -> argmax of row k."""
    t = decode_logits(target, dtype)
    tokens = np.asarray(tokens, dtype=np.int64)
    B, k1, V = t.shape
    k = k1 - 1
    a = row_argmax(t)
    out = np.full((B, k + 1), -1, dtype=np.int32)
    n_acc = np.zeros(B, dtype=np.int32)
    status = np.zeros(B, dtype=np.int32)
    for b in range(B):
        if np.any(tokens[b] < 0) or np.any(tokens[b] >= V):
            status[b] = STATUS_TOKEN
            continue
        if np.any(np.isnan(t[b])):
            status[b] = STATUS_NONFINITE
            continue
        n = 0
        while n < k and tokens[b, n] == a[b, n]:
            n += 1
        out[b, :n] = tokens[b, :n]
        out[b, n] = a[b, n]
        n_acc[b] = n
    return GreedyResult(out, n_acc, a, status)


@dataclass
class TreeResult:
    out_tokens: np.ndarray   # [B][N+1]
    n_accepted: np.ndarray   # [B] depth of the chosen node (accepted draft tokens)
    leaf: np.ndarray         # [B] chosen node, -1 = none accepted
    argmax: np.ndarray       # [B][N+1]
    status: np.ndarray       # [B]


def tree_path(parents: np.ndarray, m: int) -> List[int]:
    """Nodes from the root-level ancestor down to m."""
    path = []
    while m >= 0:
        path.append(m)
        m = int(parents[m])
    return path[::-1]


def verify_tree(target, node_tokens, parents, dtype: str) -> TreeResult:
    """Greedy tree verification by brute force over every node's root path.

    Row 0 is the target output at the context, row 1+m the output at node m.
    A node is accepted iff every node u on its root path carries the argmax of
    the row at u's parent.  The deepest accepted node wins (lowest index among
    equally deep ones); the committed tokens are its path followed by the
    argmax of its own row.  With no accepted node, the argmax of row 0 alone is
    committed.  ("Ouroboros ..." 3.4.3, "Selecting the accepted tokens": the
    longest accepted extension plus the target's correction.)
    """
    t = decode_logits(target, dtype)
    node_tokens = np.asarray(node_tokens, dtype=np.int64)
    parents = np.asarray(parents, dtype=np.int64)
    B, N1, V = t.shape
    N = N1 - 1
    a = row_argmax(t)
    out = np.full((B, N + 1), -1, dtype=np.int32)
    n_acc = np.zeros(B, dtype=np.int32)
    leaf = np.full(B, -1, dtype=np.int32)
    status = np.zeros(B, dtype=np.int32)
    for b in range(B):
        par = parents[b]
        if np.any(node_tokens[b] < 0) or np.any(node_tokens[b] >= V) or \
                any(not (-1 <= par[m] < m) for m in range(N)):
            status[b] = STATUS_TOKEN
            continue
        if np.any(np.isnan(t[b])):
            status[b] = STATUS_NONFINITE
            continue
        best, best_depth = -1, 0
        for m in range(N):
            path = tree_path(par, m)
            ok = all(node_tokens[b, u] == a[b, 0 if par[u] < 0 else par[u] + 1] for u in path)
            if ok and len(path) > best_depth:
                best, best_depth = m, len(path)
        if best < 0:
            out[b, 0] = a[b, 0]
        else:
            path = tree_path(par, best)
            out[b, :len(path)] = node_tokens[b, path]
            out[b, len(path)] = a[b, best + 1]
        n_acc[b] = best_depth
        leaf[b] = best
    return TreeResult(out, n_acc, leaf, a, status)
