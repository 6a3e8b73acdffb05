"""Additions to the verification step that the pages describe next to the rule (oracle).

TEST INFRASTRUCTURE ONLY (see the package docstring).

  * #Match and the matched runs of a greedy round -- "Ouroboros: Generating
    Longer Drafts Phrase by Phrase for Faster Speculative Decoding", Equation
    (10) and the phrase-harvesting step that follows it: d_i is compared with
    the target's own token v_i at the same position; #Match counts the
    positions where they agree, whether or not they are contiguous, and the
    runs of agreeing positions after the first disagreement are the segments a
    harvester keeps.
  * Truncation at a stop token -- "Speculative Decoding: Faster Generation
    Without Changing the Model", "Constraints must be applied consistently":
    when the committed tokens contain an end-of-sequence or stop token,
    everything after it is dropped.
  * Target-guided greedy verification -- "Double: Breaking the Acceleration
    Limit via Double Retrieval Speculative Parallelism", "Multi-token
    Pre-verify" and D.2: the verified draft prefix, then the target's
    correction, then the remaining tokens of a target-side guide, which stay
    valid because they follow the corrected path (greedy decoding only; under
    sampling the guidance is dropped after a rejection).

Readings where the pages leave a step open (also in the design notes):
  * v_i of a greedy round is the argmax of target row i (lowest index), the
    token the target itself puts at position i.
  * A "run after the first disagreement" is a maximal run of agreeing
    positions i > n, n being the accepted count (position n disagrees).
  * The guide g is aligned with the draft positions (g_i is the target-side
    token for position i).  Its tokens from n + 1 on are appended only when
    g_n equals the correction a*_n -- only then do they continue the corrected
    path -- and up to the first negative entry (the guide's end).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from .verify import STATUS_NONFINITE, STATUS_OK, STATUS_TOKEN, decode_logits, row_argmax


@dataclass
class MatchStats:
    mask: np.ndarray        # [B][k] uint8: 1 iff d_i == v_i
    n_match: np.ndarray     # [B] int32: #Match, Equation (10)
    tail_runs: np.ndarray   # [B] int32: maximal runs of matches after the first mismatch


def match_stats(target, tokens, dtype: str) -> MatchStats:
    """#Match(d_1..k, v_1..k) = sum_i [d_i = v_i] with v_i the argmax of target
    row i, and the runs of matches after the accepted prefix."""
    t = decode_logits(target, dtype)
    tokens = np.asarray(tokens, dtype=np.int64)
    B, k1, _ = t.shape
    k = k1 - 1
    v = row_argmax(t)
    mask = np.zeros((B, k), dtype=np.uint8)
    n_match = np.zeros(B, dtype=np.int32)
    runs = np.zeros(B, dtype=np.int32)
    for b in range(B):
        hits = [int(tokens[b, i] == v[b, i]) for i in range(k)]
        mask[b] = hits
        n_match[b] = sum(hits)
        n = 0
        while n < k and hits[n]:
            n += 1
        inside = False
        for i in range(n + 1, k):
            if hits[i] and not inside:
                runs[b] += 1
            inside = bool(hits[i])
    return MatchStats(mask, n_match, runs)


def truncate_at_stop(out_tokens, stop_ids):
    """Drop every committed token after the first one that is a stop id.

    out_tokens [B][W] with -1 after the committed tokens.  Returns the truncated
    copy and the committed counts [B] (the stop token itself stays committed).
    """
    out = np.array(out_tokens, dtype=np.int32, copy=True)
    stops = set(int(s) for s in stop_ids)
    B, W = out.shape
    count = np.zeros(B, dtype=np.int32)
    for b in range(B):
        c = 0
        while c < W and out[b, c] >= 0:
            c += 1
            if int(out[b, c - 1]) in stops:
                break
        out[b, c:] = -1
        count[b] = c
    return out, count


@dataclass
class GuidedResult:
    out_tokens: np.ndarray   # [B][max(k+1, L)], -1 after the committed tokens
    n_accepted: np.ndarray   # [B] accepted draft tokens
    n_committed: np.ndarray  # [B]
    status: np.ndarray       # [B]


def verify_guided(target, tokens, guide, dtype: str) -> GuidedResult:
    """Greedy verification of the draft chain, then the target-side guide.

    target [B][k+1][V]; tokens [B][k]; guide [B][L] (negative = past its end).
    Committed: x_0..x_{n-1}, the correction a*_n, and, when g_n == a*_n, the
    guide's tokens g_{n+1}, g_{n+2}, ... up to its end or the row width.
    """
    t = decode_logits(target, dtype)
    tokens = np.asarray(tokens, dtype=np.int64)
    guide = np.asarray(guide, dtype=np.int64)
    B, k1, V = t.shape
    k = k1 - 1
    L = guide.shape[1]
    W = max(k + 1, L)
    a = row_argmax(t)
    out = np.full((B, W), -1, dtype=np.int32)
    n_acc = np.zeros(B, dtype=np.int32)
    n_com = np.zeros(B, dtype=np.int32)
    status = np.zeros(B, dtype=np.int32)
    for b in range(B):
        if np.any(tokens[b] < 0) or np.any(tokens[b] >= V) or np.any(guide[b] >= V):
            status[b] = STATUS_TOKEN
            n_acc[b] = n_com[b] = -1
            continue
        if np.any(np.isnan(t[b])):
            status[b] = STATUS_NONFINITE
            n_acc[b] = n_com[b] = -1
            continue
        n = 0
        while n < k and tokens[b, n] == a[b, n]:
            n += 1
        seq = [int(x) for x in tokens[b, :n]] + [int(a[b, n])]
        if n < L and guide[b, n] == a[b, n]:
            for i in range(n + 1, L):
                if guide[b, i] < 0:
                    break
                seq.append(int(guide[b, i]))
        out[b, :len(seq)] = seq
        n_acc[b] = n
        n_com[b] = len(seq)
        status[b] = STATUS_OK
    return GuidedResult(out, n_acc, n_com, status)
