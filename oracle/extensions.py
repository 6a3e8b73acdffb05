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


# ----------------------------------------------------------------------------
# Consistent top-k / top-p filtering of p and q before verification
# ("Ouroboros: ...", random-sampling results with top-p 0.8; "Speculative
# Decoding: ...", "Logit-processor gaps" and "Constraints must be applied
# consistently": a processor applied to the target must be applied to the
# draft too, or the q the rule relies on is wrong).
#
# Readings (also in the design notes):
#   * order: temperature, then top-k, then top-p on the top-k distribution;
#   * both filters are value thresholds, so ties at a threshold are all kept:
#     top-k keeps x >= the k-th largest value (with multiplicity); top-p keeps
#     x >= the largest value tau whose mass {x >= tau} reaches top_p of the
#     mass left by top-k; -inf ids are never kept;
#   * top_k = 0 or >= the number of finite ids, and top_p = 0 or 1, leave the
#     row as it is;
#   * the filtered row is renormalised; greedy decisions do not change.
# ----------------------------------------------------------------------------

@dataclass
class RowFilter:
    keep: np.ndarray        # [V] bool
    tau: float              # the value threshold (-inf: nothing removed)
    margin: float           # distance of the top-p decision from its boundary, as a fraction of the mass
                            # (inf when no top-p decision was taken)


def filter_row(x: np.ndarray, temperature: float, top_k: int, top_p: float) -> RowFilter:
    """Kept ids of one logit row (fp64 values) under top-k then top-p."""
    x = np.asarray(x, dtype=np.float64)
    finite = np.isfinite(x)
    z = np.where(finite, x / float(temperature), -np.inf)
    m = np.max(z[finite]) if finite.any() else 0.0
    w = np.where(finite, np.exp(z - m), 0.0)
    tau = -np.inf
    if top_k and top_k < int(finite.sum()):
        tau = float(np.sort(x[finite])[::-1][top_k - 1])
    margin = np.inf
    if top_p and top_p < 1.0:
        base = finite & (x >= tau)
        mk = float(w[base].sum())
        target = top_p * mk
        values = np.unique(x[base])[::-1]                 # distinct values, descending
        cum = 0.0
        for v in values:
            grp = float(w[base & (x == v)].sum())
            if cum + grp >= target:
                # the chosen value moves when the target crosses either end of
                # its group's cumulative mass: the upper end (cum + grp) or the
                # lower end (cum), which only a group after the first has --
                # no top_p > 0 falls below a cumulative mass of 0
                upper = cum + grp - target
                margin = (min(upper, target - cum) if cum > 0 else upper) / mk
                tau = max(tau, float(v))
                break
            cum += grp
    keep = finite & (x >= tau)
    return RowFilter(keep, tau, margin)


def filtered_log_softmax(x: np.ndarray, temperature: float, top_k: int, top_p: float):
    """Natural-log probabilities of the filtered, renormalised softmax(x / T)
    (-inf outside the kept set), and the row's filter."""
    f = filter_row(x, temperature, top_k, top_p)
    z = np.where(f.keep, np.asarray(x, dtype=np.float64) / float(temperature), -np.inf)
    m = np.max(z[f.keep])
    lse = m + np.log(np.sum(np.exp(z[f.keep] - m)))
    return z - lse, f


@dataclass
class FilteredResult:
    out_tokens: np.ndarray   # [B][k+1]
    n_accepted: np.ndarray   # [B]
    status: np.ndarray       # [B]
    margins: list            # per sequence: n+1 margins (decision margins, capped by the filter margins)
    p_draft: np.ndarray      # [B][k] filtered p_i(x_i)
    q_draft: np.ndarray      # [B][k] filtered q_i(x_i)
    filter_margin: np.ndarray  # [B][2k+1]: target rows 0..k-1, draft rows 0..k-1, target row k


def verify_filtered(target, draft, tokens, dtype: str, temperature: float, seed: int, top_k: int, top_p: float,
                    seq_offset: int = 0, lenience: float = 1.0) -> FilteredResult:
    """Stochastic verification on consistently filtered p and q: every target
    row (bonus row included) and every draft row goes through the same top-k /
    top-p filter, then the rule of verify_stochastic runs on the filtered rows.
    A position's margin is its decision margin, capped by the top-p margins of
    the rows it depends on (target and draft row i for i < k, target row k)."""
    from . import verify as ov
    t = decode_logits(target, dtype)
    d = decode_logits(draft, dtype)
    tokens = np.asarray(tokens, dtype=np.int64)
    B, k1, V = t.shape
    k = k1 - 1
    out = np.full((B, k + 1), -1, dtype=np.int32)
    n_acc = np.zeros(B, dtype=np.int32)
    status = np.zeros(B, dtype=np.int32)
    p_d = np.zeros((B, k))
    q_d = np.zeros((B, k))
    fm = np.full((B, 2 * k + 1), np.inf)
    margins = []
    for b in range(B):
        margins.append(np.zeros(0))
        if np.any(tokens[b] < 0) or np.any(tokens[b] >= V):
            status[b] = STATUS_TOKEN
            continue
        if ov._bad_rows(t[b]) or ov._bad_rows(d[b]):
            status[b] = STATUS_NONFINITE
            continue
        logp = np.empty((k + 1, V))
        logq = np.empty((k, V))
        with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
            for j in range(k + 1):
                logp[j], f = filtered_log_softmax(t[b, j], temperature, top_k, top_p)
                fm[b, j if j < k else 2 * k] = f.margin
            for i in range(k):
                logq[i], f = filtered_log_softmax(d[b, i], temperature, top_k, top_p)
                fm[b, k + i] = f.margin
        p_d[b] = np.exp(logp[np.arange(k), tokens[b]])
        q_d[b] = np.exp(logq[np.arange(k), tokens[b]])
        gb = seq_offset + b
        trace = ov.SequenceTrace()
        seq, n = ov.verify_sequence(logp, logq, tokens[b], ov._philox_accept(seed, gb),
                                    ov._gumbel_draw(seed, gb, trace), lenience=lenience)
        out[b, :len(seq)] = seq
        n_acc[b] = n
        mg = ov.position_margins(seed, gb, p_d[b], q_d[b], n, k, trace.draw_gap, lenience)
        for j in range(n + 1):
            # position j follows from target and draft rows 0..j (and the bonus row at j = k)
            last = min(j, k - 1)
            cap = min(fm[b, :last + 1].min(), fm[b, k:k + last + 1].min())
            if j == k:
                cap = min(cap, fm[b, 2 * k])
            mg[j] = min(mg[j], cap)
        margins[b] = mg
    return FilteredResult(out, n_acc, status, margins, p_d, q_d, fm)
