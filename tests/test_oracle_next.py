"""Pins for the oracle's additions next to the rule (CPU only): lenience,
#Match and the matched runs, truncation at a stop token, target-guided greedy
verification.  Each is checked against what the pages state or against a
closed form / brute force the test writes itself, so that a slip in the
oracle (lenience in the wrong branch or in the residual, a shifted match
position, a run counted inside the accepted prefix, a guide appended off the
corrected path) fails here.
"""
import itertools
import re

import numpy as np
import pytest

from oracle import enumerate as oenum
from oracle import extensions as ox
from oracle import verify as ov


def _lg(p):
    with np.errstate(divide="ignore"):
        return np.log(np.asarray(p, dtype=np.float64))


def _rand_dist(rng, V, zero_frac=0.0):
    w = rng.random(V) + 0.05
    if zero_frac:
        w[rng.random(V) < zero_frac] = 0.0
        if w.sum() == 0:
            w[0] = 1.0
    return w / w.sum()


# --------------------------------------------------------------- lenience ---

def test_lenience_one_is_the_exact_rule():
    rng = np.random.default_rng(5)
    for _ in range(20):
        k, V = 3, 6
        logp = np.stack([_lg(_rand_dist(rng, V, 0.3)) for _ in range(k + 1)])
        logq = np.stack([_lg(_rand_dist(rng, V, 0.3)) for _ in range(k)])
        law1 = oenum.full_law(logp, logq, lenience=1.0)
        law0 = oenum.full_law(logp, logq)
        assert set(law1) == set(law0)
        for key in law0:
            assert law1[key] == pytest.approx(law0[key], abs=1e-15)


@pytest.mark.parametrize("l", [1.0, 1.3, 2.0, 5.0])
def test_lenience_first_token_law_closed_form(l):
    """k = 1: x ~ q is kept with probability min(1, l p(x)/q(x)); otherwise the
    replacement comes from norm(max(0, p - q)).  The first committed token's law
    is then q(v) min(1, l p(v)/q(v)) + (1 - beta) r(v)."""
    rng = np.random.default_rng(int(l * 10))
    V = 7
    for _ in range(10):
        p0, p1, q0 = _rand_dist(rng, V, 0.2), _rand_dist(rng, V), _rand_dist(rng, V, 0.2)
        law = oenum.full_law(np.stack([_lg(p0), _lg(p1)]), _lg(q0)[None], lenience=l)
        first = np.zeros(V)
        for key, pr in law.items():
            first[key[0]] += pr
        keep = np.where(q0 > 0, q0 * np.minimum(1.0, l * p0 / np.where(q0 > 0, q0, 1.0)), 0.0)
        beta = keep.sum()
        r = np.maximum(0.0, p0 - q0)
        expect = keep + ((1.0 - beta) * r / r.sum() if r.sum() > 0 else 0.0)
        np.testing.assert_allclose(first, expect, atol=1e-12)
        assert sum(law.values()) == pytest.approx(1.0, abs=1e-12)


def test_lenience_residual_is_not_scaled():
    """The pages keep the residual at norm(max(0, p - q)) under lenience; a
    residual of max(0, l p - q) gives a different law, which the closed form of
    the test above would catch."""
    V, l = 5, 2.0
    p0 = np.array([0.4, 0.3, 0.2, 0.1, 0.0])
    q0 = np.array([0.05, 0.05, 0.1, 0.3, 0.5])
    keep = q0 * np.minimum(1.0, l * p0 / q0)
    r_page = np.maximum(0.0, p0 - q0)
    r_scaled = np.maximum(0.0, l * p0 - q0)
    a = keep + (1 - keep.sum()) * r_page / r_page.sum()
    b = keep + (1 - keep.sum()) * r_scaled / r_scaled.sum()
    assert np.max(np.abs(a - b)) > 1e-3
    law = oenum.full_law(np.stack([_lg(p0), _lg(np.full(V, 1 / V))]), _lg(q0)[None], lenience=l)
    first = np.zeros(V)
    for key, pr in law.items():
        first[key[0]] += pr
    np.testing.assert_allclose(first, a, atol=1e-12)


def test_lenience_raises_acceptance_and_large_l_accepts_everything():
    rng = np.random.default_rng(11)
    k, V = 3, 5
    logp = np.stack([_lg(_rand_dist(rng, V)) for _ in range(k + 1)])
    logq = np.stack([_lg(_rand_dist(rng, V)) for _ in range(k)])

    def mean_accepted(l):
        q = np.exp(logq)
        tot = 0.0
        for xs in itertools.product(range(V), repeat=k):
            w = float(np.prod([q[i, xs[i]] for i in range(k)]))
            for key, pr in oenum.output_law(logp, logq, xs, l).items():
                # accepted drafts: the committed prefix that equals the drafts, one replacement after
                tot += w * pr * (len(key) - 1)
        return tot

    vals = [mean_accepted(l) for l in (1.0, 1.5, 3.0)]
    assert vals[0] <= vals[1] + 1e-12 <= vals[2] + 2e-12
    big = float(np.max(np.exp(logq) / np.exp(logp[:k]))) * 1.01
    assert mean_accepted(big) == pytest.approx(k, abs=1e-12)


def test_lenience_in_the_production_path():
    """The Philox path with l: a draft with q > l p is kept iff u < l p / q."""
    from oracle import philox
    V, k, seed = 4, 1, 77
    t = np.log(np.array([[0.1, 0.2, 0.3, 0.4], [0.25, 0.25, 0.25, 0.25]]))[None].astype(np.float32)
    d = np.log(np.array([[0.7, 0.1, 0.1, 0.1]]))[None].astype(np.float32)
    tokens = np.array([[0]], dtype=np.int32)
    u = philox.accept_uniform(seed, 0, 0)
    for l in (1.0, 2.0, 3.0, 6.0, 7.5):
        res = ov.verify_stochastic(t, d, tokens, "fp32", 1.0, seed, lenience=l)
        ratio = l * res.p_draft[0, 0] / res.q_draft[0, 0]
        kept = res.q_draft[0, 0] <= l * res.p_draft[0, 0] or u < ratio
        assert (res.n_accepted[0] == 1) == kept, (l, u, ratio)


# ----------------------------------------------------------------- #Match ---

def _rows_with_argmax(argmaxes, V):
    """Target logits whose row j has its unique maximum at argmaxes[j]."""
    t = np.zeros((1, len(argmaxes), V), dtype=np.float32)
    for j, a in enumerate(argmaxes):
        t[0, j, a] = 5.0
    return t


def test_match_worked_example_on_the_page(golden):
    rows = golden("ouroboros_match_example.txt")
    draft = next(r[1:] for r in rows if r[0] == "draft")
    verif = next(r[1:] for r in rows if r[0] == "verification")
    want_acc = int(next(r[1] for r in rows if r[0] == "accepted"))
    want_match = int(next(r[1] for r in rows if r[0] == "match"))
    vocab = sorted(set(draft) | set(verif))
    ids = {w: i for i, w in enumerate(vocab)}
    t = _rows_with_argmax([ids[w] for w in verif], len(vocab))
    tokens = np.array([[ids[w] for w in draft]], dtype=np.int32)
    st = ox.match_stats(t, tokens, "fp32")
    g = ov.verify_greedy(t, tokens, "fp32")
    assert g.n_accepted[0] == want_acc
    assert st.n_match[0] == want_match
    assert st.tail_runs[0] == 0
    assert list(st.mask[0]) == [1, 1, 0]


def test_match_brute_force():
    rng = np.random.default_rng(3)
    for _ in range(300):
        k = int(rng.integers(1, 12))
        V = int(rng.integers(2, 5))
        a = rng.integers(0, V, size=k + 1)
        t = _rows_with_argmax(a, V)
        tokens = np.where(rng.random(k) < 0.6, a[:k], rng.integers(0, V, size=k))[None].astype(np.int32)
        st = ox.match_stats(t, tokens, "fp32")
        hits = "".join("1" if tokens[0, i] == a[i] else "0" for i in range(k))
        n = len(hits) - len(hits.lstrip("1"))
        assert st.n_match[0] == hits.count("1")
        assert st.tail_runs[0] == len(re.findall("1+", hits[n + 1:]))
        assert st.n_match[0] >= ov.verify_greedy(t, tokens, "fp32").n_accepted[0]
        assert "".join(map(str, st.mask[0])) == hits


# -------------------------------------------------------------- stop ids ---

def test_stop_truncation_hand_built():
    out = np.array([[5, 9, 3, 7, -1], [9, 1, 2, -1, -1], [1, 2, 3, 4, 5], [-1, -1, -1, -1, -1]], dtype=np.int32)
    tr, cnt = ox.truncate_at_stop(out, [9, 4])
    assert tr.tolist() == [[5, 9, -1, -1, -1], [9, -1, -1, -1, -1], [1, 2, 3, 4, -1], [-1] * 5]
    assert cnt.tolist() == [2, 1, 4, 0]
    tr, cnt = ox.truncate_at_stop(out, [])
    assert tr.tolist() == out.tolist() and cnt.tolist() == [4, 3, 5, 0]


def test_stop_truncation_properties():
    rng = np.random.default_rng(8)
    for _ in range(200):
        W = int(rng.integers(1, 10))
        c = int(rng.integers(0, W + 1))
        out = np.full((1, W), -1, dtype=np.int32)
        out[0, :c] = rng.integers(0, 6, size=c)
        stops = list(rng.choice(6, size=int(rng.integers(0, 3)), replace=False))
        tr, cnt = ox.truncate_at_stop(out, stops)
        kept = list(tr[0, :cnt[0]])
        assert kept == list(out[0, :cnt[0]])
        assert all(x == -1 for x in tr[0, cnt[0]:])
        assert not any(x in stops for x in kept[:-1])
        assert cnt[0] == c or kept[-1] in stops


# ----------------------------------------------------- target-guided greedy ---

def test_guided_hand_built():
    V = 10
    a = [1, 2, 3, 4, 5]                     # target argmax of rows 0..4 (k = 4)
    t = _rows_with_argmax(a, V)
    cases = [
        # tokens, guide, committed, accepted
        ([1, 2, 9, 9], [1, 2, 3, 7, 8, 6], [1, 2, 3, 7, 8, 6], 2),    # correction agrees with g_2: guide appended
        ([1, 2, 9, 9], [1, 2, 8, 7, 8, 6], [1, 2, 3], 2),             # g_2 != a*_2: plain greedy
        ([1, 2, 9, 9], [1, 2, 3, 7, -1, 6], [1, 2, 3, 7], 2),         # the guide ends at its first negative entry
        ([1, 2, 3, 4], [1, 2, 3, 4, 5, 6, 0], [1, 2, 3, 4, 5, 6, 0], 4),  # all accepted: bonus, then the guide
        ([1, 2, 3, 4], [1, 2, 3], [1, 2, 3, 4, 5], 4),                # guide shorter than the accepted prefix
        ([9, 2, 3, 4], [1, 0, 0, 0, 0], [1, 0, 0, 0, 0], 0),          # first draft rejected
    ]
    for tokens, guide, committed, acc in cases:
        L = max(len(guide), 1)
        g = np.full((1, L), -1, dtype=np.int32)
        g[0, :len(guide)] = guide
        r = ox.verify_guided(t, np.array([tokens], dtype=np.int32), g, "fp32")
        assert r.n_accepted[0] == acc
        assert r.n_committed[0] == len(committed)
        assert list(r.out_tokens[0, :len(committed)]) == committed
        assert all(x == -1 for x in r.out_tokens[0, len(committed):])


def test_guided_without_guide_is_greedy():
    rng = np.random.default_rng(21)
    B, k, V = 6, 5, 7
    t = rng.normal(size=(B, k + 1, V)).astype(np.float32)
    a = ov.row_argmax(t.astype(np.float64))
    tokens = np.where(rng.random((B, k)) < 0.7, a[:, :k], rng.integers(0, V, size=(B, k))).astype(np.int32)
    g = ov.verify_greedy(t, tokens, "fp32")
    r = ox.verify_guided(t, tokens, np.full((B, 3), -1, dtype=np.int32), "fp32")
    np.testing.assert_array_equal(r.out_tokens[:, :k + 1], g.out_tokens)
    np.testing.assert_array_equal(r.n_accepted, g.n_accepted)
    np.testing.assert_array_equal(r.n_committed, g.n_accepted + 1)


def test_guided_bad_ids():
    t = _rows_with_argmax([1, 2, 3], 5)
    r = ox.verify_guided(t, np.array([[1, 2]], dtype=np.int32), np.array([[1, 2, 7]], dtype=np.int32), "fp32")
    assert r.status[0] == ov.STATUS_TOKEN and r.n_committed[0] == -1


# --------------------------------------------------------- top-k / top-p ---

def test_filter_top_k_by_brute_force():
    rng = np.random.default_rng(31)
    for _ in range(200):
        V = int(rng.integers(2, 12))
        x = rng.integers(-3, 4, size=V).astype(np.float64)        # many ties
        if rng.random() < 0.3:
            x[rng.integers(0, V)] = -np.inf
        kk = int(rng.integers(1, V + 2))
        f = ox.filter_row(x, 1.0, kk, 0.0)
        fin = np.isfinite(x)
        if kk >= fin.sum():
            assert np.array_equal(f.keep, fin)
            continue
        # brute force: the k-th largest value with multiplicity, ties kept
        kth = sorted(x[fin], reverse=True)[kk - 1]
        assert np.array_equal(f.keep, fin & (x >= kth))
        assert f.keep.sum() >= kk


def test_filter_top_p_by_brute_force():
    rng = np.random.default_rng(32)
    for _ in range(300):
        V = int(rng.integers(1, 10))
        x = rng.integers(-4, 4, size=V).astype(np.float64) * 0.5
        T = float(rng.choice([0.5, 1.0, 2.0]))
        top_p = float(rng.choice([0.1, 0.5, 0.8, 0.95, 0.999]))
        f = ox.filter_row(x, T, 0, top_p)
        w = np.exp(x / T - np.max(x / T))
        w /= w.sum()
        # brute force over every threshold among the values: the highest one reaching top_p
        best = None
        for tau in sorted(set(x), reverse=True):
            if w[x >= tau].sum() >= top_p * (1 - 1e-12):
                best = tau
                break
        assert np.array_equal(f.keep, x >= best), (x, T, top_p)
        # minimal: dropping the lowest kept value falls short of top_p
        higher = [v for v in set(x) if v > best]
        if higher:
            assert w[x >= min(higher)].sum() < top_p


def test_filter_top_k_then_top_p_and_identities():
    x = np.array([3.0, 2.0, 2.0, 1.0, 0.0, -1.0])
    w = np.exp(x - x.max())
    # top-k 3 keeps the ties at 2.0 as well: {3, 2, 2}; then top-p 0.6 of that mass
    f = ox.filter_row(x, 1.0, 3, 0.6)
    mk = w[:3].sum()
    assert w[0] / mk < 0.6 <= w[:3].sum() / mk
    assert f.keep.tolist() == [True, True, True, False, False, False]
    f = ox.filter_row(x, 1.0, 3, 0.3)
    assert w[0] / mk >= 0.3 and f.keep.tolist() == [True] + [False] * 5
    for kk, pp in [(0, 0.0), (0, 1.0), (6, 0.0), (10, 1.0)]:
        assert ox.filter_row(x, 1.0, kk, pp).keep.all()


def test_filtered_verification_is_lossless_for_the_filtered_target():
    """On consistently filtered rows, the rule commits tokens distributed as the
    filtered target (exact enumeration at V = 6, k = 2)."""
    from oracle import enumerate as oenum
    rng = np.random.default_rng(41)
    k, V = 2, 6
    for top_k, top_p in [(3, 0.0), (0, 0.7), (4, 0.8)]:
        t = rng.normal(size=(k + 1, V)) * 1.5
        d = t[:k] + rng.normal(size=(k, V))
        logp = np.stack([ox.filtered_log_softmax(t[j], 1.0, top_k, top_p)[0] for j in range(k + 1)])
        logq = np.stack([ox.filtered_log_softmax(d[i], 1.0, top_k, top_p)[0] for i in range(k)])
        law = oenum.full_law(logp, logq)
        assert sum(law.values()) == pytest.approx(1.0, abs=1e-12)
        first = np.zeros(V)
        for key, pr in law.items():
            first[key[0]] += pr
        np.testing.assert_allclose(first, np.exp(logp[0]), atol=1e-12)


def test_verify_filtered_matches_the_plain_rule_without_filters():
    import workloads as wl
    w = wl.c1_tiny(seed=5)
    a = ov.verify_stochastic(w.target, w.draft, w.tokens, w.dtype, w.temperature, 77)
    b = ox.verify_filtered(w.target, w.draft, w.tokens, w.dtype, w.temperature, 77, 0, 0.0)
    np.testing.assert_array_equal(a.out_tokens, b.out_tokens)
    np.testing.assert_array_equal(a.n_accepted, b.n_accepted)
    np.testing.assert_allclose(a.p_draft, b.p_draft, rtol=1e-12)


def test_verify_filtered_restricts_every_committed_token():
    """Committed tokens lie in the kept set of the target row at their position."""
    import workloads as wl
    w = wl.c2(seed=9)
    r = ox.verify_filtered(w.target, w.draft, w.tokens, w.dtype, w.temperature, 3, 20, 0.9)
    t = ov.decode_logits(w.target, w.dtype)
    for b in range(w.B):
        for j in range(r.n_accepted[b] + 1):
            f = ox.filter_row(t[b, j], w.temperature, 20, 0.9)
            tok = r.out_tokens[b, j]
            if j < r.n_accepted[b]:
                continue                 # an accepted draft may lie outside p's kept set only if q'(x) = 0 too
            assert f.keep[tok], (b, j, tok)
