"""Pins for the oracle's verification rule (CPU only).

Each test checks the oracle against something it does not compute itself:
hand-built cases whose outcome the rule fixes, exact enumeration of the output
law (losslessness), chi-squared laws, the closed forms the pages print, brute
force.  A plausible slip (inverted ratio, wrong residual sign, off-by-one row,
wrong bonus row, wrong tie rule) fails at least one of them.
"""
import math
from collections import defaultdict

import numpy as np
import pytest
from scipy import special, stats

import workloads as wl
from oracle import enumerate as oenum
from oracle import philox, theory
from oracle import verify as ov


def _logits(p):
    p = np.asarray(p, dtype=np.float64)
    with np.errstate(divide="ignore"):
        return np.log(p)


# ---------------------------------------------------------------- softmax ---

def test_log_softmax_against_scipy_and_invariants():
    rng = np.random.default_rng(3)
    x = rng.normal(0, 4, size=(5, 1000))
    for T in (1.0, 0.7, 2.5):
        lp, lse = ov.log_softmax(x, T)
        np.testing.assert_allclose(lp, special.log_softmax(x / T, axis=-1), atol=1e-12)
        np.testing.assert_allclose(lse, special.logsumexp(x / T, axis=-1), atol=1e-12)
        np.testing.assert_allclose(np.exp(lp).sum(-1), 1.0, atol=1e-12)
        lp2, _ = ov.log_softmax(x + 17.0, T)                    # shift invariance
        np.testing.assert_allclose(lp2, lp, atol=1e-10)


def test_bf16_decode_is_exact():
    vals = np.array([0.0, -0.0, 1.0, -2.5, 3.140625, -np.inf, 1e30], dtype=np.float32)
    bits = wl.bf16_bits_from_f32(vals)
    dec = ov.decode_logits(bits, "bf16")
    assert dec[0] == 0 and dec[2] == 1 and dec[3] == -2.5 and dec[4] == 3.140625
    assert dec[5] == -np.inf


# ------------------------------------------------------- hand-built cases ---

def _run(t, d, tokens, T=1.0, seed=1234):
    return ov.verify_stochastic(np.asarray(t, np.float32), np.asarray(d, np.float32),
                                np.asarray(tokens, np.int32), "fp32", T, seed)


def test_q_le_p_always_accepts():
    """Draft mass on the token never exceeds the target's -> every draft passes."""
    k, V = 4, 6
    p = np.array([0.05, 0.3, 0.15, 0.2, 0.1, 0.2])
    q = np.array([0.3, 0.05, 0.15, 0.1, 0.2, 0.2])          # q <= p on ids 1, 2, 3, 5
    B = 64
    tokens = np.tile(np.array([1, 2, 3, 5]), (B, 1))
    t = np.tile(_logits(p), (B, k + 1, 1))
    d = np.tile(_logits(q), (B, k, 1))
    for seed in (1, 2, 3):
        r = _run(t, d, tokens, seed=seed)
        assert np.all(r.n_accepted == k)
        assert np.all(r.out_tokens[:, :k] == tokens)
        assert all(len(m) == k + 1 for m in r.margins)


def test_target_zero_always_rejects_and_resamples_from_target_support():
    k, V, B = 3, 5, 200
    t = np.tile(_logits([0.0, 0.2, 0.3, 0.5, 0.0]), (B, k + 1, 1))
    d = np.tile(_logits([0.4, 0.2, 0.2, 0.2, 0.0]), (B, k, 1))
    tokens = np.zeros((B, k), np.int32)                        # p(0) = 0, q(0) = 0.4
    r = _run(t, d, tokens)
    assert np.all(r.n_accepted == 0)
    # residual max(0, p - q) = (0, 0, 0.1, 0.3, 0): only ids 2 and 3 can appear
    assert set(np.unique(r.out_tokens[:, 0])) <= {2, 3}
    assert np.all(r.out_tokens[:, 1:] == -1)


def test_decision_on_either_side_of_the_uniform():
    """Accept iff u < p/q: set p/q just above / below the uniform of (seed, b=0, i=0)."""
    seed = 77
    u = philox.accept_uniform(seed, 0, 0)
    for delta, want in ((+1e-4, 1), (-1e-4, 0)):
        ratio = u + delta
        q = np.array([0.5, 0.5])
        p = np.array([0.5 * ratio, 1 - 0.5 * ratio])
        t = _logits(p)[None, None, :].repeat(2, axis=1)
        d = _logits(q)[None, None, :]
        r = _run(t, d, [[0]], seed=seed)
        assert r.n_accepted[0] == want
        if want == 0:
            assert r.out_tokens[0, 0] == 1                    # residual is all on id 1
        assert abs(r.margins[0][0] - abs(delta)) < 1e-6          # logits are stored in fp32


def test_disjoint_draft_residual_equals_target():
    """q disjoint from p: p(x) = 0 forces a rejection and max(0, p - q) = p."""
    V, B = 8, 20000
    p = np.array([0.0, 0.0, 0.0, 0.1, 0.2, 0.3, 0.15, 0.25])
    q = np.array([0.5, 0.3, 0.2, 0.0, 0.0, 0.0, 0.0, 0.0])
    rng = np.random.default_rng(5)
    tokens = rng.choice(V, size=(B, 1), p=q).astype(np.int32)
    t = np.tile(_logits(p), (B, 2, 1))
    d = np.tile(_logits(q), (B, 1, 1))
    r = _run(t, d, tokens)
    assert np.all(r.n_accepted == 0)
    counts = np.bincount(r.out_tokens[:, 0], minlength=V)
    assert counts[:3].sum() == 0
    assert stats.chisquare(counts[3:], B * p[3:]).pvalue > 1e-3


def test_all_accepted_draws_bonus_from_row_k():
    """Identical draft and target rows accept everything; the bonus follows row k."""
    k, V, B = 2, 6, 20000
    rows = np.array([[0.5, 0.1, 0.1, 0.1, 0.1, 0.1],
                     [0.1, 0.5, 0.1, 0.1, 0.1, 0.1],
                     [0.05, 0.05, 0.1, 0.2, 0.25, 0.35]])     # row k differs from rows 0, 1
    t = np.tile(_logits(rows), (B, 1, 1))
    d = t[:, :k].copy()
    tokens = np.tile([0, 1], (B, 1)).astype(np.int32)
    r = _run(t, d, tokens)
    assert np.all(r.n_accepted == k)
    counts = np.bincount(r.out_tokens[:, k], minlength=V)
    assert stats.chisquare(counts, B * rows[k]).pvalue > 1e-3


def test_temperature_scales_both_rows():
    k, V = 1, 4
    t = np.array([[[1.0, 2.0, 0.5, -1.0], [0.0, 0.0, 0.0, 0.0]]])
    d = np.array([[[2.0, 1.0, 0.5, -1.0]]])
    for T in (0.5, 1.0, 3.0):
        r = _run(t, d, [[1]], T=T)
        np.testing.assert_allclose(r.p_draft[0, 0], special.softmax(t[0, 0] / T)[1], atol=1e-15)
        np.testing.assert_allclose(r.q_draft[0, 0], special.softmax(d[0, 0] / T)[1], atol=1e-15)


def test_bad_inputs_set_status():
    k, V = 2, 4
    t = np.zeros((3, k + 1, V), np.float32)
    d = np.zeros((3, k, V), np.float32)
    tokens = np.array([[0, 1], [0, 4], [1, 2]], np.int32)     # seq 1: id 4 out of range
    t[2, 1, 3] = np.nan                                         # seq 2: NaN in a verified row
    r = _run(t, d, tokens)
    assert list(r.status) == [ov.STATUS_OK, ov.STATUS_TOKEN, ov.STATUS_NONFINITE]


# ---------------------------------------------- losslessness (exact, chi2) ---

def _conditional_laws(law, k):
    """P(y_j = v | prefix, at least j+1 tokens committed), from an exact law."""
    cond = defaultdict(lambda: defaultdict(float))
    for out, pr in law.items():
        for j in range(len(out)):
            cond[(j, out[:j])][out[j]] += pr
    return cond


@pytest.mark.parametrize("k,V,mask", [(3, 8, False), (2, 8, True), (1, 5, False)])
def test_exact_enumeration_is_lossless(k, V, mask):
    """Every committed token follows the target row of its position, exactly."""
    t, d = wl.tiny_rows(k=k, V=V, seed=11 + k)
    if mask:
        t[0, 2] = -np.inf          # a masked target entry
        d[1, 5] = -np.inf          # a masked draft entry
    logp, _ = ov.log_softmax(t, 1.0)
    logq, _ = ov.log_softmax(d, 1.0)
    law = oenum.full_law(logp, logq)
    assert abs(sum(law.values()) - 1.0) < 1e-12
    p = np.exp(logp)
    for (j, prefix), dist in _conditional_laws(law, k).items():
        tot = sum(dist.values())
        for v in range(V):
            assert abs(dist.get(v, 0.0) / tot - p[j, v]) < 1e-12, (j, prefix, v)


def test_enumeration_detects_a_wrong_rule():
    """Sanity of the pin itself: the law of a rule with the ratio inverted is not lossless."""
    t, d = wl.tiny_rows(k=1, V=5, seed=3)
    logp, _ = ov.log_softmax(t, 1.0)
    logq, _ = ov.log_softmax(d, 1.0)
    law = oenum.full_law(logp, logq)
    good = sum(pr for out, pr in law.items() if out[0] == 0)
    bad_law = oenum.full_law(np.vstack([logq, logp[1:]]), logp[:1])   # roles of p and q swapped
    bad = sum(pr for out, pr in bad_law.items() if out[0] == 0)
    assert abs(good - np.exp(logp[0, 0])) < 1e-12
    assert abs(bad - np.exp(logp[0, 0])) > 1e-3


def test_production_draws_follow_target_chi2():
    """Counter-based draws through the full oracle: committed tokens ~ target rows."""
    k, V, B = 3, 8, 30000
    t, d = wl.tiny_rows(k=k, V=V, seed=21)
    p = special.softmax(t, axis=-1)
    q = special.softmax(d, axis=-1)
    rng = np.random.default_rng(8)
    tokens = np.stack([rng.choice(V, size=B, p=q[i]) for i in range(k)], axis=1).astype(np.int32)
    r = ov.verify_stochastic(np.tile(t, (B, 1, 1)).astype(np.float32), np.tile(d, (B, 1, 1)).astype(np.float32),
                             tokens, "fp32", 1.0, seed=4321)
    for j in range(k + 1):
        sel = r.n_accepted >= j
        counts = np.bincount(r.out_tokens[sel, j], minlength=V)
        pj = special.softmax(t[j].astype(np.float32).astype(np.float64))
        assert stats.chisquare(counts, counts.sum() * pj).pvalue > 1e-4, j


# ------------------------------------------------- committed-count closed form

def test_worked_values_on_the_page(golden):
    for kind, a, k, c, value, dec in golden("expected_tokens_worked.txt"):
        a, k, value, dec = float(a), int(k), float(value), int(dec)
        got = theory.expected_committed(a, k) if kind == "expected" else theory.speedup(a, k, float(c))
        assert round(got, dec) == value, (kind, a, k, got)


@pytest.mark.parametrize("a,k", [(0.8, 4), (0.6, 4), (0.8, 16), (0.6, 16), (0.3, 1)])
def test_pgf_coefficients_and_mean(a, k):
    pmf = theory.committed_pmf(a, k)
    assert abs(pmf.sum() - 1) < 1e-12
    assert abs((np.arange(k + 2) * pmf).sum() - theory.expected_committed(a, k)) < 1e-12
    for x in (0.3, 0.9, 1.7):
        assert abs(theory.pgf(a, k, x) - np.polyval(pmf[::-1], x)) < 1e-10
    # derivative of the closed-form PGF at 1 (central difference) = E[m]
    h = 1e-6
    d = (theory.pgf(a, k, 1 + h) - theory.pgf(a, k, 1 - h)) / (2 * h)
    assert abs(d - theory.expected_committed(a, k)) < 1e-6


@pytest.mark.parametrize("a", [0.6, 0.8])
def test_iid_acceptance_commits_per_the_pgf(a):
    """Inputs with acceptance exactly a: committed count ~ Theorem 4.1's law."""
    k, B = 4, 4000
    w = wl.iid_acceptance(B, k, 16, a, seed=int(a * 100))
    r = ov.verify_stochastic(w.target, w.draft, w.tokens, w.dtype, 1.0, seed=99)
    m = r.n_accepted + 1
    pmf = theory.committed_pmf(a, k)
    counts = np.bincount(m, minlength=k + 2)[1:]
    assert stats.chisquare(counts, B * pmf[1:]).pvalue > 1e-3
    sd = math.sqrt((np.arange(k + 2) ** 2 * pmf).sum() - theory.expected_committed(a, k) ** 2)
    assert abs(m.mean() - theory.expected_committed(a, k)) < 4 * sd / math.sqrt(B)


# ------------------------------------------------------------- greedy / tree

def test_argmax_first_index_rule():
    row = np.array([1.0, 3.0, -2.0, 3.0, 3.0])
    assert ov.argmax_first(row) == 1
    assert ov.row_argmax(row[None])[0] == 1
    rng = np.random.default_rng(2)
    rows = rng.integers(-3, 3, size=(200, 17)).astype(np.float64)   # many ties
    assert all(ov.argmax_first(r) == a for r, a in zip(rows, ov.row_argmax(rows)))


def test_greedy_hand_built():
    t = np.zeros((1, 4, 6), np.float32)
    t[0, 0, 2] = 5; t[0, 1, 4] = 5; t[0, 2, 1] = 5; t[0, 3, 3] = 5
    r = ov.verify_greedy(t, [[2, 4, 0]], "fp32")
    assert r.n_accepted[0] == 2 and list(r.out_tokens[0]) == [2, 4, 1, -1]
    r = ov.verify_greedy(t, [[2, 4, 1]], "fp32")
    assert r.n_accepted[0] == 3 and list(r.out_tokens[0]) == [2, 4, 1, 3]
    r = ov.verify_greedy(t, [[0, 4, 1]], "fp32")
    assert r.n_accepted[0] == 0 and list(r.out_tokens[0]) == [2, -1, -1, -1]
    t2 = np.zeros((1, 2, 6), np.float32)                      # all-equal row: id 0 wins
    r = ov.verify_greedy(t2, [[0]], "fp32")
    assert r.n_accepted[0] == 1 and list(r.out_tokens[0]) == [0, 0]


@pytest.mark.parametrize("a", [0.6, 0.8])
def test_greedy_phrase_drafts_match_closed_form(a):
    """Drafts equal to the target argmax w.p. a (k = 16): mean and law of the committed count."""
    k, rounds = 16, 150
    m = []
    for s in range(rounds):
        w = wl.c4(a, seed=1000 + s, V=257)
        r = ov.verify_greedy(w.target, w.tokens, w.dtype)
        assert np.array_equal(r.argmax, w.meta["argmax"])       # planted argmax found
        m.append(r.n_accepted + 1)
    m = np.concatenate(m)
    pmf = theory.committed_pmf(a, k)
    sd = math.sqrt((np.arange(k + 2) ** 2 * pmf).sum() - theory.expected_committed(a, k) ** 2)
    assert abs(m.mean() - theory.expected_committed(a, k)) < 4 * sd / math.sqrt(m.size)
    counts = np.bincount(m, minlength=k + 2)[1:]
    exp_ = m.size * pmf[1:]
    big = exp_ >= 5                                            # pool the sparse tail
    obs, ex = counts[big], exp_[big]
    if np.any(~big):
        obs, ex = np.append(obs, counts[~big].sum()), np.append(ex, exp_[~big].sum())
    assert stats.chisquare(obs, ex).pvalue > 1e-3


def test_tree_chain_equals_greedy():
    rng = np.random.default_rng(4)
    for s in range(20):
        k, V = 6, 40
        t = rng.integers(-3, 3, size=(3, k + 1, V)).astype(np.float32)
        a = ov.row_argmax(t.astype(np.float64))
        tokens = np.where(rng.random((3, k)) < 0.7, a[:, :k], rng.integers(0, V, (3, k))).astype(np.int32)
        g = ov.verify_greedy(t, tokens, "fp32")
        tr = ov.verify_tree(t, tokens, np.tile(np.arange(-1, k - 1), (3, 1)), "fp32")
        assert np.array_equal(g.out_tokens, tr.out_tokens[:, :k + 1])
        assert np.array_equal(g.n_accepted, tr.n_accepted)


def test_tree_hand_built():
    # context -> 0 -> 1 ; 0 -> 2 -> 3 ; context -> 4.  Row 0 = context, row 1+m = node m.
    parents = np.array([[-1, 0, 0, 2, -1]])
    V = 10
    t = np.zeros((1, 6, V), np.float32)
    win = {0: 7, 1: 3, 2: 5, 3: 9, 4: 1, 5: 2}                # argmax of row r
    for r, v in win.items():
        t[0, r, v] = 1.0
    # node 0 needs row 0's 7; nodes 1, 2 need row 1's 3; node 3 needs row 3's 9; node 4 needs 7
    tok = np.array([[7, 3, 3, 9, 7]])
    tr = ov.verify_tree(t, tok, parents, "fp32")
    assert tr.leaf[0] == 3 and tr.n_accepted[0] == 3
    assert list(tr.out_tokens[0]) == [7, 3, 9, 1, -1, -1]      # path 0, 2, 3 then row 4's argmax
    tok2 = np.array([[7, 3, 3, 4, 7]])                         # node 3 now rejected
    tr = ov.verify_tree(t, tok2, parents, "fp32")
    assert tr.leaf[0] == 1 and tr.n_accepted[0] == 2           # depth-2 tie: lowest index
    assert list(tr.out_tokens[0]) == [7, 3, 5, -1, -1, -1]
    tok3 = np.array([[0, 3, 3, 9, 0]])                         # nothing accepted
    tr = ov.verify_tree(t, tok3, parents, "fp32")
    assert tr.leaf[0] == -1 and tr.n_accepted[0] == 0 and list(tr.out_tokens[0][:2]) == [7, -1]
    tok4 = np.array([[1, 3, 3, 9, 7]])                         # only the root-level node 4
    tr = ov.verify_tree(t, tok4, parents, "fp32")
    assert tr.leaf[0] == 4 and list(tr.out_tokens[0][:3]) == [7, 2, -1]


def test_tree_c5_shape_extremes():
    par = wl.tree_shape()
    assert par.shape[0] == 26 and all(-1 <= par[m] < m for m in range(26))
    w = wl.c5(seed=3, V=300, p_match=1.0)
    tr = ov.verify_tree(w.target, w.tokens, w.parents, w.dtype)
    assert np.all(tr.n_accepted == 8) and np.all(tr.leaf == 7)   # first branch's leaf
    w = wl.c5(seed=3, V=300, p_match=0.0)
    tr = ov.verify_tree(w.target, w.tokens, w.parents, w.dtype)
    assert np.all(tr.n_accepted == 0) and np.all(tr.out_tokens[:, 0] == w.meta["argmax"][:, 0])
