"""Pins for the two oracle quantities that decide which GPU/oracle differences
the parity tests excuse (CPU only).

  * the Gumbel-max gap of a draw (top-1 minus top-2 score over the draw's
    support, fp64), recorded by the oracle's draw in ``oracle/verify.py``;
  * the top-p margin of a filtered row (distance of the top-p target from the
    cumulative masses on either side of the chosen value, relative to the mass
    the filter sees), returned by ``oracle/extensions.filter_row``.

Both are fixed here by arithmetic on hand-built rows (scores and masses chosen
so the answer is known without the oracle) and by a perturbation property
(moving the decision's input by just under the margin keeps the decision, just
over it changes it).  The mutation tests at the end plant plausible slips in a
copy of each oracle function -- the gap over fp32-rounded scores, over the
noise alone, against the third score; the top-p margin one-sided, absolute
instead of relative, or taken one value group too late -- and check that a pin
fails on every one of them.
"""
import inspect
import textwrap

import numpy as np
import pytest

from oracle import extensions as ox
from oracle import philox
from oracle import verify as ov


# ------------------------------------------------------------ Gumbel gap ---

def _draw_with(draw_factory, seed, b, j, logw, kind="residual"):
    trace = ov.SequenceTrace()
    y = draw_factory(seed, b, trace)(j, np.asarray(logw, dtype=np.float64), kind)
    return y, trace.draw_gap


def _rows_for_scores(seed, b, j, scores):
    """Log weights whose draw scores (log weight + the draw's own Gumbel noise)
    are exactly `scores` up to fp64 rounding (-inf stays outside the support)."""
    scores = np.asarray(scores, dtype=np.float64)
    g = philox.gumbel(philox.gumbel_uniforms(seed, b, j, scores.shape[0]))
    return np.where(np.isfinite(scores), scores - g, -np.inf)


def check_gap_pins(draw_factory):
    """Assert the pins of the draw gap for one draw implementation."""
    seed, b, j = 4321, 3, 2
    # two candidates a quarter apart: gap 0.25, the higher score wins
    y, gap = _draw_with(draw_factory, seed, b, j, _rows_for_scores(seed, b, j, [2.0, 1.75]))
    assert y == 0 and abs(gap - 0.25) < 1e-12, (y, gap)
    # a gap below fp32 resolution at this magnitude (ulp(3) = 2.4e-7): the
    # recorded gap is the fp64 difference, not that of the rounded scores
    y, gap = _draw_with(draw_factory, seed, b, j, _rows_for_scores(seed, b, j, [3.0, 3.0 + 3e-7, 1.0]))
    assert y == 1 and abs(gap - 3e-7) < 1e-12, (y, gap)
    # three candidates and ids outside the support (whatever their noise): gap = top-1 - top-2
    scores = [1.0, -np.inf, 0.5, 0.9, -np.inf, -np.inf]
    y, gap = _draw_with(draw_factory, seed, b, j, _rows_for_scores(seed, b, j, scores))
    assert y == 0 and abs(gap - 0.1) < 1e-12, (y, gap)
    # one candidate: nothing can overtake it
    y, gap = _draw_with(draw_factory, seed, b, j, _rows_for_scores(seed, b, j, [-np.inf, 0.3, -np.inf]))
    assert y == 1 and gap == np.inf
    # an empty residual's fallback draw always counts as a margin position
    _, gap = _draw_with(draw_factory, seed, b, j, np.zeros(5), kind="empty-residual")
    assert gap == 0.0
    # perturbation: lowering the winner by just under the gap keeps it, by just over hands the draw on
    rng = np.random.default_rng(9)
    checked = 0
    for trial in range(200):
        V = int(rng.integers(2, 40))
        logw = rng.normal(0, 2, size=V)
        logw[rng.random(V) < 0.3] = -np.inf
        if np.isfinite(logw).sum() < 2:
            continue
        y, gap = _draw_with(draw_factory, seed, trial, 0, logw)
        if not (1e-3 < gap < np.inf):
            continue
        scores = logw + philox.gumbel(philox.gumbel_uniforms(seed, trial, 0, V))
        runner = int(np.argmax(np.where(np.arange(V) == y, -np.inf, scores)))
        lo = logw.copy()
        lo[y] -= 0.99 * gap
        assert _draw_with(draw_factory, seed, trial, 0, lo)[0] == y
        lo[y] = logw[y] - 1.01 * gap
        assert _draw_with(draw_factory, seed, trial, 0, lo)[0] == runner
        checked += 1
    assert checked > 50


def test_gumbel_gap_pins():
    check_gap_pins(ov._gumbel_draw)


def test_gumbel_gap_reaches_the_margins_of_a_verification():
    """The gap a draw records becomes the margin of the drawn position."""
    seed, b = 55, 0
    k, V = 1, 4
    # p = 0 on the draft token: a certain rejection, residual = p on ids 1..3
    with np.errstate(divide="ignore"):
        t = np.log(np.array([[0.0, 0.2, 0.3, 0.5], [0.25, 0.25, 0.25, 0.25]]))
        d = np.log(np.array([[1.0, 0.0, 0.0, 0.0]]))
        r = ov.verify_stochastic(t[None].astype(np.float32), d[None].astype(np.float32),
                                 np.zeros((1, 1), np.int32), "fp32", 1.0, seed)
    logp, _ = ov.log_softmax(ov.decode_logits(t[None].astype(np.float32), "fp32")[0, 0], 1.0)
    s = logp + philox.gumbel(philox.gumbel_uniforms(seed, b, 0, V))
    top = np.sort(s[1:])[::-1]
    assert r.n_accepted[0] == 0
    # the position's margin is the smaller of its accept margin |u - p/q| = u and the gap
    u = philox.accept_uniform(seed, b, 0)
    assert abs(r.margins[0][0] - min(u, top[0] - top[1])) < 1e-9


# -------------------------------------------------------- top-p margin ---

def check_top_p_pins(filter_row):
    """Assert the pins of the top-p margin for one filter implementation."""
    def margin(w, top_p, top_k=0, T=1.0):
        return filter_row(T * np.log(np.asarray(w, dtype=np.float64)), T, top_k, top_p).margin

    # masses 0.5 | 0.3 | 0.2, target 0.75: reached inside the second value's
    # group, 0.05 short of its upper end and 0.25 past its lower end
    assert abs(margin([0.5, 0.3, 0.2], 0.75) - 0.05) < 1e-12
    assert abs(margin([0.2, 0.5, 0.3], 0.75, T=0.4) - 0.05) < 1e-12          # order and T do not matter
    # ties form one group: 0.4 | 0.6 (three equal ids); target 0.5 -> min(1.0 - 0.5, 0.5 - 0.4)
    assert abs(margin([0.2, 0.4, 0.2, 0.2], 0.5) - 0.1) < 1e-12
    # top-k 3 first: kept mass 0.9; target 0.5 * 0.9 = 0.45 lies 0.05 above 0.4 -> 0.05 / 0.9
    assert abs(margin([0.4, 0.3, 0.2, 0.1], 0.5, top_k=3) - 0.05 / 0.9) < 1e-12
    # the target on the first group: 0.6 of mass, top_p 0.55 -> 0.05 (a group
    # with no mass above it has no lower end: no top_p > 0 falls below 0)
    assert abs(margin([0.6, 0.25, 0.15], 0.55) - 0.05) < 1e-12
    assert abs(margin([0.6, 0.25, 0.15], 0.02) - 0.58) < 1e-12
    # no top-p decision taken: infinite margin
    assert margin([0.5, 0.5], 0.0) == np.inf and margin([0.5, 0.5], 1.0) == np.inf
    # perturbation: top_p moved by just under the margin keeps the threshold;
    # moved by just over it, towards the nearer boundary, changes it
    rng = np.random.default_rng(17)
    checked = 0
    for _ in range(300):
        V = int(rng.integers(3, 12))
        x = rng.integers(-4, 4, size=V).astype(np.float64) * 0.7
        T = float(rng.choice([0.5, 1.0, 2.0]))
        top_p = float(rng.uniform(0.05, 0.95))
        f = filter_row(x, T, 0, top_p)
        if not (1e-4 < f.margin < np.inf):
            continue
        for s in (-1, 1):
            p2 = top_p + s * 0.99 * f.margin
            if 0 < p2 < 1:
                assert filter_row(x, T, 0, p2).tau == f.tau
        moved = [filter_row(x, T, 0, top_p + s * 1.01 * f.margin).tau for s in (-1, 1)
                 if 0 < top_p + s * 1.01 * f.margin < 1]
        if not moved:
            continue                      # the nearer end lies beyond any valid top_p
        assert any(tau != f.tau for tau in moved), (x, T, top_p, f.margin)
        checked += 1
    assert checked > 50


def test_top_p_margin_pins():
    check_top_p_pins(ox.filter_row)


# ------------------------------------------------ planted slips (mutants) ---

def _mutant(module, name, old, new):
    """A copy of module.<name> compiled from its source with `old` replaced by `new`."""
    src = textwrap.dedent(inspect.getsource(getattr(module, name)))
    assert old in src, f"mutation target not found in {name}: {old!r}"
    ns = dict(vars(module))
    exec(compile(src.replace(old, new, 1), f"<mutant of {name}>", "exec"), ns)
    return ns[name]


GAP_SLIPS = [
    # the gap of the fp32-rounded scores instead of the fp64 ones
    ("finite = np.sort(score[np.isfinite(score)])", "finite = np.sort(s32[np.isfinite(s32)]).astype(np.float64)"),
    # the gap of the noise alone
    ("finite = np.sort(score[np.isfinite(score)])", "finite = np.sort(g[np.isfinite(score)])"),
    # top-1 minus top-3
    ("finite[-1] - finite[-2]", "finite[-1] - finite[0]"),
    # every id's score, support or not (out-of-support ids scored as if their weight were 1)
    ("finite = np.sort(score[np.isfinite(score)])",
     "finite = np.sort(np.where(np.isfinite(score), score, g))"),
]


@pytest.mark.parametrize("old,new", GAP_SLIPS)
def test_gap_pins_fail_on_planted_slips(old, new):
    with pytest.raises(AssertionError):
        check_gap_pins(_mutant(ov, "_gumbel_draw", old, new))


TOP_P_SLIPS = [
    # one-sided: only the distance to the group's upper end
    ("min(upper, target - cum) if cum > 0 else upper", "upper"),
    # one-sided: only the distance to its lower end
    ("upper = cum + grp - target", "upper = np.inf"),
    # the first group treated like the others (a lower end at mass 0)
    ("min(upper, target - cum) if cum > 0 else upper", "min(upper, target - cum)"),
    # absolute mass instead of the fraction of the filter's mass
    ("if cum > 0 else upper) / mk", "if cum > 0 else upper)"),
    # the walk stops one value group late
    ("if cum + grp >= target:", "if cum >= target:"),
    # the group's own mass left out of the upper distance
    ("upper = cum + grp - target", "upper = cum - target"),
]


@pytest.mark.parametrize("old,new", TOP_P_SLIPS)
def test_top_p_pins_fail_on_planted_slips(old, new):
    with pytest.raises(AssertionError):
        check_top_p_pins(_mutant(ox, "filter_row", old, new))
