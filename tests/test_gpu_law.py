"""The CUDA path's committed tokens follow the target's law (losslessness).

The rule's claim ("Speculative Decoding: Faster Generation Without Changing
the Model", "The acceptance rule"; the cascade page's review step) is that
verification changes nothing in the law of the output: position j, once
reached, commits a token distributed as target row j.  With context-free rows
(every sequence has the same target and draft rows, drafts drawn from the
draft rows) the committed token at position j, among the sequences whose
output reaches j, must follow p_j, and the number of accepted drafts must
follow the exact law that enumerating the rule gives.  Both are checked by
chi-squared over 200000 sequences verified in one call through the C ABI,
each drawing its own counter-based randomness.
"""
import numpy as np
import pytest
import torch
from scipy import stats

import workloads as wl
from oracle import enumerate as oe
from tests.gpu_parity import to_device, tokens_to_device

pytestmark = pytest.mark.gpu

K, V, B = 3, 8, 200_000
P_MIN = 1e-3


@pytest.fixture(scope="module")
def sv():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    import speculative_decoding_draft_online_gb300 as sv
    return sv


def log_softmax64(x):
    z = x - x.max(axis=-1, keepdims=True)
    return z - np.log(np.exp(z).sum(axis=-1, keepdims=True))


def chi2(counts, expected):
    """Chi-squared p-value, with bins expected under 5 pooled into one."""
    counts = np.asarray(counts, dtype=np.float64)
    expected = np.asarray(expected, dtype=np.float64)
    small = expected < 5
    c = np.append(counts[~small], counts[small].sum())
    e = np.append(expected[~small], expected[small].sum())
    keep = e > 0
    c, e = c[keep], e[keep]
    return stats.chisquare(c, e * c.sum() / e.sum()).pvalue


def verify_context_free(sv):
    """Verify B sequences that share their rows; drafts drawn from the draft rows."""
    t64, d64 = wl.tiny_rows(k=K, V=V, seed=7)
    t32, d32 = t64.astype(np.float32), d64.astype(np.float32)
    logp = log_softmax64(t32.astype(np.float64))
    logq = log_softmax64(d32.astype(np.float64))
    rng = np.random.default_rng(2024)
    cdf = np.cumsum(np.exp(logq), axis=1)
    u = rng.random((B, K))
    x = np.stack([np.minimum(np.searchsorted(cdf[i], u[:, i] * cdf[i, -1], side="right"), V - 1)
                  for i in range(K)], axis=1).astype(np.int32)
    target = np.ascontiguousarray(np.broadcast_to(t32, (B, K + 1, V)))
    draft = np.ascontiguousarray(np.broadcast_to(d32, (B, K, V)))
    out, n = sv.verify(to_device(target, wl.FP32), to_device(draft, wl.FP32), tokens_to_device(x), 1.0, 4321)
    torch.cuda.synchronize()
    return logp, logq, out.cpu().numpy(), n.cpu().numpy()


@pytest.fixture(scope="module")
def run(sv):
    return verify_context_free(sv)


def test_accept_count_follows_the_enumerated_law(run):
    logp, logq, out, n = run
    law = oe.full_law(logp, logq)
    pn = np.zeros(K + 1)
    for tup, pr in law.items():
        pn[len(tup) - 1] += pr
    assert abs(pn.sum() - 1.0) < 1e-12
    counts = np.bincount(n, minlength=K + 1)
    assert counts.sum() == B and np.all(n >= 0)
    assert chi2(counts, B * pn) > P_MIN


@pytest.mark.parametrize("j", range(K + 1))
def test_committed_token_follows_target_row(run, j):
    logp, _, out, n = run
    reached = n >= j
    tok = out[reached, j]
    assert np.all((tok >= 0) & (tok < V))
    counts = np.bincount(tok, minlength=V)
    assert chi2(counts, reached.sum() * np.exp(logp[j])) > P_MIN
    # positions past the committed ones are -1
    assert np.all(out[~reached, j] == -1)
