"""The bounded bulk-copy waits give up and report SPEC_ERR_TIMEOUT (GPU, through the C ABI).

A copy that never lands cannot be produced on purpose without faulting the
GPU, so the test hook spec_test_force_stage_timeouts makes every stage wait
give up at once, exactly where a wait whose 1 s limit ran out would.  The
waits that keep a CTA from leaving while its own copies are still landing in
shared memory keep their normal limit.  Checked for the two kernels that stage
rows by bulk copies -- the ring row pass of large greedy batches and the
sampling pass of stochastic calls:

  * the call returns promptly (nothing waits out a limit);
  * every sequence whose rows or draw went through a forced wait reports
    SPEC_ERR_TIMEOUT, with n_accepted = -1 and an all -1 token row;
  * the next call on the same workspace, with normal waits, matches the
    oracle: the timed-out call left every completion counter at zero.
"""
import time

import numpy as np
import pytest
import torch

import workloads as wl
from oracle import verify as ov
from tests.gpu_parity import compare_stochastic, to_device, tokens_to_device

pytestmark = pytest.mark.gpu

SPEC_ERR_TIMEOUT = -6


@pytest.fixture(scope="module")
def sv():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    import speculative_decoding_draft_online_gb300 as sv
    return sv


def _forced(sv, fn):
    """Run fn() with every stage wait forced to give up; returns (result, seconds)."""
    torch.cuda.synchronize()
    prev = sv.force_stage_timeouts(True)
    try:
        t0 = time.perf_counter()
        out = fn()
        torch.cuda.synchronize()
        return out, time.perf_counter() - t0
    finally:
        sv.force_stage_timeouts(prev)


def test_ring_row_pass_times_out_and_recovers(sv):
    """Greedy on the headline tensors (148 MB of 16-byte aligned rows: the ring row pass)."""
    w = wl.c3()
    t, x = to_device(w.target, w.dtype), tokens_to_device(w.tokens)
    ws = sv.workspace(w.B, w.k, w.V, sv.SPEC_BF16, "cuda")
    sv.verify(t, None, x, 0.0, ws=ws)                  # warm: the library's one-off set-up is done
    (out, n, ex), secs = _forced(sv, lambda: sv.verify_ex(t, None, x, 0.0, 0, ws=ws, aux=True))
    assert secs < 0.5, secs
    st = ex["status"].cpu().numpy()
    assert np.all(st == SPEC_ERR_TIMEOUT), st
    assert torch.all(n == -1) and torch.all(out == -1)
    out, n = sv.verify(t, None, x, 0.0, ws=ws)         # normal waits, same workspace
    torch.cuda.synchronize()
    ref = ov.verify_greedy(w.target, w.tokens, w.dtype)
    np.testing.assert_array_equal(out.cpu().numpy(), ref.out_tokens)
    np.testing.assert_array_equal(n.cpu().numpy(), ref.n_accepted)


@pytest.mark.parametrize("top_p", [0.0, 0.8])
def test_sampling_pass_times_out_and_recovers(sv, top_p):
    """Stochastic C2 (aligned bf16 rows: the sampling pass stages its tiles by
    bulk copies), with and without consistent top-p."""
    w = wl.c2(seed=610)
    t, d, x = to_device(w.target, w.dtype), to_device(w.draft, w.dtype), tokens_to_device(w.tokens)
    ws = sv.workspace(w.B, w.k, w.V, sv.SPEC_BF16, "cuda")
    sv.verify_ex(t, d, x, w.temperature, w.seed, ws=ws, top_p=top_p)
    (out, n, aux), secs = _forced(sv, lambda: sv.verify_ex(t, d, x, w.temperature, w.seed, ws=ws, aux=True,
                                                          top_p=top_p))
    assert secs < 0.5, secs
    st = aux["status"].cpu().numpy()
    assert np.all(st == SPEC_ERR_TIMEOUT), st
    assert torch.all(n == -1) and torch.all(out == -1)
    # the accept scan ran before the draws: p_i(x_i) is still reported
    assert np.all(np.isfinite(aux["p_draft"].cpu().numpy()))
    out, n, aux = sv.verify_ex(t, d, x, w.temperature, w.seed, ws=ws, aux=True, top_p=top_p)
    torch.cuda.synchronize()
    if top_p:
        from oracle import extensions as ox
        ref = ox.verify_filtered(w.target, w.draft, w.tokens, w.dtype, w.temperature, w.seed, 0, top_p)
    else:
        ref = ov.verify_stochastic(w.target, w.draft, w.tokens, w.dtype, w.temperature, w.seed)
    compare_stochastic(ref, out.cpu().numpy(), n.cpu().numpy(), aux["status"].cpu().numpy(), w.k)


def test_hook_is_off_by_default_and_restores(sv):
    assert sv.force_stage_timeouts(False) is False     # nothing had switched it on
    assert sv.force_stage_timeouts(True) is False
    assert sv.force_stage_timeouts(False) is True
