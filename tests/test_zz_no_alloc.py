"""spec_verify_noalloc: verification without any device allocation by the caller.

Some callers cannot allocate device memory -- a plugin inside a program that
owns all of the GPU's memory, or a path where cudaMalloc's device-wide
synchronisation is not allowed -- so they cannot hand spec_verify a workspace.
spec_verify_noalloc keeps the kernels' scratch in a fixed array inside the
library instead.  These tests call it through the C ABI and check that it
returns what spec_verify returns, on consecutive calls with different sizes
and modes (one shared scratch serves them all), inside and
around captured CUDA graphs, that it agrees with the CPU oracle on its own, and
that sizes beyond the array are refused before any launch.

This file is collected last so that a failure here leaves every other test run.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as wl
from oracle import verify as ov
from tests.gpu_parity import compare_stochastic, to_device, tokens_to_device

pytestmark = pytest.mark.gpu

SPEC_ERR_WORKSPACE = -8


@pytest.fixture(scope="module")
def abi():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    import speculative_decoding_draft_online_gb300 as sv
    lib = ctypes.CDLL(sv.LIB_PATH)                  # the C ABI itself, not the Python wrapper
    vp = ctypes.c_void_p
    lib.spec_verify_noalloc.argtypes = [vp, vp, vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_float, ctypes.c_uint64, vp, vp, vp]
    lib.spec_verify_noalloc.restype = ctypes.c_int
    return sv, lib


def _noalloc(lib, t, d, x, T, seed, dtype_code, out=None, n=None):
    B, k1, V = t.shape
    if out is None:
        out = torch.full((B, k1), -7, dtype=torch.int32, device="cuda")
        n = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    rc = lib.spec_verify_noalloc(ctypes.c_void_p(t.data_ptr()), ctypes.c_void_p(d.data_ptr()) if d is not None else None,
                                 ctypes.c_void_p(x.data_ptr()), B, k1 - 1, V, dtype_code, float(T),
                                 ctypes.c_uint64(seed), ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(n.data_ptr()),
                                 ctypes.c_void_p(stream))
    assert rc == 0, rc
    return out, n


def test_noalloc_matches_spec_verify_on_consecutive_calls(abi):
    sv, lib = abi
    s_w = wl.c2(seed=77)                              # stochastic, B=32 k=5 V=32000 bf16
    g_w = wl.c4(0.7, seed=78)                         # greedy, B=16 k=16 V=64000 bf16
    s_t, s_d, s_x = to_device(s_w.target, s_w.dtype), to_device(s_w.draft, s_w.dtype), tokens_to_device(s_w.tokens)
    g_t, g_x = to_device(g_w.target, g_w.dtype), tokens_to_device(g_w.tokens)
    calls = [(s_t, s_d, s_x, 1.0, 11), (g_t, None, g_x, 0.0, 0), (s_t, s_d, s_x, 1.0, 12), (s_t, s_d, s_x, 1.0, 12)]
    for t, d, x, T, seed in calls:
        out, n = _noalloc(lib, t, d, x, T, seed, sv.SPEC_BF16)
        ref_out, ref_n = sv.verify(t, d, x, T, seed)      # the existing entry point, caller workspace
        torch.cuda.synchronize()
        # identical kernels on identical inputs: the tolerance is equality for greedy and stochastic alike
        np.testing.assert_array_equal(out.cpu().numpy(), ref_out.cpu().numpy())
        np.testing.assert_array_equal(n.cpu().numpy(), ref_n.cpu().numpy())


def test_noalloc_agrees_with_the_oracle(abi):
    """On its own: greedy bit-exact, stochastic under the margin rule of the parity tests."""
    sv, lib = abi
    s_w = wl.c2(seed=79)
    g_w = wl.c4(0.8, seed=80)
    out, n = _noalloc(lib, to_device(s_w.target, s_w.dtype), to_device(s_w.draft, s_w.dtype),
                      tokens_to_device(s_w.tokens), s_w.temperature, s_w.seed, sv.SPEC_BF16)
    torch.cuda.synchronize()
    ref = ov.verify_stochastic(s_w.target, s_w.draft, s_w.tokens, s_w.dtype, s_w.temperature, s_w.seed)
    compare_stochastic(ref, out.cpu().numpy(), n.cpu().numpy(), np.zeros(s_w.B, np.int32), s_w.k)
    out, n = _noalloc(lib, to_device(g_w.target, g_w.dtype), None, tokens_to_device(g_w.tokens), 0.0, 0,
                      sv.SPEC_BF16)
    torch.cuda.synchronize()
    gref = ov.verify_greedy(g_w.target, g_w.tokens, g_w.dtype)
    np.testing.assert_array_equal(out.cpu().numpy(), gref.out_tokens)
    np.testing.assert_array_equal(n.cpu().numpy(), gref.n_accepted)


def test_noalloc_in_and_around_captured_graphs(abi):
    """Eager calls at one size, a graph captured at another, eager calls at the
    graph's size and replays, interleaved on one stream: every result equals
    spec_verify's on the same inputs (every execution leaves the scratch
    zeroed, whatever its sizes)."""
    sv, lib = abi
    a = wl.c2(seed=81)                                # B=32 k=5 V=32000, stochastic
    g = wl.c4(0.8, seed=82)                           # B=16 k=16 V=64000, greedy
    a_t, a_d, a_x = to_device(a.target, a.dtype), to_device(a.draft, a.dtype), tokens_to_device(a.tokens)
    g_t, g_x = to_device(g.target, g.dtype), tokens_to_device(g.tokens)
    a_ref = [r.cpu().numpy() for r in sv.verify(a_t, a_d, a_x, a.temperature, 5)]
    g_ref = [r.cpu().numpy() for r in sv.verify(g_t, None, g_x, 0.0, 0)]
    g_out = torch.full((g.B, g.k + 1), -7, dtype=torch.int32, device="cuda")
    g_n = torch.full((g.B,), -7, dtype=torch.int32, device="cuda")

    def check_a():
        out, n = _noalloc(lib, a_t, a_d, a_x, a.temperature, 5, sv.SPEC_BF16)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(out.cpu().numpy(), a_ref[0])
        np.testing.assert_array_equal(n.cpu().numpy(), a_ref[1])

    def check_g():
        torch.cuda.synchronize()
        np.testing.assert_array_equal(g_out.cpu().numpy(), g_ref[0])
        np.testing.assert_array_equal(g_n.cpu().numpy(), g_ref[1])
        g_out.fill_(-7)
        g_n.fill_(-7)

    check_a()                                         # eager at the first size
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        _noalloc(lib, g_t, None, g_x, 0.0, 0, sv.SPEC_BF16, g_out, g_n)
    torch.cuda.synchronize()
    _noalloc(lib, g_t, None, g_x, 0.0, 0, sv.SPEC_BF16, g_out, g_n)   # eager at the graph's size
    check_g()
    graph.replay()                                    # replay after an eager call at the same size
    check_g()
    check_a()                                         # eager at the first size, then a replay
    graph.replay()
    check_g()
    graph.replay()                                    # two replays in a row
    check_g()
    check_a()


def test_noalloc_refuses_sizes_beyond_its_scratch(abi):
    sv, lib = abi
    B, k, V = 4096, 8, 128256
    assert sv.workspace_size(B, k, V) > 8 << 20
    dummy = ctypes.c_void_p(0x1000)                   # never touched: the call returns before any launch
    rc = lib.spec_verify_noalloc(dummy, dummy, dummy, B, k, V, sv.SPEC_BF16, 1.0, ctypes.c_uint64(0), dummy, dummy,
                                 None)
    assert rc == SPEC_ERR_WORKSPACE


def test_noalloc_limit_at_the_headline_shape(abi):
    """The largest batch whose workspace fits the built-in scratch runs; one more is refused."""
    sv, lib = abi
    k, V = 8, 128256
    limit = 8 << 20
    B = 1
    while sv.workspace_size(B + 1, k, V) <= limit:
        B += 1
    assert sv.workspace_size(B, k, V) <= limit < sv.workspace_size(B + 1, k, V)
    dummy = ctypes.c_void_p(0x1000)
    rc = lib.spec_verify_noalloc(dummy, dummy, dummy, B + 1, k, V, sv.SPEC_BF16, 1.0, ctypes.c_uint64(0), dummy,
                                 dummy, None)
    assert rc == SPEC_ERR_WORKSPACE
    # B sequences of random rows (4 GB of logits): the call runs and agrees with spec_verify
    gen = torch.Generator(device="cuda").manual_seed(3)
    t = torch.randn((B, k + 1, V), device="cuda", generator=gen).mul_(4).to(torch.bfloat16)
    d = (t[:, :k].float() + torch.randn((B, k, V), device="cuda", generator=gen)).to(torch.bfloat16)
    x = torch.randint(0, V, (B, k), device="cuda", dtype=torch.int32, generator=gen)
    out, n = _noalloc(lib, t, d, x, 0.7, 9, sv.SPEC_BF16)
    ref_out, ref_n = sv.verify(t, d, x, 0.7, 9)
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out) and torch.equal(n, ref_n)
    del t, d
    torch.cuda.empty_cache()
