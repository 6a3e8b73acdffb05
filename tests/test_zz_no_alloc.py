"""spec_verify_noalloc: verification without any device allocation by the caller.

Some callers cannot allocate device memory -- a plugin inside a program that
owns all of the GPU's memory, or a path where cudaMalloc's device-wide
synchronisation is not allowed -- so they cannot hand spec_verify a workspace.
spec_verify_noalloc keeps the kernels' scratch in a fixed array inside the
library instead.  These tests call it through the C ABI and check that it
returns what spec_verify returns, on consecutive calls with different sizes
and modes (the shared scratch keeps the previous call's contents), and that
sizes beyond the array are refused before any launch.

This file is collected last so that a failure here leaves every other test run.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as wl
from tests.gpu_parity import to_device, tokens_to_device

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


def _noalloc(lib, t, d, x, T, seed, dtype_code):
    B, k1, V = t.shape
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


def test_noalloc_refuses_sizes_beyond_its_scratch(abi):
    sv, lib = abi
    B, k, V = 4096, 8, 128256
    assert sv.workspace_size(B, k, V) > 8 << 20
    dummy = ctypes.c_void_p(0x1000)                   # never touched: the call returns before any launch
    rc = lib.spec_verify_noalloc(dummy, dummy, dummy, B, k, V, sv.SPEC_BF16, 1.0, ctypes.c_uint64(0), dummy, dummy,
                                 None)
    assert rc == SPEC_ERR_WORKSPACE
