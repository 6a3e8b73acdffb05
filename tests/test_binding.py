"""The Python binding refuses misuse before anything reaches the library.

No GPU is needed: every case here fails in argument marshalling, so nothing
is launched.  CPU tensors, wrong shapes and wrong dtypes raise clear errors;
there is no CPU path to fall back on.
"""
import os

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LIB = os.path.join(ROOT, "speculative_decoding_draft_online_gb300", "libspecverify.so")


@pytest.fixture(scope="module")
def sv():
    if not os.path.exists(LIB):
        import __graft_entry__
        __graft_entry__.build()
    import speculative_decoding_draft_online_gb300 as sv
    return sv


def test_cpu_tensors_are_refused(sv):
    B, k, V = 2, 3, 64
    t = torch.zeros((B, k + 1, V), dtype=torch.bfloat16)
    d = torch.zeros((B, k, V), dtype=torch.bfloat16)
    x = torch.zeros((B, k), dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA"):
        sv.verify(t, d, x, 1.0, 0)
    with pytest.raises(ValueError, match="CUDA"):
        sv.verify(t, None, x, 0.0, 0)


def test_logit_dtype_must_be_bf16_or_fp32(sv):
    from speculative_decoding_draft_online_gb300 import _lib
    with pytest.raises(TypeError):
        _lib.dtype_code(torch.zeros(4, dtype=torch.float16))
    assert _lib.dtype_code(torch.zeros(4, dtype=torch.bfloat16)) == sv.SPEC_BF16
    assert _lib.dtype_code(torch.zeros(4, dtype=torch.float32)) == sv.SPEC_FP32


def test_workspace_size_rejects_invalid_sizes(sv):
    assert sv.workspace_size(0, 4, 32000) == 0
    assert sv.workspace_size(4, 0, 32000) == 0
    assert sv.workspace_size(4, 4, 0) == 0
    assert sv.workspace_size(4, 4, 32000) > 0
    with pytest.raises(ValueError):
        sv.workspace(0, 4, 32000, sv.SPEC_BF16, "cpu")


def test_bench_command_line_parses():
    """bench.py's argument parsing runs on a host without a GPU (every option the driver passes)."""
    import subprocess
    import sys as _sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([_sys.executable, os.path.join(root, "bench.py"), "--help"], capture_output=True, text=True,
                         timeout=120)
    assert out.returncode == 0, out.stderr
    for opt in ("--gpus", "--steps", "--warmup", "--impl", "--workload", "--no-per-config"):
        assert opt in out.stdout
