"""Batched speculative-decoding verification for GB300 (sm_103a).

The hot path -- row statistics, accept scan, residual / bonus sampling, greedy
match (with #Match and the target-guided variant), stop truncation and tree
verification -- runs in the CUDA kernels of libspecverify.so
behind the C ABI declared in include/spec_verify.h.  This package is the thin
Python binding of that library (torch supplies device memory and streams).
"""
from ._lib import (SPEC_BF16, SPEC_ERR_NONFINITE, SPEC_ERR_TOKEN, SPEC_FP32, LIB_PATH, SpecError, lib,  # noqa: F401
                   force_stage_timeouts, probe_read, random_stream, verify, verify_ex, verify_guided, verify_tree, workspace,
                   workspace_size)

__all__ = ["verify", "verify_ex", "verify_tree", "verify_guided", "workspace", "workspace_size", "random_stream",
           "SpecError", "SPEC_BF16", "SPEC_FP32", "LIB_PATH"]
