"""Helpers for the GPU-vs-oracle parity tests (CUDA path through the C ABI).

Tolerances (stated by the specification of this path):
  * greedy and tree outputs, token ids and accept counts: bit-exact;
  * stochastic decisions and sampled ids: equal on every sequence, except where
    the first difference sits at a committed position whose decision margin
    (|u - min(1, p/q)| of an accept decision, or the Gumbel top-1 / top-2 gap
    of a draw, both from the oracle in fp64) is below 1e-5; such positions are
    counted, and must stay under 0.01 % of the verified positions;
  * p_i(x_i) and q_i(x_i): within 1e-5 absolute.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

MARGIN = 1e-5
PROB_ATOL = 1e-5


def to_device(arr: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(arr, dtype=np.float32)).to(device)


def tokens_to_device(arr: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(arr, dtype=np.int32)).to(device)


@dataclass
class Tally:
    rows: int = 0           # verified positions compared
    margin_rows: int = 0    # first differences excused by a margin below 1e-5
    sequences: int = 0

    def add(self, other: "Tally"):
        self.rows += other.rows
        self.margin_rows += other.margin_rows
        self.sequences += other.sequences


# every comparison of the session, printed in pytest's terminal summary
SESSION = Tally()


def compare_stochastic(ref, out: np.ndarray, n: np.ndarray, status: np.ndarray, k: int) -> Tally:
    """Sequence-by-sequence comparison with the margin rule; raises on a real mismatch.

    The returned tally is also added to SESSION."""
    tally = _compare(ref, out, n, status, k)
    SESSION.add(tally)
    return tally


def _compare(ref, out: np.ndarray, n: np.ndarray, status: np.ndarray, k: int) -> Tally:
    tally = Tally()
    B = out.shape[0]
    for b in range(B):
        tally.sequences += 1
        assert status[b] == ref.status[b], f"seq {b}: status {status[b]} vs oracle {ref.status[b]}"
        if ref.status[b] != 0:
            assert n[b] == -1 and np.all(out[b] == -1), f"seq {b}: error sequence must be all -1"
            continue
        tally.rows += k + 1
        if n[b] == ref.n_accepted[b] and np.array_equal(out[b], ref.out_tokens[b]):
            continue
        # first committed position where the two runs part
        j = 0
        nr, ng = ref.n_accepted[b], n[b]
        while j <= min(nr, ng) and out[b, j] == ref.out_tokens[b, j] and (j < nr) == (j < ng):
            j += 1
        j = min(j, nr)
        margin = ref.margins[b][j]
        assert margin < MARGIN, (f"seq {b}: GPU {out[b].tolist()} n={ng} vs oracle "
                                 f"{ref.out_tokens[b].tolist()} n={nr}; first difference at {j} "
                                 f"with margin {margin:.3g}")
        tally.margin_rows += 1
    return tally


def compare_probs(ref, aux: dict, k: int):
    ok = ref.status == 0
    p = aux["p_draft"].cpu().numpy().astype(np.float64)
    q = aux["q_draft"].cpu().numpy().astype(np.float64)
    if ok.any():
        dp = np.max(np.abs(p[ok] - ref.p_draft[ok]))
        dq = np.max(np.abs(q[ok] - ref.q_draft[ok]))
        assert dp < PROB_ATOL and dq < PROB_ATOL, (dp, dq)
        lse = aux["lse"].cpu().numpy().astype(np.float64)
        ref_lse = np.concatenate([ref.lse_target[:, :k], ref.lse_draft], axis=1)
        err = np.abs(lse[ok] - ref_lse[ok]) / np.maximum(1.0, np.abs(ref_lse[ok]))
        assert np.max(err) < 2e-6, np.max(err)
