"""Seeded synthetic inputs for batched speculative-decoding verification.

This module only *builds inputs*: target logits, draft logits, draft tokens and
candidate trees with the shapes, dtypes and value distributions of the five
workloads below.  It holds none of the verification arithmetic (no acceptance
rule, no residual, no log-sum-exp of the method); both the CUDA path's tests and
the oracle read the same arrays it returns.

Where a recipe needs "a token sampled from the draft softmax", it is drawn here
by inverse-CDF sampling with numpy's own generator, which is independent of the
counter-based randomness that the verification rule itself consumes.

Storage conventions (what the C ABI takes):
  * bf16 logits are carried as ``np.uint16`` bit patterns (round-to-nearest-even
    from fp32); fp32 logits as ``np.float32``.
  * target ``[B][k+1][V]``, draft ``[B][k][V]``, tokens ``[B][k]`` int32.
  * trees: target ``[B][N+1][V]`` (row 0 = context, row 1+m = output at node m),
    ``node_tokens [B][N]``, ``parents [B][N]`` (-1 = child of the context,
    otherwise ``parents[m] < m``).

Workloads (vocabulary sizes follow the model families the pages evaluate:
32000 Llama-2/Vicuna, 64000 Yi, 128256 LLaMA-3.x, 152064 Qwen):
  C1 tiny      B=4  k=4  V=32000  fp32  T=1.0  t~N(0,3^2), d=t+N(0,1^2)
  C2           B=32 k=5  V=32000  bf16  T=1.0  t~N(0,4^2) +8 at one index/row, d=t+N(0,.5^2)
  C3 headline  B=64 k=8  V=128256 bf16  T=0.7  t~N(0,4^2) - 1.1 ln(v+1), d=t+N(0,1^2)
  C4 phrases   B=16 k=16 V=64000  bf16  greedy, draft = target argmax w.p. a
  C5 tree      B=8, 4 branches x 8 sharing a 2-token prefix (N=26), V=152064 bf16, greedy
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np

BF16 = "bf16"
FP32 = "fp32"


def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); return the uint16 bits.

    Inputs here are finite or -inf; -inf maps to 0xff80 exactly.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    b = x.view(np.uint32).astype(np.uint64)
    r = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def f32_from_bf16_bits(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to fp32 (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def logits_as_f32(arr: np.ndarray, dtype: str) -> np.ndarray:
    """Stored logits (bf16 bits or fp32) as fp32 values."""
    return f32_from_bf16_bits(arr) if dtype == BF16 else np.asarray(arr, dtype=np.float32)


def store(x_f32: np.ndarray, dtype: str) -> np.ndarray:
    return bf16_bits_from_f32(x_f32) if dtype == BF16 else np.ascontiguousarray(x_f32, np.float32)


@dataclass
class Workload:
    name: str
    mode: str                      # "stochastic" | "greedy" | "tree"
    B: int
    k: int                         # drafts per sequence (tree: N nodes)
    V: int
    dtype: str
    temperature: float
    target: np.ndarray             # [B][k+1][V]  (tree: [B][N+1][V])
    draft: Optional[np.ndarray]    # [B][k][V] or None
    tokens: np.ndarray             # [B][k] int32 (tree: node tokens [B][N])
    parents: Optional[np.ndarray] = None  # tree only, [B][N] int32
    seed: int = 1234               # verification seed (counter-based randomness)
    meta: dict = field(default_factory=dict)

    @property
    def nbytes_logits(self) -> int:
        n = self.target.nbytes
        if self.draft is not None:
            n += self.draft.nbytes
        return n


def _sample_rows(rng: np.random.Generator, logits_f32: np.ndarray, temperature: float) -> np.ndarray:
    """One categorical draw per row of ``softmax(logits / T)`` by inverse CDF.

    Input construction only: this is how a draft model would have produced its
    tokens.  Rows are processed one at a time to bound memory.
    """
    rows = logits_f32.reshape(-1, logits_f32.shape[-1])
    out = np.empty(rows.shape[0], dtype=np.int32)
    for r in range(rows.shape[0]):
        z = rows[r].astype(np.float64) / temperature
        w = np.exp(z - np.max(z))
        c = np.cumsum(w)
        u = rng.random() * c[-1]
        out[r] = min(int(np.searchsorted(c, u, side="right")), rows.shape[1] - 1)
    return out.reshape(logits_f32.shape[:-1])


def _normal(rng: np.random.Generator, shape, sigma: float) -> np.ndarray:
    return (rng.standard_normal(size=shape, dtype=np.float32) * np.float32(sigma)).astype(np.float32)


def gaussian_pair(B: int, k: int, V: int, dtype: str, temperature: float, seed: int,
                  sigma_t: float, sigma_d: float, peak: float = 0.0, zipf_s: float = 0.0,
                  name: str = "gaussian", verify_seed: int = 1234) -> Workload:
    """Target ~ N(0, sigma_t^2) (+ optional one-hot peak / Zipf-ranked bias),
    draft = target + N(0, sigma_d^2), draft tokens ~ softmax(draft / T)."""
    rng = np.random.default_rng(seed)
    t = _normal(rng, (B, k + 1, V), sigma_t)
    if peak:
        idx = rng.integers(0, V, size=(B, k + 1))
        np.put_along_axis(t, idx[..., None], np.take_along_axis(t, idx[..., None], -1) + np.float32(peak), -1)
    if zipf_s:
        t += (-zipf_s * np.log(np.arange(1, V + 1, dtype=np.float64))).astype(np.float32)
    d = t[:, :k, :] + _normal(rng, (B, k, V), sigma_d)
    tgt = store(t, dtype)
    drf = store(d, dtype)
    tokens = _sample_rows(rng, logits_as_f32(drf, dtype), temperature).astype(np.int32)
    return Workload(name, "stochastic", B, k, V, dtype, temperature, tgt, drf, tokens, seed=verify_seed,
                    meta=dict(gen_seed=seed, sigma_t=sigma_t, sigma_d=sigma_d, peak=peak, zipf_s=zipf_s))


def c1_tiny(seed: int = 101, verify_seed: int = 1234) -> Workload:
    """B=4, k=4, V=32000, fp32, T=1: t~N(0,3^2), d=t+N(0,1^2)."""
    return gaussian_pair(4, 4, 32000, FP32, 1.0, seed, 3.0, 1.0, name="C1", verify_seed=verify_seed)


def c2(seed: int = 102, verify_seed: int = 1234) -> Workload:
    """B=32, k=5, V=32000, bf16, T=1: t~N(0,4^2) with +8 at one uniform index per row, d=t+N(0,.5^2)."""
    return gaussian_pair(32, 5, 32000, BF16, 1.0, seed, 4.0, 0.5, peak=8.0, name="C2", verify_seed=verify_seed)


def c3(seed: int = 103, verify_seed: int = 1234, B: int = 64, k: int = 8, V: int = 128256) -> Workload:
    """B=64, k=8, V=128256, bf16, T=0.7: t~N(0,4^2) - 1.1 ln(v+1), d=t+N(0,1^2)."""
    return gaussian_pair(B, k, V, BF16, 0.7, seed, 4.0, 1.0, zipf_s=1.1, name="C3", verify_seed=verify_seed)


def _planted_rows(rng: np.random.Generator, shape, sigma: float, V: int):
    """Gaussian rows with a planted unique maximum at a uniform index.

    Values are clipped to [-6 sigma, 6 sigma] and the planted entry is set to
    6 sigma + 1, so the argmax of every row is known by construction (no argmax
    is computed here).
    """
    x = _normal(rng, shape + (V,), sigma)
    np.clip(x, -6 * sigma, 6 * sigma, out=x)
    top = rng.integers(0, V, size=shape)
    np.put_along_axis(x, top[..., None], np.float32(6 * sigma + 1.0), -1)
    return x, top.astype(np.int32)


def _other_id(rng: np.random.Generator, avoid: np.ndarray, V: int) -> np.ndarray:
    """A uniformly random id different from ``avoid`` (elementwise)."""
    r = rng.integers(0, V - 1, size=avoid.shape)
    return np.where(r >= avoid, r + 1, r).astype(np.int32)


def c4(a: float, seed: int = 104, B: int = 16, k: int = 16, V: int = 64000, dtype: str = BF16) -> Workload:
    """Greedy phrase-extended drafts: draft i = target argmax of row i w.p. a,
    otherwise a uniformly random other id."""
    rng = np.random.default_rng(seed)
    t, top = _planted_rows(rng, (B, k + 1), 4.0, V)
    hit = rng.random(size=(B, k)) < a
    tokens = np.where(hit, top[:, :k], _other_id(rng, top[:, :k], V)).astype(np.int32)
    return Workload(f"C4(a={a})", "greedy", B, k, V, dtype, 0.0, store(t, dtype), None, tokens,
                    meta=dict(gen_seed=seed, a=a, argmax=top))


def guided_drafts(a: float, a_guide: float, L: int, seed: int = 106, B: int = 16, k: int = 16, V: int = 64000,
                  dtype: str = BF16):
    """Target-guided greedy verification inputs: C4's rows and drafts, plus a
    target-side guide [B][L] aligned with the draft positions.  The guide's
    entry i is the planted argmax of row i w.p. a_guide (positions with a row),
    otherwise a uniform other id; past the rows it is a uniform id.  Each guide
    ends after a uniform length in [0, L] (-1 after its end)."""
    w = c4(a, seed=seed, B=B, k=k, V=V, dtype=dtype)
    rng = np.random.default_rng(seed + 1)
    top = w.meta["argmax"]
    guide = rng.integers(0, V, size=(B, L)).astype(np.int32)
    rows = min(L, k + 1)
    if rows:
        hit = rng.random(size=(B, rows)) < a_guide
        guide[:, :rows] = np.where(hit, top[:, :rows], _other_id(rng, top[:, :rows], V))
    length = rng.integers(0, L + 1, size=B)
    guide[np.arange(L)[None, :] >= length[:, None]] = -1
    return w, guide


def tree_shape(prefix: int = 2, branches: int = 4, length: int = 8) -> np.ndarray:
    """Parents of a tree: a shared chain of ``prefix`` nodes, then ``branches``
    chains continuing it so that every root-to-leaf path has ``length`` nodes."""
    parents = []
    for m in range(prefix):
        parents.append(m - 1)
    for _ in range(branches):
        prev = prefix - 1
        for _ in range(length - prefix):
            parents.append(prev)
            prev = len(parents) - 1
    return np.asarray(parents, dtype=np.int32)


def c5(seed: int = 105, B: int = 8, V: int = 152064, p_match: float = 0.7, dtype: str = BF16,
       parents: Optional[np.ndarray] = None) -> Workload:
    """Tree verification: 4 branches of length 8 sharing a 2-token prefix
    (26 nodes), one target row per node plus the context row (27 rows).
    Node token = argmax of its parent's row w.p. 0.7, else a uniform other id."""
    rng = np.random.default_rng(seed)
    par = tree_shape() if parents is None else np.asarray(parents, dtype=np.int32)
    N = par.shape[0]
    t, top = _planted_rows(rng, (B, N + 1), 4.0, V)
    row_of_parent = np.where(par < 0, 0, par + 1)
    want = top[:, row_of_parent]                       # [B][N]
    hit = rng.random(size=(B, N)) < p_match
    tokens = np.where(hit, want, _other_id(rng, want, V)).astype(np.int32)
    return Workload("C5", "tree", B, N, V, dtype, 0.0, store(t, dtype), None, tokens,
                    parents=np.broadcast_to(par, (B, N)).copy(), meta=dict(gen_seed=seed, argmax=top))


def iid_acceptance(B: int, k: int, V: int, a: float, seed: int, verify_seed: int = 1234) -> Workload:
    """Stochastic inputs whose per-draft acceptance probability is exactly ``a``.

    Each target row puts mass p on a random half of the vocabulary (-inf logits
    elsewhere).  The draft row is q = a*p + (1-a)*r with r supported on the
    other half, so sum_v min(p_v, q_v) = a.  Draft tokens are drawn from q.
    Logits are fp32 log-probabilities at T = 1.
    """
    rng = np.random.default_rng(seed)
    tgt = np.full((B, k + 1, V), -np.inf, dtype=np.float64)
    drf = np.full((B, k, V), -np.inf, dtype=np.float64)
    for b in range(B):
        for j in range(k + 1):
            perm = rng.permutation(V)
            on, off = perm[: V // 2], perm[V // 2:]
            w = np.exp(rng.standard_normal(on.size))
            p = w / w.sum()
            tgt[b, j, on] = np.log(p)
            if j < k:
                wr = np.exp(rng.standard_normal(off.size))
                r = wr / wr.sum()
                drf[b, j, on] = np.log(a * p)
                drf[b, j, off] = np.log((1.0 - a) * r)
    tgt32 = tgt.astype(np.float32)
    drf32 = drf.astype(np.float32)
    tokens = _sample_rows(rng, drf32, 1.0).astype(np.int32)
    return Workload(f"iid(a={a})", "stochastic", B, k, V, FP32, 1.0, tgt32, drf32, tokens, seed=verify_seed,
                    meta=dict(gen_seed=seed, a=a))


def tiny_rows(k: int = 3, V: int = 8, seed: int = 7, sigma_t: float = 3.0, sigma_d: float = 1.0):
    """Context-free target / draft logit rows for exhaustive enumeration (fp64)."""
    rng = np.random.default_rng(seed)
    t = rng.standard_normal((k + 1, V)) * sigma_t
    d = t[:k] + rng.standard_normal((k, V)) * sigma_d
    return t, d


CONFIGS = {
    "C1": c1_tiny,
    "C2": c2,
    "C3": c3,
    "C4": lambda seed=104: c4(0.8, seed),
    "C5": c5,
}
