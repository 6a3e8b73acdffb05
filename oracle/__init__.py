"""Oracle for batched speculative-decoding verification -- TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously correct CPU restatement, in fp64 numpy, of what the
verification path computes.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it.
The product path (the CUDA library and its Python binding) never imports, calls
or links anything here, and this package shares no code, tables or constants
with it: the only thing both sides use is the seeded input builder in
``workloads`` and the published definition of Philox4x32-10, which each side
implements on its own.

Modules
  philox   Philox4x32-10 block function and the uniforms / Gumbel noise the rule draws.
  verify   the acceptance rule, residual and bonus sampling, greedy and tree verification.
  theory   closed forms: expected committed tokens per round and its generating function.
  enumerate exact output distribution of the rule on tiny vocabularies.

Sources (page title -- section):
  * "Speculative Decoding: Faster Generation Without Changing the Model" --
    "The acceptance rule" (accept w.p. min(1, p/q), residual max(0, p-q),
    bonus token, greedy collapse) and "Predicting the speedup" (closed form).
  * "Cascade Speculative Drafting for Even Faster LLM Inference" -- the review
    step of the vertical cascade (accept if q <= p, otherwise reject with
    probability 1 - p/q; lenience l = 1 at the target) and "Theoretical
    Framework: EWIF and Generating Functions", Theorem 4.1.
  * "Ouroboros: Generating Longer Drafts Phrase by Phrase for Faster Speculative
    Decoding" -- 3.4.3 "Selecting the accepted tokens" (longest accepted branch).
  * "Double: Breaking the Acceleration Limit via Double Retrieval Speculative
    Parallelism" -- target-guided verification (greedy replacement is residual
    rejection; lossless under sampling).

Parity status: every function here is pinned by a ``-m "not gpu"`` test against
something other than itself (published Philox known-answer vectors, the
closed forms printed on the pages, exact enumeration, chi-squared laws, brute
force).  See tests/test_oracle_*.py.
"""

