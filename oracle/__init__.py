"""Reference oracle for the self-speculative decoding hot path -- TEST INFRASTRUCTURE ONLY.

This package is a plain, slow, float64 CPU restatement of what the CUDA library
computes.  It exists so that the tests, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` have an
independent answer to compare against.  Nothing else may import it: the
product path (``long_context_speculative_split_gb300``) never calls into this
package and has no CPU fallback.

It shares no code with the CUDA path (no kernels, headers, helpers, tables or
constant generators).  Inputs of any float dtype are upcast exactly to float64.

Sources (the pages this restates):
  * "MAGICDEC: BREAKING THE LATENCY-THROUGHPUT TRADEOFF FOR LONG CONTEXT
    GENERATION WITH SPECULATIVE DECODING" (paper notes, arXiv:2408.11049):
    quick-read summary (self-speculation over a compressed KV of budget K,
    Eq. 2/3 restated inline), section 3.1 (expected tokens per round
    Omega(gamma, alpha)), section 3.2 (verify and decode load the same KV),
    section 4.4 (static selection such as SnapKV; top-K attention's selection
    cost), section 5.1 (StreamingLLM-style drafting), appendix A.1 (the static
    compressed KV is built at prefill and reused for drafting).
  * "Wann beschleunigt spekulatives Decoding das LLM-Serving?", section
    "Eine Verifizierungsrunde verstehen" (left-to-right acceptance, residual
    correction at the first rejection, bonus token when all are accepted) and
    the paragraph after it (the rule preserves the target distribution).

Modules:
  attention  -- exact two-pass softmax attention (verify and draft forms) and
                the log-sum-exp merge of partial results.
  snapkv     -- observation-window scores, max-pool, top-K + window, gather.
  sampling   -- softmax, inverse-CDF draw, draft draw, modified rejection
                sampling.
  commit     -- commit / rollback of the caches after a verification round.
  streaming  -- StreamingLLM-style draft cache (attention sinks + recent rows).
  topk       -- dynamic top-K attention drafting (one draft step).

Pins: every function here is checked by ``tests/test_oracle_*.py`` against
closed forms, hand-derived fixtures in ``tests/golden/``, high-precision brute
force and statistical identities -- never against the CUDA path.
"""
