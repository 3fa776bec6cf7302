"""CPU oracle for lookahead decoding — TEST INFRASTRUCTURE, not part of the product.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may import, call or execute anything in this package.
The CUDA library never links, imports or falls back to it, and this package
imports nothing from the CUDA library: the two share no code.  The only
module both sides use is ``synth`` (seeded random inputs, none of the
method's arithmetic).

Contents (each function cites the passage of the pages it restates):

* ``model``     — plain Llama-style decoder forward (RMSNorm, RoPE, causal
  attention under an arbitrary visibility relation, SwiGLU), float64 by
  default, with an optional emulation of bf16 storage points.
* ``lookahead`` — the lookahead state machine: window levels and warm-up,
  row compiler, branch visibility, keyed n-gram extraction, per-key LRU
  pool, greedy verification, K/V publication plan, window advance, and the
  generate loops (autoregressive and lookahead, in three schedules).
* ``sampling``  — temperature/top-p warping and the exact multi-draft
  verifier with disjoint one-hot proposals.
* ``batch``     — several requests in one packed forward (each request's
  rows against its own cache and rows only), and the batched generate loop.
* ``philox``    — Philox4x32-10 counter-based generator.
* ``jacobi``    — Jacobi and Gauss–Seidel sweeps over a triangular system.

Parity status: the integer state machine, the verifiers and the Jacobi
sweeps are pinned by the worked examples, closed forms and invariants of the
pages (see tests/test_oracle_*.py).  The transformer's floating-point values
are pinned only by textbook definitions and by self-consistency between
schedules: the pages print no logits ("parity unpinned" for model numerics
beyond those definitions).
"""
