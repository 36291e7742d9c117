"""Oracle for tiered decode attention. This is TEST INFRASTRUCTURE.

It is a plain, slow, fp64 CPU implementation of what the tiered KV-cache hot
path computes, written from the pages' description of the method ("Not All
Thoughts Need HBM: Semantics-Aware Memory Hierarchy for LLM Reasoning",
gist.science summary, sections "Four-tier classification", "Importance
scoring" (the s_i equation), "Zero-approximation-error offloading"
(Proposition 1) and "System implementation" (Delta = 64); the fugumt.com
abstract of the same paper; and the ARKV summary's tri-state assignment
section for the dequantise-then-concatenate-in-original-order rule).

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import or run anything here.
The CUDA library never links, calls or reads this package, and this package
never imports the CUDA library: the two share no code.

Modules:
  fp8       -- OCP FP8-E4M3 format: decode table, round-to-nearest-even encoder
               with saturation, per-row quantise / dequantise.
  tiering   -- protected set, tier targets, tier assignment by cumulative
               score (s descending, lower index first on ties).
  attention -- decode-step attention over the retained tokens of one layer,
               reading each token from the container of its tier.
  session   -- a decode session: prefill, per-step append + attention +
               score update, and a re-tier every Delta steps.

Parity status: every function here is pinned by a ``-m "not gpu"`` test in
``tests/test_oracle_*.py`` against something other than itself (a library
routine, a closed form, a hand-derived fixture under ``tests/golden/`` or an
invariant).  None is "parity unpinned".
"""

from . import fp8, tiering, attention, session  # noqa: F401

__all__ = ["fp8", "tiering", "attention", "session"]
