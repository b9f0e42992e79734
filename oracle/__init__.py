"""Float64 CPU oracle for rotary position embedding with context-extension
rescaling and exact softmax attention.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
execute this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code, tables or constants with the CUDA library; both sides receive the same
seeded inputs and nothing else.

Every function is the plain definition the pages give, written out in numpy
float64 with no blocking, fusion or reordering beyond what the definition says:

* ``oracle.rope``      -- base frequencies, Position Interpolation, NTK-aware
  base scaling, YaRN's NTK-by-parts ramp and attention temperature, and the
  rotate-half rotation.
* ``oracle.attention`` -- the visibility predicate (causal, attention sinks plus
  sliding window, none), full-softmax attention rows, the blockwise online-
  softmax fold (used only to check invariants), and streaming decode over a
  sink + window ring-buffer cache.

Sources (cited by page title and section):

* "Context Window Scaling: YaRN, LongRoPE, and RingAttention Architectures"
  (tecvarsity) -- Section 1 (softmax attention), Section 2 (RoPE, relative
  invariance, PI), Section 3 (YaRN regimes, temperature), Section 5 and FAQ 2
  (ring blocks and causal block skip).
* "Context Length Extension" (14cs17 notes) -- Notation, Why Models Fail,
  Position Interpolation, NTK-Aware Scaling, YaRN, Sliding Window + Attention
  Sinks, Ring Attention, Exercises 1 and 2.
* "Long-context extension: stretching attention past its training window"
  (root18d) -- "Not every RoPE dimension needs the same treatment".
* Long-context guide a2-tli-4 (jovanaeducation) -- "YaRN: rescale the
  frequencies", "Attention sinks", "Ring attention".
* "Long-Context Scaling" (AI/ML animation academy) -- Production defaults
  (4 pinned sink tokens).

Pins (``tests/test_oracle_*.py``) tie every function to something other than
itself: worked examples the pages print, closed forms, invariants the pages
state, library routines for special cases, and brute force on tiny inputs.
"""

from . import rope, attention  # noqa: F401
