"""Plain, slow, fp64 CPU oracle for exact IO-aware attention.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import or call it.  It shares no
code with the CUDA library: no kernels, headers, helpers or constant tables.

Sources (the pages the method is taken from):
  * "CMU 11-868 L21 FlashAttention" lecture notes (Tri Dao guest lecture),
    slides 5, 12, 14, 24, 27-46, 57-60.
  * Book chapter "第18章 FlashAttention", sections 18.2.1-18.2.4, 18.4.1-18.4.4,
    18.5, 18.6.2 (with Table 18-21), 18.7.1, 18.8.1-18.8.3.

Modules:
  attention  -- the plain definition of attention forward / backward (S and P
                materialised), the tiled online-softmax recurrence written in the
                pages' order, and the FlashDecoding split + combine.
  plan       -- the integer plans: causal tile classes, longest-first order,
                greedy list scheduling, and decode split boundaries.
  fp8        -- the E4M3 format, the Hadamard transform of incoherent
                processing, the per-block quantiser and the FP8 forward loop
                ("第18章" §18.5 and §18.6.2; lecture slide 24).

Every function is pinned by ``tests/test_oracle_*.py`` against closed forms,
invariants, brute force and the pages' worked examples; none is "parity
unpinned".
"""

from . import attention, fp8, plan  # noqa: F401
