"""Plain float64 CPU oracle for split-KV decode attention.

TEST INFRASTRUCTURE ONLY.  This package is a slow, obviously-correct
restatement of what the decode path computes, written from three article
pages of the "Transformer System" series:

* M4.5 Decode Attention Kernels, Mask Programs, and Backend Boundaries
  (split-state algebra, split bounds, workspace ledgers, K/V address
  translation, mask tiles, causal alignment);
* M5.4 Long-Context KV Policies: Retention, Compression, Budget Allocation
  (sliding window, sink + recent retention sets);
* M8.6 Live-Data Quantization: Activations and KV Cache
  (per-token INT8 and KIVI-style INT4 K/V formats with a residual window).

Every function cites the section it follows.  Only ``tests/``,
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference``
legs of ``bench.py`` may import it.  The CUDA library never imports, links or
calls anything here, and nothing here imports the CUDA library: the two sides
share only the documented memory layout and the seeded input generators in
``workloads.py`` (which hold none of the method's arithmetic).

Parity status: every module is pinned by ``tests/test_oracle_*.py`` against
values the pages print, closed forms, invariants or brute force.  No function
here is "parity unpinned".
"""

from . import split_state, address, masks, quant, cache, attention  # noqa: F401
