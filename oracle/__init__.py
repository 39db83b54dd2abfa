"""Oracle for exact masked scaled-dot-product attention: TEST INFRASTRUCTURE ONLY.

A plain, slow, float64 CPU statement of what the CUDA library computes, written
from the pages that define the method:

  * "Exact tiled softmax attention with block-recomputed vector-Jacobian
    products" (alphabetamath) -- the Inputs paragraph (Q, K, V, scale c,
    nonempty allowed-key sets A_i), the Forward procedure and the Reverse
    procedure (p_ij, gamma_ij and the three accumulation equations);
  * "python-flash-attention-online-softmax-block-recompute" -- "The fix":
    the saved statistic L = m + log l and the backward formulas;
  * "txf-modern-flash-attention" (trentorch) -- "Constraints": exact output for
    every block size 1..n, running max and rescale rule;
  * HarshvardhanJ/FlashAttention (githubhelp) -- the backward flowchart and
    the identity D_i = dY_i . Y_i.

Modules:
  masks  -- the allowed-key sets A_i from a mask kind / window / bit rows
  dense  -- the plain dense definition (forms whole rows of S); the oracle proper
  tiled  -- the pages' block procedures (summary, merge, skip, recompute
            reverse), used only to pin ``dense`` against the pages
  philox -- the counter-based generator (Philox-4x32-10) and the dropout keep
            mask that the dropout forms of ``dense`` replay in both passes

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
reference arm of ``bench.py`` may import this package.  It shares no code with
the CUDA path and never imports it.  Every function here is pinned by the CPU
tests in ``tests/test_oracle.py`` (directly, or as a step of a pinned
procedure); none is "parity unpinned".
"""
from . import dense, masks, philox, tiled  # noqa: F401
