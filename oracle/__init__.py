"""Float64 CPU oracle for the mHC layer (test infrastructure, not product code).

This package is the independent reference that the CUDA library is checked
against.  Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import it; the library under ``mhc_pre_gb300`` never
does, and this package never imports the library.

Sources followed (page title, section):
  * "openPangu 2.0 -- architecture, training and Ascend systems" analysis
    notes, section 5.3 "mHC: reading, write-back and constrained mixing of the
    four residual streams" (RMSNorm of the stream state, the projection to
    [r_pre, r_post, r_res], sigmoid / 2*sigmoid gates, Sinkhorn of the reshaped
    n x n block) and the model table in section 01 (4 streams, 20 Sinkhorn
    rounds).
  * "Ascend mHC Triton operator" article (jinguxun.com news 8765171), the
    paragraph defining H^res / H^pre / H^post (doubly stochastic; ranges
    (0,1) and (0,2)) and the paragraph on fp32 compute for the activations.

Every function here is pinned by tests in ``tests/test_oracle_*.py`` against
closed forms, invariants, an independent fixed-point solver and central finite
differences.  Nothing in this package is "parity unpinned".
"""

from .mhc_oracle import (  # noqa: F401
    group_of_logit,
    rmsnorm_flat,
    project,
    logits_from_proj,
    gates,
    sinkhorn,
    sinkhorn_iterates,
    sinkhorn_vjp,
    mhc_pre,
    mhc_post,
    mhc_post_bwd,
    mhc_pre_bwd,
)
