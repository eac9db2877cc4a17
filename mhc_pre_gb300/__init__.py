"""GB300-native mHC (manifold-constrained hyper-connection) layer.

The compute lives in ``libmhc_gb300.so`` (hand-written CUDA for sm_103a, C ABI
declared in ``include/mhc.h``); ``binding`` marshals torch tensors to it.
``workloads`` holds the seeded synthetic inputs.  The library is loaded on
first use, so importing the package never needs a GPU.
"""

from .binding import (  # noqa: F401
    MhcError,
    mhc_post,
    mhc_post_bwd,
    mhc_pre,
    mhc_pre_bwd,
    pre_bwd_workspace_bytes,
)

__all__ = ["mhc_pre", "mhc_post", "mhc_post_bwd", "mhc_pre_bwd",
           "pre_bwd_workspace_bytes", "MhcError"]
