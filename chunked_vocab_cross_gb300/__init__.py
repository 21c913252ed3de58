"""GB300-native fused output projection + cross-entropy (memory-free LM-head loss).

The computation lives in liblce.so (hand-written sm_103a CUDA behind the C ABI
in include/lce.h); this package only marshals arguments. Calls raise if the
library has not been built: there is no CPU fallback.
"""
from ._abi import LIB_PATH, LceError, lib  # noqa: F401
from .ops import (  # noqa: F401
    FusedOptimizer, device_status, embedding, embedding_backward, embedding_forward, embedding_workspace_size,
    launch_count, lce_backward, lce_compact, lce_forward, lce_forward_backward, lce_run, linear_cross_entropy,
    profile_begin, profile_end, workspace_size,
)
