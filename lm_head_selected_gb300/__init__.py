"""GB300-native fused linear selected-token log-probability.

The computation lives in ``liblinear_logp.so`` (sm_103a CUDA kernels behind the
C ABI of ``include/linear_logp.h``); this package only marshals PyTorch tensors
into that ABI.  Build the library with ``lm_head_selected_gb300.build.build()``.
"""
from .fused import (  # noqa: F401
    fused_logp,
    fused_logp_bwd,
    fused_logp_bwd_indexed,
    fused_logp_fwd,
    fused_logp_fwd_indexed,
)
from .ops import (  # noqa: F401
    IGNORE_INDEX,
    bwd_workspace_bytes,
    device_status,
    fwd_workspace_bytes,
    linear_logp,
    linear_logp_bwd,
    linear_logp_bwd_indexed,
    linear_logp_fwd,
    linear_logp_fwd_indexed,
)
