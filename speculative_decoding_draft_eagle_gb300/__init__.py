"""EAGLE-3 training-time-test (TTT) draft-step core on GB300 (sm_103a).

Sparse-tree TTT attention (forward and backward) and the masked soft-target
cross-entropy with its in-place gradient, as a C-ABI CUDA library
(``include/stt.h``, ``libstt.so``) with a thin ctypes binding (``ops``).
"""

from .ops import (  # noqa: F401
    soft_ce_fwd_bwd_inplace,
    soft_ce_workspace_size,
    stt_attn_bwd,
    stt_attn_bwd_workspace_size,
    stt_attn_fwd,
    stt_device_error,
    stt_version,
)
