"""The draft's LM head followed by the masked soft-target cross-entropy
(oracle; test infrastructure).

Source: SpecForge review, §三 "内存高效梯度计算" (the in-place gradient of the
logits, s = sum(p*g), z <- -(p*g - pi*s)) and §四 "原地反向传播"; the logits
are the draft's LM-head output z = h W^T, the matrix whose memory the
in-place trick saves.  With hidden states h [N, Hd], head weights W [V, Hd],
targets p [N, V] and per-row upstream gradients g [N]:

    z  = h @ W^T                                   [N, V]
    (L, row_loss, dz) = soft_ce(z, p, g)           (oracle.soft_ce)
    dh = dz @ W                                    [N, Hd]
    dW = dz^T @ h                                  [V, Hd]

i.e. the loss and the gradients of L with respect to h and W.  Float64.
"""

import numpy as np

from . import soft_ce as _sce


def lm_head_soft_ce(h, W, p, g):
    """Return (L, row_loss [N], dh [N, Hd], dW [V, Hd]) in float64."""
    h = np.asarray(h, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    z = h @ W.T
    L, row_loss, dz = _sce.soft_ce(z, p, g)
    dh = dz @ W
    dW = dz.T @ h
    return L, row_loss, dh, dW
