"""Work and traffic counts used to turn measured times into throughput.

These are the measurement definitions: useful FLOPs of the attention (only
unmasked score entries count) and algorithmic HBM bytes of the soft-CE.
"""

from __future__ import annotations

from typing import Sequence

import torch

from .workloads import AttnShape


def useful_entries(T: int, Q_LEN: int, k: int) -> int:
    """Unmasked score entries of one (b, h) at TTT step k (closed form).

    Valid rows q < T see q+1 causal keys and one key in each of the k later
    blocks; padded rows q >= T see the T keys kv < T.
    """
    return T * (T + 1) // 2 + k * T + (Q_LEN - T) * T


def attn_useful_flops(shape: AttnShape, T: Sequence[int], steps=None) -> tuple:
    """(forward, backward) useful FLOPs: 4*D per unmasked entry forward, 10*D backward."""
    steps = shape.steps if steps is None else steps
    ent = sum(useful_entries(t, shape.Q_LEN, k) for t in T for k in steps) * shape.H
    return 4 * shape.D * ent, 10 * shape.D * ent


def soft_ce_algorithmic_bytes(N: int, V: int, g: torch.Tensor) -> int:
    """12*V per row with g != 0 (read z, read p, write z), 4*V per row with g == 0
    (write zeros), plus 4*N for g and 4*N for the per-row loss."""
    nz = int((g != 0).sum().item())
    return 12 * V * nz + 4 * V * (N - nz) + 8 * N
