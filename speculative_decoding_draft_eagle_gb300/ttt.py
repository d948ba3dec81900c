"""The TTT step loop as one differentiable call.

In EAGLE-3 training-time test (SpecForge review, §三 "稀疏树注意力": TTT
length 7, and §六 "训练时测试（TTT）长度的影响") the draft runs K steps; step k
attends with fresh queries q_k to the KV blocks 0..k, block j having been
produced at step j.  A block's gradient is therefore the sum over the steps
k >= j that read it.  ``ttt_attention`` runs every step's forward through the
C ABI and, in the backward, calls ``stt_attn_bwd_ex`` once per step with the
block gradients ACCUMULATED in place by the kernels (the first call, at the
last step, which covers every block, overwrites; the others add), so no
separate pass ever sums the per-step block gradients.  Gradients come back in
the inputs' dtype (bf16: STT_BWD_BF16_GRADS).  This module only orders the
calls and allocates the buffers; every arithmetic step runs in the library.
"""

from __future__ import annotations

import math
from typing import List, Optional, Sequence

import torch

from . import ops


class _TTTAttention(torch.autograd.Function):
    @staticmethod
    def forward(ctx, T, scale, n, *tensors):
        qs, Ks, Vs = tensors[:n], tensors[n:2 * n], tensors[2 * n:3 * n]
        outs, lses = [], []
        for k in range(n):
            o, l = ops.stt_attn_fwd(qs[k], list(Ks[: k + 1]), list(Vs[: k + 1]), T, scale)
            outs.append(o)
            lses.append(l)
        ctx.save_for_backward(*qs, *Ks, *Vs, *outs, *lses)
        ctx.T, ctx.scale, ctx.n = list(T), scale, n
        return tuple(outs)

    @staticmethod
    def backward(ctx, *douts):
        n, T, scale = ctx.n, ctx.T, ctx.scale
        saved = ctx.saved_tensors
        qs, Ks, Vs = saved[:n], saved[n:2 * n], saved[2 * n:3 * n]
        outs, lses = saved[3 * n:4 * n], saved[4 * n:5 * n]
        gdt = qs[0].dtype
        dKs = [torch.empty(K.shape, device=K.device, dtype=gdt) for K in Ks]
        dVs = [torch.empty(V.shape, device=V.device, dtype=gdt) for V in Vs]
        dqs: List[Optional[torch.Tensor]] = [None] * n
        ws = None
        # The last step reads every block: it overwrites all of them first,
        # every earlier step adds to the blocks it reads.
        for k in range(n - 1, -1, -1):
            dO = douts[k]
            if dO is None:
                dO = torch.zeros_like(outs[k])
            dO = dO.to(torch.bfloat16).contiguous()
            dq = torch.empty(qs[k].shape, device=qs[k].device, dtype=gdt)
            ops.stt_attn_bwd_ex(qs[k], list(Ks[: k + 1]), list(Vs[: k + 1]), T, outs[k], dO,
                                lses[k], dq, dKs[: k + 1], dVs[: k + 1], scale=scale,
                                accumulate=(k != n - 1), workspace=ws)
            dqs[k] = dq
        return (None, None, None, *dqs, *dKs, *dVs)


def ttt_attention(qs: Sequence[torch.Tensor], Ks: Sequence[torch.Tensor],
                  Vs: Sequence[torch.Tensor], T, scale: Optional[float] = None):
    """Outputs of TTT steps k = 0..K-1, differentiable in every q_k, K_j and V_j.

    qs[k]: bf16 [B, H, Q_LEN, D], the queries of step k; Ks[j], Vs[j]: bf16
    [B, H_kv, Q_LEN, D], the KV block produced at step j (len(qs) == len(Ks)
    == len(Vs) == K); T: B valid lengths.  Returns a tuple of K bf16 outputs."""
    n = len(qs)
    if n == 0 or len(Ks) != n or len(Vs) != n:
        raise ValueError("qs, Ks and Vs must each hold one tensor per TTT step")
    D = qs[0].shape[-1]
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    return _TTTAttention.apply([int(t) for t in (T.tolist() if isinstance(T, torch.Tensor) else T)],
                               scale, n, *qs, *Ks, *Vs)
