"""Seeded synthetic workloads for the TTT draft-step core.

This module holds only input generation: shapes, seeds and the value
distributions of the five workloads.  It contains none of the method's
arithmetic, so the CUDA path and the CPU oracle can both be fed from it.

Tensors are drawn with a ``torch.Generator`` on the requested device; every
tensor has its own generator seeded from (workload seed, tensor tag), so any
tensor can be regenerated alone.  The CPU and CUDA generators give different
streams: a comparison must draw once and hand the same bits to both sides.
"""

from __future__ import annotations

import dataclasses
import math
from typing import List, Sequence

import torch


@dataclasses.dataclass(frozen=True)
class AttnShape:
    B: int
    H: int
    H_kv: int
    D: int
    Q_LEN: int
    T_range: tuple          # inclusive (lo, hi) of the per-sequence valid length
    steps: tuple            # TTT steps k run by one pass of the workload

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def n_blocks(self) -> int:
        return max(self.steps) + 1


@dataclasses.dataclass(frozen=True)
class SoftCEShape:
    N: int
    V: int
    z_std: float = 2.0
    p_std: float = 2.0
    p_temp: float = 0.8
    one_hot_frac: float = 0.0
    keep_prob: float = 0.8
    mask_beyond_T: bool = False


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    index: int
    attn: AttnShape
    soft_ce: SoftCEShape

    @property
    def seed(self) -> int:
        return 1000 + self.index


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny", 1,
                 AttnShape(B=1, H=2, H_kv=1, D=64, Q_LEN=128, T_range=(100, 100), steps=(2,)),
                 SoftCEShape(N=128, V=1024)),
        Workload("llama8b", 2,
                 AttnShape(B=1, H=32, H_kv=8, D=128, Q_LEN=4096, T_range=(2048, 4096),
                           steps=tuple(range(7))),
                 SoftCEShape(N=4096, V=32000)),
        Workload("varlen", 3,
                 AttnShape(B=16, H=32, H_kv=8, D=128, Q_LEN=2048, T_range=(256, 2048),
                           steps=tuple(range(7))),
                 SoftCEShape(N=16 * 2048, V=32000, mask_beyond_T=True)),
        Workload("llama70b", 4,
                 AttnShape(B=2, H=64, H_kv=8, D=128, Q_LEN=4096, T_range=(3072, 4096),
                           steps=tuple(range(7))),
                 SoftCEShape(N=8192, V=32000, p_std=3.0, one_hot_frac=0.25)),
        Workload("long_ttt", 5,
                 AttnShape(B=1, H=32, H_kv=8, D=128, Q_LEN=8192, T_range=(8192, 8192),
                           steps=tuple(range(13))),
                 SoftCEShape(N=8192, V=151936)),
    ]
}


def _gen(device, seed: int, tag: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 7919 + tag)
    return g


def randn_bf16(shape, device, seed: int, tag: int, std: float = 1.0) -> torch.Tensor:
    """N(0, std^2) drawn in fp32 and rounded to bf16 (round to nearest even)."""
    x = torch.randn(shape, generator=_gen(device, seed, tag), device=device, dtype=torch.float32)
    if std != 1.0:
        x = x * std
    return x.to(torch.bfloat16)


def draw_T(shape: AttnShape, seed: int) -> List[int]:
    """Per-sequence valid lengths, uniform integers over T_range (inclusive), CPU generator."""
    lo, hi = shape.T_range
    g = _gen("cpu", seed, 1)
    return [int(x) for x in torch.randint(lo, hi + 1, (shape.B,), generator=g)]


# tags: 10 + j for K_j, 100 + j for V_j, 1000 + k for q of step k, 2000 + k for dO of step k
def kv_block(shape: AttnShape, which: str, j: int, device, seed: int) -> torch.Tensor:
    tag = (10 if which == "K" else 100) + j
    return randn_bf16((shape.B, shape.H_kv, shape.Q_LEN, shape.D), device, seed, tag)


def step_query(shape: AttnShape, k: int, device, seed: int) -> torch.Tensor:
    return randn_bf16((shape.B, shape.H, shape.Q_LEN, shape.D), device, seed, 1000 + k)


def step_dout(shape: AttnShape, k: int, device, seed: int) -> torch.Tensor:
    return randn_bf16((shape.B, shape.H, shape.Q_LEN, shape.D), device, seed, 2000 + k)


def attn_inputs(shape: AttnShape, device, seed: int):
    """All inputs of one pass: T, K/V blocks 0..K-1, and q/dO per step."""
    T = draw_T(shape, seed)
    Ks = [kv_block(shape, "K", j, device, seed) for j in range(shape.n_blocks)]
    Vs = [kv_block(shape, "V", j, device, seed) for j in range(shape.n_blocks)]
    qs = {k: step_query(shape, k, device, seed) for k in shape.steps}
    dOs = {k: step_dout(shape, k, device, seed) for k in shape.steps}
    return T, Ks, Vs, qs, dOs


def soft_ce_inputs(sc: SoftCEShape, device, seed: int, T: Sequence[int] = None,
                   Q_LEN: int = None):
    """z [N,V] fp32, p [N,V] fp32 (rows on the simplex), g [N] fp32.

    z ~ N(0, z_std^2).  p = softmax(N(0, p_std^2) / p_temp) per row; a fraction
    ``one_hot_frac`` of rows (chosen by a seeded permutation) is instead the
    one-hot vector at the argmax of that row's logits.  g = Bernoulli(keep_prob)
    / N per row; with ``mask_beyond_T`` the rows b*Q_LEN + q with q >= T[b] get
    g = 0.
    """
    N, V = sc.N, sc.V
    z = torch.randn((N, V), generator=_gen(device, seed, 50), device=device,
                    dtype=torch.float32) * sc.z_std
    logits = torch.randn((N, V), generator=_gen(device, seed, 51), device=device,
                         dtype=torch.float32) * sc.p_std
    p = torch.softmax(logits / sc.p_temp, dim=1)
    if sc.one_hot_frac > 0:
        n_hot = int(round(sc.one_hot_frac * N))
        perm = torch.randperm(N, generator=_gen("cpu", seed, 52))[:n_hot].to(device)
        hot = torch.zeros((n_hot, V), device=device, dtype=torch.float32)
        hot.scatter_(1, logits[perm].argmax(dim=1, keepdim=True), 1.0)
        p[perm] = hot
    del logits
    keep = torch.bernoulli(torch.full((N,), sc.keep_prob), generator=_gen("cpu", seed, 53))
    if sc.mask_beyond_T:
        assert T is not None and Q_LEN is not None and len(T) * Q_LEN == N
        pos = torch.arange(N) % Q_LEN
        lim = torch.tensor(T).repeat_interleave(Q_LEN)
        keep = torch.where(pos < lim, keep, torch.zeros_like(keep))
    g = (keep / N).to(torch.float32).to(device)
    return z, p, g


@dataclasses.dataclass(frozen=True)
class VerifyShape:
    """Rejection-sampling verification: B sequences, gamma draft tokens each,
    vocabulary V.  The target's distribution is softmax(N(0, sigma^2) / temp);
    the draft's is softmax((target logits + N(0, noise^2)) / temp), so the two
    agree roughly as a trained draft does; the draft tokens are drawn from the
    draft's distribution."""
    B: int
    gamma: int
    V: int
    sigma: float = 2.0
    noise: float = 0.5
    temp: float = 0.8


# B 64 sequences, 5 draft tokens each (num_speculative_tokens = 5 of the
# FlashSpec practice page), Qwen-sized vocabulary.
VERIFY = VerifyShape(B=64, gamma=5, V=151936)


def verify_inputs(vs: VerifyShape, device, seed: int):
    """p_target, p_draft fp32 [B, gamma, V]; draft_tokens int32 [B, gamma];
    u_accept fp32 [B, gamma] and u_sample fp32 [B], uniform in [0, 1)."""
    shape = (vs.B, vs.gamma, vs.V)
    lt = torch.randn(shape, generator=_gen(device, seed, 60), device=device) * vs.sigma
    p_t = torch.softmax(lt / vs.temp, dim=-1)
    ld = lt + torch.randn(shape, generator=_gen(device, seed, 61), device=device) * vs.noise
    p_d = torch.softmax(ld / vs.temp, dim=-1)
    del lt, ld
    toks = torch.multinomial(p_d.reshape(-1, vs.V), 1, generator=_gen(device, seed, 62))
    toks = toks.reshape(vs.B, vs.gamma).to(torch.int32)
    u_acc = torch.rand((vs.B, vs.gamma), generator=_gen(device, seed, 63), device=device)
    u_smp = torch.rand((vs.B,), generator=_gen(device, seed, 64), device=device)
    return p_t, p_d, toks, u_acc, u_smp


@dataclasses.dataclass(frozen=True)
class LmHeadShape:
    """The draft's LM head and its soft-CE: N tokens, hidden size Hd, draft
    vocabulary V.  h ~ N(0, 1) and W ~ N(0, 1/Hd) in bf16 (logits of unit
    scale); the targets and g as the soft-CE workloads draw them."""
    N: int
    Hd: int
    V: int


# Llama-3.1-8B-shaped draft: hidden 4096, draft vocabulary 32000, 4096 tokens.
LM_HEAD = LmHeadShape(N=4096, Hd=4096, V=32000)


def lm_head_inputs(ls: LmHeadShape, device, seed: int):
    """h bf16 [N, Hd], W bf16 [V, Hd], p fp32 [N, V], g fp32 [N]."""
    h = randn_bf16((ls.N, ls.Hd), device, seed, 70)
    W = randn_bf16((ls.V, ls.Hd), device, seed, 71, std=1.0 / math.sqrt(ls.Hd))
    _, p, g = soft_ce_inputs(SoftCEShape(N=ls.N, V=ls.V), device, seed)
    return h, W, p, g
