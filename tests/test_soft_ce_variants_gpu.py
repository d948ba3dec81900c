"""GPU parity of the soft-CE variants (soft_ce_fwd_bwd_inplace_ex) against
the fp64 oracle: bf16 logits and targets, and a per-element upstream
gradient G.

Bounds: the loss and the per-row losses within 1e-5 relative (fp32 sums over
inputs both sides read identically).  The gradient: fp32 output, relative L2
and max-abs within 1e-5 (of max|ref|) as for the fp32 kernel; bf16 output,
one rounding of every stored value on top: bf16 keeps 8 significant bits,
so rounding to nearest moves a value by at most 2^-8 of its magnitude, i.e.
max-abs within (2^-8 + 1e-5) max|ref| and relative L2 within 2^-8 + 1e-5.
"""

import numpy as np
import pytest
import torch

import _parity
from oracle import soft_ce as osc
from speculative_decoding_draft_eagle_gb300 import ops, workloads as wl

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from speculative_decoding_draft_eagle_gb300 import build
    build.build()


def _inputs(N, V, seed, bf16, gel, one_hot=0.0):
    z, p, g = wl.soft_ce_inputs(wl.SoftCEShape(N=N, V=V, one_hot_frac=one_hot), "cpu", seed)
    if bf16:
        z, p = z.to(torch.bfloat16), p.to(torch.bfloat16)
    if gel:
        gen = torch.Generator().manual_seed(seed + 1)
        G = (torch.rand((N, V), generator=gen) < 0.7).float() * torch.rand((N, V), generator=gen) / N
        G[0] = 0.0
        return z, p, G
    g[0] = 0.0
    return z, p, g


def _check(z, p, g, zo, L, rl, bf16, gel, tag):
    zf = z.double().numpy()
    pf = p.double().numpy()
    gf = g.double().numpy()
    if gel:
        Lr, rlr, grad = osc.soft_ce_elementwise(zf, pf, gf)
    else:
        Lr, rlr, grad = osc.soft_ce(zf, pf, gf)
    out = zo.double().numpy()
    mx = float(np.abs(grad).max())
    if bf16:
        atol, rtol = (2.0 ** -8 + 1e-5) * mx, 2.0 ** -8 + 1e-5
    else:
        atol, rtol = 1e-5 * mx, 1e-5
    _parity.close(out, grad, f"grad[{tag}]", atol=atol + 1e-30, rtol_l2=rtol, group="soft-CE variants")
    np.testing.assert_allclose(rl, rlr, rtol=1e-5, atol=1e-6)
    assert abs(L - Lr) <= 1e-5 * abs(Lr) + 1e-12
    if not gel:
        assert np.all(out[gf == 0] == 0.0)


@pytest.mark.parametrize("bf16,gel", [(True, False), (False, True), (True, True)])
@pytest.mark.parametrize("N,V", [(1, 8), (5, 1000), (9, 4096), (33, 32000), (4, 151936), (3, 1001)])
def test_variants(N, V, bf16, gel):
    z, p, g = _inputs(N, V, 100 + N + V, bf16, gel)
    zd = z.to(DEV)
    loss, rl = ops.soft_ce_fwd_bwd_inplace_ex(zd, p.to(DEV), g.to(DEV))
    torch.cuda.synchronize()
    assert ops.stt_device_error() == 0
    _check(z, p, g, zd.cpu(), loss.item(), rl.cpu().numpy(), bf16, gel, f"{N}x{V},bf16={bf16},gel={gel}")


def test_variant_flags_zero_is_the_fp32_path():
    z, p, g = _inputs(16, 2048, 5, False, False)
    zd = z.to(DEV)
    loss, rl = ops.soft_ce_fwd_bwd_inplace_ex(zd, p.to(DEV), g.to(DEV))
    torch.cuda.synchronize()
    _check(z, p, g, zd.cpu(), loss.item(), rl.cpu().numpy(), False, False, "fp32 via ex")


def test_bf16_unaligned_rows():
    """A 2-byte offset: no bulk copies, element-wise path, same results."""
    N, V = 6, 1000
    z, p, g = _inputs(N, V, 7, True, False)
    big = torch.zeros(N * V + 1, dtype=torch.bfloat16)
    big[1:] = z.reshape(-1)
    zd = big.to(DEV)[1:].view(N, V)
    loss, rl = ops.soft_ce_fwd_bwd_inplace_ex(zd, p.to(DEV), g.to(DEV))
    torch.cuda.synchronize()
    _check(z, p, g, zd.cpu(), loss.item(), rl.cpu().numpy(), True, False, "bf16 unaligned")


def test_llama8b_sized_bf16_and_per_element():
    """N 4096, V 32000 (the Llama-8B draft's soft-CE), one-hot rows mixed in."""
    for bf16, gel in [(True, False), (False, True)]:
        z, p, g = _inputs(4096, 32000, 31, bf16, gel, one_hot=0.25)
        zd = z.to(DEV)
        loss, rl = ops.soft_ce_fwd_bwd_inplace_ex(zd, p.to(DEV), g.to(DEV))
        torch.cuda.synchronize()
        assert ops.stt_device_error() == 0
        _check(z, p, g, zd.cpu(), loss.item(), rl.cpu().numpy(), bf16, gel,
               f"4096x32000,bf16={bf16},gel={gel}")
