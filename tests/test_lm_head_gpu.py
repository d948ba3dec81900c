"""GPU parity of the fused LM head + soft-CE (stt_lm_head_ce) against the
fp64 oracle (z = h W^T, soft-CE, dh = dz W, dW = dz^T h).

Bounds, from the arithmetic: z is a sum of exact bf16 x bf16 products in
fp32, so the loss and per-row losses hold to relative 1e-5 (the soft-CE's
bound).  dL/dz enters the two gradient products rounded to bf16: bf16 keeps 8
significant bits, so each element moves by at most 2^-8 of its magnitude, and
an element of dh = dz W moves by at most 2^-8 sum_v |dz_rv| |W_vd| (dW
likewise with h); the bound is that sum plus 1e-5 of the largest reference
entry for the fp32 sums."""

import numpy as np
import pytest
import torch

import _parity
from oracle import lm_head as olh
from speculative_decoding_draft_eagle_gb300 import ops, workloads as wl

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from speculative_decoding_draft_eagle_gb300 import build
    build.build()


def _run_and_check(ls, seed, zero_rows=True, tag=""):
    h, W, p, g = wl.lm_head_inputs(ls, DEV, seed)
    if zero_rows:
        g[:3] = 0.0
    loss, rl, dh, dW = ops.stt_lm_head_ce(h, W, p, g)
    torch.cuda.synchronize()
    assert ops.stt_device_error() == 0
    hf = h.double().cpu().numpy()
    Wf = W.double().cpu().numpy()
    pf = p.double().cpu().numpy()
    gf = g.double().cpu().numpy()
    del p
    L, rlr, dhr, dWr = olh.lm_head_soft_ce(hf, Wf, pf, gf)
    # the rounding bound needs |dz|: the oracle's soft-CE of the same logits
    from oracle import soft_ce as osc
    _, _, dz = osc.soft_ce(hf @ Wf.T, pf, gf)
    del pf
    adz = np.abs(dz)
    del dz
    bdh = 2.0 ** -8 * (adz @ np.abs(Wf)) + 1e-5 * np.abs(dhr).max()
    bdW = 2.0 ** -8 * (adz.T @ np.abs(hf)) + 1e-5 * np.abs(dWr).max()
    grp = "lm head + soft-CE"
    for name, gpu, ref, b in (("dh", dh, dhr, bdh), ("dW", dW, dWr, bdW)):
        d = np.abs(gpu.double().cpu().numpy() - ref)
        worst = float((d / b).max())
        _parity.record(grp, f"{name}[{tag}] (elementwise |err| / bound)", worst, 1.0, 0.0, 1.0)
        assert worst <= 1.0, f"{name}[{tag}]: worst elementwise error is {worst:.3g} of its bound"
        _parity.close(gpu.double().cpu().numpy(), ref, f"{name}[{tag}]", atol=float(b.max()),
                      rtol_l2=2.0 ** -8, group=grp)
    np.testing.assert_allclose(rl.cpu().numpy(), rlr, rtol=1e-5, atol=1e-6)
    assert abs(loss.item() - L) <= 1e-5 * abs(L)
    assert np.all(rl.cpu().numpy()[gf == 0] == 0.0)


@pytest.mark.parametrize("N,Hd,V", [(128, 64, 256), (200, 136, 1000), (300, 512, 9000),
                                    (64, 256, 16), (5, 8, 24), (257, 192, 16392)])
def test_shapes(N, Hd, V):
    """Ragged rows, a hidden size that is not a multiple of 64, vocabularies of
    one tile, ragged tiles and several gradient chunks (8192 columns each)."""
    _run_and_check(wl.LmHeadShape(N=N, Hd=Hd, V=V), 40 + N + V, tag=f"{N}x{Hd}x{V}")


def test_llama8b_draft_shape():
    """N 4096 tokens, hidden 4096, draft vocabulary 32000 (four chunks)."""
    _run_and_check(wl.LM_HEAD, 1002, tag="4096x4096x32000")


def test_empty_batch():
    h = torch.zeros((0, 64), device=DEV, dtype=torch.bfloat16)
    W = torch.ones((16, 64), device=DEV, dtype=torch.bfloat16)
    loss, rl, dh, dW = ops.stt_lm_head_ce(h, W, torch.zeros((0, 16), device=DEV),
                                          torch.zeros(0, device=DEV))
    torch.cuda.synchronize()
    assert loss.item() == 0.0
