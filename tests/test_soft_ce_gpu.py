"""GPU parity of the in-place soft-CE kernel against the fp64 oracle.

Tolerances (fp32 arithmetic): |dL| <= 1e-5 |L|; per gradient tensor relative
L2 <= 1e-5 and max-abs <= 1e-5 * max|ref|; per-row loss within 1e-5 relative
(+1e-6 absolute).  Element-wise relative error is not used for the gradient
because p*g and pi*s cancel where the target and the softmax agree.
"""

import numpy as np
import pytest
import torch

from oracle import soft_ce as osc
from speculative_decoding_draft_eagle_gb300 import ops, workloads as wl

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from speculative_decoding_draft_eagle_gb300 import build
    build.build()


def _check(z0, p, g, z_out, L_gpu, rl_gpu, rows=None):
    """Compare against the oracle; rows optionally restricts the compared rows
    (the loss is then not compared)."""
    if rows is not None:
        z0, p, g, z_out, rl_gpu = z0[rows], p[rows], g[rows], z_out[rows], rl_gpu[rows]
    L, rl, grad = osc.soft_ce(z0, p, g)
    d = z_out.astype(np.float64) - grad
    assert np.linalg.norm(d) <= 1e-5 * np.linalg.norm(grad) + 1e-30
    assert np.abs(d).max() <= 1e-5 * np.abs(grad).max() + 1e-30
    np.testing.assert_allclose(rl_gpu, rl, rtol=1e-5, atol=1e-6)
    if rows is None:
        assert abs(L_gpu - L) <= 1e-5 * abs(L) + 1e-12
    # masked rows: exact zeros
    assert np.all(z_out[g == 0] == 0.0)


def _run(z, p, g):
    zd = z.to(DEV).contiguous()
    loss, rl = ops.soft_ce_fwd_bwd_inplace(zd, p.to(DEV).contiguous(), g.to(DEV).contiguous())
    torch.cuda.synchronize()
    assert ops.stt_device_error() == 0
    return zd.cpu().numpy(), float(loss.item()), rl.cpu().numpy()


def test_tiny_workload_full():
    w = wl.WORKLOADS["tiny"]
    z, p, g = wl.soft_ce_inputs(w.soft_ce, "cpu", w.seed)
    zo, L, rl = _run(z, p, g)
    _check(z.numpy(), p.numpy(), g.numpy(), zo, L, rl)


@pytest.mark.parametrize("N,V", [(1, 1), (3, 2), (5, 7), (9, 1001), (16, 4), (4, 4096 * 3 + 4),
                                 (33, 32000), (7, 151936), (2, 409600), (64, 16383),
                                 (6, 81920 // 8 * 2 + 4)])
def test_shapes(N, V):
    """Ragged V (element-wise path), one-CTA rows, cluster splits up to 16 CTAs."""
    sc = wl.SoftCEShape(N=N, V=V)
    z, p, g = wl.soft_ce_inputs(sc, "cpu", 7 + N + V)
    g[0] = 0.0
    zo, L, rl = _run(z, p, g)
    _check(z.numpy(), p.numpy(), g.numpy(), zo, L, rl)


def test_unaligned_rows_take_elementwise_path():
    sc = wl.SoftCEShape(N=8, V=1000)
    z, p, g = wl.soft_ce_inputs(sc, "cpu", 3)
    zbig = torch.zeros(8 * 1000 + 1)
    zbig[1:] = z.reshape(-1)
    zd = zbig.to(DEV)[1:].view(8, 1000)    # 4-byte offset: not 16-byte aligned
    pd = p.to(DEV)
    loss, rl = ops.soft_ce_fwd_bwd_inplace(zd, pd, g.to(DEV))
    torch.cuda.synchronize()
    _check(z.numpy(), p.numpy(), g.numpy(), zd.cpu().numpy(), loss.item(), rl.cpu().numpy())


def test_empty_batch():
    z = torch.zeros((0, 10), device=DEV)
    loss, rl = ops.soft_ce_fwd_bwd_inplace(z, torch.zeros_like(z), torch.zeros(0, device=DEV))
    torch.cuda.synchronize()
    assert loss.item() == 0.0


def test_p_not_normalised_and_one_hot():
    sc = wl.SoftCEShape(N=64, V=5000, one_hot_frac=0.25)
    z, p, g = wl.soft_ce_inputs(sc, "cpu", 11)
    p[:10] *= 1.7
    zo, L, rl = _run(z, p, g)
    _check(z.numpy(), p.numpy(), g.numpy(), zo, L, rl)


@pytest.mark.parametrize("name", ["llama8b", "varlen", "llama70b", "long_ttt"])
def test_full_size_workloads(name):
    """Each workload at full size, generated on the GPU; every row compared
    (varlen: the loss plus every 4th row, to bound host memory)."""
    w = wl.WORKLOADS[name]
    T = wl.draw_T(w.attn, w.seed)
    z, p, g = wl.soft_ce_inputs(w.soft_ce, DEV, w.seed, T=T, Q_LEN=w.attn.Q_LEN)
    z_host = z.cpu().numpy()
    loss, rl = ops.soft_ce_fwd_bwd_inplace(z, p, g)
    torch.cuda.synchronize()
    assert ops.stt_device_error() == 0
    N = z.shape[0]
    step = 4 if N > 16384 else 1
    rows = np.arange(0, N, step)
    p_host = p[torch.from_numpy(rows).to(DEV)].cpu().numpy()
    g_host = g.cpu().numpy()
    zo = z[torch.from_numpy(rows).to(DEV)].cpu().numpy()
    assert np.all(zo[g_host[rows] == 0] == 0.0)
    Lr, rlr, grad = osc.soft_ce(z_host[rows], p_host, g_host[rows])
    d = zo.astype(np.float64) - grad
    assert np.linalg.norm(d) <= 1e-5 * np.linalg.norm(grad)
    assert np.abs(d).max() <= 1e-5 * np.abs(grad).max()
    np.testing.assert_allclose(rl.cpu().numpy()[rows], rlr, rtol=1e-5, atol=1e-6)
    # scalar loss against the oracle over all rows (row losses are exact per row)
    if step == 1:
        assert abs(loss.item() - Lr) <= 1e-5 * abs(Lr)
    else:
        L_all = 0.0
        for r0 in range(0, N, 2048):
            idx = torch.arange(r0, min(N, r0 + 2048), device=DEV)
            L_all += osc.soft_ce(z_host[r0:r0 + 2048], p[idx].cpu().numpy(), g_host[r0:r0 + 2048])[0]
        assert abs(loss.item() - L_all) <= 1e-5 * abs(L_all)
