"""The allocation-free soft-CE entry point, called through the C ABI.

Some callers cannot allocate device memory at all: an operator hosted by a
framework that passes it only its input and output buffers and keeps every
device allocation to itself, or code running in a phase where cudaMalloc is
not allowed.  `soft_ce_fwd_bwd_inplace_noalloc` serves them with the library's
own fixed scratch array instead of a caller workspace.  This test checks that
two calls in a row (the second smaller than the first, so leftovers of the
first sit in the shared scratch) give the same loss, per-row loss and gradient
as the regular workspace entry point, within the soft-CE tolerance used
elsewhere (relative 1e-5).  It is collected last and also passes alone in a
fresh process.
"""

import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _run_regular(L, z, p, g):
    N, V = z.shape
    zz = z.clone()
    rl = torch.empty(N, device=z.device)
    loss = torch.empty(1, device=z.device)
    ws = torch.empty(L.soft_ce_workspace_size(N, V), dtype=torch.uint8, device=z.device)
    st = L.soft_ce_fwd_bwd_inplace(zz.data_ptr(), p.data_ptr(), g.data_ptr(), N, V, rl.data_ptr(),
                                   loss.data_ptr(), ws.data_ptr(), ws.numel(),
                                   ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    return zz, rl, loss


def _run_noalloc(L, z, p, g):
    N, V = z.shape
    zz = z.clone()
    rl = torch.empty(N, device=z.device)
    loss = torch.empty(1, device=z.device)
    st = L.soft_ce_fwd_bwd_inplace_noalloc(zz.data_ptr(), p.data_ptr(), g.data_ptr(), N, V,
                                           rl.data_ptr(), loss.data_ptr(),
                                           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    return zz, rl, loss


def _same(a, b):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    assert np.linalg.norm(a - b) <= 1e-5 * np.linalg.norm(b) + 1e-30
    assert np.abs(a - b).max() <= 1e-5 * np.abs(b).max() + 1e-30


def test_noalloc_matches_workspace_entry_point_twice():
    from oracle import soft_ce as osc
    from speculative_decoding_draft_eagle_gb300 import _lib, build, workloads as wl
    build.build()
    L = _lib.lib()
    torch.cuda.init()
    for N, V, seed in [(3000, 32000, 1), (700, 1001, 2)]:
        z, p, g = wl.soft_ce_inputs(wl.SoftCEShape(N=N, V=V), "cuda", seed)
        g[::5] = 0.0
        z1, r1, l1 = _run_regular(L, z, p, g)
        z2, r2, l2 = _run_noalloc(L, z, p, g)
        torch.cuda.synchronize()
        _same(z2, z1)
        _same(r2, r1)
        assert abs(l2.item() - l1.item()) <= 1e-5 * abs(l1.item())
        # and against the fp64 oracle directly, so that a fault shared by both
        # entry points would not pass unseen
        Lr, rlr, gr = osc.soft_ce(z.cpu().numpy(), p.cpu().numpy(), g.cpu().numpy())
        _same(z2, torch.from_numpy(gr))
        _same(r2, torch.from_numpy(rlr))
        assert abs(l2.item() - Lr) <= 1e-5 * abs(Lr)


def test_noalloc_rejects_too_many_rows():
    from speculative_decoding_draft_eagle_gb300 import _lib, build
    build.build()
    L = _lib.lib()
    z = torch.zeros((65537, 4), device="cuda")
    st = L.soft_ce_fwd_bwd_inplace_noalloc(z.data_ptr(), z.data_ptr(), z[:, 0].contiguous().data_ptr(),
                                           65537, 4, None, z.data_ptr(), None)
    assert st == -6  # STT_ERR_WORKSPACE: the fixed scratch holds at most 65536 rows
