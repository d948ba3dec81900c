"""GPU parity of the rejection-sampling verifier (stt_verify) against the
oracle: integer outputs, compared exactly.  The draw at a rejection is an
inverse-CDF search over fp64 running sums; the GPU sums in a different order
than the oracle, so where the threshold lies within 1e-12 of the total from a
boundary of the oracle's running sums, either neighbouring token is accepted
(none of the seeded cases does)."""

import numpy as np
import pytest
import torch

from oracle import verify as ov
from speculative_decoding_draft_eagle_gb300 import ops, workloads as wl

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from speculative_decoding_draft_eagle_gb300 import build
    build.build()


def _compare(p_t, p_d, toks, ua, us):
    n_g, out_g = ops.stt_verify(p_t.to(DEV), p_d.to(DEV), toks.to(DEV), ua.to(DEV), us.to(DEV))
    torch.cuda.synchronize()
    n_g, out_g = n_g.cpu().numpy(), out_g.cpu().numpy()
    pt, pd = p_t.double().numpy(), p_d.double().numpy()
    n_r, out_r = ov.verify(pt, pd, toks.numpy(), ua.double().numpy(), us.double().numpy())
    assert np.array_equal(n_g, n_r), (n_g, n_r)
    for b in range(len(n_r)):
        if np.array_equal(out_g[b], out_r[b]):
            continue
        r = int(n_r[b])
        assert r < toks.shape[1] and np.array_equal(out_g[b, :r], out_r[b, :r])
        w = np.maximum(0.0, pt[b, r] - pd[b, r])
        if w.sum() == 0:
            w = pt[b, r]
        c = np.cumsum(w)
        t = float(us[b]) * c[-1]
        y = int(out_g[b, r])
        near = min(abs(c[y] - t), abs((c[y - 1] if y > 0 else 0.0) - t))
        assert w[y] > 0 and near <= 1e-12 * c[-1], (b, y, out_r[b, r])
    return n_g


@pytest.mark.parametrize("B,gamma,V", [(1, 1, 1), (4, 5, 7), (64, 5, 1000), (32, 5, 32000),
                                       (16, 3, 151936), (8, 32, 4096), (5, 5, 1001)])
def test_random(B, gamma, V):
    p_t, p_d, toks, ua, us = wl.verify_inputs(wl.VerifyShape(B=B, gamma=gamma, V=V), "cpu",
                                              11 + B + V)
    _compare(p_t, p_d, toks, ua, us)


def test_forced_rejections_and_edge_cases():
    B, gamma, V = 12, 4, 3000
    p_t, p_d, toks, ua, us = wl.verify_inputs(wl.VerifyShape(B=B, gamma=gamma, V=V, noise=3.0),
                                              "cpu", 5)
    ua[:4] = 0.999999          # rejections wherever p_t < p_d at the token
    us[0], us[1] = 0.0, 0.9999999
    p_d[2] = p_t[2]            # identical distributions: every token accepted
    p_t[3] = 0.5 * p_d[3]      # residual all zero at a rejection: drawn from p_t
    toks[4, 1] = V + 5         # a token outside the vocabulary: rejected
    toks[5, 0] = -1
    n = _compare(p_t, p_d, toks, ua, us)
    assert n[2] == gamma and n[4] <= 1 and n[5] == 0


def test_full_size_workload():
    """B 64, gamma 5, V 151936 (the benchmark's verification workload)."""
    p_t, p_d, toks, ua, us = wl.verify_inputs(wl.VERIFY, DEV, 1006)
    n = _compare(p_t.cpu(), p_d.cpu(), toks.cpu(), ua.cpu(), us.cpu())
    assert 0 < n.mean() < wl.VERIFY.gamma   # both outcomes occur
