"""Pins of the LM-head + soft-CE oracle (no GPU): finite differences of the
loss in h and W, and autograd of an independent torch formulation
(F.linear, log_softmax and the weighted soft-target sum)."""

import numpy as np
import torch
import torch.nn.functional as F

from oracle import lm_head as olh


def _inputs(N, Hd, V, seed):
    r = np.random.default_rng(seed)
    h = r.standard_normal((N, Hd))
    W = r.standard_normal((V, Hd)) / np.sqrt(Hd)
    lg = 2.0 * r.standard_normal((N, V)) / 0.8
    p = np.exp(lg - lg.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    g = r.binomial(1, 0.8, size=N) / N
    return h, W, p, g


def test_matches_torch_autograd():
    h, W, p, g = _inputs(7, 12, 9, 1)
    L, rl, dh, dW = olh.lm_head_soft_ce(h, W, p, g)
    ht = torch.tensor(h, requires_grad=True)
    Wt = torch.tensor(W, requires_grad=True)
    logp = F.log_softmax(F.linear(ht, Wt), dim=1)
    ell = -(torch.tensor(p) * logp).sum(1)
    gt = torch.tensor(g)
    Lt = (gt * ell).sum()
    Lt.backward()
    assert abs(L - float(Lt)) <= 1e-13 * abs(L)
    np.testing.assert_allclose(rl, np.where(g != 0, ell.detach().numpy(), 0.0), rtol=1e-13)
    np.testing.assert_allclose(dh, ht.grad.numpy(), rtol=0, atol=1e-14)
    np.testing.assert_allclose(dW, Wt.grad.numpy(), rtol=0, atol=1e-14)


def test_finite_differences():
    h, W, p, g = _inputs(3, 5, 4, 2)
    _, _, dh, dW = olh.lm_head_soft_ce(h, W, p, g)
    eps = 1e-6

    def num(x, which):
        out = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            a = olh.lm_head_soft_ce(xp, W, p, g)[0] if which == "h" else olh.lm_head_soft_ce(h, xp, p, g)[0]
            b = olh.lm_head_soft_ce(xm, W, p, g)[0] if which == "h" else olh.lm_head_soft_ce(h, xm, p, g)[0]
            out[idx] = (a - b) / (2 * eps)
        return out

    np.testing.assert_allclose(dh, num(h, "h"), rtol=1e-6, atol=1e-10)
    np.testing.assert_allclose(dW, num(W, "W"), rtol=1e-6, atol=1e-10)
