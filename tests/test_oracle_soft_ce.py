"""Pins of the soft-CE oracle: hand-worked golden rows, the closed form
g*(pi - p), the hard-label special case (torch cross_entropy), finite
differences, invariants and the g = 0 convention.  Float64 on the CPU."""

import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import soft_ce as osc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(N, V, seed, sum_p_one=True):
    r = np.random.default_rng(seed)
    z = 2.0 * r.standard_normal((N, V))
    lg = 2.0 * r.standard_normal((N, V)) / 0.8
    p = np.exp(lg - lg.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    if not sum_p_one:
        p *= r.uniform(0.3, 1.7, size=(N, 1))
    g = r.binomial(1, 0.8, size=N) / N
    return z, p, g


def test_golden_hand_rows():
    rows, L = [], None
    for line in open(os.path.join(GOLDEN, "soft_ce_hand.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        vals = [float(x) for x in line.split()]
        if len(vals) == 1:
            L = vals[0]
        else:
            rows.append(vals)
    a = np.array(rows)
    z, p, g = a[:, 0:2], a[:, 2:4], a[:, 4]
    Lo, rl, grad = osc.soft_ce(z, p, g)
    np.testing.assert_allclose(rl, a[:, 5], rtol=0, atol=1e-14)
    np.testing.assert_allclose(grad, a[:, 6:8], rtol=0, atol=1e-14)
    assert abs(Lo - L) < 1e-14


def test_closed_form_when_p_sums_to_one():
    z, p, g = _rand(33, 57, 1)
    _, _, grad = osc.soft_ce(z, p, g)
    pi = np.exp(z - z.max(1, keepdims=True))
    pi /= pi.sum(1, keepdims=True)
    np.testing.assert_allclose(grad, g[:, None] * (pi - p), rtol=0, atol=1e-15)


def test_rows_sum_to_zero_any_p():
    z, p, g = _rand(20, 31, 2, sum_p_one=False)
    _, _, grad = osc.soft_ce(z, p, g)
    np.testing.assert_allclose(grad.sum(1), 0.0, atol=1e-15)


def test_shift_invariance():
    z, p, g = _rand(10, 40, 3, sum_p_one=False)
    a = osc.soft_ce(z, p, g)
    b = osc.soft_ce(z + 7.25, p, g)
    assert abs(a[0] - b[0]) < 1e-12
    np.testing.assert_allclose(a[1], b[1], atol=1e-12)
    np.testing.assert_allclose(a[2], b[2], atol=1e-15)


def test_uniform_logits():
    _, p, _ = _rand(6, 100, 4, sum_p_one=False)
    g = np.ones(6)
    _, rl, _ = osc.soft_ce(np.full((6, 100), 0.3), p, g)
    np.testing.assert_allclose(rl, np.log(100) * p.sum(1), rtol=1e-13)


def test_one_hot_is_weighted_cross_entropy():
    """EAGLE-3 trains with hard-label CE (SpecForge review, §四 EAGLE-3 训练损失):
    one-hot p must reduce to torch's cross_entropy, and the gradient to autograd's."""
    r = np.random.default_rng(5)
    N, V = 17, 23
    z = 2 * r.standard_normal((N, V))
    lab = r.integers(0, V, N)
    p = np.zeros((N, V))
    p[np.arange(N), lab] = 1.0
    g = r.binomial(1, 0.8, N) / N
    L, rl, grad = osc.soft_ce(z, p, g)
    zt = torch.tensor(z, requires_grad=True)
    ce = F.cross_entropy(zt, torch.tensor(lab), reduction="none")
    Lt = (ce * torch.tensor(g)).sum()
    Lt.backward()
    assert abs(L - Lt.item()) < 1e-12
    np.testing.assert_allclose(rl, np.where(g != 0, ce.detach().numpy(), 0.0), atol=1e-12)
    np.testing.assert_allclose(grad, zt.grad.numpy(), atol=1e-15)


def test_finite_differences():
    z, p, g = _rand(3, 7, 6, sum_p_one=False)
    g = np.array([0.5, 1.25, 2.0])
    _, _, grad = osc.soft_ce(z, p, g)
    eps = 1e-6
    num = np.zeros_like(z)
    for idx in np.ndindex(z.shape):
        a, b = z.copy(), z.copy()
        a[idx] += eps
        b[idx] -= eps
        num[idx] = (osc.soft_ce(a, p, g)[0] - osc.soft_ce(b, p, g)[0]) / (2 * eps)
    np.testing.assert_allclose(grad, num, rtol=1e-7, atol=1e-9)


def test_row_loops_agree():
    z, p, g = _rand(5, 13, 7, sum_p_one=False)
    g[1] = 0.0
    L, rl, grad = osc.soft_ce(z, p, g)
    for r in range(5):
        l_r, gr = osc.soft_ce_row(z[r], p[r], g[r])
        assert abs(l_r - rl[r]) < 1e-12
        np.testing.assert_allclose(gr, grad[r], atol=1e-15)


def test_masked_rows_are_exact_zero():
    z, p, g = _rand(8, 50, 8)
    g[[0, 3, 7]] = 0.0
    L, rl, grad = osc.soft_ce(z, p, g)
    assert np.all(grad[[0, 3, 7]] == 0.0) and np.all(rl[[0, 3, 7]] == 0.0)
    assert abs(L - (g * rl).sum()) < 1e-12


def test_planted_sign_slip_is_caught(monkeypatch):
    """Plant a sign slip (z <- p*g - pi*s) in the oracle: the closed-form pin fails."""
    z, p, g = _rand(4, 9, 9)
    good = osc.soft_ce(z, p, g)[2]
    pi = np.exp(z - z.max(1, keepdims=True))
    pi /= pi.sum(1, keepdims=True)
    np.testing.assert_allclose(good, g[:, None] * (pi - p), atol=1e-15)
    assert not np.allclose(-good, g[:, None] * (pi - p), atol=1e-6)


# ------------------------------------------------ per-element g (variant) --

def test_elementwise_golden_hand_rows():
    rows, L = [], None
    for line in open(os.path.join(GOLDEN, "soft_ce_elementwise_hand.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        vals = [float(x) for x in line.split()]
        if len(vals) == 1:
            L = vals[0]
        else:
            rows.append(vals)
    a = np.array(rows)
    Lo, rl, grad = osc.soft_ce_elementwise(a[:, 0:2], a[:, 2:4], a[:, 4:6])
    np.testing.assert_allclose(rl, a[:, 6], rtol=0, atol=1e-14)
    np.testing.assert_allclose(grad, a[:, 7:9], rtol=0, atol=1e-14)
    assert abs(Lo - L) < 1e-14


def test_elementwise_with_row_constant_g_is_the_per_row_form():
    z, p, g = _rand(17, 45, 8, sum_p_one=False)
    L1, rl1, gr1 = osc.soft_ce(z, p, g)
    L2, rl2, gr2 = osc.soft_ce_elementwise(z, p, np.repeat(g[:, None], 45, axis=1))
    assert abs(L1 - L2) <= 1e-13 * abs(L1)
    np.testing.assert_allclose(rl2, g * rl1, rtol=1e-13, atol=1e-16)
    np.testing.assert_allclose(gr2, gr1, rtol=0, atol=1e-15)


def test_elementwise_finite_differences():
    r = np.random.default_rng(9)
    z, p, _ = _rand(3, 7, 10, sum_p_one=False)
    G = r.uniform(0.0, 2.0, size=z.shape)
    _, _, grad = osc.soft_ce_elementwise(z, p, G)
    h = 1e-6
    num = np.zeros_like(z)
    for i in range(z.shape[0]):
        for j in range(z.shape[1]):
            zp, zm = z.copy(), z.copy()
            zp[i, j] += h
            zm[i, j] -= h
            num[i, j] = (osc.soft_ce_elementwise(zp, p, G)[0] - osc.soft_ce_elementwise(zm, p, G)[0]) / (2 * h)
    np.testing.assert_allclose(grad, num, rtol=1e-7, atol=1e-9)
    np.testing.assert_allclose(grad.sum(1), 0.0, atol=1e-14)


def test_elementwise_one_hot_is_cross_entropy_weighted_at_the_target():
    r = np.random.default_rng(11)
    N, V = 12, 30
    z = 2.0 * r.standard_normal((N, V))
    t = r.integers(0, V, size=N)
    p = np.zeros((N, V))
    p[np.arange(N), t] = 1.0
    G = r.uniform(0.0, 1.0, size=(N, V))
    L, rl, grad = osc.soft_ce_elementwise(z, p, G)
    zt = torch.tensor(z, requires_grad=True)
    ce = F.cross_entropy(zt, torch.tensor(t), reduction="none")
    w = torch.tensor(G[np.arange(N), t])
    (ce * w).sum().backward()
    np.testing.assert_allclose(rl, (ce * w).detach().numpy(), rtol=1e-12)
    assert abs(L - float((ce * w).sum())) <= 1e-12 * abs(L)
    np.testing.assert_allclose(grad, zt.grad.numpy(), rtol=0, atol=1e-14)
