"""Pins of the attention oracle: library special cases (SDPA), a row-by-row
explicit-key-set formulation with autograd, finite differences, invariants and
the degenerate T = 0 case.  All float64 on the CPU."""

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import attention as oa

RNG = np.random.default_rng(1234)


def _inputs(B, H, H_kv, Q, D, k, seed=0):
    r = np.random.default_rng(seed)
    q = r.standard_normal((B, H, Q, D))
    Ks = [r.standard_normal((B, H_kv, Q, D)) for _ in range(k + 1)]
    Vs = [r.standard_normal((B, H_kv, Q, D)) for _ in range(k + 1)]
    dO = r.standard_normal((B, H, Q, D))
    return q, Ks, Vs, dO


def _row_keys(q, T, Q, k):
    """Explicit key list of query q as (block, position) pairs: the structure the
    mask pins establish (causal prefix cut at T, one diagonal key per later block)."""
    if q < T:
        return [(0, c) for c in range(q + 1)] + [(j, q) for j in range(1, k + 1)]
    return [(0, c) for c in range(T)]


def _rowwise_torch(q, Ks, Vs, T, scale):
    """Independent torch formulation: per row, gather its keys, softmax, weighted sum."""
    B, H, Q, D = q.shape
    H_kv = Ks[0].shape[1]
    G = H // H_kv
    k = len(Ks) - 1
    O = torch.zeros_like(q)
    lse = torch.full((B, H, Q), -float("inf"), dtype=q.dtype)
    outs, lses = [], []
    for b in range(B):
        for h in range(H):
            g = h // G
            for i in range(Q):
                keys = _row_keys(i, int(T[b]), Q, k)
                if not keys:
                    outs.append(((b, h, i), torch.zeros(D, dtype=q.dtype), None))
                    continue
                Kset = torch.stack([Ks[j][b, g, c] for j, c in keys])
                Vset = torch.stack([Vs[j][b, g, c] for j, c in keys])
                s = scale * (Kset @ q[b, h, i])
                outs.append(((b, h, i), torch.softmax(s, 0) @ Vset, torch.logsumexp(s, 0)))
    O = torch.stack([o for _, o, _ in outs]).reshape(B, H, Q, D)
    lse = torch.stack([l if l is not None else torch.tensor(-float("inf"), dtype=q.dtype)
                       for _, _, l in outs]).reshape(B, H, Q)
    return O, lse


def _to_t(x, grad=False):
    t = torch.tensor(x, dtype=torch.float64)
    return t.requires_grad_(grad)


def test_k0_full_length_is_causal_sdpa():
    q, Ks, Vs, _ = _inputs(1, 3, 3, 17, 8, 0)
    scale = 0.37
    O, lse = oa.forward(q, Ks, Vs, [17], scale)
    ref = F.scaled_dot_product_attention(_to_t(q), _to_t(Ks[0]), _to_t(Vs[0]), is_causal=True,
                                         scale=scale)
    np.testing.assert_allclose(O, ref.numpy(), rtol=0, atol=1e-12)


@pytest.mark.parametrize("T", [1, 5, 11, 16])
def test_k0_padded_prefix_and_padded_rows(T):
    Q = 16
    q, Ks, Vs, _ = _inputs(1, 2, 1, Q, 8, 0, seed=T)
    scale = 1 / np.sqrt(8)
    O, lse = oa.forward(q, Ks, Vs, [T], scale)
    Kr = _to_t(Ks[0]).repeat_interleave(2, dim=1)
    Vr = _to_t(Vs[0]).repeat_interleave(2, dim=1)
    # valid rows: causal attention over the first T tokens (prefix property)
    pre = F.scaled_dot_product_attention(_to_t(q)[:, :, :T], Kr[:, :, :T], Vr[:, :, :T],
                                         is_causal=True, scale=scale)
    np.testing.assert_allclose(O[:, :, :T], pre.numpy(), rtol=0, atol=1e-12)
    # padded rows: plain (non-causal) attention over the T valid keys
    if T < Q:
        pad = F.scaled_dot_product_attention(_to_t(q)[:, :, T:], Kr[:, :, :T], Vr[:, :, :T],
                                             is_causal=False, scale=scale)
        np.testing.assert_allclose(O[:, :, T:], pad.numpy(), rtol=0, atol=1e-12)


@pytest.mark.parametrize("method", ["dense", "keyset"])
@pytest.mark.parametrize("T,k", [([6, 4], 2), ([0, 3], 1), ([6, 6], 3), ([1, 5], 0)])
def test_forward_matches_rowwise_gather(method, T, k):
    q, Ks, Vs, _ = _inputs(2, 4, 2, 6, 3, k, seed=sum(T) + k)
    scale = 0.9
    O, lse = oa.forward(q, Ks, Vs, T, scale, method=method)
    Or, lr = _rowwise_torch(_to_t(q), [_to_t(x) for x in Ks], [_to_t(x) for x in Vs], T, scale)
    np.testing.assert_allclose(O, Or.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lr.numpy(), rtol=0, atol=1e-12)


@pytest.mark.parametrize("T,k", [([6, 4], 2), ([0, 3], 1), ([6, 6], 3), ([2, 5], 0)])
def test_backward_matches_autograd_of_rowwise(T, k):
    q, Ks, Vs, dO = _inputs(2, 4, 2, 6, 3, k, seed=7 + k)
    scale = 0.8
    dq, dK, dV = oa.backward(q, Ks, Vs, T, scale, dO)
    qt = _to_t(q, True)
    Kt = [_to_t(x, True) for x in Ks]
    Vt = [_to_t(x, True) for x in Vs]
    Or, _ = _rowwise_torch(qt, Kt, Vt, T, scale)
    (Or * _to_t(dO)).sum().backward()
    np.testing.assert_allclose(dq, qt.grad.numpy(), rtol=0, atol=1e-12)
    for j in range(k + 1):
        np.testing.assert_allclose(dK[j], Kt[j].grad.numpy(), rtol=0, atol=1e-12)
        np.testing.assert_allclose(dV[j], Vt[j].grad.numpy(), rtol=0, atol=1e-12)


@pytest.mark.parametrize("T,Q,k,D", [([37, 64], 64, 3, 16), ([0, 20], 20, 2, 8), ([50], 50, 5, 4),
                                     ([129], 130, 1, 32)])
def test_keyset_equals_dense(T, Q, k, D):
    B = len(T)
    q, Ks, Vs, dO = _inputs(B, 4, 2, Q, D, k, seed=Q + k)
    scale = 1 / np.sqrt(D)
    Od, ld = oa.forward(q, Ks, Vs, T, scale, method="dense")
    Ok, lk = oa.forward(q, Ks, Vs, T, scale, method="keyset")
    np.testing.assert_allclose(Ok, Od, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lk, ld, rtol=0, atol=1e-12)
    gd = oa.backward(q, Ks, Vs, T, scale, dO, method="dense")
    gk = oa.backward(q, Ks, Vs, T, scale, dO, method="keyset")
    np.testing.assert_allclose(gk[0], gd[0], rtol=0, atol=1e-12)
    for j in range(k + 1):
        np.testing.assert_allclose(gk[1][j], gd[1][j], rtol=0, atol=1e-12)
        np.testing.assert_allclose(gk[2][j], gd[2][j], rtol=0, atol=1e-12)


def test_finite_differences():
    """d sum(O*dO) / d{q, K_j, V_j} by central differences vs the direct backward."""
    T, k, Q, D = [5], 2, 6, 3
    q, Ks, Vs, dO = _inputs(1, 2, 1, Q, D, k, seed=99)
    scale = 0.7
    dq, dK, dV = oa.backward(q, Ks, Vs, T, scale, dO)

    def f(q_, Ks_, Vs_):
        O, _ = oa.forward(q_, Ks_, Vs_, T, scale)
        return float((O * dO).sum())

    eps = 1e-6

    def fd(arr, setter):
        out = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            a1, a2 = arr.copy(), arr.copy()
            a1[idx] += eps
            a2[idx] -= eps
            out[idx] = (setter(a1) - setter(a2)) / (2 * eps)
        return out

    num = fd(q, lambda a: f(a, Ks, Vs))
    np.testing.assert_allclose(dq, num, rtol=1e-6, atol=1e-8)
    for j in range(k + 1):
        numK = fd(Ks[j], lambda a: f(q, Ks[:j] + [a] + Ks[j + 1:], Vs))
        numV = fd(Vs[j], lambda a: f(q, Ks, Vs[:j] + [a] + Vs[j + 1:]))
        np.testing.assert_allclose(dK[j], numK, rtol=1e-6, atol=1e-8)
        np.testing.assert_allclose(dV[j], numV, rtol=1e-6, atol=1e-8)


def test_invariants():
    T, k, Q, D = [9, 12], 3, 12, 5
    q, Ks, Vs, dO = _inputs(2, 2, 1, Q, D, k, seed=5)
    scale = 0.5
    O, lse = oa.forward(q, Ks, Vs, T, scale)
    from oracle import mask as om
    for b in range(2):
        M = om.mask_matrix(T[b], Q, k)
        Kc = np.concatenate([x[b, 0] for x in Ks])
        Vc = np.concatenate([x[b, 0] for x in Vs])
        for h in range(2):
            S = scale * q[b, h] @ Kc.T
            P = np.where(M, np.exp(S - lse[b, h][:, None]), 0.0)
            np.testing.assert_allclose(P.sum(1), 1.0, rtol=0, atol=1e-12)   # sum_kv P = 1
            dP = dO[b, h] @ Vc.T
            dS = P * (dP - (dO[b, h] * O[b, h]).sum(1)[:, None])
            np.testing.assert_allclose(dS.sum(1), 0.0, rtol=0, atol=1e-12)  # sum_kv dS = 0
            for i in range(Q):                                              # convex hull
                att = Vc[M[i]]
                assert np.all(O[b, h, i] <= att.max(0) + 1e-12)
                assert np.all(O[b, h, i] >= att.min(0) - 1e-12)


def test_empty_rows_T0():
    q, Ks, Vs, dO = _inputs(1, 2, 1, 5, 4, 2, seed=3)
    O, lse = oa.forward(q, Ks, Vs, [0], 0.5)
    assert np.all(O == 0) and np.all(np.isneginf(lse))
    dq, dK, dV = oa.backward(q, Ks, Vs, [0], 0.5, dO)
    assert np.all(dq == 0) and all(np.all(x == 0) for x in dK + dV)


def test_gqa_mapping_matches_repeat_interleave():
    q, Ks, Vs, _ = _inputs(1, 6, 2, 9, 4, 0, seed=11)
    O, _ = oa.forward(q, Ks, Vs, [9], 0.5)
    ref = F.scaled_dot_product_attention(_to_t(q), _to_t(Ks[0]).repeat_interleave(3, 1),
                                         _to_t(Vs[0]).repeat_interleave(3, 1), is_causal=True,
                                         scale=0.5)
    np.testing.assert_allclose(O, ref.numpy(), rtol=0, atol=1e-12)


def test_planted_dropped_delta_is_caught(monkeypatch):
    """Plant a plausible slip in the oracle (the Delta term of dS dropped): the
    autograd pin's comparison must then fail."""
    T, k = [5], 1
    q, Ks, Vs, dO = _inputs(1, 2, 1, 6, 3, k, seed=21)
    orig = oa.head_backward_dense

    def no_delta(q_, Kc, Vc, M, scale, dO_, O=None, lse=None):
        O_, lse_ = oa.head_forward_dense(q_, Kc, Vc, M, scale)
        return orig(q_, Kc, Vc, M, scale, dO_, np.zeros_like(O_), lse_)
    monkeypatch.setattr(oa, "head_backward_dense", no_delta)
    dq, dK, dV = oa.backward(q, Ks, Vs, T, 0.6, dO)
    qt = _to_t(q, True)
    Or, _ = _rowwise_torch(qt, [_to_t(x) for x in Ks], [_to_t(x) for x in Vs], T, 0.6)
    (Or * _to_t(dO)).sum().backward()
    assert not np.allclose(dq, qt.grad.numpy(), atol=1e-6)
