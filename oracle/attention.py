"""Sparse-tree TTT attention, forward and backward (oracle; test infrastructure).

What is computed (SpecForge review, §三 "稀疏树注意力": FlexAttention over the
concatenated per-step KV blocks under the BlockMask M of §四 "BlockMask 构造"):

    Kc = concat(K_0, ..., K_k)            [(k+1)*Q_LEN, D]   (per batch b, KV head)
    Vc = concat(V_0, ..., V_k)
    S  = scale * q @ Kc^T,  S[~M] = -inf
    lse = log sum_kv exp(S)               (natural log)
    P  = exp(S - lse),  O = P @ Vc

The backward is the gradient of sum(O * dO) (the page trains through this
attention but never writes its backward; it is the derivative of the
definition above):

    Delta = rowsum(dO * O)
    dP = dO @ Vc^T,  dS = P * (dP - Delta)
    dq = scale * dS @ Kc,  dKc = scale * dS^T @ q,  dVc = P^T @ dO

Query head h reads KV head h // (H / H_kv); dK and dV of a KV head sum the
contributions of all its query heads.  A row whose mask is empty (T = 0) has
O = 0, lse = -inf and no gradient.

Two formulations are given:
  * ``dense``  materialises M over all (k+1)*Q_LEN keys from the formula.  It
    is the literal definition and is used at small sizes.
  * ``keyset`` evaluates the formula on block 0 only and takes the later-block
    keys from ``mask.suffix_keys`` (one diagonal key per later block for each
    query q < T).  It costs O(Q_LEN^2) instead of O(k*Q_LEN^2) and is used at
    full sizes; tests show it equal to ``dense`` to 1e-12.
All arithmetic is float64.
"""

import numpy as np

from . import mask as _mask

_CHUNK_ELEMS = 1 << 22  # score entries per row chunk (32 MiB of float64)


def _f64(x):
    return np.asarray(x, dtype=np.float64)


def _softmax_rows(S):
    """Row-wise lse and P of a score matrix that may hold -inf (masked)."""
    m = S.max(axis=1)
    empty = ~np.isfinite(m)
    m_safe = np.where(empty, 0.0, m)
    with np.errstate(invalid="ignore"):
        E = np.exp(S - m_safe[:, None])
    E[~np.isfinite(S)] = 0.0
    l = E.sum(axis=1)
    with np.errstate(divide="ignore"):
        lse = np.where(empty, -np.inf, m_safe + np.log(np.where(empty, 1.0, l)))
    P = np.where(empty[:, None], 0.0, E / np.where(empty, 1.0, l)[:, None])
    return lse, P


# ---------------------------------------------------------------------------
# dense formulation: one (query head, KV head) pair, all keys, mask from M
# ---------------------------------------------------------------------------

def head_forward_dense(q, Kc, Vc, M, scale):
    """O [Q, D] and lse [Q] for one head.  q [Q,D]; Kc, Vc [KV,D]; M [Q,KV] bool."""
    q, Kc, Vc = _f64(q), _f64(Kc), _f64(Vc)
    Q = q.shape[0]
    O = np.zeros((Q, Vc.shape[1]))
    lse = np.empty(Q)
    step = max(1, _CHUNK_ELEMS // max(1, Kc.shape[0]))
    for r0 in range(0, Q, step):
        r1 = min(Q, r0 + step)
        S = scale * (q[r0:r1] @ Kc.T)
        S[~M[r0:r1]] = -np.inf
        lse[r0:r1], P = _softmax_rows(S)
        O[r0:r1] = P @ Vc
    return O, lse


def head_backward_dense(q, Kc, Vc, M, scale, dO, O=None, lse=None):
    """dq [Q,D], dKc [KV,D], dVc [KV,D] for one head (gradient of sum(O*dO))."""
    q, Kc, Vc, dO = _f64(q), _f64(Kc), _f64(Vc), _f64(dO)
    if O is None or lse is None:
        O, lse = head_forward_dense(q, Kc, Vc, M, scale)
    O, lse = _f64(O), _f64(lse)
    Q = q.shape[0]
    dq = np.zeros_like(q)
    dKc = np.zeros_like(Kc)
    dVc = np.zeros_like(Vc)
    delta = (dO * O).sum(axis=1)
    step = max(1, _CHUNK_ELEMS // max(1, Kc.shape[0]))
    for r0 in range(0, Q, step):
        r1 = min(Q, r0 + step)
        S = scale * (q[r0:r1] @ Kc.T)
        Mc = M[r0:r1]
        fin = np.isfinite(lse[r0:r1])
        with np.errstate(invalid="ignore", over="ignore"):
            P = np.exp(S - np.where(fin, lse[r0:r1], 0.0)[:, None])
        P[~Mc] = 0.0
        P[~fin] = 0.0
        dP = dO[r0:r1] @ Vc.T
        dS = P * (dP - delta[r0:r1, None])
        dq[r0:r1] = scale * (dS @ Kc)
        dKc += scale * (dS.T @ q[r0:r1])
        dVc += P.T @ dO[r0:r1]
    return dq, dKc, dVc


# ---------------------------------------------------------------------------
# keyset formulation: block 0 from the formula, later blocks = diagonal keys
# ---------------------------------------------------------------------------

def _suffix_rows(T, Q_LEN, k):
    """Per later block j, the query rows that see key (j, q): from suffix_keys."""
    rows = np.array([q for q in range(Q_LEN) if _mask.suffix_keys(T, Q_LEN, k, q)], dtype=np.int64)
    return rows


def head_forward_keyset(q, K_blocks, V_blocks, T, scale):
    """O [Q,D] and lse [Q] for one head; K_blocks/V_blocks: k+1 arrays [Q_LEN,D]."""
    q = _f64(q)
    K = [_f64(x) for x in K_blocks]
    V = [_f64(x) for x in V_blocks]
    Q_LEN, k = q.shape[0], len(K) - 1
    valid = np.zeros(Q_LEN, dtype=bool)
    valid[_suffix_rows(T, Q_LEN, k)] = True
    O = np.zeros((Q_LEN, V[0].shape[1]))
    lse = np.empty(Q_LEN)
    step = max(1, _CHUNK_ELEMS // Q_LEN)
    for r0 in range(0, Q_LEN, step):
        r1 = min(Q_LEN, r0 + step)
        rows = np.arange(r0, r1)
        S0 = scale * (q[r0:r1] @ K[0].T)
        S0[~_mask.causal_block_mask(T, Q_LEN, rows)] = -np.inf
        Ss = np.full((r1 - r0, k), -np.inf)
        for j in range(1, k + 1):
            s = scale * np.einsum("rd,rd->r", q[r0:r1], K[j][r0:r1])
            Ss[:, j - 1] = np.where(valid[r0:r1], s, -np.inf)
        lse[r0:r1], P = _softmax_rows(np.concatenate([S0, Ss], axis=1))
        O[r0:r1] = P[:, :Q_LEN] @ V[0]
        for j in range(1, k + 1):
            O[r0:r1] += P[:, Q_LEN + j - 1, None] * V[j][r0:r1]
    return O, lse


def head_backward_keyset(q, K_blocks, V_blocks, T, scale, dO, O=None, lse=None):
    """dq [Q,D] and lists dK, dV of k+1 arrays [Q_LEN,D] for one head."""
    q, dO = _f64(q), _f64(dO)
    K = [_f64(x) for x in K_blocks]
    V = [_f64(x) for x in V_blocks]
    if O is None or lse is None:
        O, lse = head_forward_keyset(q, K, V, T, scale)
    O, lse = _f64(O), _f64(lse)
    Q_LEN, k = q.shape[0], len(K) - 1
    valid = np.zeros(Q_LEN, dtype=bool)
    valid[_suffix_rows(T, Q_LEN, k)] = True
    delta = (dO * O).sum(axis=1)
    dq = np.zeros_like(q)
    dK = [np.zeros_like(x) for x in K]
    dV = [np.zeros_like(x) for x in V]
    step = max(1, _CHUNK_ELEMS // Q_LEN)
    for r0 in range(0, Q_LEN, step):
        r1 = min(Q_LEN, r0 + step)
        rows = np.arange(r0, r1)
        fin = np.isfinite(lse[r0:r1])
        lse_c = np.where(fin, lse[r0:r1], 0.0)
        S0 = scale * (q[r0:r1] @ K[0].T)
        with np.errstate(over="ignore"):
            P0 = np.exp(S0 - lse_c[:, None])
        P0[~_mask.causal_block_mask(T, Q_LEN, rows)] = 0.0
        P0[~fin] = 0.0
        dP0 = dO[r0:r1] @ V[0].T
        dS0 = P0 * (dP0 - delta[r0:r1, None])
        dq[r0:r1] = scale * (dS0 @ K[0])
        dK[0] += scale * (dS0.T @ q[r0:r1])
        dV[0] += P0.T @ dO[r0:r1]
        for j in range(1, k + 1):
            s = scale * np.einsum("rd,rd->r", q[r0:r1], K[j][r0:r1])
            p = np.where(valid[r0:r1] & fin, np.exp(s - lse_c), 0.0)
            dp = np.einsum("rd,rd->r", dO[r0:r1], V[j][r0:r1])
            ds = p * (dp - delta[r0:r1])
            dq[r0:r1] += scale * ds[:, None] * K[j][r0:r1]
            dK[j][r0:r1] += scale * ds[:, None] * q[r0:r1]
            dV[j][r0:r1] += p[:, None] * dO[r0:r1]
    return dq, dK, dV


# ---------------------------------------------------------------------------
# full tensors: [B, H, Q_LEN, D] queries, k+1 blocks of [B, H_kv, Q_LEN, D]
# ---------------------------------------------------------------------------

def kv_head_of(h, H, H_kv):
    """KV head read by query head h (contiguous GQA groups)."""
    return h // (H // H_kv)


def forward(q, K_blocks, V_blocks, T, scale, method="dense", heads=None, batches=None):
    """O [B,H,Q,D] and lse [B,H,Q].

    ``heads`` / ``batches`` restrict the work to a subset (others left 0/nan).
    """
    q = _f64(q)
    B, H, Q_LEN, D = q.shape
    H_kv = K_blocks[0].shape[1]
    k = len(K_blocks) - 1
    O = np.zeros((B, H, Q_LEN, D))
    lse = np.full((B, H, Q_LEN), np.nan)
    for b in (range(B) if batches is None else batches):
        Tb = int(T[b])
        if method == "dense":
            M = _mask.mask_matrix(Tb, Q_LEN, k)
        for h in (range(H) if heads is None else heads):
            g = kv_head_of(h, H, H_kv)
            Kb = [_f64(Kj[b, g]) for Kj in K_blocks]
            Vb = [_f64(Vj[b, g]) for Vj in V_blocks]
            if method == "dense":
                O[b, h], lse[b, h] = head_forward_dense(
                    q[b, h], np.concatenate(Kb), np.concatenate(Vb), M, scale)
            else:
                O[b, h], lse[b, h] = head_forward_keyset(q[b, h], Kb, Vb, Tb, scale)
    return O, lse


def backward(q, K_blocks, V_blocks, T, scale, dO, O=None, lse=None, method="dense",
             heads=None, batches=None):
    """dq [B,H,Q,D] and lists dK, dV of k+1 arrays [B,H_kv,Q,D].

    With ``heads`` given, dK/dV of a KV head hold only the selected heads'
    contributions; pass all heads of a group to get that group's full dK/dV.
    """
    q, dO = _f64(q), _f64(dO)
    B, H, Q_LEN, D = q.shape
    H_kv = K_blocks[0].shape[1]
    k = len(K_blocks) - 1
    dq = np.zeros((B, H, Q_LEN, D))
    dK = [np.zeros((B, H_kv, Q_LEN, D)) for _ in range(k + 1)]
    dV = [np.zeros((B, H_kv, Q_LEN, D)) for _ in range(k + 1)]
    for b in (range(B) if batches is None else batches):
        Tb = int(T[b])
        if method == "dense":
            M = _mask.mask_matrix(Tb, Q_LEN, k)
        for h in (range(H) if heads is None else heads):
            g = kv_head_of(h, H, H_kv)
            Kb = [_f64(Kj[b, g]) for Kj in K_blocks]
            Vb = [_f64(Vj[b, g]) for Vj in V_blocks]
            Oh = None if O is None else O[b, h]
            lh = None if lse is None else lse[b, h]
            if method == "dense":
                dqh, dKc, dVc = head_backward_dense(
                    q[b, h], np.concatenate(Kb), np.concatenate(Vb), M, scale, dO[b, h], Oh, lh)
                dKl = np.split(dKc, k + 1)
                dVl = np.split(dVc, k + 1)
            else:
                dqh, dKl, dVl = head_backward_keyset(q[b, h], Kb, Vb, Tb, scale, dO[b, h], Oh, lh)
            dq[b, h] = dqh
            for j in range(k + 1):
                dK[j][b, g] += dKl[j]
                dV[j][b, g] += dVl[j]
    return dq, dK, dV


def unmasked_entries(T, Q_LEN, k):
    """Number of (q, kv) pairs with M true for one (b, h): counted from the mask.

    Used by tests; the closed form T(T+1)/2 + k*T + (Q_LEN-T)*T must agree.
    """
    return int(_mask.mask_matrix(T, Q_LEN, k).sum())
