"""Masked soft-target softmax cross-entropy with its in-place gradient
(oracle; test infrastructure).

Source: SpecForge review, §四 "掩码 Softmax 损失" and "原地反向传播", and §三
"内存高效梯度计算" (the custom kernel the page calls Algorithm 3).  Per row r
of logits z [N, V] with target distribution p [N, V] and per-row upstream
gradient g [N]:

    pi  = softmax(z_r)                     (§四, softmax(z_i) = e^{z_i} / sum_j e^{z_j})
    l_r = -sum_v p_rv * log pi_rv          (§四, L = -sum_i p_i log softmax(z_i))
    s_r = sum_v p_rv * g_r                 (§三, s = sum(p * g))
    grad_rv = -(p_rv * g_r - pi_rv * s_r)  (§三/§四, z <- -(p*g - pi*s))

and the scalar returned is L = sum_r g_r * l_r, whose derivative with respect to
z is exactly ``grad`` (when sum(p) = 1 this is g*(pi - p), §四).  g is read as
one value per row (the loss mask divided by N in the workloads).  The formula
s = sum(p * g) also admits one value per element, G [N, V]; that reading is
``soft_ce_elementwise``: the loss is L = -sum_rv G_rv p_rv log pi_rv, whose
z-gradient is again -(p*G - pi*s) with s_r = sum_v p_rv G_rv.

The per-row loss reported for a row with g_r = 0 is 0: that row is masked out
of the loss, and its gradient is exactly 0 (convention; parity unpinned).
All arithmetic is float64.
"""

import numpy as np

_CHUNK_ROWS = 256


def soft_ce(z, p, g):
    """Return (L, row_loss [N], grad [N,V]) in float64.

    z, p: [N, V]; g: [N].  Rows are processed in chunks to bound memory.
    """
    z = np.asarray(z, dtype=np.float64)
    p = np.asarray(p, dtype=np.float64)
    g = np.asarray(g, dtype=np.float64).reshape(-1)
    N, V = z.shape
    grad = np.empty((N, V))
    row_loss = np.zeros(N)
    L = 0.0
    for r0 in range(0, N, _CHUNK_ROWS):
        r1 = min(N, r0 + _CHUNK_ROWS)
        zc, pc, gc = z[r0:r1], p[r0:r1], g[r0:r1]
        m = zc.max(axis=1)
        lse = m + np.log(np.exp(zc - m[:, None]).sum(axis=1))
        log_pi = zc - lse[:, None]
        pi = np.exp(log_pi)
        ell = -(pc * log_pi).sum(axis=1)
        s = (pc * gc[:, None]).sum(axis=1)
        grad[r0:r1] = -(pc * gc[:, None] - pi * s[:, None])
        row_loss[r0:r1] = np.where(gc != 0.0, ell, 0.0)
        L += float((gc * np.where(gc != 0.0, ell, 0.0)).sum())
    return L, row_loss, grad


def soft_ce_row(z_row, p_row, g_r):
    """One row with explicit Python loops (for tiny pins and cross-checks)."""
    V = len(z_row)
    m = max(float(x) for x in z_row)
    total = 0.0
    for v in range(V):
        total += np.exp(float(z_row[v]) - m)
    lse = m + np.log(total)
    ell = 0.0
    for v in range(V):
        ell -= float(p_row[v]) * (float(z_row[v]) - lse)
    s = 0.0
    for v in range(V):
        s += float(p_row[v]) * float(g_r)
    grad = [-(float(p_row[v]) * float(g_r) - np.exp(float(z_row[v]) - lse) * s) for v in range(V)]
    return (ell if g_r != 0.0 else 0.0), np.array(grad)


def soft_ce_elementwise(z, p, G):
    """Per-element upstream gradient G [N, V] (SpecForge review, §三 "内存高效梯度计算":
    s = sum(p * g) with g of the logits' shape).  Return (L, row_loss [N], grad [N,V]):

        pi = softmax(z_r),  lse_r = log sum_v exp(z_rv)
        row_loss_r = -sum_v G_rv p_rv log pi_rv = sum_v G_rv p_rv (lse_r - z_rv)
        s_r = sum_v p_rv G_rv,  grad_rv = -(p_rv G_rv - pi_rv s_r)
        L = sum_r row_loss_r

    With G_rv = g_r for every v this is ``soft_ce`` (row_loss then carries the
    weight g_r).  Float64, rows in chunks."""
    z = np.asarray(z, dtype=np.float64)
    p = np.asarray(p, dtype=np.float64)
    G = np.asarray(G, dtype=np.float64)
    N, V = z.shape
    grad = np.empty((N, V))
    row_loss = np.zeros(N)
    for r0 in range(0, N, _CHUNK_ROWS):
        r1 = min(N, r0 + _CHUNK_ROWS)
        zc, pc, Gc = z[r0:r1], p[r0:r1], G[r0:r1]
        m = zc.max(axis=1)
        lse = m + np.log(np.exp(zc - m[:, None]).sum(axis=1))
        log_pi = zc - lse[:, None]
        pi = np.exp(log_pi)
        pg = pc * Gc
        row_loss[r0:r1] = -(pg * log_pi).sum(axis=1)
        s = pg.sum(axis=1)
        grad[r0:r1] = -(pg - pi * s[:, None])
    return float(row_loss.sum()), row_loss, grad
