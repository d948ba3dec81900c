"""Helpers shared by the GPU parity tests.

* ``close`` checks max-abs and relative-L2 error against a bound and records
  the margin of every check (also of the passing ones); the conftest prints
  the worst margin of each group at the end of the run.
* ``OraclePool`` runs the fp64 oracle on the sampled units of the full-size
  workloads in a pool of spawned processes (one BLAS thread each), fed through
  .npy files, so that every TTT step of every workload can be checked in a
  bounded time.  Spawned, never forked: the parent holds a CUDA context.
* ``emulated_backward`` repeats the backward in fp64 with the roundings the
  GPU path takes (bf16 O feeding Delta; bf16 P and dS as tensor-core
  operands); its error against the exact oracle predicts the GPU's error on
  shapes where that rounding dominates.
"""

from __future__ import annotations

import concurrent.futures as cf
import multiprocessing as mp
import os

import numpy as np

MARGINS = []  # dicts: group, name, maxabs, atol, rel, rtol

# Synthetic attention shapes of the parity tests: B, H, H_kv, Q_LEN, D, k, T.
FWD_CASES = [
    (1, 2, 1, 128, 64, 0, [128]),
    (1, 2, 2, 128, 128, 0, [128]),
    (2, 4, 2, 256, 128, 1, [256, 77]),
    (2, 4, 1, 200, 64, 3, [0, 199]),       # T = 0 and a ragged Q_LEN
    (1, 8, 2, 384, 128, 12, [1]),          # T = 1, long TTT
    (3, 2, 2, 130, 128, 2, [129, 130, 2]),
    (1, 4, 4, 64, 64, 1, [50]),            # Q_LEN smaller than one tile
    (3, 8, 2, 384, 128, 1, [384, 200, 7]),  # 24 heads: key-tile CTAs in a full and a partial head chunk
    (2, 8, 1, 512, 128, 6, [511, 300]),    # group of 8 query heads
    (1, 6, 2, 256, 128, 2, [200]),         # group of 3 (below the unrolled bound of 4)
    (1, 6, 1, 192, 128, 5, [150]),         # group of 6 (below the unrolled bound of 8)
    (1, 3, 1, 129, 64, 2, [100]),          # odd row count: a partly filled last warp
    # More work items than SMs: each persistent forward CTA walks several query
    # tiles (Q buffers reused, barrier phases carried across items), including
    # items of empty sequences (T = 0: no key tiles, zero O) next to full ones;
    # the backward takes two query heads per CTA here (1536 key-tile pairs).
    (48, 16, 4, 256, 128, 1, [256, 0, 1, 129, 200, 256, 77, 0] * 6),
    (4, 12, 3, 512, 64, 2, [512, 0, 77, 300]),  # D = 64, 192 forward items
]


def make(B, H, H_kv, Q, D, k, T, seed):
    """q, K blocks, V blocks, dO (bf16, CPU generator) and T of a synthetic shape."""
    import torch
    g = torch.Generator().manual_seed(seed)
    r = lambda *s: torch.randn(*s, generator=g).to(torch.bfloat16)  # noqa: E731
    q = r(B, H, Q, D)
    Ks = [r(B, H_kv, Q, D) for _ in range(k + 1)]
    Vs = [r(B, H_kv, Q, D) for _ in range(k + 1)]
    dO = r(B, H, Q, D)
    return q, Ks, Vs, dO, list(T)


def measure(gpu, ref):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    d = gpu - ref
    maxabs = float(np.abs(d).max()) if d.size else 0.0
    nref = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(d)) / nref if nref > 0 else float(np.linalg.norm(d))
    return maxabs, rel


def record(group, name, maxabs, atol, rel, rtol):
    MARGINS.append(dict(group=group, name=name, maxabs=maxabs, atol=atol, rel=rel, rtol=rtol))


def close(gpu, ref, name, atol=2e-2, rtol_l2=1e-2, group="shapes"):
    maxabs, rel = measure(gpu, ref)
    record(group, name, maxabs, atol, rel, rtol_l2)
    assert maxabs <= atol and rel <= rtol_l2, (
        f"{name}: maxabs={maxabs:.3g} (bound {atol:.3g}) relL2={rel:.3g} (bound {rtol_l2:.3g})")


def summary_lines():
    """Worst max-abs / bound and relative-L2 / bound per group."""
    groups = {}
    for m in MARGINS:
        groups.setdefault(m["group"], []).append(m)
    lines = []
    for gname in sorted(groups):
        ms = groups[gname]
        wa = max(ms, key=lambda m: m["maxabs"] / m["atol"] if m["atol"] else 0.0)
        wr = max(ms, key=lambda m: m["rel"] / m["rtol"] if m["rtol"] else 0.0)
        lines.append(
            f"{gname}: {len(ms)} checks; worst maxabs {wa['maxabs']:.3g}/{wa['atol']:.3g} "
            f"({wa['maxabs'] / wa['atol']:.2f} of bound, {wa['name']}); worst relL2 "
            f"{wr['rel']:.3g}/{wr['rtol']:.3g} ({wr['rel'] / wr['rtol']:.2f}, {wr['name']})")
    return lines


# ------------------------------------------------------- oracle process pool --

def bf16_bits(t):
    """torch bf16 tensor -> numpy uint16 of its bits (host)."""
    import torch
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def from_bits(u16):
    return (np.asarray(u16, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


def _unit_task(d, b, g, G, k, T, scale, tag, atol, rtol):
    """One sampled unit (batch b, KV group g, all G heads) at TTT step k: the
    oracle forward and backward from the files in d, compared with the GPU's
    outputs there.  Returns [(name, maxabs, atol, rel, rtol)]."""
    from oracle import attention as oa
    K = [from_bits(np.load(os.path.join(d, f"K{j}_b{b}_g{g}.npy"), mmap_mode="r")) for j in range(k + 1)]
    V = [from_bits(np.load(os.path.join(d, f"V{j}_b{b}_g{g}.npy"), mmap_mode="r")) for j in range(k + 1)]
    pre = os.path.join(d, f"k{k}_b{b}_g{g}_")
    q = from_bits(np.load(pre + "q.npy"))
    dO = from_bits(np.load(pre + "do.npy"))
    O_gpu = from_bits(np.load(pre + "o.npy"))
    lse_gpu = np.load(pre + "lse.npy").astype(np.float64)
    dq_gpu = np.load(pre + "dq.npy")
    out = []

    def chk(name, gpu, ref, a=atol, r=rtol):
        m, rel = measure(gpu, ref)
        out.append((name, m, a, rel, r))

    dk_ref = [np.zeros_like(x) for x in K]
    dv_ref = [np.zeros_like(x) for x in V]
    for i in range(G):
        h = g * G + i
        O, lse = oa.head_forward_keyset(q[i], K, V, T, scale)
        chk(f"O[{tag},k={k},b={b},h={h}]", O_gpu[i], O)
        fin = np.isfinite(lse)
        ok_inf = bool(np.array_equal(np.isneginf(lse_gpu[i]), ~fin))
        lerr = float(np.abs(lse_gpu[i][fin] - lse[fin]).max()) if fin.any() else 0.0
        out.append((f"lse[{tag},k={k},b={b},h={h}]", lerr if ok_inf else float("inf"), 1e-3,
                    0.0, 1.0))
        rq, rk, rv = oa.head_backward_keyset(q[i], K, V, T, scale, dO[i], O, lse)
        chk(f"dq[{tag},k={k},b={b},h={h}]", dq_gpu[i], rq)
        for j in range(k + 1):
            dk_ref[j] += rk[j]
            dv_ref[j] += rv[j]
    for j in range(k + 1):
        chk(f"dK[{tag},k={k},b={b},g={g},j={j}]", np.load(pre + f"dk{j}.npy"), dk_ref[j])
        chk(f"dV[{tag},k={k},b={b},g={g},j={j}]", np.load(pre + f"dv{j}.npy"), dv_ref[j])
    return out


class OraclePool:
    """Spawned worker processes running ``_unit_task`` with one BLAS thread."""

    _THREAD_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")

    def __init__(self, workers=None):
        n = workers or max(1, min(16, os.cpu_count() or 1))
        # Workers are spawned as tasks arrive and read these at their numpy
        # import; the parent's BLAS is already set up and is not affected.
        self._saved = {v: os.environ.get(v) for v in self._THREAD_VARS}
        for v in self._THREAD_VARS:
            os.environ[v] = "1"
        self.ex = cf.ProcessPoolExecutor(max_workers=n, mp_context=mp.get_context("spawn"))
        self.futures = []

    def submit(self, *args):
        self.futures.append(self.ex.submit(_unit_task, *args))

    def results(self):
        out = []
        for f in self.futures:
            out.extend(f.result())
        self.futures = []
        return out

    def close(self):
        self.ex.shutdown(wait=True, cancel_futures=True)
        for v, val in self._saved.items():
            if val is None:
                os.environ.pop(v, None)
            else:
                os.environ[v] = val


# ------------------------------------------------------ bf16 rounding model --

def _round_bf16(x):
    """Round float64 values to bf16 (nearest even) through float32, as torch does."""
    import torch
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).to(
        torch.float64).numpy()


def emulated_backward(q, K_blocks, V_blocks, T, scale, dO, rounding=True):
    """dq, dK, dV of the sparse-tree attention in fp64, repeating the GPU path's
    roundings when ``rounding`` is set:
      * O is stored in bf16, and Delta = rowsum(dO * O) is taken from it;
      * in block 0 (the tensor-core part) the kernel carries the attention
        scale in P: scale P enters dV = (scale P)^T dO / scale as bf16, and
        scale dS = scale P (dP - Delta) enters dK = (scale dS)^T q and
        dq = (scale dS) K as bf16;
      * the suffix keys (blocks j >= 1) are computed without operand rounding.
    With ``rounding`` off it is the exact backward.  Inputs as the oracle's
    ``backward`` (q [B,H,Q,D], K/V blocks [B,H_kv,Q,D]); dense mask."""
    from oracle import mask as om
    q = np.asarray(q, dtype=np.float64)
    dO = np.asarray(dO, dtype=np.float64)
    B, H, Q, D = q.shape
    H_kv = K_blocks[0].shape[1]
    G = H // H_kv
    k = len(K_blocks) - 1
    rb = _round_bf16 if rounding else (lambda x: x)
    dq = np.zeros_like(q)
    dK = [np.zeros((B, H_kv, Q, D)) for _ in range(k + 1)]
    dV = [np.zeros((B, H_kv, Q, D)) for _ in range(k + 1)]
    for b in range(B):
        M = om.mask_matrix(int(T[b]), Q, k)
        for h in range(H):
            g = h // G
            Kc = np.concatenate([np.asarray(x[b, g], dtype=np.float64) for x in K_blocks])
            Vc = np.concatenate([np.asarray(x[b, g], dtype=np.float64) for x in V_blocks])
            S = scale * q[b, h] @ Kc.T
            S[~M] = -np.inf
            m = S.max(axis=1)
            empty = ~np.isfinite(m)
            m = np.where(empty, 0.0, m)
            E = np.exp(S - m[:, None])
            E[~M] = 0.0
            l = E.sum(axis=1)
            P = np.where(empty[:, None], 0.0, E / np.where(empty, 1.0, l)[:, None])
            O = P @ Vc
            delta = (dO[b, h] * rb(O)).sum(axis=1)
            dP = dO[b, h] @ Vc.T
            dS = P * (dP - delta[:, None])
            causal = np.zeros(M.shape, dtype=bool)
            causal[:, :Q] = True
            Pm = np.where(causal, rb(scale * P), scale * P)
            dSm = np.where(causal, rb(scale * dS), scale * dS)
            dq[b, h] = dSm @ Kc
            dKc = dSm.T @ q[b, h]
            dVc = Pm.T @ dO[b, h] / scale
            for j in range(k + 1):
                dK[j][b, g] += dKc[j * Q:(j + 1) * Q]
                dV[j][b, g] += dVc[j * Q:(j + 1) * Q]
    return dq, dK, dV
