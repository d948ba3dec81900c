"""GPU parity of sparse-tree TTT attention (forward and backward) against the
fp64 oracle, through the C ABI.

Tolerances (bf16 inputs, fp32 accumulation): for each of O, dQ, dK_j, dV_j
max-abs <= 2e-2 and relative L2 <= 1e-2; lse max-abs <= 1e-3 (rows with no
visible key must be -inf on both sides).
"""

import numpy as np
import pytest
import torch

from oracle import attention as oa
from speculative_decoding_draft_eagle_gb300 import ops, workloads as wl

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from speculative_decoding_draft_eagle_gb300 import build
    build.build()


def f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def close(gpu, ref, name, atol=2e-2, rtol_l2=1e-2):
    gpu = np.asarray(gpu, dtype=np.float64)
    d = gpu - ref
    maxabs = float(np.abs(d).max()) if d.size else 0.0
    nref = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(d)) / nref if nref > 0 else float(np.linalg.norm(d))
    assert maxabs <= atol and rel <= rtol_l2, f"{name}: maxabs={maxabs:.3g} relL2={rel:.3g}"


def close_lse(gpu, ref):
    gpu = np.asarray(gpu, dtype=np.float64)
    inf_ref = np.isneginf(ref)
    assert np.array_equal(np.isneginf(gpu), inf_ref)
    if (~inf_ref).any():
        assert np.abs(gpu[~inf_ref] - ref[~inf_ref]).max() <= 1e-3


def make(B, H, H_kv, Q, D, k, T, seed):
    g = torch.Generator().manual_seed(seed)
    r = lambda *s: torch.randn(*s, generator=g).to(torch.bfloat16)  # noqa: E731
    q = r(B, H, Q, D)
    Ks = [r(B, H_kv, Q, D) for _ in range(k + 1)]
    Vs = [r(B, H_kv, Q, D) for _ in range(k + 1)]
    dO = r(B, H, Q, D)
    return q, Ks, Vs, dO, list(T)


def run_fwd(q, Ks, Vs, T, scale):
    out, lse = ops.stt_attn_fwd(q.to(DEV), [x.to(DEV) for x in Ks], [x.to(DEV) for x in Vs], T,
                                scale)
    torch.cuda.synchronize()
    assert ops.stt_device_error() == 0
    return out, lse


def check_fwd(q, Ks, Vs, T, scale, method="dense"):
    out, lse = run_fwd(q, Ks, Vs, T, scale)
    O_ref, lse_ref = oa.forward(f64(q), [f64(x) for x in Ks], [f64(x) for x in Vs], T, scale,
                                method=method)
    close(f64(out), O_ref, "O")
    close_lse(lse.cpu().numpy(), lse_ref)
    return out, lse


def test_tiny_workload_forward():
    w = wl.WORKLOADS["tiny"]
    T, Ks, Vs, qs, dOs = wl.attn_inputs(w.attn, "cpu", w.seed)
    k = w.attn.steps[0]
    check_fwd(qs[k], Ks[: k + 1], Vs[: k + 1], T, w.attn.scale)


FWD_CASES = [
    # B, H, H_kv, Q_LEN, D, k, T
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
]


@pytest.mark.parametrize("B,H,H_kv,Q,D,k,T", FWD_CASES)
def test_forward_shapes(B, H, H_kv, Q, D, k, T):
    q, Ks, Vs, _, T = make(B, H, H_kv, Q, D, k, T, seed=B * 1000 + Q + k)
    check_fwd(q, Ks, Vs, T, 1.0 / np.sqrt(D))


def test_forward_scale_and_large_scores():
    """A large scale forces many running-max rescales (scores spread over ~50)."""
    q, Ks, Vs, _, T = make(1, 2, 1, 256, 128, 2, [256], seed=5)
    check_fwd(q, Ks, Vs, T, 0.6)


@pytest.mark.parametrize("name", ["llama8b", "varlen", "llama70b", "long_ttt"])
def test_forward_full_size_sampled(name):
    """Full-size workload on the GPU; the oracle (key-set form) checks b in
    {0, B-1} and KV groups {0, H_kv-1} with all their query heads, at the first
    and the last TTT step."""
    w = wl.WORKLOADS[name]
    sh = w.attn
    T = wl.draw_T(sh, w.seed)
    Ks = [wl.kv_block(sh, "K", j, DEV, w.seed) for j in range(sh.n_blocks)]
    Vs = [wl.kv_block(sh, "V", j, DEV, w.seed) for j in range(sh.n_blocks)]
    G = sh.H // sh.H_kv
    heads = list(range(G)) + list(range(sh.H - G, sh.H))
    batches = sorted({0, sh.B - 1})
    for k in (sh.steps[0], sh.steps[-1]):
        q = wl.step_query(sh, k, DEV, w.seed)
        out, lse = ops.stt_attn_fwd(q, Ks[: k + 1], Vs[: k + 1], T, sh.scale)
        torch.cuda.synchronize()
        assert ops.stt_device_error() == 0
        for b in batches:
            qb = f64(q[b:b + 1, heads])
            Kb = [f64(x[b:b + 1]) for x in Ks[: k + 1]]
            Vb = [f64(x[b:b + 1]) for x in Vs[: k + 1]]
            # heads are renumbered 0..2G-1 inside the slice: map them onto KV heads
            O_ref = np.zeros_like(qb)
            l_ref = np.zeros(qb.shape[:3])
            for i, h in enumerate(heads):
                g = h // G
                O1, l1 = oa.head_forward_keyset(qb[0, i], [x[0, g] for x in Kb], [x[0, g] for x in Vb],
                                                T[b], sh.scale)
                O_ref[0, i], l_ref[0, i] = O1, l1
            close(f64(out[b:b + 1, heads]), O_ref, f"O[{name},k={k},b={b}]")
            close_lse(lse[b:b + 1, heads].cpu().numpy(), l_ref)


# ----------------------------------------------------------------- backward --

def run_bwd(q, Ks, Vs, dO, T, scale):
    qd = q.to(DEV)
    Kd = [x.to(DEV) for x in Ks]
    Vd = [x.to(DEV) for x in Vs]
    out, lse = ops.stt_attn_fwd(qd, Kd, Vd, T, scale)
    dq, dk, dv = ops.stt_attn_bwd(qd, Kd, Vd, T, out, dO.to(DEV), lse, scale)
    torch.cuda.synchronize()
    assert ops.stt_device_error() == 0
    return dq, dk, dv


def bwd_atol(ref):
    """Max-abs bound for a gradient tensor: 2e-2, or 4 bf16 ulps (2^-7 relative)
    of the tensor's largest entry when that exceeds 2.56.

    The method stores O in bf16 (round to nearest even) and the backward takes
    Delta = rowsum(dO * O) from that stored output, and P / dS enter the tensor
    cores as bf16; each contributes up to 2^-9 of relative rounding per term.
    With O(1) gradients (every workload) the flat 2e-2 binds; only degenerate
    shapes where hundreds of padded rows share a couple of keys push |dK| to
    ~10, where the bf16 storage error alone (reproduced by a CPU emulation of
    the rounding) reaches ~0.035."""
    return max(2e-2, 2.0 ** -7 * float(np.abs(ref).max()))


def check_bwd(q, Ks, Vs, dO, T, scale):
    dq, dk, dv = run_bwd(q, Ks, Vs, dO, T, scale)
    rq, rk, rv = oa.backward(f64(q), [f64(x) for x in Ks], [f64(x) for x in Vs], T, scale, f64(dO))
    close(f64(dq), rq, "dq", atol=bwd_atol(rq))
    for j in range(len(Ks)):
        close(f64(dk[j]), rk[j], f"dK[{j}]", atol=bwd_atol(rk[j]))
        close(f64(dv[j]), rv[j], f"dV[{j}]", atol=bwd_atol(rv[j]))


def test_tiny_workload_backward():
    """The tiny workload at the flat bound (2e-2 max-abs)."""
    w = wl.WORKLOADS["tiny"]
    T, Ks, Vs, qs, dOs = wl.attn_inputs(w.attn, "cpu", w.seed)
    k = w.attn.steps[0]
    q, dO = qs[k], dOs[k]
    dq, dk, dv = run_bwd(q, Ks[: k + 1], Vs[: k + 1], dO, T, w.attn.scale)
    rq, rk, rv = oa.backward(f64(q), [f64(x) for x in Ks[: k + 1]], [f64(x) for x in Vs[: k + 1]],
                             T, w.attn.scale, f64(dO))
    close(f64(dq), rq, "dq")
    for j in range(k + 1):
        close(f64(dk[j]), rk[j], f"dK[{j}]")
        close(f64(dv[j]), rv[j], f"dV[{j}]")


@pytest.mark.parametrize("B,H,H_kv,Q,D,k,T", FWD_CASES)
def test_backward_shapes(B, H, H_kv, Q, D, k, T):
    q, Ks, Vs, dO, T = make(B, H, H_kv, Q, D, k, T, seed=7 * B + Q + 3 * k)
    check_bwd(q, Ks, Vs, dO, T, 1.0 / np.sqrt(D))


def test_backward_overwrites_outputs():
    """Gradients are overwritten, not accumulated: stale contents must not leak."""
    q, Ks, Vs, dO, T = make(1, 4, 2, 256, 128, 2, [200], seed=3)
    scale = 1.0 / np.sqrt(128)
    qd, Kd, Vd = q.to(DEV), [x.to(DEV) for x in Ks], [x.to(DEV) for x in Vs]
    out, lse = ops.stt_attn_fwd(qd, Kd, Vd, T, scale)
    dq = torch.full(q.shape, 7.0, device=DEV)
    dk = [torch.full(x.shape, -3.0, device=DEV) for x in Ks]
    dv = [torch.full(x.shape, 5.0, device=DEV) for x in Vs]
    ws = torch.full((ops.stt_attn_bwd_workspace_size(1, 4, 2, 128, 256, 2),), 255, dtype=torch.uint8,
                    device=DEV)
    ops.stt_attn_bwd(qd, Kd, Vd, T, out, dO.to(DEV), lse, scale, dq=dq, dk_blocks=dk, dv_blocks=dv,
                     workspace=ws)
    torch.cuda.synchronize()
    rq, rk, rv = oa.backward(f64(q), [f64(x) for x in Ks], [f64(x) for x in Vs], T, scale, f64(dO))
    close(f64(dq), rq, "dq")
    for j in range(3):
        close(f64(dk[j]), rk[j], f"dK[{j}]")
        close(f64(dv[j]), rv[j], f"dV[{j}]")


@pytest.mark.parametrize("name", ["llama8b", "varlen", "llama70b", "long_ttt"])
def test_backward_full_size_sampled(name):
    """Full-size backward on the GPU.  The oracle computes b in {0, B-1} and KV
    groups {0, H_kv-1} with all their query heads (so dK/dV of those groups are
    complete) at the first and last TTT step."""
    w = wl.WORKLOADS[name]
    sh = w.attn
    T = wl.draw_T(sh, w.seed)
    Ks = [wl.kv_block(sh, "K", j, DEV, w.seed) for j in range(sh.n_blocks)]
    Vs = [wl.kv_block(sh, "V", j, DEV, w.seed) for j in range(sh.n_blocks)]
    G = sh.H // sh.H_kv
    groups = sorted({0, sh.H_kv - 1})
    batches = sorted({0, sh.B - 1})
    for k in (sh.steps[0], sh.steps[-1]):
        q = wl.step_query(sh, k, DEV, w.seed)
        dO = wl.step_dout(sh, k, DEV, w.seed)
        out, lse = ops.stt_attn_fwd(q, Ks[: k + 1], Vs[: k + 1], T, sh.scale)
        dq, dk, dv = ops.stt_attn_bwd(q, Ks[: k + 1], Vs[: k + 1], T, out, dO, lse, sh.scale)
        torch.cuda.synchronize()
        assert ops.stt_device_error() == 0
        for b in batches:
            for g in groups:
                Kb = [f64(x[b, g]) for x in Ks[: k + 1]]
                Vb = [f64(x[b, g]) for x in Vs[: k + 1]]
                dk_ref = [np.zeros_like(x) for x in Kb]
                dv_ref = [np.zeros_like(x) for x in Vb]
                for h in range(g * G, (g + 1) * G):
                    rq, rk, rv = oa.head_backward_keyset(f64(q[b, h]), Kb, Vb, T[b], sh.scale,
                                                         f64(dO[b, h]))
                    close(f64(dq[b, h]), rq, f"dq[{name},k={k},b={b},h={h}]")
                    for j in range(k + 1):
                        dk_ref[j] += rk[j]
                        dv_ref[j] += rv[j]
                for j in range(k + 1):
                    close(f64(dk[j][b, g]), dk_ref[j], f"dK[{name},k={k},b={b},g={g},j={j}]")
                    close(f64(dv[j][b, g]), dv_ref[j], f"dV[{name},k={k},b={b},g={g},j={j}]")
