"""GPU parity of sparse-tree TTT attention (forward and backward) against the
fp64 oracle, through the C ABI.

Tolerances (bf16 inputs, fp32 accumulation): for each of O, dQ, dK_j, dV_j
max-abs <= 2e-2 and relative L2 <= 1e-2; lse max-abs <= 1e-3 (rows with no
visible key must be -inf on both sides).
"""

import os
import tempfile

import numpy as np
import pytest
import torch

import _parity
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


def close(gpu, ref, name, atol=2e-2, rtol_l2=1e-2, group="attention shapes"):
    _parity.close(gpu, ref, name, atol, rtol_l2, group)


def close_lse(gpu, ref, group="attention shapes"):
    gpu = np.asarray(gpu, dtype=np.float64)
    inf_ref = np.isneginf(ref)
    assert np.array_equal(np.isneginf(gpu), inf_ref)
    err = float(np.abs(gpu[~inf_ref] - ref[~inf_ref]).max()) if (~inf_ref).any() else 0.0
    _parity.record(group, "lse", err, 1e-3, 0.0, 1.0)
    assert err <= 1e-3


make = _parity.make


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


FWD_CASES = _parity.FWD_CASES


@pytest.mark.parametrize("B,H,H_kv,Q,D,k,T", FWD_CASES)
def test_forward_shapes(B, H, H_kv, Q, D, k, T):
    q, Ks, Vs, _, T = make(B, H, H_kv, Q, D, k, T, seed=B * 1000 + Q + k)
    check_fwd(q, Ks, Vs, T, 1.0 / np.sqrt(D))


def test_forward_scale_and_large_scores():
    """A large scale forces many running-max rescales (scores spread over ~50)."""
    q, Ks, Vs, _, T = make(1, 2, 1, 256, 128, 2, [256], seed=5)
    check_fwd(q, Ks, Vs, T, 0.6)


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


def check_bwd(q, Ks, Vs, dO, T, scale):
    """Backward parity.  The max-abs bound of each gradient tensor is the flat
    2e-2, or twice the error of the bf16 rounding model (``emulated_backward``:
    O stored in bf16 feeds Delta, P and dS enter the tensor cores as bf16)
    where that predicted error is larger: on degenerate shapes where hundreds
    of padded rows share a couple of keys, |dK| reaches ~10 and the bf16
    storage of O alone moves it by ~0.03.  Relative L2 stays at the flat 1e-2."""
    dq, dk, dv = run_bwd(q, Ks, Vs, dO, T, scale)
    args = (f64(q), [f64(x) for x in Ks], [f64(x) for x in Vs], T, scale, f64(dO))
    rq, rk, rv = oa.backward(*args)
    eq, ek, ev = _parity.emulated_backward(*args)

    def bound(em, ref):
        return max(2e-2, 2.0 * float(np.abs(em - ref).max()))

    close(f64(dq), rq, "dq", atol=bound(eq, rq), group="attention shapes (bwd)")
    for j in range(len(Ks)):
        close(f64(dk[j]), rk[j], f"dK[{j}]", atol=bound(ek[j], rk[j]), group="attention shapes (bwd)")
        close(f64(dv[j]), rv[j], f"dV[{j}]", atol=bound(ev[j], rv[j]), group="attention shapes (bwd)")


@pytest.mark.parametrize("name", ["varlen", "llama8b"])
def test_forward_repeats_bit_identical(name):
    """The forward has no atomics and a fixed work order, so repeated launches
    on the same inputs must give bit-identical O and lse.  The persistent
    kernel carries every barrier phase across work items; a waiter that reads
    a phase too early (the many short items of varlen make item boundaries
    frequent) shows up here as rows that differ between launches."""
    w = wl.WORKLOADS[name]
    sh = w.attn
    T = wl.draw_T(sh, w.seed)
    Ks = [wl.kv_block(sh, "K", j, DEV, w.seed) for j in range(sh.n_blocks)]
    Vs = [wl.kv_block(sh, "V", j, DEV, w.seed) for j in range(sh.n_blocks)]
    for k in (0, max(sh.steps)):
        q = wl.step_query(sh, k, DEV, w.seed)
        o0, l0 = ops.stt_attn_fwd(q, Ks[: k + 1], Vs[: k + 1], T, sh.scale)
        o0, l0 = o0.clone(), l0.clone()
        for _ in range(12):
            o, l = ops.stt_attn_fwd(q, Ks[: k + 1], Vs[: k + 1], T, sh.scale)
            assert torch.equal(o.view(torch.int16), o0.view(torch.int16)), f"O differs, k={k}"
            assert torch.equal(l.view(torch.int32), l0.view(torch.int32)), f"lse differs, k={k}"
        assert ops.stt_device_error() == 0


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


FULL = ["llama8b", "varlen", "llama70b", "long_ttt"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_every_step(name):
    """Full-size workload, forward and backward on the GPU at EVERY TTT step k.
    The oracle checks the sampled units b in {0, B-1} x KV groups {0, H_kv-1}
    with all their query heads (so dK/dV of those groups are complete) and all
    rows: O, lse, dq per head and dK_j, dV_j per group, at the flat bounds
    (max-abs 2e-2, relative L2 1e-2; lse max-abs 1e-3).  The oracle runs in a
    pool of spawned processes while the GPU goes on with the next step."""
    w = wl.WORKLOADS[name]
    sh = w.attn
    T = wl.draw_T(sh, w.seed)
    Ks = [wl.kv_block(sh, "K", j, DEV, w.seed) for j in range(sh.n_blocks)]
    Vs = [wl.kv_block(sh, "V", j, DEV, w.seed) for j in range(sh.n_blocks)]
    G = sh.H // sh.H_kv
    groups = sorted({0, sh.H_kv - 1})
    batches = sorted({0, sh.B - 1})
    d = tempfile.mkdtemp(prefix=f"stt_{name}_")
    for b in batches:
        for g in groups:
            for j in range(sh.n_blocks):
                np.save(os.path.join(d, f"K{j}_b{b}_g{g}.npy"), _parity.bf16_bits(Ks[j][b, g]))
                np.save(os.path.join(d, f"V{j}_b{b}_g{g}.npy"), _parity.bf16_bits(Vs[j][b, g]))
    pool = _parity.OraclePool()
    try:
        # longest units first: the oracle's cost grows a little with k
        for k in sorted(sh.steps, reverse=True):
            q = wl.step_query(sh, k, DEV, w.seed)
            dO = wl.step_dout(sh, k, DEV, w.seed)
            out, lse = ops.stt_attn_fwd(q, Ks[: k + 1], Vs[: k + 1], T, sh.scale)
            dq, dk, dv = ops.stt_attn_bwd(q, Ks[: k + 1], Vs[: k + 1], T, out, dO, lse, sh.scale)
            torch.cuda.synchronize()
            assert ops.stt_device_error() == 0
            for b in batches:
                for g in groups:
                    hs = slice(g * G, (g + 1) * G)
                    pre = os.path.join(d, f"k{k}_b{b}_g{g}_")
                    np.save(pre + "q.npy", _parity.bf16_bits(q[b, hs]))
                    np.save(pre + "do.npy", _parity.bf16_bits(dO[b, hs]))
                    np.save(pre + "o.npy", _parity.bf16_bits(out[b, hs]))
                    np.save(pre + "lse.npy", lse[b, hs].cpu().numpy())
                    np.save(pre + "dq.npy", dq[b, hs].cpu().numpy())
                    for j in range(k + 1):
                        np.save(pre + f"dk{j}.npy", dk[j][b, g].cpu().numpy())
                        np.save(pre + f"dv{j}.npy", dv[j][b, g].cpu().numpy())
                    pool.submit(d, b, g, G, k, T[b], sh.scale, name, 2e-2, 1e-2)
            del q, dO, out, lse, dq, dk, dv
        res = pool.results()
    finally:
        pool.close()
        import shutil
        shutil.rmtree(d, ignore_errors=True)
    steps_seen = sorted({int(r[0].split("k=")[1].split(",")[0]) for r in res})
    assert steps_seen == sorted(sh.steps)
    bad = []
    for nm, maxabs, atol, rel, rtol in res:
        _parity.record(f"full size {name}", nm, maxabs, atol, rel, rtol)
        if not (maxabs <= atol and rel <= rtol):
            bad.append(f"{nm}: maxabs={maxabs:.3g}/{atol:.3g} relL2={rel:.3g}/{rtol:.3g}")
    assert not bad, "\n".join(bad[:20])
