"""GPU parity of the backward's options and of the TTT step loop, through the
C ABI, against the fp64 oracle.

* STT_BWD_ACCUMULATE_KV: dK_j / dV_j are added to the buffers' contents.
* STT_BWD_BF16_GRADS: bf16 gradients (fp32 sums in the workspace, one
  rounding at the end).
* ``ttt.ttt_attention``: autograd over TTT steps k = 0..K-1, each block's
  gradient summed over the steps that read it by the accumulate flag.

Bounds: the attention bounds (max-abs 2e-2, or twice the bf16 rounding
model's predicted error where larger; relative L2 1e-2), plus, for bf16
outputs, the rounding of each stored value: bf16 keeps 8 significant bits,
so each rounding moves a value by at most 2^-8 of its magnitude, once per
call that writes it (for accumulated buffers, of the sum with what was
there before).
"""

import numpy as np
import pytest
import torch

import _parity
from oracle import attention as oa
from speculative_decoding_draft_eagle_gb300 import ops

pytestmark = pytest.mark.gpu
DEV = "cuda"
CASE = (2, 4, 2, 256, 128, 2, [256, 77])


@pytest.fixture(scope="module", autouse=True)
def _built():
    from speculative_decoding_draft_eagle_gb300 import build
    build.build()


def f64(t):
    return t.detach().double().cpu().numpy()


def _setup(case, seed):
    B, H, H_kv, Q, D, k, T = case
    q, Ks, Vs, dO, T = _parity.make(B, H, H_kv, Q, D, k, T, seed)
    scale = 1.0 / np.sqrt(D)
    qd, Kd, Vd, dOd = q.to(DEV), [x.to(DEV) for x in Ks], [x.to(DEV) for x in Vs], dO.to(DEV)
    out, lse = ops.stt_attn_fwd(qd, Kd, Vd, T, scale)
    args = (f64(q), [f64(x) for x in Ks], [f64(x) for x in Vs], T, scale, f64(dO))
    ref = oa.backward(*args)
    emu = _parity.emulated_backward(*args)
    return (qd, Kd, Vd, dOd, out, lse, T, scale), ref, emu


def _bounds(em, ref, n_round=0, base=None):
    """(max-abs, relative-L2) bounds of one gradient tensor."""
    atol = max(2e-2, 2.0 * float(np.abs(em - ref).max()))
    tot = ref if base is None else base + ref
    nref = float(np.linalg.norm(ref))
    atol += n_round * 2.0 ** -8 * float(np.abs(tot).max())
    rtol = 1e-2 + (n_round * 2.0 ** -8 * float(np.linalg.norm(tot)) / nref if nref > 0 else 0.0)
    return atol, rtol


@pytest.mark.parametrize("bf16", [False, True])
def test_accumulate_adds_to_block_gradients(bf16):
    (qd, Kd, Vd, dOd, out, lse, T, scale), (rq, rk, rv), (eq, ek, ev) = _setup(CASE, 11)
    dt = torch.bfloat16 if bf16 else torch.float32
    g = torch.Generator(device=DEV).manual_seed(5)
    base_k = [torch.randn(x.shape, generator=g, device=DEV).to(dt) for x in Kd]
    base_v = [torch.randn(x.shape, generator=g, device=DEV).to(dt) for x in Vd]
    dk = [x.clone() for x in base_k]
    dv = [x.clone() for x in base_v]
    dq = torch.full(qd.shape, 3.0, device=DEV, dtype=dt)   # dq is overwritten, never added to
    ops.stt_attn_bwd_ex(qd, Kd, Vd, T, out, dOd, lse, dq, dk, dv, scale=scale, accumulate=True)
    assert ops.stt_device_error() == 0
    nr = 1 if bf16 else 0
    grp = "bwd options (bf16)" if bf16 else "bwd options (fp32)"
    _parity.close(f64(dq), rq, "dq", *_bounds(eq, rq, nr), group=grp)
    for j in range(len(Kd)):
        bk, bv = f64(base_k[j]), f64(base_v[j])
        _parity.close(f64(dk[j]) - bk, rk[j], f"dK[{j}]", *_bounds(ek[j], rk[j], nr, bk), group=grp)
        _parity.close(f64(dv[j]) - bv, rv[j], f"dV[{j}]", *_bounds(ev[j], rv[j], nr, bv), group=grp)


def test_bf16_gradients_overwrite():
    (qd, Kd, Vd, dOd, out, lse, T, scale), (rq, rk, rv), (eq, ek, ev) = _setup(CASE, 12)
    dq = torch.full(qd.shape, 7.0, device=DEV, dtype=torch.bfloat16)
    dk = [torch.full(x.shape, -3.0, device=DEV, dtype=torch.bfloat16) for x in Kd]
    dv = [torch.full(x.shape, 5.0, device=DEV, dtype=torch.bfloat16) for x in Vd]
    ops.stt_attn_bwd_ex(qd, Kd, Vd, T, out, dOd, lse, dq, dk, dv, scale=scale)
    assert ops.stt_device_error() == 0
    grp = "bwd options (bf16)"
    _parity.close(f64(dq), rq, "dq", *_bounds(eq, rq, 1), group=grp)
    for j in range(len(Kd)):
        _parity.close(f64(dk[j]), rk[j], f"dK[{j}]", *_bounds(ek[j], rk[j], 1), group=grp)
        _parity.close(f64(dv[j]), rv[j], f"dV[{j}]", *_bounds(ev[j], rv[j], 1), group=grp)


@pytest.mark.parametrize("grad_dtype", [torch.bfloat16])
def test_ttt_step_loop_autograd(grad_dtype):
    """K = 4 TTT steps through torch.autograd: every q_k, K_j and V_j gradient
    against the oracle's backward of each step, summed over the steps."""
    from speculative_decoding_draft_eagle_gb300.ttt import ttt_attention
    B, H, H_kv, Q, D, n = 2, 4, 2, 256, 128, 4
    T = [256, 150]
    g = torch.Generator().manual_seed(21)
    r = lambda *s: torch.randn(*s, generator=g).to(torch.bfloat16)  # noqa: E731
    qs = [r(B, H, Q, D) for _ in range(n)]
    Ks = [r(B, H_kv, Q, D) for _ in range(n)]
    Vs = [r(B, H_kv, Q, D) for _ in range(n)]
    dOs = [r(B, H, Q, D) for _ in range(n)]
    qd = [x.to(DEV).requires_grad_() for x in qs]
    Kd = [x.to(DEV).requires_grad_() for x in Ks]
    Vd = [x.to(DEV).requires_grad_() for x in Vs]
    outs = ttt_attention(qd, Kd, Vd, T)
    torch.autograd.backward(list(outs), [x.to(DEV) for x in dOs])
    assert ops.stt_device_error() == 0
    scale = 1.0 / np.sqrt(D)
    rk = [np.zeros((B, H_kv, Q, D)) for _ in range(n)]
    rv = [np.zeros((B, H_kv, Q, D)) for _ in range(n)]
    grp = "ttt step loop (bf16 grads)"
    for k in range(n):
        O_ref, _ = oa.forward(f64(qs[k]), [f64(x) for x in Ks[: k + 1]], [f64(x) for x in Vs[: k + 1]],
                              T, scale, method="keyset")
        _parity.close(f64(outs[k]), O_ref, f"O[k={k}]", group=grp)
        dq, dk, dv = oa.backward(f64(qs[k]), [f64(x) for x in Ks[: k + 1]],
                                 [f64(x) for x in Vs[: k + 1]], T, scale, f64(dOs[k]))
        _parity.close(f64(qd[k].grad), dq, f"dq[k={k}]", atol=2e-2 + 2.0 ** -8 * np.abs(dq).max(),
                      rtol_l2=1e-2 + 2.0 ** -8, group=grp)
        for j in range(k + 1):
            rk[j] += dk[j]
            rv[j] += dv[j]
    for j in range(n):
        nr = n - j  # steps j..n-1 each round block j's running sum once
        _parity.close(f64(Kd[j].grad), rk[j], f"dK[{j}]",
                      atol=2e-2 + nr * 2.0 ** -8 * np.abs(rk[j]).max(),
                      rtol_l2=1e-2 + nr * 2.0 ** -8, group=grp)
        _parity.close(f64(Vd[j].grad), rv[j], f"dV[{j}]",
                      atol=2e-2 + nr * 2.0 ** -8 * np.abs(rv[j]).max(),
                      rtol_l2=1e-2 + nr * 2.0 ** -8, group=grp)


def test_first_call_on_a_fresh_thread():
    """A thread whose first CUDA work is a library call (the autograd engine's
    worker threads are such threads): the tensor maps must still encode."""
    import threading
    case = (1, 4, 2, 256, 128, 3, [200])
    res = {}

    def work():
        try:
            (qd, Kd, Vd, dOd, out, lse, T, scale), (rq, rk, rv), _ = _setup(case, 17)
            dq = torch.empty(qd.shape, device=DEV, dtype=torch.bfloat16)
            dk = [torch.empty(x.shape, device=DEV, dtype=torch.bfloat16) for x in Kd]
            dv = [torch.empty(x.shape, device=DEV, dtype=torch.bfloat16) for x in Vd]
            ops.stt_attn_bwd_ex(qd, Kd, Vd, T, out, dOd, lse, dq, dk, dv, scale=scale)
            torch.cuda.synchronize()
            res["out"] = (dq, dk, rq, rk)
        except Exception as e:  # pragma: no cover - reported below
            res["err"] = e

    for _ in range(2):
        t = threading.Thread(target=work)
        t.start()
        t.join()
        assert "err" not in res, res.get("err")
        dq, dk, rq, rk = res["out"]
        _parity.close(f64(dq), rq, "dq (fresh thread)", atol=2e-2 + 2.0 ** -8 * np.abs(rq).max(),
                      rtol_l2=1e-2 + 2.0 ** -8, group="bwd options (bf16)")
