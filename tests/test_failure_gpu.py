"""Failure detection on the GPU without a fault: a bounded wait is made to run
out on purpose, and the kernel must return, report the site in the device
error word and leave the context usable.

The attention forward is launched with the STT_INJECT_FWD_WITHHOLD_Q hook
(its producer never loads the query tile, so the wait for that tile cannot be
satisfied) and a 1 ms wait budget.  Nothing faults, traps or spins: every
wait is bounded, every copy already issued is waited for, and no tensor-core
product is issued.  The next normal launch must then match the oracle with a
clean error word.
"""

import numpy as np
import pytest
import torch

from oracle import attention as oa
from speculative_decoding_draft_eagle_gb300 import ops, workloads as wl

pytestmark = pytest.mark.gpu

STT_INJECT_FWD_WITHHOLD_Q = 0x1
STT_DEVERR_FWD_WAIT = 0x1


@pytest.fixture(scope="module", autouse=True)
def _built():
    from speculative_decoding_draft_eagle_gb300 import build
    build.build()


def _inputs():
    w = wl.WORKLOADS["tiny"]
    T, Ks, Vs, qs, _ = wl.attn_inputs(w.attn, "cpu", w.seed)
    k = w.attn.steps[0]
    return T, Ks[: k + 1], Vs[: k + 1], qs[k], w.attn.scale


def test_bounded_wait_runs_out_and_context_survives():
    T, Ks, Vs, q, scale = _inputs()
    qd, Kd, Vd = q.cuda(), [x.cuda() for x in Ks], [x.cuda() for x in Vs]
    assert ops.stt_device_error() == 0
    try:
        ops.stt_debug_set_wait_budget(1_000_000)      # 1 ms
        ops.stt_debug_inject(STT_INJECT_FWD_WITHHOLD_Q)
        ops.stt_attn_fwd(qd, Kd, Vd, T, scale)         # the launch itself succeeds
        word = ops.stt_device_error()                  # synchronises: the kernel returned
    finally:
        ops.stt_debug_inject(0)
        ops.stt_debug_set_wait_budget(0)
    assert word & STT_DEVERR_FWD_WAIT, f"error word {word:#x}"
    # the error word was read and cleared; a normal launch is clean and correct
    out, lse = ops.stt_attn_fwd(qd, Kd, Vd, T, scale)
    assert ops.stt_device_error() == 0
    f = lambda t: t.detach().float().cpu().numpy().astype(np.float64)  # noqa: E731
    O_ref, lse_ref = oa.forward(f(q), [f(x) for x in Ks], [f(x) for x in Vs], T, scale)
    assert np.abs(f(out) - O_ref).max() <= 2e-2


def test_status_code_of_a_timeout():
    """The C entry point returns STT_ERR_TIMEOUT (-5) with the site in the word."""
    import ctypes
    from speculative_decoding_draft_eagle_gb300 import _lib
    T, Ks, Vs, q, scale = _inputs()
    qd, Kd, Vd = q.cuda(), [x.cuda() for x in Ks], [x.cuda() for x in Vs]
    L = _lib.lib()
    try:
        assert L.stt_debug_set_wait_budget(1_000_000) == 0
        assert L.stt_debug_inject(STT_INJECT_FWD_WITHHOLD_Q) == 0
        ops.stt_attn_fwd(qd, Kd, Vd, T, scale)
        w = ctypes.c_uint32(0)
        st = L.stt_device_error(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream),
                                ctypes.byref(w))
    finally:
        L.stt_debug_inject(0)
        L.stt_debug_set_wait_budget(0)
    assert st == -5 and (w.value & STT_DEVERR_FWD_WAIT)
    w2 = ctypes.c_uint32(7)
    assert L.stt_device_error(None, ctypes.byref(w2)) == 0 and w2.value == 0
