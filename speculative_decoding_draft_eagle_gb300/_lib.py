"""ctypes loader of the in-tree ``libstt.so`` (the C ABI of include/stt.h).

There is no fallback: if the library is missing or fails to load, every entry
point raises.  Build it with ``__graft_entry__.build()`` or
``python -m speculative_decoding_draft_eagle_gb300.build``.
"""

from __future__ import annotations

import ctypes
import os
import threading

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libstt.so")

STATUS = {
    0: "STT_OK",
    -1: "STT_ERR_INVALID_ARG",
    -2: "STT_ERR_UNSUPPORTED",
    -3: "STT_ERR_MISALIGNED",
    -4: "STT_ERR_CUDA",
    -5: "STT_ERR_TIMEOUT",
    -6: "STT_ERR_WORKSPACE",
}

# every symbol include/stt.h declares
EXPORTS = (
    "stt_status_string",
    "stt_version",
    "stt_last_cuda_error",
    "stt_device_error",
    "stt_debug_set_wait_budget",
    "stt_debug_inject",
    "stt_attn_fwd",
    "stt_attn_bwd_workspace_size",
    "stt_attn_bwd",
    "stt_attn_bwd_ex_workspace_size",
    "stt_attn_bwd_ex",
    "soft_ce_workspace_size",
    "soft_ce_fwd_bwd_inplace",
    "soft_ce_fwd_bwd_inplace_ex",
    "soft_ce_fwd_bwd_inplace_noalloc",
    "stt_verify",
    "stt_lm_head_ce_workspace_size",
    "stt_lm_head_ce",
    "stt_profile_start",
    "stt_profile_stop",
    "stt_kernel_name",
)

_lock = threading.Lock()
_lib = None


class SttError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn} failed: {STATUS.get(status, status)} ({msg})")
        self.status = status


def _declare(L):
    c = ctypes
    vp, i32, i64, f32, sz = c.c_void_p, c.c_int, c.c_int64, c.c_float, c.c_size_t
    L.stt_status_string.argtypes = [i32]
    L.stt_status_string.restype = c.c_char_p
    L.stt_version.argtypes = []
    L.stt_version.restype = i32
    L.stt_last_cuda_error.argtypes = [c.POINTER(c.c_char_p)]
    L.stt_last_cuda_error.restype = i32
    L.stt_device_error.argtypes = [vp, c.POINTER(c.c_uint32)]
    L.stt_device_error.restype = i32
    L.stt_debug_set_wait_budget.argtypes = [c.c_uint64]
    L.stt_debug_set_wait_budget.restype = i32
    L.stt_debug_inject.argtypes = [c.c_uint32]
    L.stt_debug_inject.restype = i32
    L.stt_attn_fwd.argtypes = [vp, c.POINTER(vp), c.POINTER(vp), c.POINTER(c.c_int32),
                               i32, i32, i32, i32, i32, i32, f32, vp, vp, vp]
    L.stt_attn_fwd.restype = i32
    L.stt_attn_bwd_workspace_size.argtypes = [i32] * 6
    L.stt_attn_bwd_workspace_size.restype = sz
    L.stt_attn_bwd.argtypes = [vp, c.POINTER(vp), c.POINTER(vp), c.POINTER(c.c_int32),
                               i32, i32, i32, i32, i32, i32, f32, vp, vp, vp, vp,
                               c.POINTER(vp), c.POINTER(vp), vp, sz, vp]
    L.stt_attn_bwd.restype = i32
    L.stt_attn_bwd_ex_workspace_size.argtypes = [i32] * 6 + [c.c_uint32]
    L.stt_attn_bwd_ex_workspace_size.restype = sz
    L.stt_attn_bwd_ex.argtypes = [vp, c.POINTER(vp), c.POINTER(vp), c.POINTER(c.c_int32),
                                  i32, i32, i32, i32, i32, i32, f32, vp, vp, vp, vp,
                                  c.POINTER(vp), c.POINTER(vp), c.c_uint32, vp, sz, vp]
    L.stt_attn_bwd_ex.restype = i32
    L.soft_ce_workspace_size.argtypes = [i64, i64]
    L.soft_ce_workspace_size.restype = sz
    L.soft_ce_fwd_bwd_inplace.argtypes = [vp, vp, vp, i64, i64, vp, vp, vp, sz, vp]
    L.soft_ce_fwd_bwd_inplace.restype = i32
    L.soft_ce_fwd_bwd_inplace_ex.argtypes = [vp, vp, vp, i64, i64, c.c_uint32, vp, vp, vp, sz, vp]
    L.soft_ce_fwd_bwd_inplace_ex.restype = i32
    L.stt_lm_head_ce_workspace_size.argtypes = [i64, i64, i64]
    L.stt_lm_head_ce_workspace_size.restype = sz
    L.stt_lm_head_ce.argtypes = [vp, vp, vp, vp, i64, i64, i64, vp, vp, vp, vp, vp, sz, vp]
    L.stt_lm_head_ce.restype = i32
    L.stt_verify.argtypes = [vp, vp, vp, vp, vp, i32, i32, i64, vp, vp, vp]
    L.stt_verify.restype = i32
    L.soft_ce_fwd_bwd_inplace_noalloc.argtypes = [vp, vp, vp, i64, i64, vp, vp, vp]
    L.soft_ce_fwd_bwd_inplace_noalloc.restype = i32
    L.stt_profile_start.argtypes = [i32]
    L.stt_profile_start.restype = i32
    L.stt_profile_stop.argtypes = [c.POINTER(i32), c.POINTER(i32), c.POINTER(f32), i32]
    L.stt_profile_stop.restype = i32
    L.stt_kernel_name.argtypes = [i32]
    L.stt_kernel_name.restype = c.c_char_p


def load(path: str):
    """Load a copy of the library from `path`; raises if it is missing."""
    if not os.path.exists(path):
        raise RuntimeError(
            f"CUDA library not built: {path} is missing "
            "(run __graft_entry__.build() first); there is no CPU fallback")
    L = ctypes.CDLL(path)
    _declare(L)
    return L


def lib():
    """The in-tree library, loaded once.  Raises if it is missing."""
    global _lib
    with _lock:
        if _lib is None:
            _lib = load(LIB_PATH)
        return _lib


def check(fn: str, status: int):
    if status != 0:
        msg = lib().stt_status_string(status).decode()
        name = ctypes.c_char_p()
        code = lib().stt_last_cuda_error(ctypes.byref(name))
        if code:
            msg += f"; CUDA error {code} {name.value.decode() if name.value else ''}"
        raise SttError(fn, status, msg)
