"""Python binding of the C ABI, with the same names: argument marshalling only.

Every computation runs in the CUDA library; torch supplies device memory,
streams and output allocation.  Functions take torch CUDA tensors and enqueue
on the current torch stream (or ``stream=``).
"""

from __future__ import annotations

import ctypes
import math
from typing import List, Optional, Sequence, Tuple

import torch

from ._lib import check, lib

__all__ = [
    "stt_attn_fwd",
    "stt_attn_bwd",
    "stt_attn_bwd_workspace_size",
    "stt_attn_bwd_ex",
    "stt_attn_bwd_ex_workspace_size",
    "soft_ce_fwd_bwd_inplace",
    "soft_ce_fwd_bwd_inplace_ex",
    "soft_ce_fwd_bwd_inplace_noalloc",
    "soft_ce_workspace_size",
    "stt_verify",
    "stt_lm_head_ce",
    "stt_device_error",
    "stt_debug_set_wait_budget",
    "stt_debug_inject",
    "stt_version",
]


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _need(t: torch.Tensor, name: str, dtype: torch.dtype, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _ptr_array(ts: Sequence[torch.Tensor]):
    arr = (ctypes.c_void_p * len(ts))()
    for i, t in enumerate(ts):
        arr[i] = t.data_ptr()
    return arr


def _attn_dims(q, k_blocks, v_blocks, T):
    if q.dim() != 4:
        raise ValueError("q must be [B, H, Q_LEN, D]")
    B, H, Q_LEN, D = q.shape
    if len(k_blocks) == 0 or len(k_blocks) != len(v_blocks):
        raise ValueError("k_blocks and v_blocks must both hold k+1 tensors")
    H_kv = k_blocks[0].shape[1]
    _need(q, "q", torch.bfloat16)
    for j, (kb, vb) in enumerate(zip(k_blocks, v_blocks)):
        _need(kb, f"k_blocks[{j}]", torch.bfloat16, (B, H_kv, Q_LEN, D))
        _need(vb, f"v_blocks[{j}]", torch.bfloat16, (B, H_kv, Q_LEN, D))
    Tl = [int(x) for x in (T.tolist() if isinstance(T, torch.Tensor) else T)]
    if len(Tl) != B:
        raise ValueError("T must hold B values")
    T_arr = (ctypes.c_int32 * B)(*Tl)
    return B, H, H_kv, D, Q_LEN, len(k_blocks) - 1, T_arr


def stt_attn_fwd(q: torch.Tensor, k_blocks: Sequence[torch.Tensor],
                 v_blocks: Sequence[torch.Tensor], T, scale: Optional[float] = None,
                 out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                 stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Sparse-tree TTT attention forward at step k = len(k_blocks) - 1.

    Returns (out bf16 [B,H,Q_LEN,D], lse fp32 [B,H,Q_LEN])."""
    B, H, H_kv, D, Q_LEN, k, T_arr = _attn_dims(q, k_blocks, v_blocks, T)
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, Q_LEN), device=q.device, dtype=torch.float32)
    _need(out, "out", torch.bfloat16, q.shape)
    _need(lse, "lse", torch.float32, (B, H, Q_LEN))
    ka, va = _ptr_array(k_blocks), _ptr_array(v_blocks)
    st = lib().stt_attn_fwd(_ptr(q), ka, va, T_arr, B, H, H_kv, D, Q_LEN, k, scale, _ptr(out),
                            _ptr(lse), _stream(stream))
    check("stt_attn_fwd", st)
    return out, lse


def stt_attn_bwd_workspace_size(B, H, H_kv, D, Q_LEN, k) -> int:
    return int(lib().stt_attn_bwd_workspace_size(B, H, H_kv, D, Q_LEN, k))


def stt_attn_bwd(q: torch.Tensor, k_blocks: Sequence[torch.Tensor],
                 v_blocks: Sequence[torch.Tensor], T, out: torch.Tensor, dout: torch.Tensor,
                 lse: torch.Tensor, scale: Optional[float] = None,
                 dq: Optional[torch.Tensor] = None, dk_blocks: Optional[List[torch.Tensor]] = None,
                 dv_blocks: Optional[List[torch.Tensor]] = None,
                 workspace: Optional[torch.Tensor] = None, stream=None):
    """Backward of stt_attn_fwd.  Returns (dq, dk_blocks, dv_blocks), all fp32."""
    B, H, H_kv, D, Q_LEN, k, T_arr = _attn_dims(q, k_blocks, v_blocks, T)
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    _need(out, "out", torch.bfloat16, q.shape)
    _need(dout, "dout", torch.bfloat16, q.shape)
    _need(lse, "lse", torch.float32, (B, H, Q_LEN))
    dev = q.device
    if dq is None:
        dq = torch.empty(q.shape, device=dev, dtype=torch.float32)
    kv_shape = (B, H_kv, Q_LEN, D)
    if dk_blocks is None:
        dk_blocks = [torch.empty(kv_shape, device=dev, dtype=torch.float32) for _ in range(k + 1)]
    if dv_blocks is None:
        dv_blocks = [torch.empty(kv_shape, device=dev, dtype=torch.float32) for _ in range(k + 1)]
    _need(dq, "dq", torch.float32, q.shape)
    for j in range(k + 1):
        _need(dk_blocks[j], f"dk_blocks[{j}]", torch.float32, kv_shape)
        _need(dv_blocks[j], f"dv_blocks[{j}]", torch.float32, kv_shape)
    need = stt_attn_bwd_workspace_size(B, H, H_kv, D, Q_LEN, k)
    if workspace is None:
        workspace = torch.empty(need, device=dev, dtype=torch.uint8)
    st = lib().stt_attn_bwd(_ptr(q), _ptr_array(k_blocks), _ptr_array(v_blocks), T_arr, B, H,
                            H_kv, D, Q_LEN, k, scale, _ptr(out), _ptr(dout), _ptr(lse), _ptr(dq),
                            _ptr_array(dk_blocks), _ptr_array(dv_blocks), _ptr(workspace),
                            workspace.numel() * workspace.element_size(), _stream(stream))
    check("stt_attn_bwd", st)
    return dq, dk_blocks, dv_blocks


STT_BWD_ACCUMULATE_KV = 0x1
STT_BWD_BF16_GRADS = 0x2


def stt_attn_bwd_ex_workspace_size(B, H, H_kv, D, Q_LEN, k, flags) -> int:
    return int(lib().stt_attn_bwd_ex_workspace_size(B, H, H_kv, D, Q_LEN, k, flags))


def stt_attn_bwd_ex(q: torch.Tensor, k_blocks: Sequence[torch.Tensor],
                    v_blocks: Sequence[torch.Tensor], T, out: torch.Tensor, dout: torch.Tensor,
                    lse: torch.Tensor, dq: torch.Tensor, dk_blocks: Sequence[torch.Tensor],
                    dv_blocks: Sequence[torch.Tensor], scale: Optional[float] = None,
                    accumulate: bool = False, workspace: Optional[torch.Tensor] = None,
                    stream=None):
    """Backward of stt_attn_fwd into caller-given gradient buffers, all fp32 or all
    bf16 (the dtype of ``dq`` selects STT_BWD_BF16_GRADS).  With ``accumulate``
    the block gradients are added to dk_blocks / dv_blocks (STT_BWD_ACCUMULATE_KV);
    dq is always overwritten."""
    B, H, H_kv, D, Q_LEN, k, T_arr = _attn_dims(q, k_blocks, v_blocks, T)
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    _need(out, "out", torch.bfloat16, q.shape)
    _need(dout, "dout", torch.bfloat16, q.shape)
    _need(lse, "lse", torch.float32, (B, H, Q_LEN))
    gd = dq.dtype
    if gd not in (torch.float32, torch.bfloat16):
        raise ValueError("gradients must be float32 or bfloat16")
    _need(dq, "dq", gd, q.shape)
    if len(dk_blocks) != k + 1 or len(dv_blocks) != k + 1:
        raise ValueError("dk_blocks and dv_blocks must hold k+1 tensors")
    kv_shape = (B, H_kv, Q_LEN, D)
    for j in range(k + 1):
        _need(dk_blocks[j], f"dk_blocks[{j}]", gd, kv_shape)
        _need(dv_blocks[j], f"dv_blocks[{j}]", gd, kv_shape)
    flags = (STT_BWD_ACCUMULATE_KV if accumulate else 0) | (
        STT_BWD_BF16_GRADS if gd == torch.bfloat16 else 0)
    need = stt_attn_bwd_ex_workspace_size(B, H, H_kv, D, Q_LEN, k, flags)
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(need, device=q.device, dtype=torch.uint8)
    st = lib().stt_attn_bwd_ex(_ptr(q), _ptr_array(k_blocks), _ptr_array(v_blocks), T_arr, B, H,
                               H_kv, D, Q_LEN, k, scale, _ptr(out), _ptr(dout), _ptr(lse),
                               _ptr(dq), _ptr_array(dk_blocks), _ptr_array(dv_blocks), flags,
                               _ptr(workspace), workspace.numel() * workspace.element_size(),
                               _stream(stream))
    check("stt_attn_bwd_ex", st)
    return dq, dk_blocks, dv_blocks


def soft_ce_workspace_size(N: int, V: int) -> int:
    return int(lib().soft_ce_workspace_size(N, V))


def soft_ce_fwd_bwd_inplace(z: torch.Tensor, p: torch.Tensor, g: torch.Tensor,
                            row_loss: Optional[torch.Tensor] = None,
                            loss: Optional[torch.Tensor] = None,
                            workspace: Optional[torch.Tensor] = None, want_row_loss: bool = True,
                            stream=None):
    """In-place soft-CE: z is overwritten with dL/dz.  Returns (loss [1], row_loss [N] or None)."""
    if z.dim() != 2:
        raise ValueError("z must be [N, V]")
    N, V = z.shape
    _need(z, "z", torch.float32)
    _need(p, "p", torch.float32, (N, V))
    _need(g, "g", torch.float32, (N,))
    dev = z.device
    if loss is None:
        loss = torch.empty(1, device=dev, dtype=torch.float32)
    _need(loss, "loss", torch.float32)
    if row_loss is None and want_row_loss:
        row_loss = torch.empty(N, device=dev, dtype=torch.float32)
    if row_loss is not None:
        _need(row_loss, "row_loss", torch.float32, (N,))
    need = soft_ce_workspace_size(N, V)
    if workspace is None:
        workspace = torch.empty(need, device=dev, dtype=torch.uint8)
    st = lib().soft_ce_fwd_bwd_inplace(_ptr(z), _ptr(p), _ptr(g), N, V, _ptr(row_loss),
                                       _ptr(loss), _ptr(workspace),
                                       workspace.numel() * workspace.element_size(),
                                       _stream(stream))
    check("soft_ce_fwd_bwd_inplace", st)
    return loss, row_loss


STT_CE_BF16 = 0x1
STT_CE_G_PER_ELEMENT = 0x2


def soft_ce_fwd_bwd_inplace_ex(z: torch.Tensor, p: torch.Tensor, g: torch.Tensor,
                               row_loss: Optional[torch.Tensor] = None,
                               loss: Optional[torch.Tensor] = None,
                               workspace: Optional[torch.Tensor] = None, stream=None):
    """In-place soft-CE in any of the admitted forms: z and p both fp32 or both
    bf16 (STT_CE_BF16), g fp32 of shape [N] (per row) or [N, V] (per element,
    STT_CE_G_PER_ELEMENT).  z is overwritten with dL/dz in its own dtype.
    Returns (loss [1], row_loss [N])."""
    if z.dim() != 2:
        raise ValueError("z must be [N, V]")
    N, V = z.shape
    if z.dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("z must be float32 or bfloat16")
    _need(z, "z", z.dtype)
    _need(p, "p", z.dtype, (N, V))
    if g.dim() == 2:
        _need(g, "g", torch.float32, (N, V))
    else:
        _need(g, "g", torch.float32, (N,))
    flags = (STT_CE_BF16 if z.dtype == torch.bfloat16 else 0) | (
        STT_CE_G_PER_ELEMENT if g.dim() == 2 else 0)
    dev = z.device
    if loss is None:
        loss = torch.empty(1, device=dev, dtype=torch.float32)
    if row_loss is None:
        row_loss = torch.empty(N, device=dev, dtype=torch.float32)
    _need(loss, "loss", torch.float32)
    _need(row_loss, "row_loss", torch.float32, (N,))
    need = soft_ce_workspace_size(N, V)
    if workspace is None:
        workspace = torch.empty(need, device=dev, dtype=torch.uint8)
    st = lib().soft_ce_fwd_bwd_inplace_ex(_ptr(z), _ptr(p), _ptr(g), N, V, flags, _ptr(row_loss),
                                          _ptr(loss), _ptr(workspace),
                                          workspace.numel() * workspace.element_size(),
                                          _stream(stream))
    check("soft_ce_fwd_bwd_inplace_ex", st)
    return loss, row_loss


def soft_ce_fwd_bwd_inplace_noalloc(z: torch.Tensor, p: torch.Tensor, g: torch.Tensor,
                                    row_loss: Optional[torch.Tensor] = None,
                                    loss: Optional[torch.Tensor] = None, stream=None):
    """Same as soft_ce_fwd_bwd_inplace but without a workspace: the library's own
    fixed scratch is used (at most 65536 rows), for callers that cannot allocate
    device memory.  Calls must not overlap on the GPU."""
    if z.dim() != 2:
        raise ValueError("z must be [N, V]")
    N, V = z.shape
    _need(z, "z", torch.float32)
    _need(p, "p", torch.float32, (N, V))
    _need(g, "g", torch.float32, (N,))
    if loss is None:
        loss = torch.empty(1, device=z.device, dtype=torch.float32)
    _need(loss, "loss", torch.float32)
    if row_loss is not None:
        _need(row_loss, "row_loss", torch.float32, (N,))
    st = lib().soft_ce_fwd_bwd_inplace_noalloc(_ptr(z), _ptr(p), _ptr(g), N, V, _ptr(row_loss),
                                               _ptr(loss), _stream(stream))
    check("soft_ce_fwd_bwd_inplace_noalloc", st)
    return loss, row_loss


STT_ERR_TIMEOUT = -5


def stt_lm_head_ce(h: torch.Tensor, W: torch.Tensor, p: torch.Tensor, g: torch.Tensor,
                   dh: Optional[torch.Tensor] = None, dW: Optional[torch.Tensor] = None,
                   row_loss: Optional[torch.Tensor] = None, loss: Optional[torch.Tensor] = None,
                   workspace: Optional[torch.Tensor] = None, stream=None):
    """Draft LM head z = h W^T fused with the soft-CE: loss and the fp32 gradients
    of h [N, Hd] and W [V, Hd] (both bf16), z never materialised.
    Returns (loss [1], row_loss [N], dh [N, Hd], dW [V, Hd])."""
    if h.dim() != 2 or W.dim() != 2:
        raise ValueError("h must be [N, Hd] and W [V, Hd]")
    N, Hd = h.shape
    V = W.shape[0]
    _need(h, "h", torch.bfloat16)
    _need(W, "W", torch.bfloat16, (V, Hd))
    _need(p, "p", torch.float32, (N, V))
    _need(g, "g", torch.float32, (N,))
    dev = h.device
    if dh is None:
        dh = torch.empty((N, Hd), device=dev, dtype=torch.float32)
    if dW is None:
        dW = torch.empty((V, Hd), device=dev, dtype=torch.float32)
    if row_loss is None:
        row_loss = torch.empty(N, device=dev, dtype=torch.float32)
    if loss is None:
        loss = torch.empty(1, device=dev, dtype=torch.float32)
    _need(dh, "dh", torch.float32, (N, Hd))
    _need(dW, "dW", torch.float32, (V, Hd))
    _need(row_loss, "row_loss", torch.float32, (N,))
    _need(loss, "loss", torch.float32)
    need = int(lib().stt_lm_head_ce_workspace_size(N, Hd, V))
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(need, device=dev, dtype=torch.uint8)
    st = lib().stt_lm_head_ce(_ptr(h), _ptr(W), _ptr(p), _ptr(g), N, Hd, V, _ptr(dh), _ptr(dW),
                              _ptr(row_loss), _ptr(loss), _ptr(workspace),
                              workspace.numel() * workspace.element_size(), _stream(stream))
    check("stt_lm_head_ce", st)
    return loss, row_loss, dh, dW


def stt_verify(p_target: torch.Tensor, p_draft: torch.Tensor, draft_tokens: torch.Tensor,
               u_accept: torch.Tensor, u_sample: torch.Tensor,
               n_accepted: Optional[torch.Tensor] = None,
               out_tokens: Optional[torch.Tensor] = None, stream=None):
    """Rejection-sampling verification of draft tokens.  p_target, p_draft fp32
    [B, gamma, V]; draft_tokens int32 [B, gamma]; u_accept fp32 [B, gamma];
    u_sample fp32 [B].  Returns (n_accepted int32 [B], out_tokens int32 [B, gamma])."""
    if p_target.dim() != 3:
        raise ValueError("p_target must be [B, gamma, V]")
    B, gamma, V = p_target.shape
    _need(p_target, "p_target", torch.float32)
    _need(p_draft, "p_draft", torch.float32, (B, gamma, V))
    _need(draft_tokens, "draft_tokens", torch.int32, (B, gamma))
    _need(u_accept, "u_accept", torch.float32, (B, gamma))
    _need(u_sample, "u_sample", torch.float32, (B,))
    dev = p_target.device
    if n_accepted is None:
        n_accepted = torch.empty(B, device=dev, dtype=torch.int32)
    if out_tokens is None:
        out_tokens = torch.empty((B, gamma), device=dev, dtype=torch.int32)
    _need(n_accepted, "n_accepted", torch.int32, (B,))
    _need(out_tokens, "out_tokens", torch.int32, (B, gamma))
    st = lib().stt_verify(_ptr(p_target), _ptr(p_draft), _ptr(draft_tokens), _ptr(u_accept),
                          _ptr(u_sample), B, gamma, V, _ptr(n_accepted), _ptr(out_tokens),
                          _stream(stream))
    check("stt_verify", st)
    return n_accepted, out_tokens


def stt_device_error(stream=None) -> int:
    """Synchronises the stream, then reads and clears the device error word
    (0 when no bounded wait ran out).  STT_ERR_TIMEOUT is reported through
    the returned word's STT_DEVERR_*_WAIT bits, not raised."""
    w = ctypes.c_uint32(0)
    st = lib().stt_device_error(_stream(stream), ctypes.byref(w))
    if st != STT_ERR_TIMEOUT:
        check("stt_device_error", st)
    return int(w.value)


def stt_debug_set_wait_budget(ns: int) -> None:
    """Bounded-wait budget of every kernel on the current device (0: default)."""
    check("stt_debug_set_wait_budget", lib().stt_debug_set_wait_budget(int(ns)))


def stt_debug_inject(what: int) -> None:
    """Test hook: STT_INJECT_* bits (0 switches injection off)."""
    check("stt_debug_inject", lib().stt_debug_inject(int(what)))


def stt_version() -> int:
    return int(lib().stt_version())
