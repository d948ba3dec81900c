"""Host-only checks of the C ABI: the library loads, exports every symbol the
header declares, and rejects bad arguments before touching the GPU."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from speculative_decoding_draft_eagle_gb300 import build, _lib
    build.build()
    return _lib.lib()


def _header_symbols():
    src = open(os.path.join(ROOT, "include", "stt.h")).read()
    return sorted(set(re.findall(r"^STT_API\s+[\w \*]*?\b(\w+)\s*\(", src, re.M)))


def test_header_declares_expected_api():
    from speculative_decoding_draft_eagle_gb300 import _lib
    assert _header_symbols() == sorted(_lib.EXPORTS)


def test_every_declared_symbol_is_exported(L):
    for name in _header_symbols():
        assert hasattr(L, name), name


def test_status_strings(L):
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert L.stt_status_string(code)
    assert L.stt_status_string(123) == b"unknown status"
    assert L.stt_version() >= 100


def _T(vals):
    return (ctypes.c_int32 * len(vals))(*vals)


def _ptrs(vals):
    return (ctypes.c_void_p * len(vals))(*vals)


def test_attn_fwd_rejects_bad_arguments(L):
    good = 0x1000
    kb, vb = _ptrs([good, good]), _ptrs([good, good])
    f = L.stt_attn_fwd
    base = dict(q=good, kb=kb, vb=vb, T=_T([5]), B=1, H=4, Hkv=2, D=128, Q=8, k=1, s=0.1,
                out=good, lse=good)

    def call(**kw):
        a = dict(base, **kw)
        return f(a["q"], a["kb"], a["vb"], a["T"], a["B"], a["H"], a["Hkv"], a["D"], a["Q"], a["k"],
                 a["s"], a["out"], a["lse"], None)
    assert call(q=None) == -1
    assert call(H=3) == -1                 # H % H_kv != 0
    assert call(D=96) == -2                # unsupported head dim
    assert call(T=_T([9])) == -1           # T > Q_LEN
    assert call(T=_T([-1])) == -1
    assert call(k=-1) == -1
    assert call(k=32) == -1
    assert call(B=0) == -1
    assert call(q=good + 8) == -3          # misaligned
    assert call(kb=_ptrs([good, good + 4])) == -3
    assert call(kb=_ptrs([good, 0])) == -1
    assert call(s=float("nan")) == -1
    assert call(s=0.0) == -1               # the kernels need scale > 0
    assert call(s=-0.1) == -1
    assert call(out=None) == -1
    assert call(H=64, Hkv=4) == -2         # group of 16 query heads: unsupported


def test_attn_bwd_workspace_and_rejects(L):
    assert L.stt_attn_bwd_workspace_size(2, 4, 2, 128, 100, 3) >= 2 * 4 * 100 * 4
    good = 0x1000
    kb = _ptrs([good, good])
    st = L.stt_attn_bwd(good, kb, kb, _T([5]), 1, 4, 2, 128, 8, 1, 0.1, good, good, good, good,
                        kb, kb, None, 0, None)
    assert st == -6                        # workspace missing
    st = L.stt_attn_bwd(good, kb, kb, _T([5]), 1, 4, 2, 128, 8, 1, 0.1, good, None, good, good,
                        kb, kb, good, 1 << 20, None)
    assert st == -1


def test_soft_ce_rejects_bad_arguments(L):
    good = 0x1000
    f = L.soft_ce_fwd_bwd_inplace
    assert f(good, good, good, -1, 10, None, good, good, 1 << 20, None) == -1
    assert f(good, good, good, 4, 0, None, good, good, 1 << 20, None) == -1
    assert f(good, good, good, 4, 10, None, None, good, 1 << 20, None) == -1
    assert f(None, good, good, 4, 10, None, good, good, 1 << 20, None) == -1
    assert f(good, good, good, 4, 10, None, good, None, 0, None) == -6
    assert f(good, good, good, 4, 10, None, good, good, 4, None) == -6
    assert f(good, good, good, 4, 10_000_000, None, good, good, 1 << 20, None) == -2
    assert L.soft_ce_workspace_size(1000, 7) >= 4000


def test_binding_fails_loudly_without_library(tmp_path):
    from speculative_decoding_draft_eagle_gb300 import _lib
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        _lib.load(str(tmp_path / "missing.so"))


def test_debug_inject_rejects_unknown_bits(L):
    assert L.stt_debug_inject(0x80) == -1
    assert L.stt_debug_inject(0) == 0


def test_attn_bwd_ex_rejects_bad_flags_and_workspace(L):
    good = 0x1000
    kb = _ptrs([good, good])
    args = (good, kb, kb, _T([5]), 1, 4, 2, 128, 8, 1, 0.1, good, good, good, good, kb, kb)
    assert L.stt_attn_bwd_ex(*args, 0x4, good, 1 << 20, None) == -1    # unknown flag
    assert L.stt_attn_bwd_ex(*args, 0x2, good, 16, None) == -6         # bf16 needs a larger workspace
    assert L.stt_attn_bwd_ex(*args, 0x1, good + 16, 1 << 20, None) == -3  # not 256-byte aligned
    small = L.stt_attn_bwd_ex_workspace_size(1, 4, 2, 128, 8, 1, 0)
    big = L.stt_attn_bwd_ex_workspace_size(1, 4, 2, 128, 8, 1, 2)
    assert small == L.stt_attn_bwd_workspace_size(1, 4, 2, 128, 8, 1)
    assert big >= small + (4 + 2 + 2) * 8 * 128 * 4


def test_soft_ce_ex_rejects_bad_arguments(L):
    good = 0x1000
    f = L.soft_ce_fwd_bwd_inplace_ex
    assert f(good, good, good, 4, 10, 0x8, None, good, good, 1 << 20, None) == -1   # unknown flag
    assert f(good, good, good, -1, 10, 0x1, None, good, good, 1 << 20, None) == -1
    assert f(good, good, good, 4, 10, 0x1, None, good, None, 0, None) == -6
    assert f(good, good, good, 4, 10_000_000, 0x2, None, good, good, 1 << 20, None) == -2


def test_verify_rejects_bad_arguments(L):
    good = 0x1000
    f = L.stt_verify
    assert f(good, good, good, good, good, 0, 5, 100, good, good, None) == 0   # B = 0: nothing to do
    assert f(good, good, good, good, good, 2, 0, 100, good, good, None) == -1
    assert f(good, good, good, good, good, 2, 33, 100, good, good, None) == -1
    assert f(good, good, good, good, good, 2, 5, 0, good, good, None) == -1
    assert f(None, good, good, good, good, 2, 5, 100, good, good, None) == -1
    assert f(good + 2, good, good, good, good, 2, 5, 100, good, good, None) == -3


def test_lm_head_ce_rejects_bad_arguments(L):
    good = 0x1000
    f = L.stt_lm_head_ce
    big = 1 << 30
    assert f(good, good, good, good, -1, 64, 256, good, good, None, good, good, big, None) == -1
    assert f(good, good, good, good, 8, 60, 256, good, good, None, good, good, big, None) == -2
    assert f(good, good, good, good, 8, 64, 250, good, good, None, good, good, big, None) == -2
    assert f(good, good, good, good, 8, 64, 256, good, good, None, good, None, 0, None) == -6
    assert f(good + 8, good, good, good, 8, 64, 256, good, good, None, good, good, big, None) == -3
    assert L.stt_lm_head_ce_workspace_size(4096, 4096, 32000) >= 4096 * 125 * 16
