"""Host-side checks of the C ABI: the library builds, loads, exports every declared
symbol, and rejects bad arguments before touching the GPU."""
import ctypes
import os
import re

import pytest

import jagged_attention_recsys_gb300 as jfa
from jagged_attention_recsys_gb300 import build as jbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    jbuild.build()
    return jfa.lib()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "jfa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(jfa_[a-z_0-9]+)\s*\(", text)))


def test_exports_every_declared_symbol(L):
    names = declared_symbols()
    assert len(names) >= 12
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(jfa.EXPORTS)


def test_status_strings(L):
    for code in range(7):
        assert jfa.status_string(code)
    assert jfa.status_string(99) == "unknown status"


def P(**kw):
    base = dict(batch=2, total_q=10, total_k=10, heads=2, dim_qk=64, dim_v=64,
                dtype=jfa.JFA_BF16, scale=0.125, causal=0)
    base.update(kw)
    return jfa.jfa_params(base["batch"], base["total_q"], base["total_k"], base["heads"],
                          base["dim_qk"], base["dim_v"], base["scale"], base["causal"],
                          base["dtype"])


def test_workspace_size_monotone(L):
    a = jfa.jfa_workspace_size(P())
    b = jfa.jfa_workspace_size(P(total_q=100000, total_k=100000))
    assert 0 < a < b
    assert L.jfa_workspace_size(None) == 0
    assert jfa.jfa_workspace_size(P(heads=0)) == 0


def test_path_selection(L):
    assert jfa.jfa_path_for(P(dtype=jfa.JFA_F32, dim_qk=32, dim_v=32)) == 0
    assert jfa.jfa_path_for(P(dim_qk=129)) == -1
    assert jfa.jfa_path_for(P(dim_v=0)) == -1
    assert jfa.jfa_path_for(P(dtype=7)) == -1


def _call_fwd(L, p, ptr=16, ws_ptr=256, ws_bytes=1 << 20):
    vp = ctypes.c_void_p
    return L.jfa_fwd(ctypes.byref(p) if p is not None else None, vp(ptr), vp(ptr), vp(ptr),
                     vp(ptr), vp(ptr), vp(ptr), vp(ws_ptr), ws_bytes, None)


def test_invalid_arguments_rejected_on_host(L):
    # None of these reach a CUDA call: the checks run first and return.
    assert _call_fwd(L, None) == jfa.JFA_ERR_INVALID_ARG
    assert _call_fwd(L, P(heads=0)) == jfa.JFA_ERR_INVALID_ARG
    assert _call_fwd(L, P(batch=-1)) == jfa.JFA_ERR_INVALID_ARG
    assert _call_fwd(L, P(total_k=11)) == jfa.JFA_ERR_INVALID_ARG  # self-attention
    assert _call_fwd(L, P(dim_qk=200)) == jfa.JFA_ERR_UNSUPPORTED
    # work-list items H * (10 // 32 + 2 + 1) = 3H must stay within the 32-bit item index
    assert _call_fwd(L, P(heads=715827883)) == jfa.JFA_ERR_UNSUPPORTED  # 3H = 2^31 + 1
    assert _call_fwd(L, P(heads=715827882)) == jfa.JFA_ERR_WORKSPACE  # 3H = 2^31 - 2
    assert _call_fwd(L, P(causal=2)) == jfa.JFA_ERR_INVALID_ARG
    assert _call_fwd(L, P(scale=float("nan"))) == jfa.JFA_ERR_INVALID_ARG
    assert _call_fwd(L, P(scale=0.0)) == jfa.JFA_ERR_INVALID_ARG
    assert _call_fwd(L, P(scale=-0.1)) == jfa.JFA_ERR_INVALID_ARG
    assert _call_fwd(L, P(batch=0)) == jfa.JFA_ERR_INVALID_ARG  # totals must be 0 too
    assert _call_fwd(L, P(), ptr=8) == jfa.JFA_ERR_INVALID_ARG  # not 16-byte aligned
    assert _call_fwd(L, P(), ptr=0) == jfa.JFA_ERR_INVALID_ARG  # null
    assert _call_fwd(L, P(), ws_ptr=0) == jfa.JFA_ERR_WORKSPACE
    assert _call_fwd(L, P(), ws_ptr=128) == jfa.JFA_ERR_WORKSPACE  # not 256-aligned
    assert _call_fwd(L, P(), ws_bytes=16) == jfa.JFA_ERR_WORKSPACE


def test_cross_rejects_causal(L):
    vp = ctypes.c_void_p
    p = P(causal=1, total_k=30)
    rc = L.jfa_cross_fwd(ctypes.byref(p), vp(16), vp(16), vp(16), vp(16), vp(16), vp(16),
                         vp(16), vp(256), 1 << 20, None)
    assert rc == jfa.JFA_ERR_UNSUPPORTED


def test_pooled_checks_on_host(L):
    vp = ctypes.c_void_p
    # 3 sequences, m = 4 shared query rows: o has 12 rows
    p = P(batch=3, total_q=12, total_k=30)
    assert L.jfa_pooled_workspace_size(ctypes.byref(p), 4) > L.jfa_workspace_size(ctypes.byref(p))
    assert L.jfa_pooled_workspace_size(ctypes.byref(p), 5) == 0  # total_q != B*m

    def fwd(p, m=4, ptr=16, ws_bytes=1 << 24):
        return L.jfa_pooled_fwd(ctypes.byref(p), m, vp(ptr), vp(ptr), vp(ptr), vp(ptr), vp(ptr),
                                vp(ptr), vp(256), ws_bytes, None)

    assert fwd(p, m=0) == jfa.JFA_ERR_INVALID_ARG
    assert fwd(p, m=5) == jfa.JFA_ERR_INVALID_ARG
    assert fwd(P(batch=3, total_q=12, total_k=30, causal=1)) == jfa.JFA_ERR_UNSUPPORTED
    assert fwd(p, ptr=8) == jfa.JFA_ERR_INVALID_ARG  # misaligned: nothing is launched
    assert fwd(p, ws_bytes=1024) == jfa.JFA_ERR_WORKSPACE


def test_profile_read_rejects_bad_kind(L):
    n = ctypes.c_int64()
    ms = ctypes.c_double()
    assert L.jfa_profile_read(99, ctypes.byref(n), ctypes.byref(ms)) == jfa.JFA_ERR_INVALID_ARG


def _flagged(flags, **kw):
    p = P(**kw)
    p.flags = flags
    return p


def test_plan_and_flags_checked_on_host(L):
    vp = ctypes.c_void_p
    # unknown flag bits are argument errors in every call
    assert _call_fwd(L, _flagged(2)) == jfa.JFA_ERR_INVALID_ARG
    assert _call_fwd(L, _flagged(3)) == jfa.JFA_ERR_INVALID_ARG
    assert _call_fwd(L, _flagged(jfa.JFA_PLANNED), ptr=8) == jfa.JFA_ERR_INVALID_ARG

    def plan(p, oq=16, ok=16, ws_ptr=256, ws_bytes=1 << 20):
        return L.jfa_plan(ctypes.byref(p) if p is not None else None, vp(oq), vp(ok), vp(ws_ptr),
                          ws_bytes, None)

    assert plan(None) == jfa.JFA_ERR_INVALID_ARG
    assert plan(P(), oq=0) == jfa.JFA_ERR_INVALID_ARG
    assert plan(P(), ok=8) == jfa.JFA_ERR_INVALID_ARG
    assert plan(P(causal=1, total_k=30)) == jfa.JFA_ERR_INVALID_ARG  # causal: equal totals
    assert plan(_flagged(4)) == jfa.JFA_ERR_INVALID_ARG
    assert plan(P(), ws_ptr=128) == jfa.JFA_ERR_WORKSPACE
    assert plan(P(), ws_bytes=16) == jfa.JFA_ERR_WORKSPACE
    assert L.jfa_block_plan(ctypes.byref(P()), vp(0), vp(256), 1 << 24, None) == jfa.JFA_ERR_INVALID_ARG
    assert L.jfa_block_plan(ctypes.byref(P()), vp(16), vp(256), 64, None) == jfa.JFA_ERR_WORKSPACE
    # calls that cannot use a plan say so before anything is launched
    rc = L.jfa_fwd_noalloc(ctypes.byref(_flagged(jfa.JFA_PLANNED)), vp(16), vp(16), vp(16),
                           vp(16), vp(16), vp(16), None)
    assert rc == jfa.JFA_ERR_UNSUPPORTED
    rc = L.jfa_fwd_noalloc(ctypes.byref(_flagged(2)), vp(16), vp(16), vp(16), vp(16), vp(16),
                           vp(16), None)
    assert rc == jfa.JFA_ERR_INVALID_ARG
    rc = L.jfa_pooled_fwd(ctypes.byref(_flagged(jfa.JFA_PLANNED, batch=3, total_q=12, total_k=30)),
                          4, vp(16), vp(16), vp(16), vp(16), vp(16), vp(16), vp(256), 1 << 24, None)
    assert rc == jfa.JFA_ERR_UNSUPPORTED
