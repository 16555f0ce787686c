"""Python binding of libjfa (Jagged Flash Attention for GB300): argument marshalling only.

Every function here has the name of the C entry point it calls (see
``include/jfa.h``) and forwards torch CUDA tensors as raw device pointers on
the current CUDA stream.  No attention arithmetic happens in Python and there
is no fallback: if the compiled library is missing or no CUDA device is
present, the calls raise.

Build the library with ``python -m jagged_attention_recsys_gb300.build``.
"""
from __future__ import annotations

import ctypes
import math
import os

import numpy as np
import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libjfa.so")

JFA_OK = 0
JFA_ERR_INVALID_ARG = 1
JFA_ERR_UNSUPPORTED = 2
JFA_ERR_WORKSPACE = 3
JFA_ERR_BAD_OFFSETS = 4
JFA_ERR_TIMEOUT = 5
JFA_ERR_CUDA = 6

JFA_F32 = 0
JFA_BF16 = 1

JFA_PLANNED = 1

KERNEL_KINDS = {"schedule": 0, "fwd": 1, "bwd_d": 2, "bwd_dkdv": 3, "bwd_dq": 4, "aux": 5}

# Every symbol include/jfa.h declares.
EXPORTS = ("jfa_workspace_size", "jfa_fwd", "jfa_bwd", "jfa_cross_fwd", "jfa_cross_bwd",
           "jfa_gdpa_fwd", "jfa_gdpa_bwd", "jfa_status_check", "jfa_status_string",
           "jfa_profile_enable", "jfa_profile_reset", "jfa_profile_read", "jfa_path_for",
           "jfa_fwd_noalloc", "jfa_bbs_plan", "jfa_pooled_workspace_size", "jfa_pooled_fwd",
           "jfa_pooled_bwd", "jfa_block_workspace_size", "jfa_block_fwd", "jfa_block_bwd",
           "jfa_test_hold", "jfa_block_rope_fwd", "jfa_block_rope_bwd", "jfa_plan",
           "jfa_block_plan")


class JfaError(RuntimeError):
    def __init__(self, code, where):
        self.code = code
        super().__init__("%s: %s (status %d)" % (where, status_string(code), code))


class jfa_params(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int64), ("total_q", ctypes.c_int64),
                ("total_k", ctypes.c_int64), ("heads", ctypes.c_int32),
                ("dim_qk", ctypes.c_int32), ("dim_v", ctypes.c_int32),
                ("scale", ctypes.c_float), ("causal", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("flags", ctypes.c_int32)]


_lib = None


def lib():
    """The loaded libjfa (ctypes.CDLL); raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libjfa is not built (%s missing); run "
                               "`python -m jagged_attention_recsys_gb300.build`" % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        vp, i64p, fp = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p
        P = ctypes.POINTER(jfa_params)
        sz = ctypes.c_size_t
        L.jfa_workspace_size.argtypes = [P]
        L.jfa_workspace_size.restype = sz
        L.jfa_path_for.argtypes = [P]
        L.jfa_path_for.restype = ctypes.c_int
        L.jfa_fwd.argtypes = [P, vp, vp, vp, i64p, vp, fp, vp, sz, vp]
        L.jfa_bwd.argtypes = [P, vp, vp, vp, vp, fp, vp, i64p, vp, vp, vp, vp, sz, vp]
        L.jfa_cross_fwd.argtypes = [P, vp, vp, vp, i64p, i64p, vp, fp, vp, sz, vp]
        L.jfa_cross_bwd.argtypes = [P, vp, vp, vp, vp, fp, vp, i64p, i64p, vp, vp, vp, vp, sz, vp]
        L.jfa_gdpa_fwd.argtypes = [P, vp, vp, vp, i64p, i64p, vp, vp, sz, vp]
        L.jfa_gdpa_bwd.argtypes = [P, vp, vp, vp, vp, i64p, i64p, vp, vp, vp, vp, sz, vp]
        for f in ("jfa_fwd", "jfa_bwd", "jfa_cross_fwd", "jfa_cross_bwd", "jfa_gdpa_fwd",
                  "jfa_gdpa_bwd"):
            getattr(L, f).restype = ctypes.c_int
        L.jfa_fwd_noalloc.argtypes = [P, vp, vp, vp, i64p, vp, fp, vp]
        L.jfa_fwd_noalloc.restype = ctypes.c_int
        L.jfa_status_check.argtypes = [vp, vp]
        L.jfa_status_check.restype = ctypes.c_int
        L.jfa_status_string.argtypes = [ctypes.c_int]
        L.jfa_status_string.restype = ctypes.c_char_p
        L.jfa_test_hold.argtypes = [ctypes.c_int]
        L.jfa_test_hold.restype = ctypes.c_int
        L.jfa_profile_enable.argtypes = [ctypes.c_int]
        L.jfa_profile_enable.restype = ctypes.c_int
        L.jfa_profile_reset.argtypes = []
        L.jfa_profile_reset.restype = ctypes.c_int
        L.jfa_profile_read.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_int64),
                                       ctypes.POINTER(ctypes.c_double)]
        L.jfa_profile_read.restype = ctypes.c_int
        L.jfa_bbs_plan.argtypes = [vp, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, vp, vp, vp]
        L.jfa_bbs_plan.restype = ctypes.c_int
        i32 = ctypes.c_int32
        L.jfa_pooled_workspace_size.argtypes = [P, i32]
        L.jfa_pooled_workspace_size.restype = sz
        L.jfa_pooled_fwd.argtypes = [P, i32, vp, vp, vp, i64p, vp, fp, vp, sz, vp]
        L.jfa_pooled_fwd.restype = ctypes.c_int
        L.jfa_pooled_bwd.argtypes = [P, i32, vp, vp, vp, vp, fp, vp, i64p, vp, vp, vp, vp, sz, vp]
        L.jfa_pooled_bwd.restype = ctypes.c_int
        L.jfa_block_workspace_size.argtypes = [P]
        L.jfa_block_workspace_size.restype = sz
        L.jfa_block_fwd.argtypes = [P, vp, vp, vp, i64p, vp, fp, vp, sz, vp]
        L.jfa_block_fwd.restype = ctypes.c_int
        L.jfa_block_bwd.argtypes = [P, vp, vp, vp, vp, fp, vp, i64p, vp, vp, vp, vp, sz, vp]
        L.jfa_block_bwd.restype = ctypes.c_int
        L.jfa_block_rope_fwd.argtypes = [P, vp, vp, vp, i64p, vp, fp, vp, sz, vp]
        L.jfa_block_rope_fwd.restype = ctypes.c_int
        L.jfa_block_rope_bwd.argtypes = [P, vp, vp, vp, vp, fp, vp, i64p, vp, vp, vp, vp, sz, vp]
        L.jfa_block_rope_bwd.restype = ctypes.c_int
        L.jfa_plan.argtypes = [P, i64p, i64p, vp, sz, vp]
        L.jfa_plan.restype = ctypes.c_int
        L.jfa_block_plan.argtypes = [P, i64p, vp, sz, vp]
        L.jfa_block_plan.restype = ctypes.c_int
        _lib = L
    return _lib


def status_string(code: int) -> str:
    return lib().jfa_status_string(int(code)).decode()


def _check(code, where):
    if code != JFA_OK:
        raise JfaError(code, where)


def _dtype_code(t: torch.dtype) -> int:
    if t == torch.float32:
        return JFA_F32
    if t == torch.bfloat16:
        return JFA_BF16
    raise TypeError("libjfa takes fp32 or bf16 tensors, got %s" % t)


def make_params(batch, total_q, total_k, heads, dim_qk, dim_v, dtype, scale=None, causal=False):
    if scale is None:
        scale = 1.0 / math.sqrt(dim_qk)
    return jfa_params(int(batch), int(total_q), int(total_k), int(heads), int(dim_qk),
                      int(dim_v), float(scale), int(bool(causal)), _dtype_code(dtype))


def params_for(q, k, v, offs_q, scale=None, causal=False):
    return make_params(offs_q.numel() - 1, q.shape[0], k.shape[0], q.shape[1], q.shape[2],
                       v.shape[2], q.dtype, scale, causal)


def jfa_workspace_size(p: jfa_params) -> int:
    return int(lib().jfa_workspace_size(ctypes.byref(p)))


def jfa_path_for(p: jfa_params) -> int:
    return int(lib().jfa_path_for(ctypes.byref(p)))


def jfa_bbs_plan(cost, sub=128, ranks=1):
    """Base Batch Shuffling plan (host only): returns (sub_rank, sub_slot, rank_cost) numpy
    arrays for per-sample costs `cost`, `sub` samples per sub-batch and `ranks` ranks."""
    c = np.ascontiguousarray(np.asarray(cost, dtype=np.int64))
    n_sub = -(-c.size // int(sub)) if int(sub) > 0 else 0
    sub_rank = np.zeros(max(n_sub, 1), np.int32)
    sub_slot = np.zeros(max(n_sub, 1), np.int32)
    rank_cost = np.zeros(max(int(ranks), 1), np.int64)
    _check(lib().jfa_bbs_plan(c.ctypes.data if c.size else None, c.size, int(sub), int(ranks),
                              sub_rank.ctypes.data, sub_slot.ctypes.data, rank_cost.ctypes.data),
           "jfa_bbs_plan")
    return sub_rank[:n_sub], sub_slot[:n_sub], rank_cost[:int(ranks)]


def workspace(p: jfa_params, device="cuda") -> torch.Tensor:
    """A device workspace large enough for every call with these params."""
    return torch.empty(max(jfa_workspace_size(p), 256), dtype=torch.uint8, device=device)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check_tensors(q, k, v, offs_q, offs_k=None):
    for t in (q, k, v):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous CUDA tensors")
    for o in (offs_q, offs_k):
        if o is not None and (o.dtype != torch.int64 or not o.is_cuda):
            raise ValueError("offsets must be int64 CUDA tensors")


def _prep(q, k, v, offs_q, offs_k, ws, scale, causal, planned=False):
    _check_tensors(q, k, v, offs_q, offs_k)
    p = params_for(q, k, v, offs_q, scale, causal)
    if planned:
        if ws is None:
            raise ValueError("a planned call needs the workspace its plan was built in")
        p.flags = JFA_PLANNED
    if ws is None:
        ws = workspace(p, q.device)
    return p, ws


def jfa_plan(q, k, v, offs_q, offs_k=None, *, scale=None, causal=False, ws=None, stream=None):
    """Builds the work lists of the forward and backward calls on these inputs' shapes and
    offsets into ``ws`` (allocated if None) and returns ``ws``; later calls given
    ``planned=True``, the same offsets and this workspace skip their own scheduling.
    offs_k=None means self-attention."""
    offs_k = offs_q if offs_k is None else offs_k
    p, ws = _prep(q, k, v, offs_q, offs_k, ws, scale, causal)
    _check(lib().jfa_plan(ctypes.byref(p), _ptr(offs_q), _ptr(offs_k), _ptr(ws), ws.numel(),
                          _stream(stream)), "jfa_plan")
    return ws


def jfa_fwd(q, k, v, offs, *, scale=None, causal=False, o=None, lse=None, ws=None, stream=None,
            planned=False):
    """Softmax self-attention forward; returns (o, lse)."""
    p, ws = _prep(q, k, v, offs, None, ws, scale, causal, planned)
    if o is None:
        o = torch.empty(q.shape[0], q.shape[1], v.shape[2], dtype=q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty(q.shape[0], q.shape[1], dtype=torch.float32, device=q.device)
    _check(lib().jfa_fwd(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(offs), _ptr(o),
                         _ptr(lse), _ptr(ws), ws.numel(), _stream(stream)), "jfa_fwd")
    return o, lse


def jfa_fwd_noalloc(q, k, v, offs, *, scale=None, causal=False, o=None, lse=None, stream=None):
    """jfa_fwd without a workspace (scratch in a static device array); returns (o, lse).

    For callers that cannot allocate device memory; pass preallocated ``o`` and ``lse``
    to keep the call itself free of allocations.
    """
    p = params_for(q, k, v, offs, scale, causal)
    if o is None:
        o = torch.empty(q.shape[0], q.shape[1], v.shape[2], dtype=q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty(q.shape[0], q.shape[1], dtype=torch.float32, device=q.device)
    _check(lib().jfa_fwd_noalloc(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(offs),
                                 _ptr(o), _ptr(lse), _stream(stream)), "jfa_fwd_noalloc")
    return o, lse


def jfa_bwd(q, k, v, o, lse, dout, offs, *, scale=None, causal=False, dq=None, dk=None,
            dv=None, ws=None, stream=None, planned=False):
    """Softmax self-attention backward; returns (dq, dk, dv)."""
    p, ws = _prep(q, k, v, offs, None, ws, scale, causal, planned)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _check(lib().jfa_bwd(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                         _ptr(dout), _ptr(offs), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ws),
                         ws.numel(), _stream(stream)), "jfa_bwd")
    return dq, dk, dv


def jfa_cross_fwd(q, k, v, offs_q, offs_k, *, scale=None, o=None, lse=None, ws=None,
                  stream=None, planned=False):
    """Softmax cross-attention forward (independent key offsets); returns (o, lse)."""
    p, ws = _prep(q, k, v, offs_q, offs_k, ws, scale, False, planned)
    if o is None:
        o = torch.empty(q.shape[0], q.shape[1], v.shape[2], dtype=q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty(q.shape[0], q.shape[1], dtype=torch.float32, device=q.device)
    _check(lib().jfa_cross_fwd(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(offs_q),
                               _ptr(offs_k), _ptr(o), _ptr(lse), _ptr(ws), ws.numel(),
                               _stream(stream)), "jfa_cross_fwd")
    return o, lse


def jfa_cross_bwd(q, k, v, o, lse, dout, offs_q, offs_k, *, scale=None, dq=None, dk=None,
                  dv=None, ws=None, stream=None, planned=False):
    """Backward of jfa_cross_fwd; returns (dq, dk, dv)."""
    p, ws = _prep(q, k, v, offs_q, offs_k, ws, scale, False, planned)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _check(lib().jfa_cross_bwd(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                               _ptr(dout), _ptr(offs_q), _ptr(offs_k), _ptr(dq), _ptr(dk),
                               _ptr(dv), _ptr(ws), ws.numel(), _stream(stream)), "jfa_cross_bwd")
    return dq, dk, dv


def jfa_gdpa_fwd(q, k, v, offs_q, offs_k=None, *, scale=None, causal=False, o=None, ws=None,
                 stream=None, planned=False):
    """SiLU(s)/L attention forward; returns o.  offs_k=None means self-attention."""
    offs_k = offs_q if offs_k is None else offs_k
    p, ws = _prep(q, k, v, offs_q, offs_k, ws, scale, causal, planned)
    if o is None:
        o = torch.empty(q.shape[0], q.shape[1], v.shape[2], dtype=q.dtype, device=q.device)
    _check(lib().jfa_gdpa_fwd(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(offs_q),
                              _ptr(offs_k), _ptr(o), _ptr(ws), ws.numel(), _stream(stream)),
           "jfa_gdpa_fwd")
    return o


def jfa_gdpa_bwd(q, k, v, dout, offs_q, offs_k=None, *, scale=None, causal=False, dq=None,
                 dk=None, dv=None, ws=None, stream=None, planned=False):
    """Backward of jfa_gdpa_fwd; returns (dq, dk, dv)."""
    offs_k = offs_q if offs_k is None else offs_k
    p, ws = _prep(q, k, v, offs_q, offs_k, ws, scale, causal, planned)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _check(lib().jfa_gdpa_bwd(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(dout),
                              _ptr(offs_q), _ptr(offs_k), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ws),
                              ws.numel(), _stream(stream)), "jfa_gdpa_bwd")
    return dq, dk, dv


def jfa_status_check(ws, stream=None) -> int:
    """Synchronises the stream and returns the device status word of the last call on ``ws``."""
    return int(lib().jfa_status_check(_ptr(ws), _stream(stream)))


def jfa_test_hold(on: bool):
    """Test hook of the kernels' bounded waits (see jfa_test_hold in include/jfa.h)."""
    _check(lib().jfa_test_hold(int(bool(on))), "jfa_test_hold")


def jfa_profile_enable(on: bool = True):
    _check(lib().jfa_profile_enable(int(bool(on))), "jfa_profile_enable")


def jfa_profile_reset():
    _check(lib().jfa_profile_reset(), "jfa_profile_reset")


def jfa_profile_read(kind: str):
    """(launches, total_ms) of one kernel kind since the last reset."""
    n = ctypes.c_int64(0)
    ms = ctypes.c_double(0.0)
    _check(lib().jfa_profile_read(KERNEL_KINDS[kind], ctypes.byref(n), ctypes.byref(ms)),
           "jfa_profile_read")
    return int(n.value), float(ms.value)


# ----------------------------------------------------------------------------- pooled attention
def pooled_params(q, k, v, offs_k, scale=None):
    """Params of a pooled call: q [m,H,Dqk] shared rows; B = len(offs_k)-1; o has B*m rows."""
    B, m = offs_k.numel() - 1, q.shape[0]
    return make_params(B, B * m, k.shape[0], q.shape[1], q.shape[2], v.shape[2], q.dtype, scale,
                       False), m


def pooled_workspace(p: jfa_params, m: int, device="cuda") -> torch.Tensor:
    n = int(lib().jfa_pooled_workspace_size(ctypes.byref(p), int(m)))
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device)


def _pooled_prep(q, k, v, offs_k, ws, scale):
    _check_tensors(q, k, v, offs_k)
    p, m = pooled_params(q, k, v, offs_k, scale)
    if ws is None:
        ws = pooled_workspace(p, m, q.device)
    return p, m, ws


def jfa_pooled_fwd(q, k, v, offs_k, *, scale=None, o=None, lse=None, ws=None, stream=None):
    """Pooled multi-head attention forward: the m rows of q attend every sequence;
    returns (o [B*m,H,Dv], lse [B*m,H])."""
    p, m, ws = _pooled_prep(q, k, v, offs_k, ws, scale)
    if o is None:
        o = torch.empty(p.total_q, q.shape[1], v.shape[2], dtype=q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty(p.total_q, q.shape[1], dtype=torch.float32, device=q.device)
    _check(lib().jfa_pooled_fwd(ctypes.byref(p), m, _ptr(q), _ptr(k), _ptr(v), _ptr(offs_k),
                                _ptr(o), _ptr(lse), _ptr(ws), ws.numel(), _stream(stream)),
           "jfa_pooled_fwd")
    return o, lse


def jfa_pooled_bwd(q, k, v, o, lse, dout, offs_k, *, scale=None, dq=None, dk=None, dv=None,
                   ws=None, stream=None):
    """Backward of jfa_pooled_fwd; returns (dq [m,H,Dqk] summed over sequences, dk, dv)."""
    p, m, ws = _pooled_prep(q, k, v, offs_k, ws, scale)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _check(lib().jfa_pooled_bwd(ctypes.byref(p), m, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                _ptr(dout), _ptr(offs_k), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ws),
                                ws.numel(), _stream(stream)), "jfa_pooled_bwd")
    return dq, dk, dv


# ----------------------------------------------------------------------------- BlockAttention
def block_workspace(p: jfa_params, device="cuda") -> torch.Tensor:
    n = int(lib().jfa_block_workspace_size(ctypes.byref(p)))
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device)


def _block_prep(q, k, v, offs, ws, scale, causal, planned=False):
    _check_tensors(q, k, v, offs)
    p = params_for(q, k, v, offs, scale, causal)
    if planned:
        if ws is None:
            raise ValueError("a planned call needs the workspace its plan was built in")
        p.flags = JFA_PLANNED
    return p, block_workspace(p, q.device) if ws is None else ws


def jfa_block_plan(q, k, v, offs, *, scale=None, causal=False, ws=None, stream=None):
    """The block offsets, rotary table and work lists of the BlockAttention calls on these
    inputs, built into ``ws`` (allocated if None); returns ``ws``."""
    p, ws = _block_prep(q, k, v, offs, ws, scale, causal)
    _check(lib().jfa_block_plan(ctypes.byref(p), _ptr(offs), _ptr(ws), ws.numel(),
                                _stream(stream)), "jfa_block_plan")
    return ws


def jfa_block_fwd(q, k, v, offs, *, scale=None, causal=False, o=None, lse=None, ws=None,
                  stream=None, rope=False, planned=False):
    """BlockAttention forward (softmax within fixed 64-row blocks); returns (o, lse).
    With ``rope``, the fused rotary position embedding (jfa_block_rope_fwd)."""
    p, ws = _block_prep(q, k, v, offs, ws, scale, causal, planned)
    if o is None:
        o = torch.empty(q.shape[0], q.shape[1], v.shape[2], dtype=q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty(q.shape[0], q.shape[1], dtype=torch.float32, device=q.device)
    name = "jfa_block_rope_fwd" if rope else "jfa_block_fwd"
    _check(getattr(lib(), name)(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(offs), _ptr(o),
                                _ptr(lse), _ptr(ws), ws.numel(), _stream(stream)), name)
    return o, lse


def jfa_block_bwd(q, k, v, o, lse, dout, offs, *, scale=None, causal=False, dq=None, dk=None,
                  dv=None, ws=None, stream=None, rope=False, planned=False):
    """Backward of jfa_block_fwd; returns (dq, dk, dv).  With ``rope``, the backward of the
    fused rotary position embedding as well (jfa_block_rope_bwd)."""
    p, ws = _block_prep(q, k, v, offs, ws, scale, causal, planned)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    name = "jfa_block_rope_bwd" if rope else "jfa_block_bwd"
    _check(getattr(lib(), name)(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                _ptr(dout), _ptr(offs), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ws),
                                ws.numel(), _stream(stream)), name)
    return dq, dk, dv
