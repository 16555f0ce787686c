"""Plain fp64 CPU oracle for jagged attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, the smoke check in ``__graft_entry__`` and the CPU-baseline leg
of ``bench.py`` may import this package.  The product path (the CUDA library
``libjfa`` and its Python binding) never imports, links or calls it, and the
two share no code: the arithmetic lives in ``jfa_oracle.c`` (plain loops in
double precision, one (sequence, head) pair at a time) and this module only
marshals numpy arrays into it.

Sources for the definitions (restated in ``jfa_oracle.c``):
Meta GEM MFU co-design write-up (piletech.kr/articles/112134), details
section: jagged-input bullet, Jagged Flash Attention bullet (attention directly
on variable-length tensors; self / cross / asymmetric-QKV patterns) and the
Generalized Dot-Product Attention bullet (non-softmax activation).  The
library fixes that activation to SiLU(u)/L with L the sequence length.

Pooled multi-head attention (``pooled_fwd`` / ``pooled_bwd``) is the cross-attention
above with every sequence's query block equal to the same shared rows, and the
shared rows' gradient summed over sequences.

BlockAttention (``block_fwd`` / ``block_bwd``) is softmax self-attention in which a row
sees only the keys of its own fixed 64-row block of the sequence: the definition above
applied to every block as a sequence of its own.

Rotary position embedding (``rope``) and BlockAttention with it (``block_rope_fwd`` /
``block_rope_bwd``): the BlockAttention bullet pairs the blocks with a fused rotary
position embedding but gives none of its parameters, so the oracle takes the embedding's
published definition (RoFormer, Su et al. 2021, section 3.4): coordinate pairs
(x[2i], x[2i+1]) of a row at position p rotated by the angle p * base^(-2i/D), base
10000, applied to q and k; position p counts rows from the start of the row's sequence.

Every oracle function here has independent pins in ``tests/test_oracle_pins.py``
(50-digit brute force, finite differences, padded dense attention through
torch autograd, closed forms and invariants).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "jfa_oracle.c")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "libjfa_oracle.so")

ACT_SOFTMAX = 0
ACT_SILU_OVER_LEN = 1

_ERRORS = {1: "bad arguments", 2: "bad offsets", 3: "out of memory"}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (OpenMP, -O3, portable flags) and return its path."""
    os.makedirs(_LIB_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        cmd = ["gcc", "-O3", "-std=c11", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64p = ctypes.POINTER(ctypes.c_int64)
            dp = ctypes.POINTER(ctypes.c_double)
            common = [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, i64p, i64p,
                      dp, dp, dp]
            lib.oracle_fwd.argtypes = common + [ctypes.c_double, ctypes.c_int32, ctypes.c_int32,
                                                dp, dp]
            lib.oracle_fwd.restype = ctypes.c_int
            lib.oracle_bwd.argtypes = common + [dp, ctypes.c_double, ctypes.c_int32,
                                                ctypes.c_int32, dp, dp, dp]
            lib.oracle_bwd.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _i64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.int64))


def _ptr(a, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _shapes(q, k, v, offs_q, offs_k):
    if q.ndim != 3 or k.ndim != 3 or v.ndim != 3:
        raise ValueError("q, k, v must be [T, H, D]")
    B = offs_q.shape[0] - 1
    if offs_k.shape[0] != B + 1 or B < 0:
        raise ValueError("offs_q and offs_k must both have B+1 entries")
    Tq, H, Dqk = q.shape
    Tk, Hk, Dk = k.shape
    if Hk != H or Dk != Dqk or v.shape[0] != Tk or v.shape[1] != H:
        raise ValueError("inconsistent q/k/v shapes")
    if B >= 0 and (offs_q[-1] != Tq or offs_k[-1] != Tk):
        raise ValueError("offsets must end at the row counts")
    return B, Tq, Tk, H, Dqk, v.shape[2]


def fwd(q, k, v, offs_q, offs_k=None, scale=None, causal=False, act=ACT_SOFTMAX):
    """Forward pass.  q [Tq,H,Dqk], k [Tk,H,Dqk], v [Tk,H,Dv]; returns (o [Tq,H,Dv], lse [Tq,H])."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    offs_q = _i64(offs_q)
    offs_k = offs_q if offs_k is None else _i64(offs_k)
    B, Tq, Tk, H, Dqk, Dv = _shapes(q, k, v, offs_q, offs_k)
    if scale is None:
        scale = 1.0 / np.sqrt(Dqk)
    o = np.zeros((Tq, H, Dv), dtype=np.float64)
    lse = np.zeros((Tq, H), dtype=np.float64)
    lib = _load()
    dp = ctypes.c_double
    rc = lib.oracle_fwd(B, H, Dqk, Dv, _ptr(offs_q, ctypes.c_int64), _ptr(offs_k, ctypes.c_int64),
                        _ptr(q, dp), _ptr(k, dp), _ptr(v, dp), float(scale), int(bool(causal)),
                        int(act), _ptr(o, dp), _ptr(lse, dp))
    if rc:
        raise ValueError("oracle_fwd: " + _ERRORS.get(rc, str(rc)))
    return o, lse


def bwd(q, k, v, dout, offs_q, offs_k=None, scale=None, causal=False, act=ACT_SOFTMAX):
    """Backward pass.  Returns (dq, dk, dv) with the shapes of q, k, v."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    offs_q = _i64(offs_q)
    offs_k = offs_q if offs_k is None else _i64(offs_k)
    B, Tq, Tk, H, Dqk, Dv = _shapes(q, k, v, offs_q, offs_k)
    if dout.shape != (Tq, H, Dv):
        raise ValueError("dout must be [Tq, H, Dv]")
    if scale is None:
        scale = 1.0 / np.sqrt(Dqk)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    lib = _load()
    dp = ctypes.c_double
    rc = lib.oracle_bwd(B, H, Dqk, Dv, _ptr(offs_q, ctypes.c_int64), _ptr(offs_k, ctypes.c_int64),
                        _ptr(q, dp), _ptr(k, dp), _ptr(v, dp), _ptr(dout, dp), float(scale),
                        int(bool(causal)), int(act), _ptr(dq, dp), _ptr(dk, dp), _ptr(dv, dp))
    if rc:
        raise ValueError("oracle_bwd: " + _ERRORS.get(rc, str(rc)))
    return dq, dk, dv



def pooled_fwd(q, k, v, offs_k, scale=None):
    """Pooled multi-head attention forward: the m rows of q [m,H,Dqk] are the query block of
    every sequence (Meta GEM MFU write-up, details section, jagged-input bullet: pooled
    multi-head attention is one of the attention patterns).  Softmax, non-causal.
    Returns (o [B*m,H,Dv], lse [B*m,H]); sequence b's outputs are rows b*m .. b*m+m-1."""
    q = _f64(q)
    offs_k = _i64(offs_k)
    B, m = offs_k.shape[0] - 1, q.shape[0]
    q_rep = np.tile(q, (max(B, 0), 1, 1))
    offs_q = np.arange(B + 1, dtype=np.int64) * m
    return fwd(q_rep, k, v, offs_q, offs_k, scale=scale)


def pooled_bwd(q, k, v, dout, offs_k, scale=None):
    """Pooled multi-head attention backward: (dq [m,H,Dqk], dk, dv).  The shared queries'
    gradient is the sum over sequences of each sequence's query-block gradient."""
    q = _f64(q)
    offs_k = _i64(offs_k)
    B, m = offs_k.shape[0] - 1, q.shape[0]
    q_rep = np.tile(q, (max(B, 0), 1, 1))
    offs_q = np.arange(B + 1, dtype=np.int64) * m
    dq_rep, dk, dv = bwd(q_rep, k, v, dout, offs_q, offs_k, scale=scale)
    dq = dq_rep.reshape(max(B, 0), m, *q.shape[1:]).sum(axis=0) if B > 0 else np.zeros_like(q)
    return dq, dk, dv


BLOCK = 64  # BlockAttention block length (tokens)


def block_offsets(offs, block=BLOCK):
    """Offsets of the fixed blocks: every sequence cut into pieces of `block` rows from its
    first row on (the last piece of a sequence may be shorter)."""
    offs = _i64(offs)
    out = [0]
    for b in range(offs.shape[0] - 1):
        start, end = int(offs[b]), int(offs[b + 1])
        for s in range(start, end, block):
            out.append(min(s + block, end))
    return np.asarray(out, dtype=np.int64)


def block_fwd(q, k, v, offs, scale=None, causal=False):
    """BlockAttention forward (Meta GEM MFU write-up, details section, BlockAttention bullet:
    attention within fixed 64-token blocks, linear in the sequence length): softmax
    self-attention of every row over the keys of its own block (and, if causal, not after
    it).  Returns (o, lse) like ``fwd``."""
    bo = block_offsets(offs)
    return fwd(q, k, v, bo, bo, scale=scale, causal=causal)


def block_bwd(q, k, v, dout, offs, scale=None, causal=False):
    """BlockAttention backward: (dq, dk, dv)."""
    bo = block_offsets(offs)
    return bwd(q, k, v, dout, bo, bo, scale=scale, causal=causal)


ROPE_BASE = 10000.0  # RoFormer's base for the rotation frequencies


def rope(x, offs, base=ROPE_BASE, inverse=False):
    """Rotary position embedding of x [T, H, D] (D even), rows grouped into sequences by offs:
    row t of sequence b sits at position p = t - offs[b], and its pair i, the coordinates
    (2i, 2i+1), is rotated by the angle p * theta_i with theta_i = base^(-2i/D) (RoFormer,
    Su et al. 2021, section 3.4).  inverse=True rotates by the opposite angle, which is the
    transpose: it maps a gradient with respect to the rotated rows back to the rows."""
    x = _f64(x)
    offs = _i64(offs)
    T, H, D = x.shape
    if D % 2:
        raise ValueError("rope needs an even head dimension, got %d" % D)
    pos = np.zeros(T)
    for b in range(offs.shape[0] - 1):
        start, end = int(offs[b]), int(offs[b + 1])
        pos[start:end] = np.arange(end - start)
    theta = base ** (-2.0 * np.arange(D // 2) / D)
    angle = pos[:, None] * theta[None, :]
    c = np.cos(angle)[:, None, :]
    s = np.sin(angle)[:, None, :]
    if inverse:
        s = -s
    x0, x1 = x[..., 0::2], x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = x0 * c - x1 * s
    out[..., 1::2] = x0 * s + x1 * c
    return out


def block_rope_fwd(q, k, v, offs, scale=None, causal=False, base=ROPE_BASE):
    """BlockAttention with the rotary position embedding applied to q and k first (Meta GEM
    MFU write-up, details section, BlockAttention bullet: fixed blocks combined with a fused
    rotary position embedding).  Returns (o, lse) like ``block_fwd``."""
    return block_fwd(rope(q, offs, base), rope(k, offs, base), v, offs, scale=scale, causal=causal)


def block_rope_bwd(q, k, v, dout, offs, scale=None, causal=False, base=ROPE_BASE):
    """Backward of ``block_rope_fwd``: (dq, dk, dv).  The gradients with respect to the rotated
    q and k are rotated back (the rotation's transpose)."""
    dqr, dkr, dv = block_bwd(rope(q, offs, base), rope(k, offs, base), v, dout, offs, scale=scale,
                             causal=causal)
    return rope(dqr, offs, base, inverse=True), rope(dkr, offs, base, inverse=True), dv
