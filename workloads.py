"""Seeded synthetic jagged-attention workloads, shared by the tests and the benchmark.

This module holds no attention arithmetic: it only draws sequence lengths and
input values, builds offsets, and counts FLOPs and bytes.  Both the CUDA path
and the CPU oracle receive the arrays it returns.

The pages this library follows measure on production ads traffic, which is not
public; these seeded batches stand in for it.  Lengths come from
``numpy.random.default_rng(seed)`` in a fixed draw order, so the sizes
reproduce exactly; values are i.i.d. N(0, 1) drawn with a seeded
``torch.Generator`` in the order Q, K, V, dO, then cast to the compute dtype.

Workloads (named by what they are):

``tiny``    B=4 self-attention, lengths {1, 7, 33, 64}, H=2, D=32, fp32, softmax.
``d64``     B=256 self-attention, lengths uniform in [1, 512], H=4, D=64, bf16, softmax.
``causal``  B=1024 causal self-attention over long user histories, lengths
            lognormal(5.5, 0.8) rounded and clipped to [1, 2048], H=8, D=128, bf16.
``cross``   B=512 asymmetric-QKV cross-attention, query lengths uniform in [1, 64],
            key lengths uniform in [1, 4096], H=4, Dqk=128, Dv=64, bf16, softmax.
``gdpa``    B=256 causal non-softmax attention P = SiLU(QK^T/sqrt(D))/L, lengths uniform
            in [256, 4096], H=8, D=128, bf16.
``pooled``  B=512 pooled multi-head attention: 32 shared learned query rows per head attend
            every sequence, key lengths uniform in [1, 4096], H=4, Dqk=128, Dv=64, bf16,
            softmax.  Q holds the 32 shared rows; O and dO have 32 rows per sequence.
``block``   BlockAttention over the causal workload's sequences (B=1024, lognormal lengths
            clipped to [1, 2048], H=8, D=128, bf16): every row attends only the keys of its
            own 64-row block, causally.
``block_rope``  the same, with the rotary position embedding of q and k.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

ACT_SOFTMAX = 0
ACT_SILU_OVER_LEN = 1


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    heads: int
    dim_qk: int
    dim_v: int
    causal: bool
    act: int
    dtype: torch.dtype
    cross: bool
    pooled: int = 0  # shared query rows per sequence (pooled attention); 0 = not pooled
    block: int = 0   # BlockAttention block length; 0 = whole sequences
    rope: bool = False  # rotary position embedding of q and k (BlockAttention)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.dim_qk)


WORKLOADS = {
    "tiny": Workload("tiny", 4, 2, 32, 32, False, ACT_SOFTMAX, torch.float32, False),
    "d64": Workload("d64", 256, 4, 64, 64, False, ACT_SOFTMAX, torch.bfloat16, False),
    "causal": Workload("causal", 1024, 8, 128, 128, True, ACT_SOFTMAX, torch.bfloat16, False),
    "cross": Workload("cross", 512, 4, 128, 64, False, ACT_SOFTMAX, torch.bfloat16, True),
    "gdpa": Workload("gdpa", 256, 8, 128, 128, True, ACT_SILU_OVER_LEN, torch.bfloat16, False),
    "pooled": Workload("pooled", 512, 4, 128, 64, False, ACT_SOFTMAX, torch.bfloat16, True, 32),
    "block": Workload("block", 1024, 8, 128, 128, True, ACT_SOFTMAX, torch.bfloat16, False, 0, 64),
    "block_rope": Workload("block_rope", 1024, 8, 128, 128, True, ACT_SOFTMAX, torch.bfloat16,
                           False, 0, 64, True),
}


def lengths(name: str, seed: int = 0):
    """Per-sequence (query, key) lengths of a named workload, as int64 numpy arrays."""
    rng = np.random.default_rng(seed)
    if name == "tiny":
        lq = np.array([1, 7, 33, 64], dtype=np.int64)
        return lq, lq.copy()
    if name == "d64":
        lq = rng.integers(1, 512, 256, endpoint=True).astype(np.int64)
        return lq, lq.copy()
    if name in ("causal", "block", "block_rope"):
        lq = np.clip(np.rint(rng.lognormal(5.5, 0.8, 1024)), 1, 2048).astype(np.int64)
        return lq, lq.copy()
    if name == "cross":
        lq = rng.integers(1, 64, 512, endpoint=True).astype(np.int64)
        lk = rng.integers(1, 4096, 512, endpoint=True).astype(np.int64)
        return lq, lk
    if name == "gdpa":
        lq = rng.integers(256, 4096, 256, endpoint=True).astype(np.int64)
        return lq, lq.copy()
    if name == "pooled":
        lk = rng.integers(1, 4096, 512, endpoint=True).astype(np.int64)
        return np.full(512, 32, dtype=np.int64), lk
    raise KeyError(name)


def offsets(lens) -> np.ndarray:
    """Exclusive prefix sum of the lengths, int64 [B+1]."""
    lens = np.asarray(lens, dtype=np.int64)
    out = np.zeros(lens.shape[0] + 1, dtype=np.int64)
    np.cumsum(lens, out=out[1:])
    return out


def values(tq: int, tk: int, heads: int, dim_qk: int, dim_v: int, dtype: torch.dtype,
           seed: int = 0, device="cpu"):
    """Q [tq,H,Dqk], K [tk,H,Dqk], V [tk,H,Dv], dO [tq,H,Dv], N(0,1), drawn in that order."""
    g = torch.Generator(device=device).manual_seed(seed)
    shapes = [(tq, heads, dim_qk), (tk, heads, dim_qk), (tk, heads, dim_v), (tq, heads, dim_v)]
    out = []
    for s in shapes:
        t = torch.randn(s, generator=g, dtype=torch.float32, device=device)
        out.append(t.to(dtype))
    return tuple(out)


def make_batch(w: Workload, lq=None, lk=None, seed: int = 0, device="cpu"):
    """A full input batch for workload ``w`` (or for explicit lengths, if given)."""
    if lq is None:
        lq, lk = lengths(w.name, seed)
    lq = np.asarray(lq, dtype=np.int64)
    lk = lq.copy() if lk is None else np.asarray(lk, dtype=np.int64)
    oq, ok = offsets(lq), offsets(lk)
    q, k, v, do = values(int(oq[-1]), int(ok[-1]), w.heads, w.dim_qk, w.dim_v, w.dtype, seed, device)
    if w.pooled:
        q = q[:w.pooled].contiguous()  # the shared query rows; every lq equals w.pooled
    return dict(lq=lq, lk=lk, offs_q=oq, offs_k=ok, q=q, k=k, v=v, do=do)


def valid_pairs(lq, lk, causal: bool, block: int = 0) -> float:
    """Number of (query, key) pairs that take part in attention, per head.  With ``block``,
    attention stays inside each sequence's consecutive blocks of that many rows."""
    lq = np.asarray(lq, dtype=np.float64)
    lk = np.asarray(lk, dtype=np.float64)
    if block:
        full, rest = np.floor(lq / block), lq % block
        per = (lambda n: n * (n + 1) / 2) if causal else (lambda n: n * n)
        return float(np.sum(full * per(block) + per(rest)))
    if causal:
        return float(np.sum(lq * (lq + 1) / 2))
    return float(np.sum(lq * lk))


def executed_pairs(lq, lk, causal: bool, block: int = 0, tile: int = 128,
                   trim_queries: bool = False) -> float:
    """(query, key) pairs the tensor-core kernels cover with their MMA tiles, per head:
    every tile x tile tile of a sequence's query x key grid that holds at least one valid
    pair (for causal attention, the tiles on and below the diagonal).  With
    ``trim_queries`` (the dK/dV pass, whose products run over a step's valid queries
    only), a tile's query side counts the valid queries rounded up to 16.  With
    ``block``, the sequences are cut into pieces of ``tile`` rows (tile / block blocks,
    masked to their own block inside the tile), each a sequence of its own.
    valid_pairs / executed_pairs is the share of the executed MMA area that does useful
    work."""
    lq = [int(x) for x in np.asarray(lq).ravel()]
    lk = [int(x) for x in np.asarray(lk).ravel()]
    if block:
        cut = lambda n: [tile] * (n // tile) + ([n % tile] if n % tile else [])
        lq = [x for n in lq for x in cut(n)]
        lk = list(lq)

    def rows(a, t):  # query rows a tile at query-tile index t covers
        return ((min(tile, a - t * tile) + 15) // 16 * 16) if trim_queries else tile

    total = 0
    for a, b in zip(lq, lk):
        nq, nk = -(-a // tile), -(-b // tile)
        for t in range(nq):
            keys = min(nk, t + 1) if causal else nk
            total += keys * tile * rows(a, t)
    return float(total)


def useful_flops(w: Workload, lq, lk):
    """(forward, backward) useful FLOPs: no padding and no masked area.

    Forward: QK^T and PV, 2*P*H*(Dqk+Dv).  Backward: one recompute of S, then dV, dP,
    dQ and dK, 2*P*H*(3*Dqk+2*Dv) (2.5 times the forward when Dqk = Dv, the usual
    count for flash attention).  The atomic-free backward computes S and dP once in
    each of its two passes; the second time is not counted.  P = valid pairs per head.
    """
    p = valid_pairs(lq, lk, w.causal, w.block)
    return 2.0 * p * w.heads * (w.dim_qk + w.dim_v), 2.0 * p * w.heads * (3 * w.dim_qk + 2 * w.dim_v)


def algorithmic_bytes(w: Workload, tq: int, tk: int):
    """(forward, backward) minimum HBM bytes the method must move.

    Forward reads Q, K, V and writes O and the fp32 log-sum-exp.  Backward reads
    Q, K, V, O, dO and the log-sum-exp, writes dQ, dK, dV and the fp32 row term D.
    """
    e = torch.tensor([], dtype=w.dtype).element_size()
    H, dq, dv = w.heads, w.dim_qk, w.dim_v
    fwd = e * H * (tq * dq + tk * dq + tk * dv + tq * dv) + 4 * H * tq
    bwd = e * H * (2 * tq * dq + 2 * tk * dq + 2 * tk * dv + 2 * tq * dv) + 8 * H * tq
    return fwd, bwd
