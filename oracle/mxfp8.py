"""MXFP8 quantisation and MXFP8 attention forward, in plain numpy fp64 -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, the smoke check and the benchmark's CPU legs may import this module; the
product path never does, and nothing here is shared with the CUDA side.

Source.  Meta GEM MFU co-design write-up (piletech.kr/articles/112134), details section,
MXFP8 training bullet: training uses the GPU's native low-precision format MXFP8; the
softmax output is quantised online (reusing operations the kernel already performs) in
32 x 32 blocks with warp-level quantisation.  The page gives no formula.  The format
itself is the OCP Microscaling (MX) format, v1.0: a block of 32 values shares one scale
X = 2^e stored as E8M0 (an 8-bit exponent, bias 127, e in [-127, 127]); each value is
stored as FP8 E4M3 (1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits; normal
numbers 2^-6 .. 448, subnormals m * 2^-9 for m = 1..7, no infinities).

Readings where the page is silent (each is listed in the design notes):

* Element rounding: round to nearest, ties to even mantissa, as IEEE conversions do.
  Values beyond the largest normal (448) saturate to +-448.
* Block scale: the smallest power of two X with max|x| / X <= 448, i.e.
  e = ceil(log2(max|x| / 448)), clamped to [-127, 127]; an all-zero block takes e = -127.
  (OCP's example conversion takes e = floor(log2 max|x|) - 8 and saturates the block
  maximum when its mantissa is 1.75 or more -- for softmax weights, whose block maxima sit
  near 1, that clips the largest weights by up to 12.5%.  The rounded-up scale never
  saturates: every normal element keeps a relative error of at most 2^-4.)
* Block shapes.  The tensor cores take one scale per 32 consecutive elements along the
  contraction dimension ("1 x 32").  Q and K are blocked along the head dimension; V,
  whose contraction dimension in P V is the key index, is blocked along 32 consecutive
  key rows of one sequence (per column); the softmax output P is blocked in 32 x 32
  tiles of a sequence's (query row, key) grid, the page's warp-level blocks: one warp
  holds 32 query rows, one per thread, so the tile's maximum is a warp reduction.  A
  32 x 32 tile is a special case of 1 x 32 blocks: its 32 rows each take the tile's
  scale for those 32 keys (``mx_quantize_tiles`` is written that way and pinned).
  Blocks start at a sequence's first row and key; the last block of a sequence may be
  shorter.
* What is quantised in the forward: P~ = exp(s - m) with m the exact row maximum over
  the valid keys (values in (0, 1]); the row sum l = sum_j P~_ij is taken before
  quantisation; o_i = sum_j Q(P~)_ij Q(V)_j / l_i; lse_i = m_i + ln l_i.  The scores use
  the quantised Q and K.
"""
from __future__ import annotations

import math

import numpy as np

E4M3_MAX = 448.0
E4M3_MIN_NORMAL_EXP = -6   # smallest normal 2^-6
E4M3_MANTISSA_BITS = 3
E8M0_MIN_EXP = -127
E8M0_MAX_EXP = 127
BLOCK = 32


def e4m3_decode(code: int) -> float:
    """The value of an E4M3 bit pattern (0..255), from the format's definition: sign, 4-bit
    exponent field E with bias 7, 3-bit mantissa field M; E = 0 is subnormal (M/8 * 2^-6);
    S.1111.111 is NaN (there are no infinities)."""
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return s * (m / 8.0) * 2.0 ** -6
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def e4m3_quantize(y):
    """Round fp64 values to the nearest E4M3 value (ties to even), saturating at +-448.

    For |y| >= 2^-6 the spacing of E4M3 values in y's binade [2^e, 2^(e+1)) is 2^(e-3);
    below 2^-6 (subnormals) it is 2^-9.  y divided by its spacing is exact in fp64, and
    numpy's rint rounds half to even.
    """
    y = np.asarray(y, dtype=np.float64)
    a = np.abs(y)
    _, ex = np.frexp(a)            # a = f * 2^ex with f in [0.5, 1): floor(log2 a) = ex - 1
    e = ex.astype(np.int64) - 1
    e = np.maximum(e, E4M3_MIN_NORMAL_EXP)   # subnormal range shares the 2^-6 binade's spacing
    spacing = np.ldexp(1.0, e - E4M3_MANTISSA_BITS)
    q = np.rint(a / spacing) * spacing
    q = np.minimum(q, E4M3_MAX)
    q = np.where(a == 0, 0.0, q)
    return np.copysign(q, y)


def block_scale_exp(amax):
    """E8M0 exponent of a block with largest magnitude ``amax``: the smallest e with
    amax / 2^e <= 448, clamped to [-127, 127]; -127 for an all-zero block."""
    amax = np.asarray(amax, dtype=np.float64)
    out = np.full(amax.shape, E8M0_MIN_EXP, dtype=np.int64)
    nz = amax > 0
    r = amax[nz] / E4M3_MAX
    # ceil(log2 r) exactly: r = f 2^k with f in [0.5, 1) -> log2 r in [k-1, k); it equals k-1
    # only when f == 0.5 (r a power of two)
    f, k = np.frexp(r)
    e = np.where(f == 0.5, k - 1, k).astype(np.int64)
    out[nz] = np.clip(e, E8M0_MIN_EXP, E8M0_MAX_EXP)
    return out


def mx_quantize_rows(x, block=BLOCK):
    """MX quantisation of a 2-D array along its last axis in blocks of ``block`` consecutive
    elements (the last block may be shorter).  Returns (dequantised values, exponents
    [rows, n_blocks])."""
    x = np.asarray(x, dtype=np.float64)
    rows, n = x.shape
    nb = -(-n // block) if n else 0
    out = np.empty_like(x)
    exps = np.empty((rows, nb), dtype=np.int64)
    for c in range(nb):
        sl = slice(c * block, min(n, (c + 1) * block))
        e = block_scale_exp(np.max(np.abs(x[:, sl]), axis=1))
        exps[:, c] = e
        scale = np.ldexp(1.0, e)[:, None]
        out[:, sl] = e4m3_quantize(x[:, sl] / scale) * scale
    return out, exps


def mx_quantize_tiles(x, tile_rows=BLOCK, block=BLOCK):
    """MX quantisation of a 2-D array in tiles of ``tile_rows`` x ``block`` elements with one
    scale per tile, written as 1 x ``block`` blocks whose ``tile_rows`` rows share the
    tile's scale (the largest magnitude of the whole tile).  Returns (dequantised values,
    exponents [n_row_tiles, n_blocks])."""
    x = np.asarray(x, dtype=np.float64)
    rows, n = x.shape
    nb = -(-n // block) if n else 0
    nt = -(-rows // tile_rows) if rows else 0
    out = np.empty_like(x)
    exps = np.empty((nt, nb), dtype=np.int64)
    for t in range(nt):
        rs = slice(t * tile_rows, min(rows, (t + 1) * tile_rows))
        for c in range(nb):
            cs = slice(c * block, min(n, (c + 1) * block))
            e = int(block_scale_exp(np.max(np.abs(x[rs, cs])))) if x[rs, cs].size else E8M0_MIN_EXP
            exps[t, c] = e
            scale = math.ldexp(1.0, e)
            out[rs, cs] = e4m3_quantize(x[rs, cs] / scale) * scale
    return out, exps


def _identity(x):
    return np.asarray(x, dtype=np.float64)


def attention_fwd(q, k, v, offs, scale=None, causal=False, quantize=True):
    """MXFP8 softmax self-attention forward over a jagged batch, one (sequence, head) at a
    time.  q, k [T, H, Dqk], v [T, H, Dv] fp64 (the values the caller passes, e.g. bf16);
    offs int64 [B+1].  Returns (o [T, H, Dv], lse [T, H]).

    With ``quantize=False`` every quantiser is the identity and the result is plain
    softmax attention (the same definition as the C oracle), which pins the arithmetic
    around the quantisers.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    offs = np.asarray(offs, dtype=np.int64)
    T, H, Dqk = q.shape
    Dv = v.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(Dqk)
    o = np.zeros((T, H, Dv))
    lse = np.full((T, H), -np.inf)
    rows_q = (lambda a: mx_quantize_rows(a)[0]) if quantize else _identity
    tiles_p = (lambda a: mx_quantize_tiles(a)[0]) if quantize else _identity
    for b in range(len(offs) - 1):
        a, e = int(offs[b]), int(offs[b + 1])
        L = e - a
        if L == 0:
            continue
        for h in range(H):
            qh = rows_q(q[a:e, h, :])            # 1 x 32 blocks along Dqk
            kh = rows_q(k[a:e, h, :])
            vh = rows_q(v[a:e, h, :].T).T         # 1 x 32 blocks along the key index
            s = scale * (qh @ kh.T)               # [L, L]
            valid = np.ones((L, L), dtype=bool)
            if causal:
                valid = np.tril(valid)
            m = np.max(np.where(valid, s, -np.inf), axis=1)
            pt = np.where(valid, np.exp(s - m[:, None]), 0.0)
            l = np.sum(pt, axis=1)
            pq = tiles_p(pt)                      # 32 x 32 tiles of the (row, key) grid
            o[a:e, h, :] = (pq @ vh) / l[:, None]
            lse[a:e, h] = m + np.log(l)
    return o, lse
