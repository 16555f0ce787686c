"""Pins of the MXFP8 oracle (oracle/mxfp8.py) against the format's definition, brute force,
hand-worked values, invariants and the plain attention oracle.  CPU only.

The quantiser is checked against the E4M3 bit-pattern definition (every finite code decoded
by sign, biased exponent and mantissa fields), not against its own arithmetic: each finite
value must map to itself, and arbitrary values to the nearest finite value with ties to the
even mantissa, saturating at +-448.
"""
import math

import numpy as np
import pytest

import oracle
from oracle import mxfp8 as mx


def _finite_codes():
    return [c for c in range(256) if not math.isnan(mx.e4m3_decode(c))]


def test_decode_table_landmarks():
    # fixed by the format: bias 7, 3 mantissa bits, S.1111.111 NaN, no infinities
    assert mx.e4m3_decode(0x00) == 0.0
    assert mx.e4m3_decode(0x38) == 1.0            # E = 7, M = 0
    assert mx.e4m3_decode(0x7E) == 448.0          # E = 15, M = 6: the largest normal
    assert math.isnan(mx.e4m3_decode(0x7F)) and math.isnan(mx.e4m3_decode(0xFF))
    assert mx.e4m3_decode(0x08) == 2.0 ** -6      # smallest normal
    assert mx.e4m3_decode(0x01) == 2.0 ** -9      # smallest subnormal
    assert mx.e4m3_decode(0x07) == 7 * 2.0 ** -9  # largest subnormal
    assert mx.e4m3_decode(0xB8) == -1.0
    assert len(_finite_codes()) == 254


def test_every_finite_value_is_fixed():
    vals = np.array([mx.e4m3_decode(c) for c in _finite_codes()])
    assert np.array_equal(mx.e4m3_quantize(vals), vals)


def _nearest_brute(y, codes, vals):
    """Nearest finite E4M3 value by exhaustive search; ties to the code with an even
    mantissa field."""
    d = np.abs(vals - y)
    best = d.min()
    cand = [c for c, dd in zip(codes, d) if dd == best]
    if len(cand) > 1:
        even = [c for c in cand if (c & 1) == 0]
        cand = even or cand
    return mx.e4m3_decode(cand[0])


def test_rounding_matches_exhaustive_nearest():
    codes = _finite_codes()
    vals = np.array([mx.e4m3_decode(c) for c in codes])
    rng = np.random.default_rng(0)
    ys = np.concatenate([
        rng.uniform(-500, 500, 400),
        np.sign(rng.standard_normal(400)) * np.exp2(rng.uniform(-12, 9.5, 400)),
        # midpoints between neighbouring values: ties
        (np.sort(vals)[1:] + np.sort(vals)[:-1]) / 2,
    ])
    got = mx.e4m3_quantize(ys)
    for y, g in zip(ys, got):
        want = _nearest_brute(y, codes, vals)
        assert g == want or (g == 0.0 and want == 0.0), (y, g, want)


def test_hand_worked_roundings():
    q = mx.e4m3_quantize
    assert q(0.1) == 0.1015625        # 0.1 = 1.6 * 2^-4; spacing 2^-7; 12.8 -> 13
    assert q(1.0 / 3.0) == 0.34375    # spacing 2^-5; 10.67 -> 11
    assert q(2.0 ** -10) == 0.0       # half the subnormal spacing: tie to the even 0
    assert q(3 * 2.0 ** -10) == 2.0 ** -8   # 1.5 spacings -> 2 (even)
    assert q(5 * 2.0 ** -10) == 2.0 ** -8   # 2.5 spacings -> 2 (even)
    assert q(460.0) == 448.0          # saturates
    assert q(-1e9) == -448.0
    assert q(1.0625) == 1.0           # tie between 1.0 (M=0) and 1.125 (M=1): even
    assert q(1.1875) == 1.25          # tie between 1.125 (M=1) and 1.25 (M=2): even


def test_block_scale_rule():
    e = lambda a: int(mx.block_scale_exp(np.array(a)))
    assert e(448.0) == 0
    assert e(449.0) == 1
    assert e(1.0) == -8               # ceil(log2(1/448)) = ceil(-8.807)
    assert e(0.875) == -9             # 0.875/448 = 2^-9 exactly
    assert e(0.0) == -127
    assert e(1e300) == 127 and e(1e-300) == -127


def test_block_error_bound_and_scale_invariance():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((40, 96)) * np.exp2(rng.uniform(-20, 20, (40, 1)))
    x[3, 5:20] = 0.0
    xq, ex = mx.mx_quantize_rows(x)
    for c in range(3):
        sl = slice(32 * c, 32 * c + 32)
        X = np.exp2(ex[:, c])[:, None]
        assert np.all(np.max(np.abs(x[:, sl]), axis=1) <= 448.0 * X[:, 0])
        assert np.all(np.abs(xq[:, sl] - x[:, sl]) <= 2.0 ** -4 * np.abs(x[:, sl]) + 2.0 ** -10 * X)
    # power-of-two scaling commutes with the quantiser (no clamping in this range)
    for k in (-7, 3, 11):
        assert np.array_equal(mx.mx_quantize_rows(x * 2.0 ** k)[0], xq * 2.0 ** k)


def test_ragged_last_block():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((3, 40))
    xq, ex = mx.mx_quantize_rows(x)
    assert ex.shape == (3, 2)
    a, _ = mx.mx_quantize_rows(x[:, 32:])       # the 8-wide tail is a block of its own
    assert np.array_equal(xq[:, 32:], a)


def test_tiles_reduce_to_rows_and_share_the_tile_scale():
    rng = np.random.default_rng(3)
    x = rng.random((70, 50))
    # one-row tiles are exactly the 1 x 32 quantisation
    assert np.array_equal(mx.mx_quantize_tiles(x, tile_rows=1)[0], mx.mx_quantize_rows(x)[0])
    # a tile whose rows all equal one row quantises every row as that row alone
    r = rng.random(50)
    t = np.tile(r, (32, 1))
    assert np.array_equal(mx.mx_quantize_tiles(t)[0], np.tile(mx.mx_quantize_rows(r[None])[0], (32, 1)))
    # each tile's exponent comes from the tile's largest value: planting a larger value in
    # one row changes the scale of all 32 rows of that tile and of no other tile
    y = x.copy()
    y[40, 10] = 1000.0
    _, e0 = mx.mx_quantize_tiles(x)
    _, e1 = mx.mx_quantize_tiles(y)
    diff = np.argwhere(e0 != e1)
    assert diff.tolist() == [[1, 0]]
    assert e1[1, 0] == int(mx.block_scale_exp(np.array(1000.0)))


def _batch(lens, H=2, D=64, Dv=64, seed=0):
    rng = np.random.default_rng(seed)
    offs = np.zeros(len(lens) + 1, dtype=np.int64)
    offs[1:] = np.cumsum(lens)
    T = int(offs[-1])
    q = rng.standard_normal((T, H, D))
    k = rng.standard_normal((T, H, D))
    v = rng.standard_normal((T, H, Dv))
    return q, k, v, offs


@pytest.mark.parametrize("causal", [False, True])
def test_unquantised_path_is_the_plain_oracle(causal):
    q, k, v, offs = _batch([1, 0, 33, 70, 7])
    o, lse = mx.attention_fwd(q, k, v, offs, causal=causal, quantize=False)
    ro, rlse = oracle.fwd(q, k, v, offs, scale=1 / 8.0, causal=causal)
    assert np.max(np.abs(o - ro)) < 1e-12
    assert np.max(np.abs(lse - rlse)) < 1e-12


def test_length_one_gives_the_quantised_value_row():
    q, k, v, offs = _batch([1, 1, 1], seed=4)
    o, lse = mx.attention_fwd(q, k, v, offs)
    for t in range(3):
        for h in range(2):
            vq = mx.mx_quantize_rows(v[t:t + 1, h, :].T)[0].T
            assert np.array_equal(o[t, h], vq[0])
    # lse of one key = its score from the quantised q and k
    qq = mx.mx_quantize_rows(q[0:1, 0, :])[0]
    kq = mx.mx_quantize_rows(k[0:1, 0, :])[0]
    assert abs(lse[0, 0] - float((qq @ kq.T)[0, 0]) / 8.0) < 1e-12


def test_zero_queries_give_the_mean_of_the_quantised_values():
    # all scores equal: every weight is exactly 1 before and after quantisation
    q, k, v, offs = _batch([5, 40], seed=5)
    q[:] = 0.0
    o, _ = mx.attention_fwd(q, k, v, offs, causal=True)
    for b in range(2):
        a, e = int(offs[b]), int(offs[b + 1])
        for h in range(2):
            vq = mx.mx_quantize_rows(v[a:e, h, :].T)[0].T
            prefix = np.cumsum(vq, axis=0) / np.arange(1, e - a + 1)[:, None]
            assert np.max(np.abs(o[a:e, h] - prefix)) < 1e-12


def test_quantised_attention_stays_near_the_exact_one():
    # E4M3 keeps 3 mantissa bits: relative errors up to 2^-4 per value; over a batch the
    # errors average out to a few per cent of |o| (measured here, for the record)
    q, k, v, offs = _batch([64, 100, 3], seed=6)
    o, _ = mx.attention_fwd(q, k, v, offs)
    ro, _ = oracle.fwd(q, k, v, offs, scale=1 / 8.0)
    rel = np.linalg.norm(o - ro) / np.linalg.norm(ro)
    assert 1e-3 < rel < 0.08, rel
