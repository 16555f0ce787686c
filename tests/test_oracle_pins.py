"""Pins for the fp64 CPU oracle: checks against something other than the oracle itself.

The pages print no worked example, so the oracle is pinned by mathematics:
  * a hand-worked two-token example with closed-form values (tests/golden),
  * 50-digit brute force with mpmath (no max subtraction; gradients by
    high-precision central differences, not by the analytic formulas),
  * fp64 central finite differences of the oracle's own forward pass,
  * padded dense attention with an explicit mask, differentiated by torch autograd,
  * closed forms (length 1, zero queries, constant values), invariants
    (sequence order, head split, key shift, log-sum-exp consistency) and the
    length-0 conventions.
Each is chosen so that a plausible slip in the oracle (a dropped term, a wrong
sign, index or normaliser, a transposed operand, an off-by-one causal mask)
fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
SM, GD = oracle.ACT_SOFTMAX, oracle.ACT_SILU_OVER_LEN


def _offs(lens):
    o = np.zeros(len(lens) + 1, dtype=np.int64)
    o[1:] = np.cumsum(lens)
    return o


def _rand(lq, lk, H, Dqk, Dv, seed):
    rng = np.random.default_rng(seed)
    tq, tk = int(sum(lq)), int(sum(lk))
    q = rng.standard_normal((tq, H, Dqk))
    k = rng.standard_normal((tk, H, Dqk))
    v = rng.standard_normal((tk, H, Dv))
    do = rng.standard_normal((tq, H, Dv))
    return q, k, v, do


# --------------------------------------------------------------------------------------
# Hand-worked example (closed form)
# --------------------------------------------------------------------------------------
def _ev(x):
    if isinstance(x, list):
        return [_ev(y) for y in x]
    return eval(x, {"__builtins__": {}}, {"log": math.log})


@pytest.mark.parametrize("variant", ["softmax", "softmax_causal", "gdpa", "gdpa_causal"])
def test_hand_worked_example(variant):
    g = json.load(open(os.path.join(GOLDEN, "hand_worked_2x2.json")))
    q, k, v, do = (np.array(_ev(g[n])) for n in ("q", "k", "v", "dout"))
    offs = np.array([0, 2])
    act = GD if variant.startswith("gdpa") else SM
    causal = variant.endswith("causal")
    o, lse = oracle.fwd(q, k, v, offs, scale=g["scale"], causal=causal, act=act)
    exp = g[variant]
    np.testing.assert_allclose(o, np.array(_ev(exp["o"])), rtol=0, atol=1e-14)
    if "lse" in exp:
        np.testing.assert_allclose(lse, np.array(_ev(exp["lse"])), rtol=0, atol=1e-14)
    if "dq" in exp:
        dq, dk, dv = oracle.bwd(q, k, v, do, offs, scale=g["scale"], causal=causal, act=act)
        for got, name in ((dq, "dq"), (dk, "dk"), (dv, "dv")):
            np.testing.assert_allclose(got, np.array(_ev(exp[name])), rtol=0, atol=1e-14)


# --------------------------------------------------------------------------------------
# 50-digit brute force (mpmath)
# --------------------------------------------------------------------------------------
def _mp_forward(mp, q, k, v, lq, lk, H, scale, causal, act):
    """Direct evaluation of the definitions in 50-digit arithmetic, no max subtraction."""
    oq, ok = _offs(lq), _offs(lk)
    tq, dv = len(q), len(v[0][0])
    o = [[[mp.mpf(0)] * dv for _ in range(H)] for _ in range(tq)]
    lse = [[mp.mpf(0)] * H for _ in range(tq)]
    for b in range(len(lq)):
        for h in range(H):
            for i in range(lq[b]):
                cols = [j for j in range(lk[b]) if (not causal or j <= i)]
                qi = q[oq[b] + i][h]
                u = {j: scale * mp.fsum(qi[d] * k[ok[b] + j][h][d] for d in range(len(qi)))
                     for j in cols}
                if act == SM:
                    z = mp.fsum(mp.exp(u[j]) for j in cols)
                    w = {j: mp.exp(u[j]) / z for j in cols}
                    lse[oq[b] + i][h] = mp.log(z) if cols else mp.mpf("-inf")
                else:
                    w = {j: u[j] / (1 + mp.exp(-u[j])) / lq[b] for j in cols}
                for c in range(dv):
                    o[oq[b] + i][h][c] = mp.fsum(w[j] * v[ok[b] + j][h][c] for j in cols)
    return o, lse


@pytest.mark.parametrize("act,causal", [(SM, False), (SM, True), (GD, False), (GD, True)])
def test_mpmath_brute_force(act, causal):
    mpmath = pytest.importorskip("mpmath")
    mp = mpmath.mp
    mp.dps = 50
    lq = [3, 1, 5]
    lk = lq if causal else [2, 4, 5]
    H, Dqk, Dv = 2, 3, 4
    q, k, v, do = _rand(lq, lk, H, Dqk, Dv, seed=11)
    scale = 0.7
    o, lse = oracle.fwd(q, k, v, _offs(lq), _offs(lk), scale=scale, causal=causal, act=act)
    Q, K, V, DO = ([[[mp.mpf(float(x)) for x in row] for row in t] for t in a]
                   for a in (q, k, v, do))
    mo, mlse = _mp_forward(mp, Q, K, V, lq, lk, H, mp.mpf(scale), causal, act)
    np.testing.assert_allclose(o, np.array(mo, dtype=float), rtol=0, atol=1e-13)
    if act == SM:
        np.testing.assert_allclose(lse, np.array(mlse, dtype=float), rtol=0, atol=1e-13)

    # Gradients of the scalar loss <O, dO> by 50-digit central differences.
    dq, dk, dv = oracle.bwd(q, k, v, do, _offs(lq), _offs(lk), scale=scale, causal=causal, act=act)
    h = mp.mpf("1e-20")

    def loss(Qx, Kx, Vx):
        ox, _ = _mp_forward(mp, Qx, Kx, Vx, lq, lk, H, mp.mpf(scale), causal, act)
        return mp.fsum(ox[t][hh][c] * DO[t][hh][c] for t in range(len(ox)) for hh in range(H)
                       for c in range(Dv))

    rng = np.random.default_rng(5)
    for which, grad in ((0, dq), (1, dk), (2, dv)):
        base = [Q, K, V][which]
        for _ in range(4):  # a few random entries per tensor
            t = int(rng.integers(0, len(base)))
            hh = int(rng.integers(0, H))
            d = int(rng.integers(0, len(base[0][0])))
            plus = [[[x for x in r] for r in m] for m in base]
            minus = [[[x for x in r] for r in m] for m in base]
            plus[t][hh][d] += h
            minus[t][hh][d] -= h
            args_p = [Q, K, V]
            args_m = [Q, K, V]
            args_p[which] = plus
            args_m[which] = minus
            fd = (loss(*args_p) - loss(*args_m)) / (2 * h)
            assert abs(float(fd) - grad[t, hh, d]) <= 1e-12 * max(1.0, abs(float(fd)))


# --------------------------------------------------------------------------------------
# fp64 finite differences of the oracle's own forward
# --------------------------------------------------------------------------------------
@pytest.mark.parametrize("act,causal,cross", [(SM, False, False), (SM, True, False),
                                              (SM, False, True), (GD, False, False),
                                              (GD, True, False), (GD, False, True)])
def test_finite_differences(act, causal, cross):
    lq = [9, 1, 17, 4]
    lk = [13, 6, 3, 20] if cross else lq
    H, Dqk, Dv = 2, 8, 6 if cross else 8
    q, k, v, do = _rand(lq, lk, H, Dqk, Dv, seed=3)
    oq, ok = _offs(lq), _offs(lk)
    kw = dict(scale=0.4, causal=causal, act=act)
    dq, dk, dv = oracle.bwd(q, k, v, do, oq, ok, **kw)

    def loss(qx, kx, vx):
        return float(np.sum(oracle.fwd(qx, kx, vx, oq, ok, **kw)[0] * do))

    rng = np.random.default_rng(9)
    eps = 1e-6
    for which, grad in ((0, dq), (1, dk), (2, dv)):
        for _ in range(3):
            u = rng.standard_normal(grad.shape)
            args_p = [q, k, v]
            args_m = [q, k, v]
            args_p[which] = args_p[which] + eps * u
            args_m[which] = args_m[which] - eps * u
            fd = (loss(*args_p) - loss(*args_m)) / (2 * eps)
            an = float(np.sum(grad * u))
            assert abs(fd - an) <= 1e-7 * max(1.0, abs(an)), (which, fd, an)


# --------------------------------------------------------------------------------------
# Padded dense attention + explicit mask, gradients by torch autograd (fp64)
# --------------------------------------------------------------------------------------
def _padded_reference(q, k, v, do, lq, lk, H, scale, causal, act):
    B = len(lq)
    mq, mk = max(max(lq), 1), max(max(lk), 1)
    oq, ok = _offs(lq), _offs(lk)
    Dqk, Dv = q.shape[2], v.shape[2]
    Qp = torch.zeros(B, H, mq, Dqk, dtype=torch.float64)
    Kp = torch.zeros(B, H, mk, Dqk, dtype=torch.float64)
    Vp = torch.zeros(B, H, mk, Dv, dtype=torch.float64)
    DOp = torch.zeros(B, H, mq, Dv, dtype=torch.float64)
    mask = torch.zeros(B, 1, mq, mk, dtype=torch.bool)
    for b in range(B):
        Qp[b, :, :lq[b]] = torch.from_numpy(q[oq[b]:oq[b + 1]]).permute(1, 0, 2)
        Kp[b, :, :lk[b]] = torch.from_numpy(k[ok[b]:ok[b + 1]]).permute(1, 0, 2)
        Vp[b, :, :lk[b]] = torch.from_numpy(v[ok[b]:ok[b + 1]]).permute(1, 0, 2)
        DOp[b, :, :lq[b]] = torch.from_numpy(do[oq[b]:oq[b + 1]]).permute(1, 0, 2)
        m = torch.zeros(mq, mk, dtype=torch.bool)
        m[:lq[b], :lk[b]] = True
        if causal:
            m &= torch.ones(mq, mk, dtype=torch.bool).tril()
        mask[b, 0] = m
    Qp.requires_grad_(True)
    Kp.requires_grad_(True)
    Vp.requires_grad_(True)
    S = scale * Qp @ Kp.transpose(-1, -2)
    if act == SM:
        Sm = S.masked_fill(~mask, float("-inf"))
        P = torch.softmax(Sm, dim=-1).nan_to_num(0.0)
        lse = torch.logsumexp(Sm, dim=-1)
    else:
        L = torch.tensor(lq, dtype=torch.float64).view(B, 1, 1, 1).clamp(min=1)
        P = (torch.nn.functional.silu(S) / L) * mask
        lse = None
    O = P @ Vp
    (O * DOp).sum().backward()

    def unpad(X, lens, offs):
        out = np.zeros((int(offs[-1]), H, X.shape[-1]))
        for b in range(B):
            out[offs[b]:offs[b + 1]] = X[b, :, :lens[b]].permute(1, 0, 2).detach().numpy()
        return out

    res = dict(o=unpad(O, lq, oq), dq=unpad(Qp.grad, lq, oq), dk=unpad(Kp.grad, lk, ok),
               dv=unpad(Vp.grad, lk, ok))
    if lse is not None:
        res["lse"] = unpad(lse.unsqueeze(-1), lq, oq)[..., 0]
    return res


@pytest.mark.parametrize("act,causal,cross", [(SM, False, False), (SM, True, False),
                                              (SM, False, True), (GD, False, False),
                                              (GD, True, False), (GD, False, True)])
def test_padded_dense_autograd(act, causal, cross):
    lq = [1, 7, 33, 64, 2]
    lk = [5, 64, 1, 40, 17] if cross else lq
    H, Dqk, Dv = 2, 16, 8 if cross else 16
    q, k, v, do = _rand(lq, lk, H, Dqk, Dv, seed=21)
    oq, ok = _offs(lq), _offs(lk)
    scale = 1.0 / math.sqrt(Dqk)
    o, lse = oracle.fwd(q, k, v, oq, ok, scale=scale, causal=causal, act=act)
    dq, dk, dv = oracle.bwd(q, k, v, do, oq, ok, scale=scale, causal=causal, act=act)
    ref = _padded_reference(q, k, v, do, lq, lk, H, scale, causal, act)
    for got, name in ((o, "o"), (dq, "dq"), (dk, "dk"), (dv, "dv")):
        np.testing.assert_allclose(got, ref[name], rtol=0, atol=1e-12, err_msg=name)
    if act == SM:
        np.testing.assert_allclose(lse, ref["lse"], rtol=0, atol=1e-12)


def test_matches_torch_sdpa():
    """Equal-length batch: torch's own scaled_dot_product_attention routine, fp64."""
    B, L, H, D = 3, 11, 2, 8
    q, k, v, do = _rand([L] * B, [L] * B, H, D, D, seed=4)
    for causal in (False, True):
        o, _ = oracle.fwd(q, k, v, _offs([L] * B), causal=causal)
        tq = torch.from_numpy(q).view(B, L, H, D).transpose(1, 2)
        tk = torch.from_numpy(k).view(B, L, H, D).transpose(1, 2)
        tv = torch.from_numpy(v).view(B, L, H, D).transpose(1, 2)
        ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal)
        np.testing.assert_allclose(o, ref.transpose(1, 2).reshape(B * L, H, D).numpy(),
                                   rtol=0, atol=1e-12)


# --------------------------------------------------------------------------------------
# Closed forms and invariants
# --------------------------------------------------------------------------------------
def test_length_one_softmax():
    q, k, v, do = _rand([1, 1], [1, 1], 2, 4, 4, seed=1)
    offs = _offs([1, 1])
    o, lse = oracle.fwd(q, k, v, offs)
    np.testing.assert_array_equal(o, v)
    s = np.einsum("thd,thd->th", q, k) / 2.0
    np.testing.assert_allclose(lse, s, rtol=0, atol=1e-15)
    dq, dk, dv = oracle.bwd(q, k, v, do, offs)
    np.testing.assert_array_equal(dv, do)
    assert np.all(dq == 0) and np.all(dk == 0)


def test_length_one_gdpa():
    q, k, v, do = _rand([1], [1], 1, 4, 3, seed=2)
    o, _ = oracle.fwd(q, k, v, _offs([1]), act=GD)
    u = float(np.dot(q[0, 0], k[0, 0])) / 2.0
    silu = u / (1.0 + math.exp(-u))
    np.testing.assert_allclose(o[0, 0], silu * v[0, 0], rtol=1e-15, atol=1e-15)


@pytest.mark.parametrize("causal", [False, True])
def test_zero_queries_give_uniform_average(causal):
    lq = [5, 12]
    q, k, v, _ = _rand(lq, lq, 2, 4, 3, seed=6)
    q[:] = 0.0
    o, lse = oracle.fwd(q, k, v, _offs(lq), causal=causal)
    offs = _offs(lq)
    for b in range(2):
        for i in range(lq[b]):
            n = i + 1 if causal else lq[b]
            ref = v[offs[b]:offs[b] + n].mean(axis=0)
            np.testing.assert_allclose(o[offs[b] + i], ref, rtol=0, atol=1e-14)
            np.testing.assert_allclose(lse[offs[b] + i], math.log(n), rtol=0, atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_constant_values(causal):
    lq = [6, 9]
    q, k, v, do = _rand(lq, lq, 2, 4, 3, seed=7)
    v[:] = np.array([1.5, -2.0, 0.25])
    o, _ = oracle.fwd(q, k, v, _offs(lq), causal=causal)
    np.testing.assert_allclose(o, np.broadcast_to(v[:1], o.shape), rtol=0, atol=1e-14)
    dq, dk, _ = oracle.bwd(q, k, v, do, _offs(lq), causal=causal)
    assert np.abs(dq).max() < 1e-13 and np.abs(dk).max() < 1e-13


@pytest.mark.parametrize("causal", [False, True])
def test_key_shift_invariance_and_dk_sum(causal):
    lq = [6, 17, 1]
    q, k, v, do = _rand(lq, lq, 2, 5, 3, seed=8)
    offs = _offs(lq)
    o, _ = oracle.fwd(q, k, v, offs, causal=causal)
    k2 = k.copy()
    for b in range(3):
        k2[offs[b]:offs[b + 1]] += np.random.default_rng(b).standard_normal((1, 2, 5))
    o2, _ = oracle.fwd(q, k2, v, offs, causal=causal)
    np.testing.assert_allclose(o, o2, rtol=0, atol=1e-13)
    _, dk, _ = oracle.bwd(q, k, v, do, offs, causal=causal)
    for b in range(3):
        assert np.abs(dk[offs[b]:offs[b + 1]].sum(axis=0)).max() < 1e-13


@pytest.mark.parametrize("causal", [False, True])
def test_lse_consistency(causal):
    lq = [20, 3]
    q, k, v, _ = _rand(lq, lq, 2, 8, 8, seed=10)
    offs = _offs(lq)
    _, lse = oracle.fwd(q, k, v, offs, scale=0.3, causal=causal)
    for b in range(2):
        for h in range(2):
            for i in range(lq[b]):
                n = i + 1 if causal else lq[b]
                s = 0.3 * k[offs[b]:offs[b] + n, h] @ q[offs[b] + i, h]
                assert abs(np.exp(s - lse[offs[b] + i, h]).sum() - 1.0) < 1e-14


@pytest.mark.parametrize("act", [SM, GD])
def test_sequence_order_invariance(act):
    lq = [4, 19, 1, 30]
    lk = [8, 2, 25, 3]
    H, Dqk, Dv = 2, 8, 4
    q, k, v, do = _rand(lq, lk, H, Dqk, Dv, seed=12)
    oq, ok = _offs(lq), _offs(lk)
    o, lse = oracle.fwd(q, k, v, oq, ok, act=act)
    dq, dk, dv = oracle.bwd(q, k, v, do, oq, ok, act=act)
    perm = [2, 0, 3, 1]

    def permute(x, offs):
        return np.concatenate([x[offs[p]:offs[p + 1]] for p in perm])

    lq2 = [lq[p] for p in perm]
    lk2 = [lk[p] for p in perm]
    oq2, ok2 = _offs(lq2), _offs(lk2)
    q2, do2 = permute(q, oq), permute(do, oq)
    k2, v2 = permute(k, ok), permute(v, ok)
    o2, lse2 = oracle.fwd(q2, k2, v2, oq2, ok2, act=act)
    dq2, dk2, dv2 = oracle.bwd(q2, k2, v2, do2, oq2, ok2, act=act)
    np.testing.assert_array_equal(o2, permute(o, oq))
    np.testing.assert_array_equal(lse2, permute(lse, oq))
    np.testing.assert_array_equal(dq2, permute(dq, oq))
    np.testing.assert_array_equal(dk2, permute(dk, ok))
    np.testing.assert_array_equal(dv2, permute(dv, ok))


def test_head_split_invariance():
    lq = [7, 13]
    q, k, v, do = _rand(lq, lq, 2, 8, 8, seed=13)
    offs = _offs(lq)
    o, lse = oracle.fwd(q, k, v, offs, causal=True)
    dq, dk, dv = oracle.bwd(q, k, v, do, offs, causal=True)
    for h in range(2):
        sl = slice(h, h + 1)
        o1, lse1 = oracle.fwd(q[:, sl], k[:, sl], v[:, sl], offs, causal=True)
        dq1, dk1, dv1 = oracle.bwd(q[:, sl], k[:, sl], v[:, sl], do[:, sl], offs, causal=True)
        np.testing.assert_array_equal(o1, o[:, sl])
        np.testing.assert_array_equal(lse1, lse[:, sl])
        np.testing.assert_array_equal(dq1, dq[:, sl])
        np.testing.assert_array_equal(dk1, dk[:, sl])
        np.testing.assert_array_equal(dv1, dv[:, sl])


# --------------------------------------------------------------------------------------
# Length-0 conventions
# --------------------------------------------------------------------------------------
def test_empty_sequences_do_not_change_others():
    lq = [5, 0, 7, 0]
    q, k, v, do = _rand(lq, lq, 2, 4, 4, seed=14)
    o, lse = oracle.fwd(q, k, v, _offs(lq))
    o2, lse2 = oracle.fwd(q, k, v, _offs([5, 7]))
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(lse, lse2)
    g = oracle.bwd(q, k, v, do, _offs(lq))
    g2 = oracle.bwd(q, k, v, do, _offs([5, 7]))
    for a, b in zip(g, g2):
        np.testing.assert_array_equal(a, b)


def test_cross_with_no_keys():
    lq, lk = [3, 2], [0, 4]
    q, k, v, do = _rand(lq, lk, 1, 4, 4, seed=15)
    o, lse = oracle.fwd(q, k, v, _offs(lq), _offs(lk))
    assert np.all(o[:3] == 0) and np.all(np.isneginf(lse[:3]))
    dq, dk, dv = oracle.bwd(q, k, v, do, _offs(lq), _offs(lk))
    assert np.all(dq[:3] == 0)
    o_g, _ = oracle.fwd(q, k, v, _offs(lq), _offs(lk), act=GD)
    assert np.all(o_g[:3] == 0)


def test_empty_batch():
    e = np.zeros((0, 1, 4))
    o, lse = oracle.fwd(e, e, e, np.array([0]))
    assert o.shape == (0, 1, 4) and lse.shape == (0, 1)
    dq, dk, dv = oracle.bwd(e, e, e, e, np.array([0]))
    assert dq.shape == (0, 1, 4)


def test_bad_offsets_rejected():
    q = np.zeros((4, 1, 2))
    with pytest.raises(ValueError):
        oracle.fwd(q, q, q, np.array([0, 3, 2, 4]))
    with pytest.raises(ValueError):
        oracle.fwd(q, q, q, np.array([0, 1, 4]), np.array([0, 2, 4]), causal=True)


# --------------------------------------------------------------------------------------
# Pooled multi-head attention: shared queries, through torch autograd per sequence
# --------------------------------------------------------------------------------------
def test_pooled_matches_shared_query_autograd():
    """m shared query rows attend each sequence; torch autograd sums the shared rows'
    gradient over sequences by itself.  A sequence without keys contributes o = 0."""
    m, H, Dqk, Dv = 5, 2, 16, 8
    lk = [7, 1, 0, 40, 13]
    rng = np.random.default_rng(33)
    q = rng.standard_normal((m, H, Dqk))
    k = rng.standard_normal((sum(lk), H, Dqk))
    v = rng.standard_normal((sum(lk), H, Dv))
    do = rng.standard_normal((len(lk) * m, H, Dv))
    ok = _offs(lk)
    scale = 1.0 / math.sqrt(Dqk)
    o, lse = oracle.pooled_fwd(q, k, v, ok, scale=scale)
    dq, dk, dv = oracle.pooled_bwd(q, k, v, do, ok, scale=scale)

    tq = torch.tensor(q, requires_grad=True)
    tk = torch.tensor(k, requires_grad=True)
    tv = torch.tensor(v, requires_grad=True)
    outs = []
    for b, n in enumerate(lk):
        if n == 0:
            outs.append(torch.zeros(m, H, Dv, dtype=torch.float64))
            continue
        kb, vb = tk[ok[b]:ok[b + 1]], tv[ok[b]:ok[b + 1]]
        s = torch.einsum("ihd,jhd->hij", tq, kb) * scale
        outs.append(torch.einsum("hij,jhd->ihd", torch.softmax(s, dim=-1), vb))
    out = torch.cat(outs)
    (out * torch.tensor(do)).sum().backward()
    np.testing.assert_allclose(o, out.detach().numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dv, tv.grad.numpy(), rtol=0, atol=1e-12)
    assert np.all(np.isneginf(lse[2 * m:3 * m]))  # the sequence without keys


# --------------------------------------------------------------------------------------
# BlockAttention: dense attention over the whole sequence with a block-diagonal mask
# --------------------------------------------------------------------------------------
def test_block_offsets_cut_each_sequence():
    assert oracle.block_offsets([0, 3, 3, 200, 264]).tolist() == [0, 3, 67, 131, 195, 200, 264]


@pytest.mark.parametrize("causal", [False, True])
def test_block_matches_block_diagonal_mask(causal):
    """Each row attends the keys of its own 64-row block (0-63, 64-127, ... from the start
    of its sequence), through torch autograd on the whole sequence with an explicit mask."""
    lens = [1, 64, 65, 200, 0, 130]
    H, D = 2, 8
    rng = np.random.default_rng(41)
    T = sum(lens)
    q, k, v, do = (rng.standard_normal((T, H, D)) for _ in range(4))
    offs = _offs(lens)
    scale = 1.0 / math.sqrt(D)
    o, lse = oracle.block_fwd(q, k, v, offs, scale=scale, causal=causal)
    dq, dk, dv = oracle.block_bwd(q, k, v, do, offs, scale=scale, causal=causal)
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    outs, lses = [], []
    for b, L in enumerate(lens):
        if L == 0:
            continue
        sl = slice(offs[b], offs[b + 1])
        i = torch.arange(L)
        mask = (i[:, None] // 64) == (i[None, :] // 64)
        if causal:
            mask &= i[None, :] <= i[:, None]
        s = torch.einsum("ihd,jhd->hij", tq[sl], tk[sl]) * scale
        s = s.masked_fill(~mask, float("-inf"))
        outs.append(torch.einsum("hij,jhd->ihd", torch.softmax(s, dim=-1), tv[sl]))
        lses.append(torch.logsumexp(s, dim=-1).T)
    out = torch.cat(outs)
    (out * torch.tensor(do)).sum().backward()
    np.testing.assert_allclose(o, out.detach().numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, torch.cat(lses).detach().numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dv, tv.grad.numpy(), rtol=0, atol=1e-12)


# --------------------------------------------------------------------------------------
# Rotary position embedding (RoFormer's definition) and BlockAttention with it
# --------------------------------------------------------------------------------------
def _rope_complex_d8(x, offs):
    """The rotation in RoFormer's complex form for D = 8 and base 10000: pair i is the complex
    number x[2i] + i x[2i+1], multiplied by e^(i p theta_i); with D = 8 the frequencies are
    10000^(-2i/8) = 10^-i exactly."""
    T, H, D = x.shape
    assert D == 8
    pos = np.concatenate([np.arange(offs[b + 1] - offs[b]) for b in range(len(offs) - 1)])
    theta = np.array([1.0, 0.1, 0.01, 0.001])
    z = x[..., 0::2] + 1j * x[..., 1::2]
    z = z * np.exp(1j * pos[:, None, None] * theta[None, None, :])
    out = np.empty_like(x)
    out[..., 0::2], out[..., 1::2] = z.real, z.imag
    return out


def test_rope_complex_form():
    rng = np.random.default_rng(50)
    offs = _offs([5, 0, 130, 1])
    x = rng.standard_normal((int(offs[-1]), 3, 8))
    np.testing.assert_allclose(oracle.rope(x, offs), _rope_complex_d8(x, offs), rtol=0, atol=1e-13)


def test_rope_pairs_adjacent_coordinates_counterclockwise():
    # a unit vector on the second coordinate of pair 0, at position 3 of its sequence:
    # rotated by 3 radians to (-sin 3, cos 3); no other coordinate moves
    x = np.zeros((4, 1, 6))
    x[3, 0, 1] = 1.0
    y = oracle.rope(x, [0, 4])
    expect = np.zeros(6)
    expect[0], expect[1] = -math.sin(3.0), math.cos(3.0)
    np.testing.assert_allclose(y[3, 0], expect, rtol=0, atol=1e-15)
    assert not y[:3].any()


def test_rope_positions_restart_per_sequence_and_preserve_norms():
    rng = np.random.default_rng(51)
    offs = _offs([3, 7, 2])
    x = rng.standard_normal((12, 2, 16))
    y = oracle.rope(x, offs)
    for start in offs[:-1]:  # position 0 of every sequence: the identity
        np.testing.assert_array_equal(y[start], x[start])
    pair_norm = lambda a: np.hypot(a[..., 0::2], a[..., 1::2])
    np.testing.assert_allclose(pair_norm(y), pair_norm(x), rtol=1e-14)


def test_rope_inverse_is_the_transpose():
    rng = np.random.default_rng(52)
    offs = _offs([9, 40])
    x, y = rng.standard_normal((2, 49, 2, 32))
    lhs = np.sum(oracle.rope(x, offs) * y)
    rhs = np.sum(x * oracle.rope(y, offs, inverse=True))
    assert abs(lhs - rhs) <= 1e-12 * (abs(lhs) + 1)
    np.testing.assert_allclose(oracle.rope(oracle.rope(x, offs), offs, inverse=True), x,
                               rtol=0, atol=1e-13)


def test_rope_scores_depend_on_relative_position_only():
    # the same q and k vectors placed at (m, n) and at (m + s, n + s) give the same score
    rng = np.random.default_rng(53)
    D = 64
    q, k = rng.standard_normal((2, D))
    L = 300
    for m, n, s in ((10, 4, 200), (0, 37, 150), (99, 99, 1)):
        xq, xk = np.zeros((L, 1, D)), np.zeros((L, 1, D))
        xq[m, 0], xk[n, 0] = q, k
        xq2, xk2 = np.zeros((L, 1, D)), np.zeros((L, 1, D))
        xq2[m + s, 0], xk2[n + s, 0] = q, k
        a = oracle.rope(xq, [0, L])[m, 0] @ oracle.rope(xk, [0, L])[n, 0]
        b = oracle.rope(xq2, [0, L])[m + s, 0] @ oracle.rope(xk2, [0, L])[n + s, 0]
        assert abs(a - b) <= 1e-11 * (abs(a) + 1), (m, n, s, a, b)


@pytest.mark.parametrize("causal", [False, True])
def test_block_rope_matches_autograd(causal):
    """BlockAttention with q and k rotated (complex form, in torch) through torch autograd on
    the whole sequence with a block-diagonal mask: o, lse and the gradients of the
    unrotated q, k, v."""
    lens = [1, 64, 65, 200, 0, 130]
    H, D = 2, 8
    rng = np.random.default_rng(54)
    T = sum(lens)
    q, k, v, do = (rng.standard_normal((T, H, D)) for _ in range(4))
    offs = _offs(lens)
    scale = 1.0 / math.sqrt(D)
    o, lse = oracle.block_rope_fwd(q, k, v, offs, scale=scale, causal=causal)
    dq, dk, dv = oracle.block_rope_bwd(q, k, v, do, offs, scale=scale, causal=causal)

    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    theta = torch.tensor([1.0, 0.1, 0.01, 0.001], dtype=torch.float64)

    def rot(t, L):
        z = torch.view_as_complex(t.reshape(L, H, D // 2, 2).contiguous())
        ang = torch.arange(L, dtype=torch.float64)[:, None, None] * theta
        return torch.view_as_real(z * torch.polar(torch.ones_like(ang), ang)).reshape(L, H, D)

    outs, lses = [], []
    for b, L in enumerate(lens):
        if L == 0:
            continue
        sl = slice(offs[b], offs[b + 1])
        i = torch.arange(L)
        mask = (i[:, None] // 64) == (i[None, :] // 64)
        if causal:
            mask &= i[None, :] <= i[:, None]
        s = torch.einsum("ihd,jhd->hij", rot(tq[sl], L), rot(tk[sl], L)) * scale
        s = s.masked_fill(~mask, float("-inf"))
        outs.append(torch.einsum("hij,jhd->ihd", torch.softmax(s, dim=-1), tv[sl]))
        lses.append(torch.logsumexp(s, dim=-1).T)
    out = torch.cat(outs)
    (out * torch.tensor(do)).sum().backward()
    np.testing.assert_allclose(o, out.detach().numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, torch.cat(lses).detach().numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dv, tv.grad.numpy(), rtol=0, atol=1e-12)


def test_block_rope_same_with_positions_counted_per_block():
    """Scores under the rotation depend only on the offset between query and key, and both
    lie in one block: counting positions from the block's first row gives the same
    outputs and gradients as counting from the sequence's first row."""
    lens = [70, 3, 129]
    H, D = 2, 16
    rng = np.random.default_rng(55)
    T = sum(lens)
    q, k, v, do = (rng.standard_normal((T, H, D)) for _ in range(4))
    offs = _offs(lens)
    bo = oracle.block_offsets(offs)
    o, lse = oracle.block_rope_fwd(q, k, v, offs, causal=True)
    o2, lse2 = oracle.block_fwd(oracle.rope(q, bo), oracle.rope(k, bo), v, offs, causal=True)
    np.testing.assert_allclose(o, o2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse2, rtol=0, atol=1e-12)
    grads = oracle.block_rope_bwd(q, k, v, do, offs, causal=True)
    dqr, dkr, dv2 = oracle.block_bwd(oracle.rope(q, bo), oracle.rope(k, bo), v, do, offs, causal=True)
    grads2 = (oracle.rope(dqr, bo, inverse=True), oracle.rope(dkr, bo, inverse=True), dv2)
    for a, b in zip(grads, grads2):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)
