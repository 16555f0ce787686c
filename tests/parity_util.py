"""Helpers for the GPU parity tests: run libjfa and the fp64 oracle on the same inputs."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import workloads

# Tolerances.  fp32 inputs: max-abs error <= 1e-5 on O, dQ, dK, dV.  bf16 inputs with fp32
# accumulation: O max-abs <= 2e-2 and relative L2 <= 1e-2; each gradient relative L2 <= 1e-2.
F32_ATOL = 1e-5
BF16_O_ATOL = 2e-2
BF16_REL_L2 = 1e-2


def to64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def rel_l2(got, ref):
    den = float(np.linalg.norm(ref))
    num = float(np.linalg.norm(got - ref))
    return num / den if den > 0 else num


def run_gpu(w: workloads.Workload, batch, ws=None, check_status=False):
    """Forward and backward on the GPU through the C ABI binding; returns the outputs.
    With ``check_status``, one workspace serves both calls and the device status word
    is checked after each."""
    import jagged_attention_recsys_gb300 as jfa

    dev = batch["q"].device
    oq = torch.as_tensor(batch["offs_q"], device=dev)
    ok = torch.as_tensor(batch["offs_k"], device=dev)
    q, k, v, do = batch["q"], batch["k"], batch["v"], batch["do"]
    sc = w.scale
    if check_status:
        ws = jfa.workspace(jfa.params_for(q, k, v, oq, sc, w.causal), dev) if ws is None else ws
        got = run_gpu(w, batch, ws)
        assert jfa.jfa_status_check(ws) == jfa.JFA_OK
        return got
    if w.act == workloads.ACT_SILU_OVER_LEN:
        o = jfa.jfa_gdpa_fwd(q, k, v, oq, ok, scale=sc, causal=w.causal, ws=ws)
        dq, dk, dv = jfa.jfa_gdpa_bwd(q, k, v, do, oq, ok, scale=sc, causal=w.causal, ws=ws)
        lse = None
    elif w.cross:
        o, lse = jfa.jfa_cross_fwd(q, k, v, oq, ok, scale=sc, ws=ws)
        dq, dk, dv = jfa.jfa_cross_bwd(q, k, v, o, lse, do, oq, ok, scale=sc, ws=ws)
    else:
        o, lse = jfa.jfa_fwd(q, k, v, oq, scale=sc, causal=w.causal, ws=ws)
        dq, dk, dv = jfa.jfa_bwd(q, k, v, o, lse, do, oq, scale=sc, causal=w.causal, ws=ws)
    torch.cuda.synchronize()
    return dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv)


def run_oracle(w: workloads.Workload, q, k, v, do, offs_q, offs_k):
    o, lse = oracle.fwd(q, k, v, offs_q, offs_k, scale=w.scale, causal=w.causal, act=w.act)
    dq, dk, dv = oracle.bwd(q, k, v, do, offs_q, offs_k, scale=w.scale, causal=w.causal,
                            act=w.act)
    return dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv)


def compare(w: workloads.Workload, got, ref, fp32: bool, strict_o: bool = False):
    """Asserts the tolerances; returns the error figures.

    The O max-abs bound of 2e-2 is stated for the named workloads, whose outputs are O(1).
    bf16 output rounding alone is half an ulp of |o|, so for other cases (for example
    SiLU/L cross-attention with one query and thousands of keys, |o| ~ 60) the bound is
    scaled by max(1, max |o|).  ``strict_o`` applies the plain bound.
    """
    errs = {}
    for name in ("o", "dq", "dk", "dv"):
        g, r = got[name], ref[name]
        assert np.all(np.isfinite(g)), name + " has non-finite values"
        errs[name + "_maxabs"] = float(np.max(np.abs(g - r))) if g.size else 0.0
        errs[name + "_rel_l2"] = rel_l2(g, r) if g.size else 0.0
    if got.get("lse") is not None and ref.get("lse") is not None and got["lse"].size:
        fin = np.isfinite(ref["lse"])
        assert np.array_equal(fin, np.isfinite(got["lse"])), "lse -inf pattern differs"
        if fin.any():
            errs["lse_maxabs"] = float(np.max(np.abs(got["lse"][fin] - ref["lse"][fin])))
    if fp32:
        for name in ("o", "dq", "dk", "dv"):
            assert errs[name + "_maxabs"] <= F32_ATOL, (name, errs)
        if "lse_maxabs" in errs:
            assert errs["lse_maxabs"] <= F32_ATOL, errs
    else:
        mag = 1.0 if strict_o else max(1.0, float(np.max(np.abs(ref["o"]))) if ref["o"].size else 1.0)
        assert errs["o_maxabs"] <= BF16_O_ATOL * mag, errs
        assert errs["o_rel_l2"] <= BF16_REL_L2, errs
        for name in ("dq", "dk", "dv"):
            assert errs[name + "_rel_l2"] <= BF16_REL_L2, (name, errs)
        if "lse_maxabs" in errs:
            assert errs["lse_maxabs"] <= 2e-2, errs
    return errs


def full_check(w: workloads.Workload, lq, lk=None, seed=0, device="cuda", strict_o=False):
    """Whole batch on GPU and in the oracle; element-by-element comparison."""
    batch = workloads.make_batch(w, lq, lk, seed=seed, device=device)
    got = run_gpu(w, batch)
    got = {n: (to64(t) if t is not None else None) for n, t in got.items()}
    q, k, v, do = (to64(batch[n]) for n in ("q", "k", "v", "do"))
    ref = run_oracle(w, q, k, v, do, batch["offs_q"], batch["offs_k"])
    return compare(w, got, ref, fp32=(w.dtype == torch.float32), strict_o=strict_o)


def sample_indices(lq, count=6, seed=0):
    """Longest, shortest and a few seeded random sequences."""
    lq = np.asarray(lq)
    order = np.argsort(lq, kind="stable")
    pick = {int(order[-1]), int(order[0])}
    if len(lq) > 1:
        pick.add(int(order[-2]))
    rng = np.random.default_rng(seed + 1)
    while len(pick) < min(count, len(lq)):
        pick.add(int(rng.integers(0, len(lq))))
    return sorted(pick)


def sampled_check(w: workloads.Workload, batch, got, idx, strict_o=True):
    """Compares the GPU result of a full batch with the oracle on a few whole sequences."""
    oq, ok = batch["offs_q"], batch["offs_k"]
    lq = [int(oq[b + 1] - oq[b]) for b in idx]
    lk = [int(ok[b + 1] - ok[b]) for b in idx]
    rq = np.concatenate([np.arange(oq[b], oq[b + 1]) for b in idx]).astype(np.int64)
    rk = np.concatenate([np.arange(ok[b], ok[b + 1]) for b in idx]).astype(np.int64)
    tq = torch.as_tensor(rq, device=batch["q"].device)
    tk = torch.as_tensor(rk, device=batch["q"].device)
    q, do = to64(batch["q"][tq]), to64(batch["do"][tq])
    k, v = to64(batch["k"][tk]), to64(batch["v"][tk])
    sub_q = workloads.offsets(lq)
    sub_k = workloads.offsets(lk)
    ref = run_oracle(w, q, k, v, do, sub_q, sub_k)
    g = dict(o=to64(got["o"][tq]), dq=to64(got["dq"][tq]), dk=to64(got["dk"][tk]),
             dv=to64(got["dv"][tk]),
             lse=to64(got["lse"][tq]) if got.get("lse") is not None else None)
    return compare(w, g, ref, fp32=(w.dtype == torch.float32), strict_o=strict_o)


def whole_batch_check(w: workloads.Workload, batch, got, seqs=None, max_rows=60000,
                      strict_o=True, oracle_fn=None):
    """Every sequence of a (full-size) batch against the oracle, at the tolerances above,
    with the error metrics taken over the whole batch (or over the sequences ``seqs``).

    The sequences are processed in chunks of at most ``max_rows`` query and key rows each,
    so that host memory stays bounded: each chunk's rows are converted to fp64, run
    through the oracle and compared; squared errors and norms are accumulated, so the
    relative L2 errors are those of the whole batch.  Returns the figures, including the
    worst sequence for each tensor (largest max-abs error for O, largest relative L2 error
    among sequences with a nonzero reference for the gradients).  ``strict_o`` applies the
    plain O max-abs bound (the named workloads); otherwise it is scaled by
    max(1, max |o|) as in ``compare``.  ``oracle_fn(w, q, k, v, do, offs_q, offs_k)``
    replaces the plain oracle (for example BlockAttention with the rotary embedding).
    """
    oq, ok = np.asarray(batch["offs_q"]), np.asarray(batch["offs_k"])
    dev = batch["q"].device
    seqs = list(range(len(oq) - 1)) if seqs is None else list(seqs)
    names = ("o", "dq", "dk", "dv")
    acc = {n: [0.0, 0.0, 0.0] for n in names}  # sum sq err, sum sq ref, max abs err
    o_mag = 0.0  # largest |o| of the reference
    worst = {n: (0.0, -1) for n in names}
    lse_err = 0.0
    chunk = []

    def flush(chunk):
        nonlocal lse_err, o_mag
        lq = [int(oq[b + 1] - oq[b]) for b in chunk]
        lk = [int(ok[b + 1] - ok[b]) for b in chunk]
        rq = np.concatenate([np.arange(oq[b], oq[b + 1]) for b in chunk]).astype(np.int64)
        rk = np.concatenate([np.arange(ok[b], ok[b + 1]) for b in chunk]).astype(np.int64)
        tq = torch.as_tensor(rq, device=dev)
        tk = torch.as_tensor(rk, device=dev)
        q, do = to64(batch["q"][tq]), to64(batch["do"][tq])
        k, v = to64(batch["k"][tk]), to64(batch["v"][tk])
        sub_q, sub_k = workloads.offsets(lq), workloads.offsets(lk)
        ref = (oracle_fn or run_oracle)(w, q, k, v, do, sub_q, sub_k)
        g = dict(o=to64(got["o"][tq]), dq=to64(got["dq"][tq]), dk=to64(got["dk"][tk]),
                 dv=to64(got["dv"][tk]))
        if ref["o"].size:
            o_mag = max(o_mag, float(np.max(np.abs(ref["o"]))))
        for n in names:
            gg, rr = g[n], ref[n]
            assert np.all(np.isfinite(gg)), n + " has non-finite values"
            d = gg - rr
            acc[n][0] += float(np.sum(d * d))
            acc[n][1] += float(np.sum(rr * rr))
            if d.size:
                acc[n][2] = max(acc[n][2], float(np.max(np.abs(d))))
            offs = sub_q if n in ("o", "dq") else sub_k
            for i, b in enumerate(chunk):
                a, e = int(offs[i]), int(offs[i + 1])
                if e == a:
                    continue
                if n == "o":
                    val = float(np.max(np.abs(d[a:e])))
                else:
                    den = float(np.linalg.norm(rr[a:e]))
                    if den == 0.0:
                        continue
                    val = float(np.linalg.norm(d[a:e])) / den
                if val > worst[n][0]:
                    worst[n] = (val, b)
        if got.get("lse") is not None:
            gl, rl = to64(got["lse"][tq]), ref["lse"]
            fin = np.isfinite(rl)
            assert np.array_equal(fin, np.isfinite(gl)), "lse -inf pattern differs"
            if fin.any():
                lse_err = max(lse_err, float(np.max(np.abs(gl[fin] - rl[fin]))))

    rows_q = rows_k = 0
    for b in seqs:
        nq, nk = int(oq[b + 1] - oq[b]), int(ok[b + 1] - ok[b])
        if chunk and (rows_q + nq > max_rows or rows_k + nk > max_rows):
            flush(chunk)
            chunk, rows_q, rows_k = [], 0, 0
        chunk.append(b)
        rows_q += nq
        rows_k += nk
    if chunk:
        flush(chunk)

    fig = {}
    for n in names:
        se, sr, mx = acc[n]
        fig[n + "_rel_l2"] = (se ** 0.5) / (sr ** 0.5) if sr > 0 else se ** 0.5
        fig[n + "_maxabs"] = mx
        fig[n + "_worst_seq"] = {"seq": worst[n][1], ("maxabs" if n == "o" else "rel_l2"): worst[n][0]}
    fig["lse_maxabs"] = lse_err
    fig["o_ref_maxabs"] = o_mag
    fig["sequences"] = len(seqs)
    if w.dtype == torch.float32:
        for n in names:
            assert fig[n + "_maxabs"] <= F32_ATOL, (n, fig)
    else:
        assert fig["o_maxabs"] <= BF16_O_ATOL * (1.0 if strict_o else max(1.0, o_mag)), fig
        assert fig["o_rel_l2"] <= BF16_REL_L2, fig
        for n in ("dq", "dk", "dv"):
            assert fig[n + "_rel_l2"] <= BF16_REL_L2, (n, fig)
        assert fig["lse_maxabs"] <= 2e-2, fig
    return fig


def stratified_subset(lq, longest=8, shortest=8, random=16, seed=0):
    """The labelled subset used where the whole batch is too costly for the oracle: the
    `longest` longest and `shortest` shortest sequences and `random` others drawn with a
    seeded generator (ties broken by index)."""
    lq = np.asarray(lq)
    order = np.argsort(lq, kind="stable")
    pick = set(int(i) for i in order[-longest:]) | set(int(i) for i in order[:shortest])
    rest = [i for i in range(len(lq)) if i not in pick]
    rng = np.random.default_rng(seed)
    pick |= set(int(i) for i in rng.choice(rest, size=min(random, len(rest)), replace=False))
    return sorted(pick)
