"""Work lists built once (jfa_plan, jfa_block_plan) and used by several calls: every
planned call gives bit-identical results to the same call that schedules for itself,
however many times the plan is used, in both the fixed and the claimed assignment.
GPU only."""
import numpy as np
import pytest
import torch

import jagged_attention_recsys_gb300 as jfa
import workloads

pytestmark = pytest.mark.gpu

GD = workloads.ACT_SILU_OVER_LEN
SM = workloads.ACT_SOFTMAX


def _claims(ws):
    # status, n_q, n_k, claim[fwd], claim[dkdv], claim[dq]
    return ws[:24].view(torch.int32).cpu().numpy().tolist()


def _calls(w, b, oq, ok, ws, planned):
    q, k, v, do = b["q"], b["k"], b["v"], b["do"]
    sc, c = w.scale, w.causal
    if w.act == GD:
        o = jfa.jfa_gdpa_fwd(q, k, v, oq, ok, scale=sc, causal=c, ws=ws, planned=planned)
        g = jfa.jfa_gdpa_bwd(q, k, v, do, oq, ok, scale=sc, causal=c, ws=ws, planned=planned)
        return [o, *g]
    if w.cross:
        o, lse = jfa.jfa_cross_fwd(q, k, v, oq, ok, scale=sc, ws=ws, planned=planned)
        g = jfa.jfa_cross_bwd(q, k, v, o, lse, do, oq, ok, scale=sc, ws=ws, planned=planned)
        return [o, lse, *g]
    o, lse = jfa.jfa_fwd(q, k, v, oq, scale=sc, causal=c, ws=ws, planned=planned)
    g = jfa.jfa_bwd(q, k, v, o, lse, do, oq, scale=sc, causal=c, ws=ws, planned=planned)
    return [o, lse, *g]


CASES = [
    # name, heads, Dqk, Dv, causal, act, dtype, cross, lengths (q, k)
    ("softmax_d64", 4, 64, 64, False, SM, torch.bfloat16, False, None),
    ("causal_d128", 2, 128, 128, True, SM, torch.bfloat16, False, None),
    ("cross_asym", 2, 128, 64, False, SM, torch.bfloat16, True, "cross"),
    ("gdpa_claimed", 2, 128, 128, True, GD, torch.bfloat16, False, "long"),
    ("gdpa_fixed", 2, 128, 128, True, GD, torch.bfloat16, False, None),
    ("fp32_cross", 2, 32, 48, False, SM, torch.float32, True, "cross"),
]


def _lengths(kind, rng):
    if kind == "long":  # items of many steps: the lists are claimed
        return rng.integers(1500, 3000, 6), None
    if kind == "cross":
        lq = rng.integers(0, 90, 60)
        return lq, rng.integers(0, 700, 60)
    return rng.integers(0, 400, 300), None


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_planned_calls_match_unplanned_bitwise(case):
    name, H, dqk, dv, causal, act, dtype, cross, kind = case
    rng = np.random.default_rng(11)
    lq, lk = _lengths(kind, rng)
    w = workloads.Workload(name, 0, H, dqk, dv, causal, act, dtype, cross)
    b = workloads.make_batch(w, lq, lk, seed=11, device="cuda")
    oq = torch.as_tensor(b["offs_q"], device="cuda")
    ok = torch.as_tensor(b["offs_k"], device="cuda") if cross else oq
    p = jfa.params_for(b["q"], b["k"], b["v"], oq, w.scale, causal)
    ref = _calls(w, b, oq, ok, jfa.workspace(p), planned=False)
    ws = jfa.jfa_plan(b["q"], b["k"], b["v"], oq, ok, scale=w.scale, causal=causal)
    planned_claims = _claims(ws)[3:6]
    if name == "gdpa_claimed":
        assert planned_claims == [0, 0, 0]  # the SiLU/L kernels take these items by claiming
    if name == "gdpa_fixed":
        assert planned_claims == [-1, -1, -1]
    for _ in range(3):  # one plan, used again and again
        got = _calls(w, b, oq, ok, ws, planned=True)
        torch.cuda.synchronize()
        for i, (x, y) in enumerate(zip(ref, got)):
            assert torch.equal(x, y), (name, i)
        assert jfa.jfa_status_check(ws) == jfa.JFA_OK
        # a kernel that claimed items rewound its counter to 0 at the end of its launch
        assert _claims(ws)[3:6] == planned_claims


@pytest.mark.parametrize("rope", [False, True])
def test_planned_block_calls_match_unplanned_bitwise(rope):
    rng = np.random.default_rng(4)
    lq = rng.integers(0, 700, 80)
    w = workloads.Workload("blk", 0, 2, 128, 128, True, SM, torch.bfloat16, False, 0, 64)
    b = workloads.make_batch(w, lq, seed=4, device="cuda")
    oq = torch.as_tensor(b["offs_q"], device="cuda")
    q, k, v, do = b["q"], b["k"], b["v"], b["do"]

    def calls(ws, planned):
        o, lse = jfa.jfa_block_fwd(q, k, v, oq, causal=True, ws=ws, rope=rope, planned=planned)
        g = jfa.jfa_block_bwd(q, k, v, o, lse, do, oq, causal=True, ws=ws, rope=rope,
                              planned=planned)
        return [o, lse, *g]

    ref = calls(None, False)
    ws = jfa.jfa_block_plan(q, k, v, oq, causal=True)
    for _ in range(2):
        got = calls(ws, True)
        torch.cuda.synchronize()
        for i, (x, y) in enumerate(zip(ref, got)):
            assert torch.equal(x, y), i
        assert jfa.jfa_status_check(ws) == jfa.JFA_OK


def test_plan_of_bad_offsets_makes_planned_calls_compute_nothing():
    w = workloads.Workload("bad", 0, 2, 64, 64, False, SM, torch.bfloat16, False)
    b = workloads.make_batch(w, np.array([100, 50, 70]), seed=2, device="cuda")
    bad = torch.tensor([0, 100, 90, 220], dtype=torch.int64, device="cuda")  # decreasing
    q, k, v = b["q"], b["k"], b["v"]
    ws = jfa.jfa_plan(q, k, v, bad)
    assert jfa.jfa_status_check(ws) == jfa.JFA_ERR_BAD_OFFSETS
    o = torch.full((q.shape[0], q.shape[1], v.shape[2]), 7.0, dtype=q.dtype, device="cuda")
    lse = torch.full((q.shape[0], q.shape[1]), 7.0, dtype=torch.float32, device="cuda")
    jfa.jfa_fwd(q, k, v, bad, o=o, lse=lse, ws=ws, planned=True)
    assert jfa.jfa_status_check(ws) == jfa.JFA_ERR_BAD_OFFSETS
    assert bool((o == 7.0).all()) and bool((lse == 7.0).all())
    # a call that schedules for itself, on good offsets, clears it
    good = torch.as_tensor(b["offs_q"], device="cuda")
    jfa.jfa_fwd(q, k, v, good, ws=ws)
    assert jfa.jfa_status_check(ws) == jfa.JFA_OK


def test_planned_call_without_workspace_is_refused():
    w = workloads.Workload("nows", 0, 2, 64, 64, False, SM, torch.bfloat16, False)
    b = workloads.make_batch(w, np.array([10, 20]), seed=0, device="cuda")
    oq = torch.as_tensor(b["offs_q"], device="cuda")
    with pytest.raises(ValueError):
        jfa.jfa_fwd(b["q"], b["k"], b["v"], oq, planned=True)


@pytest.mark.parametrize("name", ["d64", "causal", "cross", "gdpa", "block", "block_rope"])
def test_full_size_bench_step_matches_unplanned_calls(name):
    """The step bench.py times (one plan, then the planned forward and backward calls), on
    the full-size workload, gives the outputs of calls that each build their own lists, bit
    for bit; those are the calls the whole-batch oracle tests check."""
    import bench

    w = workloads.WORKLOADS[name]
    lq, lk = workloads.lengths(w.name, seed=0)
    b = workloads.make_batch(w, lq, lk, seed=0, device="cuda")
    d = dict(q=b["q"], k=b["k"], v=b["v"], do=b["do"],
             oq=torch.as_tensor(b["offs_q"], device="cuda"),
             ok=torch.as_tensor(b["offs_k"], device="cuda"))
    q, k, v, do, oq, ok = d["q"], d["k"], d["v"], d["do"], d["oq"], d["ok"]
    d["o"] = torch.empty(q.shape[0], q.shape[1], v.shape[2], dtype=q.dtype, device="cuda")
    d["lse"] = torch.empty(q.shape[0], q.shape[1], dtype=torch.float32, device="cuda")
    d["dq"], d["dk"], d["dv"] = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    p = jfa.params_for(q, k, v, oq, w.scale, w.causal)
    ws = jfa.block_workspace(p) if w.block else jfa.workspace(p)
    bench.gpu_step_fn(jfa, w, d, ws)()
    torch.cuda.synchronize()
    assert jfa.jfa_status_check(ws) == jfa.JFA_OK
    sc, c = w.scale, w.causal
    if w.block:
        o, lse = jfa.jfa_block_fwd(q, k, v, oq, scale=sc, causal=c, rope=w.rope)
        g = jfa.jfa_block_bwd(q, k, v, o, lse, do, oq, scale=sc, causal=c, rope=w.rope)
        ref = [o, lse, *g]
    elif w.act == GD:
        o = jfa.jfa_gdpa_fwd(q, k, v, oq, ok, scale=sc, causal=c)
        ref = [o, None, *jfa.jfa_gdpa_bwd(q, k, v, do, oq, ok, scale=sc, causal=c)]
    elif w.cross:
        o, lse = jfa.jfa_cross_fwd(q, k, v, oq, ok, scale=sc)
        ref = [o, lse, *jfa.jfa_cross_bwd(q, k, v, o, lse, do, oq, ok, scale=sc)]
    else:
        o, lse = jfa.jfa_fwd(q, k, v, oq, scale=sc, causal=c)
        ref = [o, lse, *jfa.jfa_bwd(q, k, v, o, lse, do, oq, scale=sc, causal=c)]
    torch.cuda.synchronize()
    for nm, x in zip(("o", "lse", "dq", "dk", "dv"), ref):
        if x is not None:
            assert torch.equal(x, d[nm]), (name, nm)
