"""Work distribution of the tensor-core kernels: the scheduler's choice between claimed
and fixed assignment, and that claimed lists give bit-identical results from run to run
and match the oracle.  GPU only."""
import numpy as np
import pytest
import torch

import jagged_attention_recsys_gb300 as jfa
import workloads
from parity_util import run_gpu, whole_batch_check

pytestmark = pytest.mark.gpu

GD = workloads.ACT_SILU_OVER_LEN


def _header(ws):
    # status, n_q, n_k, claim[fwd], claim[dkdv], claim[dq]
    return ws[:24].view(torch.int32).cpu().numpy().tolist()


def _gdpa_batch(lens, seed=0):
    w = workloads.Workload("feed", 0, 2, 128, 128, True, GD, torch.bfloat16, False)
    b = workloads.make_batch(w, np.array(lens), seed=seed, device="cuda")
    oq = torch.as_tensor(b["offs_q"], device="cuda")
    return w, b, oq


def _run(w, b, oq, ws):
    o = jfa.jfa_gdpa_fwd(b["q"], b["k"], b["v"], oq, causal=True, ws=ws)
    dq, dk, dv = jfa.jfa_gdpa_bwd(b["q"], b["k"], b["v"], b["do"], oq, causal=True, ws=ws)
    torch.cuda.synchronize()
    return o, dq, dk, dv


def test_long_items_are_claimed_and_every_item_taken():
    # causal lengths of 16 tiles: the lists average 8.5 steps per item, above the threshold
    w, b, oq = _gdpa_batch([2048, 2048, 2048])
    p = jfa.params_for(b["q"], b["k"], b["v"], oq, causal=True)
    ws = jfa.workspace(p)
    _run(w, b, oq, ws)
    status, n_q, n_k, c_fwd, c_dkdv, c_dq = _header(ws)
    assert status == 0
    assert n_q == n_k == 3 * 16 * 2
    # each CTA's claimer takes indices until one is past the end, and the CTA that takes
    # the last of those sets the counter back to 0: every counter reads 0 afterwards
    assert [c_fwd, c_dkdv, c_dq] == [0, 0, 0]


def test_short_items_keep_the_fixed_assignment():
    # one or two tiles per sequence: the lists average under two steps per item
    w, b, oq = _gdpa_batch([100, 200, 37, 129] * 8)
    p = jfa.params_for(b["q"], b["k"], b["v"], oq, causal=True)
    ws = jfa.workspace(p)
    _run(w, b, oq, ws)
    status, n_q, n_k, c_fwd, c_dkdv, c_dq = _header(ws)
    assert status == 0 and n_q > 0 and n_k > 0
    assert c_fwd == c_dkdv == c_dq == -1


def test_claimed_lists_are_bitwise_deterministic_and_match_the_oracle():
    lens = [4096, 3000, 2048, 1800, 777, 300]
    w, b, oq = _gdpa_batch(lens, seed=3)
    p = jfa.params_for(b["q"], b["k"], b["v"], oq, causal=True)
    ws = jfa.workspace(p)
    ref = run_gpu(w, b, ws)
    assert _header(ws)[3] >= 0  # claimed
    for _ in range(3):
        got = run_gpu(w, b, ws)
        for name in ("o", "dq", "dk", "dv"):
            assert torch.equal(ref[name], got[name]), name
    whole_batch_check(w, b, ref, seqs=[0, 4, 5], strict_o=False)


def test_softmax_cross_over_long_keys_keeps_the_fixed_order():
    """Softmax cross-attention over long key sequences: the scheduler marks the q-list
    (many steps per item) for claiming, but the softmax kernels are compiled without the
    claimer and walk it in the fixed order, leaving the counters as planned; repeated
    planned calls give the same results bit for bit, and they match the oracle."""
    rng = np.random.default_rng(8)
    lq = rng.integers(1, 64, 400)
    lk = rng.integers(1500, 4096, 400)
    w = workloads.Workload("feedx", 0, 2, 128, 64, False, workloads.ACT_SOFTMAX, torch.bfloat16, True)
    b = workloads.make_batch(w, lq, lk, seed=8, device="cuda")
    oq = torch.as_tensor(b["offs_q"], device="cuda")
    ok = torch.as_tensor(b["offs_k"], device="cuda")
    ws = jfa.jfa_plan(b["q"], b["k"], b["v"], oq, ok)
    status, n_q, n_k, c_fwd, c_dkdv, c_dq = _header(ws)
    assert status == 0 and c_fwd == 0 and c_dq == 0  # marked for claiming
    ref = None
    for _ in range(3):
        o, lse = jfa.jfa_cross_fwd(b["q"], b["k"], b["v"], oq, ok, ws=ws, planned=True)
        g = jfa.jfa_cross_bwd(b["q"], b["k"], b["v"], o, lse, b["do"], oq, ok, ws=ws, planned=True)
        torch.cuda.synchronize()
        assert _header(ws)[3:6] == [0, c_dkdv, 0]
        got = dict(o=o, lse=lse, dq=g[0], dk=g[1], dv=g[2])
        if ref is None:
            ref = got
        for name in got:
            assert torch.equal(ref[name], got[name]), name
    whole_batch_check(w, b, ref, seqs=[0, 1, 399], strict_o=True)
