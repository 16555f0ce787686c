"""The kernels' bounded waits give up cleanly, and the GPU stays usable afterwards.

Every mbarrier wait inside the tensor-core kernels is bounded (about two seconds).  A
wait that runs out records JFA_ERR_TIMEOUT in the workspace's status word, raises the
CTA's abort flag so that its other roles leave their loops, waits for the CTA's own
TMA loads and MMAs in flight, frees its tensor memory and returns: no trap, no fault,
the context stays valid.  The library's test hook (jfa_test_hold) makes the forward
kernel's MMA issuer wait first on a barrier that nothing arrives on, before it issues
any MMA; this test checks the status that comes back and then runs normal calls on the
same GPU and workspace against the oracle.
"""
import numpy as np
import pytest
import torch

import workloads
from parity_util import compare, run_oracle, to64, full_check

pytestmark = pytest.mark.gpu


def test_forward_wait_gives_up_reports_timeout_and_gpu_stays_usable():
    import jagged_attention_recsys_gb300 as jfa

    w = workloads.Workload("hold", 0, 2, 128, 128, True, workloads.ACT_SOFTMAX,
                           torch.bfloat16, False)
    lens = [300, 1, 129, 64]
    batch = workloads.make_batch(w, lens, seed=9, device="cuda")
    oq = torch.as_tensor(batch["offs_q"], device="cuda")
    q, k, v = batch["q"], batch["k"], batch["v"]
    p = jfa.params_for(q, k, v, oq, causal=True)
    ws = jfa.workspace(p)
    o = torch.full((q.shape[0], q.shape[1], v.shape[2]), float("nan"), dtype=q.dtype,
                   device="cuda")
    lse = torch.full(q.shape[:2], float("nan"), device="cuda")
    jfa.jfa_test_hold(True)
    try:
        jfa.jfa_fwd(q, k, v, oq, causal=True, o=o, lse=lse, ws=ws)
        st = jfa.jfa_status_check(ws)
    finally:
        jfa.jfa_test_hold(False)
    assert st == jfa.JFA_ERR_TIMEOUT, jfa.status_string(st)
    # nothing was computed: no MMA was issued before the issuer gave up
    assert torch.isnan(o.float()).all() and torch.isnan(lse).all()

    # the same GPU and workspace serve a normal call, which matches the oracle
    jfa.jfa_fwd(q, k, v, oq, causal=True, o=o, lse=lse, ws=ws)
    assert jfa.jfa_status_check(ws) == jfa.JFA_OK
    ref = run_oracle(w, *(to64(batch[n]) for n in ("q", "k", "v", "do")), batch["offs_q"],
                     batch["offs_k"])
    got_o, ref_o = to64(o), ref["o"]
    assert float(np.max(np.abs(got_o - ref_o))) <= 2e-2
    fin = np.isfinite(ref["lse"])
    assert float(np.max(np.abs(to64(lse)[fin] - ref["lse"][fin]))) <= 2e-2
    # and a whole forward + backward on fresh buffers
    full_check(w, lens, seed=9)


def test_claimed_forward_wait_gives_up_and_gpu_stays_usable():
    """The same with claimed work items (SiLU/L, long sequences): the claimer and every
    reader of the item ring leave through the abort path, and the counter-based
    distribution works again on the next call."""
    import jagged_attention_recsys_gb300 as jfa

    w = workloads.Workload("hold_gdpa", 0, 2, 128, 128, True, workloads.ACT_SILU_OVER_LEN,
                           torch.bfloat16, False)
    lens = [2048, 1500, 3000, 2048]
    batch = workloads.make_batch(w, lens, seed=10, device="cuda")
    oq = torch.as_tensor(batch["offs_q"], device="cuda")
    q, k, v = batch["q"], batch["k"], batch["v"]
    p = jfa.params_for(q, k, v, oq, causal=True)
    ws = jfa.workspace(p)
    o = torch.full((q.shape[0], q.shape[1], v.shape[2]), float("nan"), dtype=q.dtype,
                   device="cuda")
    jfa.jfa_test_hold(True)
    try:
        jfa.jfa_gdpa_fwd(q, k, v, oq, causal=True, o=o, ws=ws)
        st = jfa.jfa_status_check(ws)
    finally:
        jfa.jfa_test_hold(False)
    assert st == jfa.JFA_ERR_TIMEOUT, jfa.status_string(st)
    assert ws[12:16].view(torch.int32).item() >= 0  # the list was in the claimed mode
    assert torch.isnan(o.float()).all()

    jfa.jfa_gdpa_fwd(q, k, v, oq, causal=True, o=o, ws=ws)
    assert jfa.jfa_status_check(ws) == jfa.JFA_OK
    full_check(w, lens, seed=10)
