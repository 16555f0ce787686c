"""The device-built jagged tile scheduler against a plain-Python statement of its rule.

Rule: every (sequence b, head h, tile t) is one item; its cost is the number of inner
steps the kernel runs for it.  Sequences are ordered by total cost, heaviest first (cost
bucketed into 128 levels relative to the heaviest sequence, ties by b); the tiles of a
sequence are contiguous, heaviest first; the H heads of a tile are adjacent.  The list is
read back from the caller's workspace.
"""
import numpy as np
import pytest
import torch

import workloads
from sched_model import expected

pytestmark = pytest.mark.gpu


def _align(x, a=256):
    return (x + a - 1) // a * a


def read_lists(ws, B, Tq, Tk, H):
    """(status, q-list, k-list) from the workspace; each item is 8 int32 values."""
    raw = ws.cpu().numpy()
    hdr = raw[:256].view(np.int32)
    n_q, n_k = int(hdr[1]), int(hdr[2])
    off = 256 + _align(16 * B) + _align(16 * (B + 1))
    max_q = H * (Tq // 32 + B + 1)
    lq_ = raw[off:off + 32 * n_q].view(np.int32).reshape(-1, 8)
    off2 = off + _align(32 * max_q)
    lk_ = raw[off2:off2 + 32 * n_k].view(np.int32).reshape(-1, 8)
    return int(hdr[0]), [tuple(x) for x in lq_], [tuple(x) for x in lk_]


def with_rows(items, lq, lk):
    """Appends (q0, k0, lq, lk) of the item's sequence, as the scheduler does."""
    oq = np.concatenate([[0], np.cumsum(lq)])
    ok = np.concatenate([[0], np.cumsum(lk)])
    return [(b, h, t, c, int(oq[b]), int(ok[b]), int(lq[b]), int(lk[b])) for b, h, t, c in items]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("seed", [0, 1])
def test_tensor_core_lists(causal, seed):
    import jagged_attention_recsys_gb300 as jfa

    rng = np.random.default_rng(seed)
    lq = rng.integers(0, 700, 37)
    lq[3] = 0
    lq[5] = 1
    H = 3
    w = workloads.Workload("s", 0, H, 64, 64, causal, 0, torch.bfloat16, False)
    batch = workloads.make_batch(w, lq, seed=seed, device="cuda")
    oq = torch.as_tensor(batch["offs_q"], device="cuda")
    p = jfa.params_for(batch["q"], batch["k"], batch["v"], oq, causal=causal)
    ws = jfa.workspace(p)
    o, lse = jfa.jfa_fwd(batch["q"], batch["k"], batch["v"], oq, causal=causal, ws=ws)
    st, got_q, _ = read_lists(ws, len(lq), int(oq[-1]), int(oq[-1]), H)
    assert st == 0
    assert got_q == with_rows(expected(list(lq), list(lq), H, 128, 128, causal, False), lq, lq)
    jfa.jfa_bwd(batch["q"], batch["k"], batch["v"], o, lse, batch["do"], oq, causal=causal, ws=ws)
    st, got_q, got_k = read_lists(ws, len(lq), int(oq[-1]), int(oq[-1]), H)
    assert st == 0
    assert got_q == with_rows(expected(list(lq), list(lq), H, 128, 128, causal, False), lq, lq)
    assert got_k == with_rows(expected(list(lq), list(lq), H, 128, 128, causal, True), lq, lq)


def test_cuda_core_lists_cross():
    import jagged_attention_recsys_gb300 as jfa

    rng = np.random.default_rng(5)
    lq = rng.integers(0, 90, 20)
    lk = rng.integers(0, 300, 20)
    H = 2
    w = workloads.Workload("s", 0, H, 32, 32, False, 0, torch.float32, True)
    batch = workloads.make_batch(w, lq, lk, seed=5, device="cuda")
    oq = torch.as_tensor(batch["offs_q"], device="cuda")
    ok = torch.as_tensor(batch["offs_k"], device="cuda")
    p = jfa.params_for(batch["q"], batch["k"], batch["v"], oq)
    ws = jfa.workspace(p)
    o, lse = jfa.jfa_cross_fwd(batch["q"], batch["k"], batch["v"], oq, ok, ws=ws)
    jfa.jfa_cross_bwd(batch["q"], batch["k"], batch["v"], o, lse, batch["do"], oq, ok, ws=ws)
    st, got_q, got_k = read_lists(ws, len(lq), int(oq[-1]), int(ok[-1]), H)
    assert st == 0
    assert got_q == with_rows(expected(list(lq), list(lk), H, 64, 32, False, False), lq, lk)
    assert got_k == with_rows(expected(list(lq), list(lk), H, 64, 32, False, True), lq, lk)


@pytest.mark.parametrize("nseq", [2500, 7000])
def test_large_batch_many_rounds(nseq):
    """More sequences than scheduler threads (several scan rounds), and more than the
    shared-memory cache holds (per-sequence data in the workspace)."""
    import jagged_attention_recsys_gb300 as jfa

    rng = np.random.default_rng(9)
    lq = rng.integers(1, 300, nseq)
    H = 1
    w = workloads.Workload("s", 0, H, 64, 64, True, 0, torch.bfloat16, False)
    batch = workloads.make_batch(w, lq, seed=9, device="cuda")
    oq = torch.as_tensor(batch["offs_q"], device="cuda")
    p = jfa.params_for(batch["q"], batch["k"], batch["v"], oq, causal=True)
    ws = jfa.workspace(p)
    jfa.jfa_fwd(batch["q"], batch["k"], batch["v"], oq, causal=True, ws=ws)
    st, got_q, _ = read_lists(ws, len(lq), int(oq[-1]), int(oq[-1]), H)
    assert st == 0
    assert got_q == with_rows(expected(list(lq), list(lq), H, 128, 128, True, False), lq, lq)


@pytest.mark.parametrize("causal", [False, True])
def test_lists_written_by_many_slices(causal):
    """A batch whose lists are large enough to be written by several CTAs, each taking a
    share of the units after computing the whole order itself; the lists must be exactly
    those of the rule, both from a planned build (q- and k-list at once) and from the
    forward's own build (q-list alone)."""
    import jagged_attention_recsys_gb300 as jfa

    rng = np.random.default_rng(21)
    lq = rng.integers(0, 700, 1500)
    lq[7] = 0
    H = 8
    w = workloads.Workload("s", 0, H, 64, 64, causal, 0, torch.bfloat16, False)
    batch = workloads.make_batch(w, lq, seed=21, device="cuda")
    oq = torch.as_tensor(batch["offs_q"], device="cuda")
    T = int(oq[-1])
    assert H * (T // 128 + len(lq)) >= 8 * 4096  # several slices per list
    want_q = with_rows(expected(list(lq), list(lq), H, 128, 128, causal, False), lq, lq)
    want_k = with_rows(expected(list(lq), list(lq), H, 128, 128, causal, True), lq, lq)
    ws = jfa.jfa_plan(batch["q"], batch["k"], batch["v"], oq, causal=causal)
    st, got_q, got_k = read_lists(ws, len(lq), T, T, H)
    assert st == 0
    assert got_q == want_q
    assert got_k == want_k
    ws2 = jfa.workspace(jfa.params_for(batch["q"], batch["k"], batch["v"], oq, causal=causal))
    jfa.jfa_fwd(batch["q"], batch["k"], batch["v"], oq, causal=causal, ws=ws2)
    st, got_q, _ = read_lists(ws2, len(lq), T, T, H)
    assert st == 0
    assert got_q == want_q
