"""GPU parity: libjfa (through its C ABI) against the fp64 CPU oracle, element by element.

Small cases span several tiles and ragged tails and run the whole batch through the
oracle.  Mid-size batches give every persistent CTA several work items, so that the
kernels' hand-offs between items (deferred epilogues, tiles loaded for the next item,
products issued across item boundaries) are compared with the oracle too.  The
full-size workloads run on the GPU in the launch configuration the benchmark times and
are compared with the oracle over every sequence (the SiLU/L workload, whose oracle
cost is about 12 fp64 TFLOP, over a labelled stratified subset of 32 sequences).
"""
import numpy as np
import pytest
import torch

import workloads
from workloads import ACT_SILU_OVER_LEN as GD, ACT_SOFTMAX as SM, Workload

from parity_util import (compare, full_check, run_gpu, sample_indices, sampled_check,
                         stratified_subset, to64, whole_batch_check)

pytestmark = pytest.mark.gpu

BF16, F32 = torch.bfloat16, torch.float32


def W(dq, dv, causal=False, act=SM, dtype=BF16, cross=False, heads=2):
    return Workload("case", 0, heads, dq, dv, causal, act, dtype, cross)


# ----------------------------------------------------------------------------- fp32 path
def test_tiny_fp32_workload():
    w = workloads.WORKLOADS["tiny"]
    lq, lk = workloads.lengths("tiny")
    full_check(w, lq, lk, strict_o=True)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("act", [SM, GD])
@pytest.mark.parametrize("dims", [(32, 32), (48, 20), (128, 64)])
def test_fp32_self(causal, act, dims):
    lq = [1, 7, 33, 64, 65, 130, 0, 5]
    full_check(W(*dims, causal=causal, act=act, dtype=F32), lq)


@pytest.mark.parametrize("act", [SM, GD])
def test_fp32_cross(act):
    lq = [3, 64, 1, 0, 40]
    lk = [100, 1, 0, 7, 129]
    full_check(W(64, 32, act=act, dtype=F32, cross=True), lq, lk)


# ----------------------------------------------------------------------------- bf16 path
TILE_EDGES = [1, 2, 63, 64, 65, 127, 128, 129, 255, 256, 257, 300, 511]


@pytest.mark.parametrize("dims", [(64, 64), (128, 128), (128, 64), (64, 128)])
@pytest.mark.parametrize("causal", [False, True])
def test_bf16_self_softmax(dims, causal):
    full_check(W(*dims, causal=causal), TILE_EDGES, seed=1)


@pytest.mark.parametrize("dims", [(64, 64), (128, 128), (128, 64), (64, 128)])
@pytest.mark.parametrize("causal", [False, True])
def test_bf16_gdpa(dims, causal):
    full_check(W(*dims, causal=causal, act=GD), TILE_EDGES, seed=2)


@pytest.mark.parametrize("act", [SM, GD])
def test_bf16_cross_asymmetric(act):
    lq = [1, 64, 17, 63, 128, 129, 5]
    lk = [4096, 1, 300, 129, 64, 1000, 2]
    full_check(W(128, 64, act=act, cross=True, heads=4), lq, lk, seed=3)


def test_bf16_zero_length_sequences():
    full_check(W(128, 128, causal=True), [0, 130, 0, 0, 1, 0], seed=4)


def test_cross_with_empty_key_sequences():
    lq = [5, 70, 3]
    lk = [0, 40, 0]
    full_check(W(128, 64, cross=True), lq, lk, seed=5)
    full_check(W(64, 64, cross=True, dtype=F32), lq, lk, seed=5)


def test_single_sequence_single_row():
    full_check(W(64, 64), [1], seed=6)
    full_check(W(64, 64, causal=True, act=GD), [1], seed=6)


# ----------------------------------------------------------------------------- edge cases
def test_empty_batch():
    import jagged_attention_recsys_gb300 as jfa

    e = torch.empty(0, 2, 64, dtype=BF16, device="cuda")
    offs = torch.zeros(1, dtype=torch.int64, device="cuda")
    o, lse = jfa.jfa_fwd(e, e, e, offs)
    dq, dk, dv = jfa.jfa_bwd(e, e, e, o, lse, e, offs)
    assert o.shape == (0, 2, 64) and dq.shape == (0, 2, 64)


def test_bad_offsets_reported_and_outputs_untouched():
    import jagged_attention_recsys_gb300 as jfa

    T, H, D = 40, 2, 64
    q = torch.randn(T, H, D, device="cuda").to(BF16)
    offs = torch.tensor([0, 30, 20, 40], dtype=torch.int64, device="cuda")  # not monotone
    o = torch.full((T, H, D), 7.0, dtype=BF16, device="cuda")
    lse = torch.zeros(T, H, device="cuda")
    p = jfa.params_for(q, q, q, offs)
    ws = jfa.workspace(p)
    jfa.jfa_fwd(q, q, q, offs, o=o, lse=lse, ws=ws)
    assert jfa.jfa_status_check(ws) == jfa.JFA_ERR_BAD_OFFSETS
    assert torch.all(o == 7.0)
    good = torch.tensor([0, 20, 30, 40], dtype=torch.int64, device="cuda")
    jfa.jfa_fwd(q, q, q, good, o=o, lse=lse, ws=ws)
    assert jfa.jfa_status_check(ws) == jfa.JFA_OK
    last = torch.tensor([0, 20, 30, 39], dtype=torch.int64, device="cuda")  # offs[B] != T
    jfa.jfa_fwd(q, q, q, last, o=o, lse=lse, ws=ws)
    assert jfa.jfa_status_check(ws) == jfa.JFA_ERR_BAD_OFFSETS


def test_causal_gdpa_needs_equal_lengths():
    import jagged_attention_recsys_gb300 as jfa

    q = torch.randn(10, 1, 64, device="cuda").to(BF16)
    oq = torch.tensor([0, 4, 10], dtype=torch.int64, device="cuda")
    ok = torch.tensor([0, 5, 10], dtype=torch.int64, device="cuda")
    p = jfa.params_for(q, q, q, oq, causal=True)
    ws = jfa.workspace(p)
    jfa.jfa_gdpa_fwd(q, q, q, oq, ok, causal=True, ws=ws)
    assert jfa.jfa_status_check(ws) == jfa.JFA_ERR_BAD_OFFSETS


def test_neighbour_rows_not_overwritten():
    """Outputs pre-filled with NaN: every row of every sequence must be written, exactly once."""
    import jagged_attention_recsys_gb300 as jfa

    w = W(128, 128, causal=True)
    batch = workloads.make_batch(w, [129, 3, 128, 1], seed=7, device="cuda")
    oq = torch.as_tensor(batch["offs_q"], device="cuda")
    q, k, v, do = batch["q"], batch["k"], batch["v"], batch["do"]
    o = torch.full_like(q, float("nan"))
    lse = torch.full(q.shape[:2], float("nan"), device="cuda")
    jfa.jfa_fwd(q, k, v, oq, causal=True, o=o, lse=lse)
    dq, dk, dv = (torch.full_like(t, float("nan")) for t in (q, k, v))
    jfa.jfa_bwd(q, k, v, o, lse, do, oq, causal=True, dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    for t in (o, lse, dq, dk, dv):
        assert torch.isfinite(t).all()


def test_deterministic_bitwise():
    w = W(128, 128, causal=True, heads=3)
    batch = workloads.make_batch(w, [300, 17, 129, 64], seed=8, device="cuda")
    a = run_gpu(w, batch)
    b = run_gpu(w, batch)
    for n in ("o", "lse", "dq", "dk", "dv"):
        assert torch.equal(a[n], b[n]), n


# ----------------------------------------------------------------------------- mid size
# 600 sequences of lengths U[1, 300] at H = 2 give about 2,000 q-tile and k-tile items,
# 13 per CTA of the 152 persistent CTAs; cross-attention with query lengths U[1, 64] and
# key lengths U[1, 600] gives 1,200 q-tile items (8 per CTA) and about 3,400 k-tile items.
def _mid_lengths(seed, n=600, hi=300):
    rng = np.random.default_rng(seed)
    return rng.integers(1, hi, n, endpoint=True).astype(np.int64)


@pytest.mark.parametrize("dims", [(64, 64), (128, 128)])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("act", [SM, GD])
def test_mid_size_many_items_per_cta(dims, causal, act):
    w = W(*dims, causal=causal, act=act)
    lq = _mid_lengths(10 + dims[0] + 2 * causal + act)
    batch = workloads.make_batch(w, lq, seed=11, device="cuda")
    got = run_gpu(w, batch, check_status=True)
    whole_batch_check(w, batch, got, strict_o=False)


@pytest.mark.parametrize("act", [SM, GD])
def test_mid_size_cross_many_items_per_cta(act):
    w = W(128, 64, act=act, cross=True)
    rng = np.random.default_rng(20 + act)
    lq = rng.integers(1, 64, 600, endpoint=True).astype(np.int64)
    lk = rng.integers(1, 600, 600, endpoint=True).astype(np.int64)
    batch = workloads.make_batch(w, lq, lk, seed=12, device="cuda")
    got = run_gpu(w, batch, check_status=True)
    whole_batch_check(w, batch, got, strict_o=False)


# ----------------------------------------------------------------------------- full size
@pytest.mark.parametrize("name", ["d64", "causal", "cross"])
def test_full_size_workload_whole_batch(name):
    """Every sequence of the named workload, as the benchmark runs it, against the oracle;
    the error metrics are taken over the whole batch."""
    w = workloads.WORKLOADS[name]
    batch = workloads.make_batch(w, device="cuda")
    got = run_gpu(w, batch, check_status=True)
    fig = whole_batch_check(w, batch, got)
    print("\n%s whole batch: %s" % (name, fig))


def test_full_size_gdpa_stratified_subset():
    """The SiLU/L workload at full size on the GPU; against the oracle on its labelled
    stratified subset: the 8 longest and 8 shortest sequences and 16 drawn with seed 0."""
    w = workloads.WORKLOADS["gdpa"]
    batch = workloads.make_batch(w, device="cuda")
    got = run_gpu(w, batch, check_status=True)
    for t in got.values():
        if t is not None:
            assert torch.isfinite(t).all()
    idx = stratified_subset(batch["lq"])
    assert len(idx) == 32
    fig = whole_batch_check(w, batch, got, seqs=idx)
    print("\ngdpa stratified subset (32 of 256 sequences): %s" % fig)


# ----------------------------------------------------------------------------- pooled
def _pooled_run(m, lk, H, Dqk, Dv, dtype, seed):
    import jagged_attention_recsys_gb300 as jfa

    B = len(lk)
    ok = workloads.offsets(lk)
    q, k, v, do = workloads.values(B * m, int(ok[-1]), H, Dqk, Dv, dtype, seed, "cuda")
    q = q[:m].contiguous()  # the shared query rows
    okd = torch.as_tensor(ok, device="cuda")
    o, lse = jfa.jfa_pooled_fwd(q, k, v, okd)
    dq, dk, dv = jfa.jfa_pooled_bwd(q, k, v, o, lse, do, okd)
    torch.cuda.synchronize()
    got = dict(o=to64(o), lse=to64(lse), dq=to64(dq), dk=to64(dk), dv=to64(dv))
    import oracle

    qq, kk, vv, dd = (to64(t) for t in (q, k, v, do))
    ro, rlse = oracle.pooled_fwd(qq, kk, vv, ok)
    rdq, rdk, rdv = oracle.pooled_bwd(qq, kk, vv, dd, ok)
    ref = dict(o=ro, lse=rlse, dq=rdq, dk=rdk, dv=rdv)
    return got, ref


@pytest.mark.parametrize("dims,m", [((128, 64), 32), ((64, 64), 1), ((128, 128), 130)])
def test_bf16_pooled(dims, m):
    """m shared query rows over ragged key sequences (one empty, one longer than a tile)."""
    got, ref = _pooled_run(m, [1, 0, 300, 4096, 129, 64, 17], 2, *dims, BF16, seed=4)
    compare(W(*dims, cross=True), got, ref, fp32=False)


def test_fp32_pooled():
    got, ref = _pooled_run(5, [3, 0, 40, 129], 2, 32, 16, F32, seed=5)
    compare(W(32, 16, dtype=F32, cross=True), got, ref, fp32=True)


def test_fp32_pooled_rows_not_a_multiple_of_16_bytes():
    # 3 shared rows of one head, Dqk = 5: the broadcast copies 60 bytes per sequence in
    # 4-byte words
    got, ref = _pooled_run(3, [3, 0, 7, 70], 1, 5, 3, F32, seed=6)
    compare(W(5, 3, dtype=F32, cross=True, heads=1), got, ref, fp32=True)


def test_full_size_pooled_workload():
    """The pooled workload at full size (512 sequences, 32 shared rows, keys up to 4096):
    o, lse, dk, dv equal, bit for bit, the cross-attention path given the shared rows
    broadcast to every sequence; dq equals the fp64 sum of that path's per-sequence query
    gradients; a sample of whole sequences matches the oracle."""
    import jagged_attention_recsys_gb300 as jfa

    w = workloads.WORKLOADS["pooled"]
    batch = workloads.make_batch(w, device="cuda")
    q, k, v, do = batch["q"], batch["k"], batch["v"], batch["do"]
    B, m = len(batch["lk"]), w.pooled
    okd = torch.as_tensor(batch["offs_k"], device="cuda")
    oqd = torch.as_tensor(batch["offs_q"], device="cuda")
    o, lse = jfa.jfa_pooled_fwd(q, k, v, okd)
    dq, dk, dv = jfa.jfa_pooled_bwd(q, k, v, o, lse, do, okd)
    q_rep = q.repeat(B, 1, 1)
    o2, lse2 = jfa.jfa_cross_fwd(q_rep, k, v, oqd, okd)
    dq2, dk2, dv2 = jfa.jfa_cross_bwd(q_rep, k, v, o2, lse2, do, oqd, okd)
    torch.cuda.synchronize()
    for a, b, n in ((o, o2, "o"), (lse, lse2, "lse"), (dk, dk2, "dk"), (dv, dv2, "dv")):
        assert torch.equal(a, b), n
    assert torch.isfinite(dq.float()).all()
    # the sum over sequences has a fixed order: a second call gives the same bits
    dq_again, _, _ = jfa.jfa_pooled_bwd(q, k, v, o, lse, do, okd)
    torch.cuda.synchronize()
    assert torch.equal(dq, dq_again)
    ref_dq = dq2.double().view(B, m, *q.shape[1:]).sum(0)
    err = float(torch.linalg.vector_norm(dq.double() - ref_dq) / torch.linalg.vector_norm(ref_dq))
    print("\npooled dq against the fp64 sum of the per-sequence cross gradients: rel-L2 %.3g" % err)
    assert err <= 4e-3, err  # bf16 rounding of those per-sequence terms and of the sum
    rep = dict(batch, q=q_rep)
    fig = whole_batch_check(w, rep, dict(o=o, lse=lse, dq=dq2, dk=dk, dv=dv))
    print("\npooled whole batch: %s" % fig)


# ----------------------------------------------------------------------------- BlockAttention
def _block_run(lens, H, Dqk, Dv, dtype, causal, seed):
    import jagged_attention_recsys_gb300 as jfa
    import oracle

    offs = workloads.offsets(lens)
    q, k, v, do = workloads.values(int(offs[-1]), int(offs[-1]), H, Dqk, Dv, dtype, seed, "cuda")
    od = torch.as_tensor(offs, device="cuda")
    o, lse = jfa.jfa_block_fwd(q, k, v, od, causal=causal)
    dq, dk, dv = jfa.jfa_block_bwd(q, k, v, o, lse, do, od, causal=causal)
    torch.cuda.synchronize()
    got = dict(o=to64(o), lse=to64(lse), dq=to64(dq), dk=to64(dk), dv=to64(dv))
    qq, kk, vv, dd = (to64(t) for t in (q, k, v, do))
    ro, rlse = oracle.block_fwd(qq, kk, vv, offs, causal=causal)
    rdq, rdk, rdv = oracle.block_bwd(qq, kk, vv, dd, offs, causal=causal)
    return got, dict(o=ro, lse=rlse, dq=rdq, dk=rdk, dv=rdv)


@pytest.mark.parametrize("dims", [(64, 64), (128, 128)])
@pytest.mark.parametrize("causal", [False, True])
def test_bf16_block(dims, causal):
    """Blocks of 64 rows from the start of every sequence; lengths around block and tile edges."""
    got, ref = _block_run(TILE_EDGES + [0, 1000], 2, *dims, BF16, causal, seed=6)
    compare(W(*dims, causal=causal), got, ref, fp32=False)


def test_fp32_block():
    got, ref = _block_run([1, 63, 64, 65, 130, 0, 200], 2, 32, 32, F32, True, seed=7)
    compare(W(32, 32, causal=True, dtype=F32), got, ref, fp32=True)


def test_block_bad_offsets_reported():
    import jagged_attention_recsys_gb300 as jfa

    q, k, v, do = workloads.values(100, 100, 2, 64, 64, BF16, 0, "cuda")
    bad = torch.as_tensor([0, 60, 40, 100], device="cuda")  # not monotone
    p = jfa.params_for(q, k, v, bad)
    ws = jfa.block_workspace(p)
    o = torch.full((100, 2, 64), 7.0, dtype=BF16, device="cuda")
    lse = torch.zeros(100, 2, dtype=torch.float32, device="cuda")
    jfa.jfa_block_fwd(q, k, v, bad, o=o, lse=lse, ws=ws)
    assert jfa.jfa_status_check(ws) == jfa.JFA_ERR_BAD_OFFSETS
    assert torch.all(o == 7.0)  # untouched


def test_full_size_block_workload():
    """BlockAttention over the causal workload's 1024 sequences (H=8, D=128) on the GPU;
    every block of every sequence against the oracle's definition (causal softmax
    attention within each 64-row block), error metrics over the whole batch."""
    import jagged_attention_recsys_gb300 as jfa
    import oracle

    w = workloads.WORKLOADS["block"]
    batch = workloads.make_batch(w, device="cuda")
    od = torch.as_tensor(batch["offs_q"], device="cuda")
    q, k, v, do = batch["q"], batch["k"], batch["v"], batch["do"]
    p = jfa.params_for(q, k, v, od, causal=True)
    ws = jfa.block_workspace(p)
    o, lse = jfa.jfa_block_fwd(q, k, v, od, causal=True, ws=ws)
    dq, dk, dv = jfa.jfa_block_bwd(q, k, v, o, lse, do, od, causal=True, ws=ws)
    assert jfa.jfa_status_check(ws) == jfa.JFA_OK
    bo = oracle.block_offsets(batch["offs_q"])
    blocks = dict(batch, offs_q=bo, offs_k=bo)
    wb = W(128, 128, causal=True, heads=w.heads)
    fig = whole_batch_check(wb, blocks, dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv))
    print("\nblock whole batch (%d blocks): %s" % (len(bo) - 1, fig))


# ----------------------------------------------------------------------------- BlockAttention + RoPE
def _block_rope_oracle(w, q, k, v, do, offs_q, offs_k):
    import oracle

    o, lse = oracle.block_rope_fwd(q, k, v, offs_q, scale=w.scale, causal=w.causal)
    dq, dk, dv = oracle.block_rope_bwd(q, k, v, do, offs_q, scale=w.scale, causal=w.causal)
    return dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv)


def _block_rope_gpu(batch, causal, ws=None):
    import jagged_attention_recsys_gb300 as jfa

    od = torch.as_tensor(batch["offs_q"], device="cuda")
    q, k, v, do = batch["q"], batch["k"], batch["v"], batch["do"]
    p = jfa.params_for(q, k, v, od, causal=causal)
    ws = jfa.block_workspace(p) if ws is None else ws
    o, lse = jfa.jfa_block_fwd(q, k, v, od, causal=causal, ws=ws, rope=True)
    dq, dk, dv = jfa.jfa_block_bwd(q, k, v, o, lse, do, od, causal=causal, ws=ws, rope=True)
    assert jfa.jfa_status_check(ws) == jfa.JFA_OK
    return dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv)


@pytest.mark.parametrize("dim", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_bf16_block_rope(dim, causal):
    """BlockAttention with the fused rotary embedding against the oracle (RoFormer's rotation
    of q and k, positions counted from each sequence's first row), lengths around block and
    tile edges, and a sequence of many blocks."""
    w = W(dim, dim, causal=causal)
    batch = workloads.make_batch(w, TILE_EDGES + [0, 1000], seed=13, device="cuda")
    got = _block_rope_gpu(batch, causal)
    got = {n: to64(t) for n, t in got.items()}
    ref = _block_rope_oracle(w, *(to64(batch[n]) for n in ("q", "k", "v", "do")), batch["offs_q"],
                             batch["offs_k"])
    compare(w, got, ref, fp32=False)


def test_block_rope_differs_from_plain_block():
    """The rotation changes the result (a kernel that skipped it would match plain
    BlockAttention instead)."""
    w = W(64, 64, causal=True)
    batch = workloads.make_batch(w, [64, 40], seed=14, device="cuda")
    got = _block_rope_gpu(batch, True)
    import jagged_attention_recsys_gb300 as jfa

    od = torch.as_tensor(batch["offs_q"], device="cuda")
    o_plain, _ = jfa.jfa_block_fwd(batch["q"], batch["k"], batch["v"], od, causal=True)
    torch.cuda.synchronize()
    assert float((got["o"].float() - o_plain.float()).abs().max()) > 0.05


def test_block_rope_rejects_fp32():
    import jagged_attention_recsys_gb300 as jfa

    q, k, v, do = workloads.values(70, 70, 2, 32, 32, F32, 0, "cuda")
    od = torch.as_tensor(workloads.offsets([70]), device="cuda")
    with pytest.raises(jfa.JfaError) as e:
        jfa.jfa_block_fwd(q, k, v, od, rope=True)
    assert e.value.code == jfa.JFA_ERR_UNSUPPORTED


def test_full_size_block_rope_workload():
    """BlockAttention with the rotary embedding over the causal workload's 1024 sequences
    (H=8, D=128): every sequence against the oracle, error metrics over the whole batch."""
    w = workloads.WORKLOADS["block_rope"]
    batch = workloads.make_batch(w, device="cuda")
    got = _block_rope_gpu(batch, True)
    wb = W(128, 128, causal=True, heads=w.heads)
    fig = whole_batch_check(wb, batch, got, oracle_fn=_block_rope_oracle)
    print("\nblock_rope whole batch: %s" % fig)


# ----------------------------------------------------------------------------- CUDA graphs
@pytest.mark.parametrize("planned", [False, True])
@pytest.mark.parametrize("name", ["d64", "gdpa"])
def test_cuda_graph_replay_matches_separate_calls(name, planned):
    """The library's calls capture into a CUDA graph (nothing synchronises with the host),
    and a replay gives the same outputs, bit for bit, as the calls made one by one; with
    ``planned``, the captured step is a plan and the planned calls."""
    import jagged_attention_recsys_gb300 as jfa

    w = workloads.WORKLOADS[name]
    lq = [1, 130, 64, 300, 7]
    batch = workloads.make_batch(w, lq, lq, seed=3, device="cuda")
    q, k, v, do = batch["q"], batch["k"], batch["v"], batch["do"]
    oq = torch.as_tensor(batch["offs_q"], device="cuda")
    p = jfa.params_for(q, k, v, oq, causal=w.causal)
    ws = jfa.workspace(p)
    outs = dict(o=torch.empty(q.shape[0], q.shape[1], v.shape[2], dtype=q.dtype, device="cuda"),
                lse=torch.empty(q.shape[0], q.shape[1], dtype=torch.float32, device="cuda"),
                dq=torch.empty_like(q), dk=torch.empty_like(k), dv=torch.empty_like(v))

    def step():
        if planned:
            jfa.jfa_plan(q, k, v, oq, causal=w.causal, ws=ws)
        if w.act == workloads.ACT_SILU_OVER_LEN:
            jfa.jfa_gdpa_fwd(q, k, v, oq, causal=w.causal, o=outs["o"], ws=ws, planned=planned)
            jfa.jfa_gdpa_bwd(q, k, v, do, oq, causal=w.causal, dq=outs["dq"], dk=outs["dk"],
                             dv=outs["dv"], ws=ws, planned=planned)
        else:
            jfa.jfa_fwd(q, k, v, oq, causal=w.causal, o=outs["o"], lse=outs["lse"], ws=ws,
                        planned=planned)
            jfa.jfa_bwd(q, k, v, outs["o"], outs["lse"], do, oq, causal=w.causal, dq=outs["dq"],
                        dk=outs["dk"], dv=outs["dv"], ws=ws, planned=planned)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    eager = {n: t.clone() for n, t in outs.items()}
    for t in outs.values():
        t.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for t in outs.values():
        t.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert jfa.jfa_status_check(ws) == 0
    for n in ("o", "dq", "dk", "dv") + (("lse",) if w.act == workloads.ACT_SOFTMAX else ()):
        assert torch.equal(outs[n], eager[n]), n
