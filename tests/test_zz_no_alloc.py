"""jfa_fwd_noalloc: the forward for callers that cannot allocate device memory.

Such callers (a plugin inside an application that owns the device allocator, a
serving process that must not allocate after start-up) cannot hand jfa_fwd a
workspace, so this entry point keeps its scratch in a fixed array compiled into
the library.  Its results must equal jfa_fwd's.  This file is collected last so
that a run stopping at the first failure has already run every other test; it
also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads
from parity_util import BF16_O_ATOL, BF16_REL_L2, rel_l2, to64

pytestmark = pytest.mark.gpu


def _call_noalloc(jfa, p, q, k, v, offs, o, lse):
    """Through the C ABI directly: raw device pointers and the current stream."""
    vp = ctypes.c_void_p
    stream = vp(torch.cuda.current_stream().cuda_stream)
    return jfa.lib().jfa_fwd_noalloc(ctypes.byref(p), vp(q.data_ptr()), vp(k.data_ptr()),
                                     vp(v.data_ptr()), vp(offs.data_ptr()), vp(o.data_ptr()),
                                     vp(lse.data_ptr()), stream)


@pytest.mark.parametrize("causal", [True, False])
def test_noalloc_matches_workspace_forward_twice(causal):
    import jagged_attention_recsys_gb300 as jfa

    w = workloads.Workload("noalloc", 0, 3, 128, 128, causal, workloads.ACT_SOFTMAX,
                           torch.bfloat16, False)
    # Two calls in a row on different batches: the shared scratch must not carry
    # anything from the first call into the second.
    for seed, lens in ((0, [300, 1, 129, 64, 0, 511]), (1, [7, 1000, 128])):
        batch = workloads.make_batch(w, lens, seed=seed, device="cuda")
        offs = torch.as_tensor(batch["offs_q"], device="cuda")
        q, k, v = batch["q"], batch["k"], batch["v"]
        ref_o, ref_lse = jfa.jfa_fwd(q, k, v, offs, causal=causal)
        p = jfa.params_for(q, k, v, offs, causal=causal)
        o = torch.full_like(ref_o, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        rc = _call_noalloc(jfa, p, q, k, v, offs, o, lse)
        assert rc == jfa.JFA_OK, jfa.status_string(rc)
        torch.cuda.synchronize()
        g, r = to64(o), to64(ref_o)
        assert np.all(np.isfinite(g))
        assert float(np.max(np.abs(g - r))) <= BF16_O_ATOL
        assert rel_l2(g, r) <= BF16_REL_L2
        gl, rl = to64(lse), to64(ref_lse)
        assert float(np.max(np.abs(gl - rl))) <= 2e-2
        # same kernels, same order: in fact bitwise equal
        assert torch.equal(o, ref_o) and torch.equal(lse, ref_lse)


def test_noalloc_rejects_requests_beyond_its_scratch():
    import jagged_attention_recsys_gb300 as jfa

    # ~2^31 rows x 8 heads needs far more than the fixed scratch; rejected on the host.
    p = jfa.make_params(1, 1 << 30, 1 << 30, 8, 128, 128, torch.bfloat16)
    vp = ctypes.c_void_p
    rc = jfa.lib().jfa_fwd_noalloc(ctypes.byref(p), vp(256), vp(256), vp(256), vp(256),
                                   vp(256), vp(256), None)
    assert rc == jfa.JFA_ERR_WORKSPACE


def test_noalloc_many_sequences_matches_workspace_forward():
    """More sequences than the scheduler keeps in shared memory (6,144), so its
    per-sequence arrays go to the scratch: here the fixed array.  Bitwise equal to
    jfa_fwd with a workspace, twice in a row."""
    import jagged_attention_recsys_gb300 as jfa

    w = workloads.Workload("noalloc", 0, 2, 64, 64, False, workloads.ACT_SOFTMAX,
                           torch.bfloat16, False)
    rng = np.random.default_rng(3)
    for seed in (0, 1):
        lens = rng.integers(0, 9, 7000).astype(np.int64)
        batch = workloads.make_batch(w, lens, seed=seed, device="cuda")
        offs = torch.as_tensor(batch["offs_q"], device="cuda")
        q, k, v = batch["q"], batch["k"], batch["v"]
        ref_o, ref_lse = jfa.jfa_fwd(q, k, v, offs)
        p = jfa.params_for(q, k, v, offs)
        o = torch.full_like(ref_o, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        rc = _call_noalloc(jfa, p, q, k, v, offs, o, lse)
        assert rc == jfa.JFA_OK, jfa.status_string(rc)
        torch.cuda.synchronize()
        assert torch.equal(o, ref_o) and torch.equal(lse, ref_lse)


def test_noalloc_bad_offsets_leave_outputs_untouched():
    """Offsets that are not a jagged layout: the call computes nothing (the status word is
    in the fixed array, out of the caller's reach), so NaN-filled outputs stay NaN; a
    following valid call through the same array computes normally."""
    import jagged_attention_recsys_gb300 as jfa

    T, H, D = 40, 2, 64
    q = torch.randn(T, H, D, device="cuda").to(torch.bfloat16)
    bad = torch.tensor([0, 30, 20, 40], dtype=torch.int64, device="cuda")  # not monotone
    p = jfa.params_for(q, q, q, bad)
    o = torch.full((T, H, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((T, H), float("nan"), device="cuda")
    assert _call_noalloc(jfa, p, q, q, q, bad, o, lse) == jfa.JFA_OK
    torch.cuda.synchronize()
    assert torch.isnan(o.float()).all() and torch.isnan(lse).all()
    good = torch.tensor([0, 20, 30, 40], dtype=torch.int64, device="cuda")
    assert _call_noalloc(jfa, p, q, q, q, good, o, lse) == jfa.JFA_OK
    ref_o, ref_lse = jfa.jfa_fwd(q, q, q, good)
    torch.cuda.synchronize()
    assert torch.equal(o, ref_o) and torch.equal(lse, ref_lse)
