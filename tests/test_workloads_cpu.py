"""The seeded input recipe and the FLOP count of the metric, on the CPU.

The sizes below are the seed-0 draws the benchmark and the full-size parity tests use;
a change to the recipe (draw order, distribution, clipping) changes them.
"""
import numpy as np
import pytest
import torch

import workloads

SIZES = {  # name: (B, T_q, T_k)
    "tiny": (4, 105, 105),
    "d64": (256, 68452, 68452),
    "causal": (1024, 323911, 323911),
    "block": (1024, 323911, 323911),
    "cross": (512, 17331, 1067204),
    "gdpa": (256, 577927, 577927),
    "pooled": (512, 16384, 1092721),
}


@pytest.mark.parametrize("name", sorted(SIZES))
def test_seed0_sizes(name):
    lq, lk = workloads.lengths(name, seed=0)
    B, tq, tk = SIZES[name]
    assert len(lq) == len(lk) == B
    assert int(lq.sum()) == tq and int(lk.sum()) == tk


@pytest.mark.parametrize("name,lo,hi", [("d64", 1, 512), ("causal", 1, 2048), ("gdpa", 256, 4096)])
def test_length_ranges(name, lo, hi):
    lq, lk = workloads.lengths(name, seed=0)
    assert lq.min() >= lo and lq.max() <= hi and np.array_equal(lq, lk)


def test_cross_and_pooled_ranges():
    lq, lk = workloads.lengths("cross")
    assert 1 <= lq.min() and lq.max() <= 64 and 1 <= lk.min() and lk.max() <= 4096
    lq, lk = workloads.lengths("pooled")
    assert (lq == 32).all() and 1 <= lk.min() and lk.max() <= 4096


def test_draws_are_reproducible():
    a = workloads.lengths("causal", seed=3)
    b = workloads.lengths("causal", seed=3)
    assert all(np.array_equal(x, y) for x, y in zip(a, b))
    v1 = workloads.values(5, 7, 2, 8, 4, torch.bfloat16, seed=9)
    v2 = workloads.values(5, 7, 2, 8, 4, torch.bfloat16, seed=9)
    assert all(torch.equal(x, y) for x, y in zip(v1, v2))
    assert [tuple(t.shape) for t in v1] == [(5, 2, 8), (7, 2, 8), (7, 2, 4), (5, 2, 4)]


def test_offsets():
    assert workloads.offsets([3, 0, 5]).tolist() == [0, 3, 3, 8]
    assert workloads.offsets([]).tolist() == [0]


def test_valid_pairs_hand_worked():
    vp = workloads.valid_pairs
    assert vp([3], [3], False) == 9
    assert vp([3], [3], True) == 6  # 1 + 2 + 3
    assert vp([2, 1], [3, 0], False) == 6  # cross: 2*3 + 1*0
    # blocks of 2 over a length-5 sequence: blocks of 2, 2 and 1 rows
    assert vp([5], [5], True, block=2) == 3 + 3 + 1
    assert vp([5], [5], False, block=2) == 4 + 4 + 1
    assert vp([64, 65], [64, 65], True, block=64) == 2 * 64 * 65 / 2 + 1


def test_useful_flops_hand_worked():
    # one sequence of 3 rows, causal: 6 pairs; H=2, Dqk=4, Dv=2
    w = workloads.Workload("t", 1, 2, 4, 2, True, workloads.ACT_SOFTMAX, torch.float32, False)
    fwd, bwd = workloads.useful_flops(w, [3], [3])
    assert fwd == 2 * 6 * 2 * (4 + 2)  # QK^T and PV
    assert bwd == 2 * 6 * 2 * (3 * 4 + 2 * 2)  # S, dQ, dK on Dqk; dV, dP on Dv
    w = workloads.Workload("t", 1, 1, 8, 8, False, workloads.ACT_SOFTMAX, torch.float32, False)
    fwd, bwd = workloads.useful_flops(w, [5], [5])
    assert bwd == 2.5 * fwd


def test_executed_pairs_hand_worked():
    ep = workloads.executed_pairs
    assert ep([100], [100], False) == 128 * 128
    assert ep([129], [300], False) == 2 * 3 * 128 * 128
    # causal, 300 rows: q-tiles 0, 1, 2 cover 1, 2, 3 key tiles
    assert ep([300], [300], True) == 6 * 128 * 128
    assert ep([0, 5], [0, 5], True) == 128 * 128
    # blocks of 64 over 130 rows, two blocks per 128-row tile: pieces of 128 and 2 rows
    assert ep([130], [130], True, block=64) == 2 * 128 * 128
    assert ep([300, 64], [300, 64], False, block=64) == 4 * 128 * 128


def test_tile_occupancy_of_the_workloads():
    """The share of executed 128 x 128 MMA area that holds valid pairs, seed-0 draws."""
    occ = {}
    for name in ("d64", "causal", "cross", "gdpa", "pooled", "block"):
        w = workloads.WORKLOADS[name]
        lq, lk = workloads.lengths(name)
        occ[name] = workloads.valid_pairs(lq, lk, w.causal, w.block) / workloads.executed_pairs(
            lq, lk, w.causal, w.block)
    expect = {"d64": 0.723, "causal": 0.656, "cross": 0.265, "gdpa": 0.918, "pooled": 0.243,
              "block": 0.205}
    for name, v in expect.items():
        assert abs(occ[name] - v) < 5e-4, (name, occ[name])


def test_executed_pairs_trimmed_queries_hand_worked():
    ep = workloads.executed_pairs
    # dK/dV: a step's products cover its valid queries rounded up to 16
    assert ep([100], [100], False, trim_queries=True) == 128 * 112
    assert ep([130], [300], False, trim_queries=True) == 3 * 128 * (128 + 16)
    # causal, 300 queries: query tiles of 128, 128, 44 -> 48 rows; 1 + 2 + 3 key tiles
    assert ep([300], [300], True, trim_queries=True) == 128 * (1 * 128 + 2 * 128 + 3 * 48)
