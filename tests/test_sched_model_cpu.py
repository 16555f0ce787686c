"""The scheduler's plain-Python rule (`sched_model.expected`) on hand-worked cases.

The GPU tests hold the device-built work lists to this rule item for item; these cases
pin the rule itself: costs, the heavy-first order of sequences, the tile order inside a
sequence, and heads adjacent.
"""
from sched_model import expected


def _seq_order(items):
    out = []
    for b, *_ in items:
        if not out or out[-1] != b:
            out.append(b)
    return out


def test_query_tiles_non_causal():
    # lengths 130, 10, 300 with 128-row tiles and 128-key steps: 2, 1 and 3 q-tiles of
    # cost ceil(L/128) = 2, 1, 3 each; totals 4, 1, 9 -> order 2, 0, 1
    items = expected([130, 10, 300], [130, 10, 300], 2, 128, 128, False, False)
    assert _seq_order(items) == [2, 0, 1]
    assert items[:6] == [(2, 0, 0, 3), (2, 1, 0, 3), (2, 0, 1, 3), (2, 1, 1, 3),
                         (2, 0, 2, 3), (2, 1, 2, 3)]
    assert items[6:] == [(0, 0, 0, 2), (0, 1, 0, 2), (0, 0, 1, 2), (0, 1, 1, 2),
                         (1, 0, 0, 1), (1, 1, 0, 1)]


def test_query_tiles_causal_heaviest_tile_first():
    # causal: q-tile t sees the keys up to its last row, ceil(min(L, 128(t+1))/128) steps;
    # sequence 2 (300 rows): tiles cost 1, 2, 3 and are taken last tile first
    items = expected([130, 10, 300], [130, 10, 300], 1, 128, 128, True, False)
    assert items == [(2, 0, 2, 3), (2, 0, 1, 2), (2, 0, 0, 1),
                     (0, 0, 1, 2), (0, 0, 0, 1),
                     (1, 0, 0, 1)]


def test_key_tiles_causal():
    # k-tile t of a causal sequence is visited by the q-rows from its first key on:
    # ceil(L/step) - t*tile/step steps; 300 rows, 128-key tiles, 64-row steps: 5, 3, 1
    items = expected([300, 64], [300, 64], 1, 128, 64, True, True)
    assert items == [(0, 0, 0, 5), (0, 0, 1, 3), (0, 0, 2, 1), (1, 0, 0, 1)]


def test_key_tiles_cross_non_causal():
    # cross: k-tiles of the key lengths, each visited by every q-step of the sequence
    items = expected([64, 3], [200, 500], 1, 128, 32, False, True)
    # totals: seq 0: 2 tiles x ceil(64/32) = 4; seq 1: 4 tiles x 1 = 4 -> tie, by index
    assert items == [(0, 0, 0, 2), (0, 0, 1, 2),
                     (1, 0, 0, 1), (1, 0, 1, 1), (1, 0, 2, 1), (1, 0, 3, 1)]


def test_buckets_merge_near_ties_and_keep_index_order():
    # one q-tile per sequence costing ceil(Lk/1) = Lk steps: totals 1000, 999, 1000 fall
    # in levels 127, 126 (999*127//1000), 127 of the 128 -> 0 and 2 tie, by index
    items = expected([1, 1, 1], [1000, 999, 1000], 1, 128, 1, False, False)
    assert _seq_order(items) == [0, 2, 1]
    # totals 993, 1000, 995: levels 126, 127, 126 -> 995 and 993 share a level, so
    # index order decides between them
    items = expected([1, 1, 1], [993, 1000, 995], 1, 128, 1, False, False)
    assert _seq_order(items) == [1, 0, 2]
    # equal work everywhere: index order
    items = expected([5, 5, 5, 5], [5, 5, 5, 5], 1, 128, 128, False, False)
    assert _seq_order(items) == [0, 1, 2, 3]


def test_empty_sequences_have_no_items():
    items = expected([0, 7, 0], [0, 7, 0], 3, 128, 128, True, False)
    assert [(b, h) for b, h, _, _ in items] == [(1, 0), (1, 1), (1, 2)]
    assert expected([], [], 2, 128, 128, False, False) == []
