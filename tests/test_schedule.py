"""Pins of the split-KV partition rule (oracle/schedule.py).

The rule is the library's own (the pages leave the scheduler open), so these
tests pin the plain-Python statement to the properties any valid partition
must have: every key tile processed by exactly one part, an item's pieces
contiguous and owned by consecutive parts with piece indices 0..n-1, no part
over its budget, empty items written exactly once, and split counts that
match the pieces.
"""
import numpy as np
import pytest

from oracle import schedule as S


CASES = [
    # seqlens, H, T, parts, topk, causal
    ([256, 256], 64, 1, 8, 0, False),
    ([4096] * 16, 128, 1, 76, 0, False),
    ([1, 64, 65, 0, 129, 5000], 128, 1, 7, 0, False),
    ([0, 0, 0], 64, 1, 4, 0, False),
    ([16384] * 3, 64, 4, 10, 0, True),
    ([3, 130, 64], 64, 3, 5, 0, True),
    ([65536] * 4, 64, 1, 9, 2048, False),
    ([100, 300], 64, 2, 3, 70, False),
    ([7], 128, 1, 76, 0, False),
]


def _check(seqlens, H, T, P, topk, causal):
    items = S.item_list(seqlens, H, T, topk, causal)
    md, ns = S.schedule(seqlens, H, T, P, topk, causal)
    assert len(md) == P and len(ns) == len(items) + 1
    pcs = S.pieces(md, items)
    owned = {}
    per_item = {}
    for p, i, t0, t1, k in pcs:
        per_item.setdefault(i, []).append((p, t0, t1, k))
        for t in range(t0, t1):
            assert (i, t) not in owned, "tile processed twice"
            owned[(i, t)] = p
    for i, it in enumerate(items):
        n = it[3]
        got = per_item.get(i, [])
        if n == 0:
            assert len(got) == 1, "empty item must be written exactly once"
            assert ns[i + 1] - ns[i] == 1
            continue
        for t in range(n):
            assert (i, t) in owned, "tile never processed"
        got.sort()
        assert [g[3] for g in got] == list(range(len(got)))
        assert ns[i + 1] - ns[i] == len(got)
        for a, b in zip(got[:-1], got[1:]):
            assert a[2] == b[1], "pieces of an item must be contiguous"
            assert b[0] == a[0] + 1, "consecutive parts"
    W = sum(S.FIXED_COST + it[3] for it in items)
    L = -(-W // P)
    load = np.zeros(P, dtype=int)
    for (i, t), p in owned.items():
        load[p] += 1
    assert load.max() <= L
    assert ns[-1] <= len(items) + P - 1
    return items, md, ns


@pytest.mark.parametrize("case", CASES)
def test_partition_properties(case):
    _check(*case)


def test_partition_random():
    rng = np.random.default_rng(3)
    for _ in range(200):
        B = int(rng.integers(1, 12))
        H = int(rng.choice([64, 128]))
        T = int(rng.integers(1, 5))
        causal = bool(rng.integers(0, 2))
        topk = int(rng.choice([0, 0, 64, 100])) if not causal else 0
        lo = topk if topk else 0
        sl = [int(x) for x in rng.integers(lo, 3000, size=B)]
        P = int(rng.integers(1, 80))
        _check(sl, H, T, P, topk, causal)


def test_items_rows_and_tiles():
    """M tiles of at most 128 rows, row = t*H + h, ordered m-tile-major;
    causal tiles follow the last query token of the tile; top-k items are
    one query token each, ordered b-major."""
    it = S.item_list([700, 300, 50], 64, 4, 0, False)
    assert [(b, r0) for b, r0, _, _ in it] == [(0, 0), (1, 0), (2, 0), (0, 128), (1, 128), (2, 128)]
    it = S.item_list([300, 200], 64, 2, 70, False)
    assert [(b, r0) for b, r0, _, _ in it] == [(0, 0), (0, 64), (1, 0), (1, 64)]
    it = S.item_list([1000], 64, 4, 0, True)
    assert [(r0, c) for _, r0, c, _ in it] == [(0, 128), (128, 128)]
    assert it[0][3] == -(-(1000 - 4 + 1 + 1) // 64)
    assert it[1][3] == -(-1000 // 64)
    it = S.item_list([300, 10], 128, 2, 100, False)
    assert len(it) == 4 and all(x[3] == 2 and x[2] == 128 for x in it)
    it = S.item_list([5], 64, 3, 0, False)
    assert [(r0, c) for _, r0, c, _ in it] == [(0, 128), (128, 64)]
    it = S.item_list([2], 64, 4, 0, True)
    assert it[0][3] == 0 and it[1][3] == 1
