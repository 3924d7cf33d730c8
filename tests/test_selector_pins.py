"""Pins of the CPU statement of the comparison selectors (oracle/selectors.py): hand-worked
cases, brute force on tiny inputs, invariances and special cases. No GPU needed."""
import itertools
import math

import numpy as np
import pytest

from oracle import selectors as SEL


def _scores(G, per_block, n=None):
    """s_hat [G, n] with every token of block c of head i at per_block[i][c]."""
    per_block = np.asarray(per_block, float)
    nb = per_block.shape[1]
    n = n or nb * 64
    s = np.zeros((G, n))
    for c in range(nb):
        s[:, c * 64:min(n, (c + 1) * 64)] = per_block[:, c:c + 1]
    return s


def test_forced_blocks_follow_the_window_edges():
    f = SEL.forced_blocks(300, 65, 37)  # tokens 0..64 and 263..299
    assert f.tolist() == [True, True, False, False, True]
    assert SEL.forced_blocks(300, 0, 0).tolist() == [False] * 5
    assert SEL.forced_blocks(40, 64, 0).tolist() == [True]


def test_topk_hand_worked():
    # head 0 block maxima 1, 5, 3, 2; head 1: 4, 0, 0, 6 -> importance 4, 5, 3, 6
    s = _scores(2, [[1, 5, 3, 2], [4, 0, 0, 6]])
    s[0, 10] = 4.5  # one token of block 0 of head 0 above the rest of its block
    keep, imp = SEL.select_topk(s, 256, 0, 0, 2)
    assert imp.tolist() == [4.5, 5, 3, 6]
    assert keep.tolist() == [0, 1, 0, 1]
    keep, _ = SEL.select_topk(s, 256, 0, 0, 3)
    assert keep.tolist() == [1, 1, 0, 1]


def test_topk_ties_prefer_lower_blocks_and_budget_edges():
    s = _scores(1, [[2, 2, 2, 2, 2]])
    assert SEL.select_topk(s, 320, 0, 0, 2)[0].tolist() == [1, 1, 0, 0, 0]
    assert SEL.select_topk(s, 320, 0, 0, 0)[0].tolist() == [0] * 5
    assert SEL.select_topk(s, 320, 0, 0, 99)[0].tolist() == [1] * 5


def test_topk_keeps_forced_blocks_outside_the_budget():
    s = _scores(1, [[-9, 1, 3, 2, -9]])
    keep, _ = SEL.select_topk(s, 320, 64, 64, 1)  # blocks 0 and 4 forced
    assert keep.tolist() == [1, 0, 1, 0, 1]
    keep, _ = SEL.select_topk(s, 300, 1, 1, 0)
    assert keep.tolist() == [1, 0, 0, 0, 1]


def test_topp_hand_worked_masses():
    # every token of a block shares one score: block masses are proportional to e^score, so
    # scores log 5, log 3, log 2 give masses 0.5, 0.3, 0.2
    s = _scores(1, [[math.log(5), math.log(3), math.log(2)]])
    keep, mass, before = SEL.select_topp(s, 192, 0, 0, 0.6)
    np.testing.assert_allclose(mass[0], [0.5, 0.3, 0.2], rtol=1e-12)
    np.testing.assert_allclose(before[0], [0.0, 0.5, 0.8], rtol=1e-12, atol=1e-15)
    assert keep.tolist() == [1, 1, 0]
    assert SEL.select_topp(s, 192, 0, 0, 0.45)[0].tolist() == [1, 0, 0]
    assert SEL.select_topp(s, 192, 0, 0, 0.85)[0].tolist() == [1, 1, 1]
    # the block order is by mass, not by position
    s2 = _scores(1, [[math.log(2), math.log(5), math.log(3)]])
    assert SEL.select_topp(s2, 192, 0, 0, 0.6)[0].tolist() == [0, 1, 1]


def test_topp_unions_heads_and_forced_blocks():
    s = _scores(2, [[9, 0, 0, 0], [0, 0, 9, 0]])
    keep, _, _ = SEL.select_topp(s, 256, 0, 0, 0.5)
    assert keep.tolist() == [1, 0, 1, 0]
    keep, _, _ = SEL.select_topp(s, 256, 0, 64, 0.5)  # block 3 forced
    assert keep.tolist() == [1, 0, 1, 1]


def test_topp_ragged_last_block_mass():
    # 130 tokens: the last block holds 2 tokens; equal scores give masses 64/130, 64/130, 2/130
    s = np.zeros((1, 130))
    _, mass, _ = SEL.select_topp(s, 130, 0, 0, 0.9)
    np.testing.assert_allclose(mass[0], [64 / 130, 64 / 130, 2 / 130], rtol=1e-12)


@pytest.mark.parametrize("seed", range(6))
def test_topp_prefix_is_the_shortest_by_brute_force(seed):
    rng = np.random.default_rng(seed)
    G, nb = 3, 6
    n = nb * 64 - int(rng.integers(0, 60))
    s = rng.standard_normal((G, n)) * 2.0
    for p in (0.3, 0.7, 0.95):
        keep, mass, before = SEL.select_topp(s, n, 0, 0, p)
        union = np.zeros(nb, bool)
        for i in range(G):
            mine = before[i] < p
            union |= mine
            # the shortest subset whose mass reaches p, found by enumeration
            shortest = next(r for r in range(1, nb + 1)
                            if any(mass[i, list(c)].sum() >= p
                                   for c in itertools.combinations(range(nb), r)))
            assert mine.sum() == shortest
            assert mass[i, mine].sum() >= p - 1e-12
            # and it holds the heaviest blocks
            assert mass[i, mine].min() >= mass[i, ~mine].max(initial=-1)
        assert np.array_equal(keep.astype(bool), union)


@pytest.mark.parametrize("seed", range(4))
def test_topk_by_brute_force(seed):
    rng = np.random.default_rng(100 + seed)
    G, nb = 2, 7
    n = nb * 64 - 5
    s = rng.standard_normal((G, n))
    imp = np.array([s[:, c * 64:min(n, c * 64 + 64)].max() for c in range(nb)])
    for k in range(nb + 1):
        keep, got_imp = SEL.select_topk(s, n, 0, 0, k)
        np.testing.assert_array_equal(got_imp, imp)
        # the kept set is the size-k subset of largest total importance (distinct values here)
        best = max(itertools.combinations(range(nb), k), key=lambda c: imp[list(c)].sum())
        assert sorted(np.nonzero(keep)[0].tolist()) == sorted(best)


def test_invariances_and_monotonicity():
    rng = np.random.default_rng(7)
    G, n = 4, 1000
    s = rng.standard_normal((G, n)) * 3
    shift = rng.standard_normal((G, 1)) * 10
    for p in (0.2, 0.5, 0.9):
        a = SEL.select_topp(s, n, 64, 128, p)[0]
        b = SEL.select_topp(s + shift, n, 64, 128, p)[0]  # softmax ignores a per-head shift
        assert np.array_equal(a, b)
    prev = None
    for p in (0.1, 0.3, 0.6, 0.9, 1.0):
        cur = SEL.select_topp(s, n, 64, 128, p)[0]
        if prev is not None:
            assert np.all(cur >= prev)
        prev = cur
    assert prev.all()  # p = 1 keeps every block
    prev = None
    for k in range(0, 17, 3):
        cur = SEL.select_topk(s, n, 64, 128, k)[0]
        assert np.array_equal(cur, SEL.select_topk(s + 5.0, n, 64, 128, k)[0])
        if prev is not None:
            assert np.all(cur >= prev)
        prev = cur
