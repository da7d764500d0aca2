"""Pins of the oracle's top-k selection (the indexer's topk step of "[Feat]
[NVIDIA] DeepSeek-V4.1: Prefill support CP with multistream forward prepare
(4/N)"; the pages give no tie rule, so ties go to the smaller column): brute
force over all k-subsets on tiny rows, ties to the smaller column, the
signed-zero order, short rows, and the result being a valid top-k."""
import itertools

import numpy as np

from oracle import oracle as orc


def test_brute_force_over_all_subsets():
    rng = np.random.default_rng(0)
    for trial in range(30):
        n = int(rng.integers(1, 9))
        k = int(rng.integers(1, 6))
        x = rng.integers(-3, 4, n).astype(np.float32)  # many ties
        got = orc.topk_select(x[None, :], [n], k)[0]
        if n <= k:
            assert list(got[:n]) == list(range(n)) and (got[n:] == -1).all()
            continue
        # the best subset: largest values, then the smallest columns among ties
        best = max(itertools.combinations(range(n), k),
                   key=lambda c: (sorted(x[list(c)], reverse=True), [-j for j in c]))
        assert list(got) == sorted(best), (x, k, got, best)


def test_ties_go_to_the_smaller_column():
    x = np.array([[1, 5, 5, 5, 2, 5]], np.float32)
    assert list(orc.topk_select(x, [6], 2)[0]) == [1, 2]
    assert list(orc.topk_select(x, [6], 5)[0]) == [1, 2, 3, 4, 5]
    # only the first row_len columns are candidates
    assert list(orc.topk_select(x, [4], 2)[0]) == [1, 2]


def test_signed_zero_order_and_negatives():
    x = np.array([[-0.0, 0.0, -1.0, -0.0, -2.0]], np.float32)
    # +0 above -0 above -1
    assert list(orc.topk_select(x, [5], 1)[0]) == [1]
    assert list(orc.topk_select(x, [5], 3)[0]) == [0, 1, 3]


def test_random_rows_are_valid_top_k():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((20, 3000)).astype(np.float32)
    lens = rng.integers(1, 3001, 20)
    k = 300
    got = orc.topk_select(x, lens, k)
    for i in range(20):
        n = int(lens[i])
        sel = got[i][got[i] >= 0]
        assert len(sel) == min(n, k) and (np.diff(sel) > 0).all() and sel.max() < n
        if n > k:
            rest = np.setdiff1d(np.arange(n), sel)
            assert x[i, sel].min() >= x[i, rest].max()
