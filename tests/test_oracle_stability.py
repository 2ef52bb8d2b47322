"""Pins of the oracle's temporal-stability functions (RCO, window mean, classification).

FlexiCache blog summary (MLSys'26), "Core insight: attention heads differ in
temporal stability": top-K sets of a head are compared a few steps apart with
the Random-Corrected Overlap, 1 for identical sets and 0 for the overlap that
random sets would have; it is aggregated over a window, and the least stable
quarter of the heads is unstable.  The formula is not printed; the reading is
RCO = (|A n B| - |A||B|/P) / (min(|A|,|B|) - |A||B|/P).

The pins check what fixes the reading without retyping it: identical sets give
1; a subset gives 1 (the largest possible overlap); the mean over ALL pairs of
subsets, enumerated exhaustively, is exactly 0 (chance overlap), also for
unequal sizes and for a page count that grew between the steps; more overlap
means a higher value; the window mean follows the pairs' order; the
classification takes the lowest round(frac * n) with ties to the lower index.
"""
import itertools

import numpy as np
import pytest





def test_identical_sets_score_one(oracle_mod):
    rng = np.random.default_rng(1)
    for P, K in [(10, 3), (64, 8), (2048, 128), (5, 4)]:
        a = np.sort(rng.choice(P, K, replace=False))
        assert oracle_mod.rco(a, a, P) == 1.0
        assert oracle_mod.rco(a, a, P + 7) == 1.0  # also after the sequence grew


def test_a_subset_reaches_the_largest_possible_overlap(oracle_mod):
    assert oracle_mod.rco([2, 5], [1, 2, 5, 9], 20) == 1.0
    assert oracle_mod.rco([1, 2, 5, 9], [5, 2], 20) == 1.0


def test_every_page_selected_scores_one(oracle_mod):
    assert oracle_mod.rco(list(range(6)), list(range(6)), 6) == 1.0
    assert oracle_mod.rco([], [], 0) == 1.0


def test_mean_over_all_subset_pairs_is_zero(oracle_mod):
    # chance overlap: the exhaustive mean of RCO over every pair of subsets of these sizes is 0
    for P, ka, kb in [(7, 3, 3), (6, 2, 2), (8, 2, 5), (9, 4, 1)]:
        vals = [oracle_mod.rco(a, b, P) for a in itertools.combinations(range(P), ka)
                for b in itertools.combinations(range(P), kb)]
        assert abs(np.mean(vals)) < 1e-12
        assert min(vals) < 0 < max(vals) <= 1.0


def test_chance_uses_the_larger_page_count_when_the_sequence_grew(oracle_mod):
    # A from the first Pa pages, B from Pb > Pa pages: exhaustive mean 0 with P = Pb
    Pa, Pb, k = 5, 8, 2
    vals = [oracle_mod.rco(a, b, Pb) for a in itertools.combinations(range(Pa), k)
            for b in itertools.combinations(range(Pb), k)]
    assert abs(np.mean(vals)) < 1e-12


def test_more_overlap_scores_higher(oracle_mod):
    P, a = 50, [0, 1, 2, 3, 4, 5, 6, 7]
    prev = -np.inf
    for shared in range(0, 9):
        b = list(range(shared)) + list(range(40, 40 + 8 - shared))
        v = oracle_mod.rco(a, b, P)
        assert v > prev
        prev = v
    assert prev == 1.0


def test_window_mean_takes_pairs_lag_apart_newest_first(oracle_mod):
    # three steps newest first; lag 1 pairs (0,1) and (1,2); lag 2 pair (0,2)
    idx = np.array([[1, 2, 3, 0], [1, 2, 9, 0], [5, 6, 7, 8]], dtype=np.int32)
    cnt = np.array([3, 3, 4], dtype=np.int32)
    pages = np.array([12, 12, 10], dtype=np.int32)
    want1 = (oracle_mod.rco([1, 2, 3], [1, 2, 9], 12) + oracle_mod.rco([1, 2, 9], [5, 6, 7, 8], 12)) / 2
    assert oracle_mod.unit_stability(idx, cnt, pages, 1) == pytest.approx(want1, abs=0, rel=1e-15)
    assert oracle_mod.unit_stability(idx, cnt, pages, 2) == oracle_mod.rco([1, 2, 3], [5, 6, 7, 8], 12)
    # two identical steps: 1
    assert oracle_mod.unit_stability(idx[:1].repeat(2, 0), cnt[:1].repeat(2), pages[:1].repeat(2), 1) == 1.0
    # disjoint sets of 3 among 12: the overlap 0 lies below chance (9/12)
    assert oracle_mod.rco([1, 2, 3], [7, 8, 9], 12) < 0


def test_classification_takes_the_lowest_with_ties_to_the_lower_index(oracle_mod):
    s = [0.5, 0.1, 0.1, 0.9]
    assert oracle_mod.classify(s, 0.5).tolist() == [0, 1, 1, 0]
    assert oracle_mod.classify(s, 0.25).tolist() == [0, 1, 0, 0]
    assert oracle_mod.classify(s, 0.375).tolist() == [0, 1, 1, 0]  # 1.5 rounds up to 2
    assert oracle_mod.classify(s, 0.0).tolist() == [0, 0, 0, 0]
    assert oracle_mod.classify(s, 1.0).tolist() == [1, 1, 1, 1]
    rng = np.random.default_rng(3)
    v = rng.random(256)
    m = oracle_mod.classify(v, 0.25)
    assert m.sum() == 64 and v[m == 1].max() < v[m == 0].min()
