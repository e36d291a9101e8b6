"""Pins of the placement oracle (catalog cut, filler packing) against facts that do not
come from the oracle itself: a hand-worked cut, Fisher's result that the best 2-group
split of ordered data is contiguous (checked against every subset split), invariances,
exact small cases, and Graham's bound for longest-first list scheduling checked
against brute-force optima."""
import itertools
import math
import random

import pytest

from oracle import placement as P


def test_cut_worked_example():
    # x = ln T = 0, 1, 4 (one sequence each): {0} | {1, 4} -> 4.5; {0, 1} | {4} -> 0.5
    k, d = P.catalog_cut([1.0, math.e, math.e ** 4], [1, 1, 1])
    assert k == 2 and abs(d - 0.5) < 1e-12
    assert abs(P.dispersion([1.0, math.e, math.e ** 4], [1, 1, 1], 1) - 4.5) < 1e-12


def test_cut_two_clusters_has_zero_dispersion_at_the_gap():
    times = [2.0, 2.0, 2.0, 900.0, 900.0]
    k, d = P.catalog_cut(times, [5, 1, 3, 2, 7])
    assert k == 3 and d <= 1e-20   # zero up to rounding of the means


@pytest.mark.parametrize("seed", range(6))
def test_cut_is_the_best_of_all_two_set_splits(seed):
    # Fisher (1958): for one-dimensional data the least-squares two-group partition is
    # contiguous in sorted order, so the best contiguous cut is the best of all splits
    rng = random.Random(seed)
    n = rng.randint(2, 8)
    times = sorted(math.exp(rng.uniform(-3, 8)) for _ in range(n))
    counts = [rng.randint(1, 5) for _ in range(n)]
    k, d = P.catalog_cut(times, counts)
    best = math.inf
    for mask in range(1, 2 ** n - 1):
        A = [b for b in range(n) if mask >> b & 1]
        B = [b for b in range(n) if not mask >> b & 1]
        tot = 0.0
        for idx in (A, B):
            m = sum(counts[b] * math.log(times[b]) for b in idx) / sum(counts[b] for b in idx)
            tot += sum(counts[b] * (math.log(times[b]) - m) ** 2 for b in idx)
        best = min(best, tot)
    assert abs(d - best) <= 1e-9 * max(1.0, best)


def test_cut_invariances():
    times, counts = [1.0, 3.0, 4.0, 50.0, 70.0, 2000.0], [9, 4, 4, 2, 2, 1]
    k, d = P.catalog_cut(times, counts)
    k2, d2 = P.catalog_cut([7.5 * t for t in times], counts)   # ln shift
    k3, d3 = P.catalog_cut(times, [2 * c for c in counts])     # every sequence twice
    assert k == k2 == k3 and abs(d - d2) < 1e-9 and abs(d3 - 2 * d) < 1e-9
    assert P.catalog_cut([5.0], [3]) == (1, 0.0)


def test_pack_single_rank_and_one_each():
    a, L, M, over, mk = P.pack_fillers([3.0, 1.0, 2.0], [1.0, 1.0, 1.0], 1, M_cap=10.0)
    assert a == [0, 0, 0] and mk == 6.0 and over == 0
    # equal fillers on empty ranks: each goes to the lowest of the equally open ranks
    a, L, M, over, mk = P.pack_fillers([2.0] * 4, [0.5] * 4, 4, M_cap=1.0)
    assert a == [0, 1, 2, 3] and L == [2.0] * 4 and over == 0


def test_pack_places_longest_first():
    # 1, 1, 1, 1, 4 on two ranks: longest first puts the 4 alone and reaches the optimum
    # 4; shortest first would end at 6
    a, L, M, over, mk = P.pack_fillers([1.0, 1.0, 1.0, 1.0, 4.0], [0.0] * 5, 2, M_cap=1.0)
    assert mk == 4.0 and a[4] == 0 and a[:4] == [1, 1, 1, 1]


def test_pack_memory_binds():
    # four equal fillers, two ranks, memory for two fillers per rank, time for all:
    # memory is the bottleneck, so they alternate
    a, L, M, over, mk = P.pack_fillers([1.0] * 4, [5.0] * 4, 2, F=100.0, M_cap=10.0)
    assert sorted(a) == [0, 0, 1, 1] and M == [10.0, 10.0] and over == 0
    # a fifth does not fit anywhere: placed and counted
    a, L, M, over, mk = P.pack_fillers([1.0] * 5, [5.0] * 5, 2, F=100.0, M_cap=10.0)
    assert over == 1


def test_pack_fills_the_lightest_anchor_rank_first():
    a, L, M, over, mk = P.pack_fillers([1.0], [0.0], 3, rank_time=[5.0, 2.0, 4.0], M_cap=1.0)
    assert a == [1] and L == [5.0, 3.0, 4.0]


@pytest.mark.parametrize("seed", range(8))
def test_pack_within_grahams_bound(seed):
    # with memory slack everywhere the score orders ranks by time slack, so the greedy is
    # longest-processing-time-first list scheduling: makespan <= (4/3 - 1/(3N)) OPT
    rng = random.Random(100 + seed)
    N = rng.choice([2, 3])
    n = rng.randint(N + 1, 7)
    t = [rng.randint(1, 20) * 1.0 for _ in range(n)]
    a, L, M, over, mk = P.pack_fillers(t, [0.0] * n, N, M_cap=1.0)
    opt = min(max(sum(t[s] for s in range(n) if asg[s] == r) for r in range(N))
              for asg in itertools.product(range(N), repeat=n))
    assert mk <= (4.0 / 3.0 - 1.0 / (3 * N)) * opt + 1e-9
    assert abs(sum(L) - sum(t)) < 1e-9 and all(x in range(N) for x in a)
