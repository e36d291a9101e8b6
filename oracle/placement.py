"""Plain Python oracle of the host placement slice (catalog cut, filler packing).

TEST INFRASTRUCTURE ONLY.  Only tests/ may import this module.  It shares no code with the C++ slice and imports nothing from the package.

What it computes (method: "Zellige: Moldable Sequence Placement for Mixed Image-Video
DiT Training"; the pages name both rules without printing them):
  * Catalog cut (pith.science review, "Free parameters", and its ref. [28], Fisher's
    grouping: the cut is the split under which the log run times of whole sequences
    vary least inside each set).  Reading: buckets sorted by whole-sequence time T; every sequence is one
    observation x = ln T; the dispersion of a cut is the sum over the two sets of the
    squared deviations from each set's mean; the set below the cut holds the fillers.
  * Filler Packing (pith.science review, referee report on Eq. (8), and "What carries
    the argument": whole fillers are placed one by one, scored by their tighter
    resource, compute headroom normalised by F or memory headroom by M_cap).  Reading: fillers in
    decreasing time, each to the rank whose smaller normalised slack after taking it is
    largest; F defaults to the makespan lower bound.
Ties: smallest cut; earlier filler first; lowest rank.
"""
from __future__ import annotations

import math


def dispersion(times, counts, k):
    """Within-set dispersion of ln T for the cut after the k-th bucket (k in 1..n-1):
    every sequence counted once, each set measured against its own mean."""
    def ssd(idx):
        n = sum(counts[b] for b in idx)
        if n == 0:
            return 0.0
        mean = sum(counts[b] * math.log(times[b]) for b in idx) / n
        return sum(counts[b] * (math.log(times[b]) - mean) ** 2 for b in idx)
    return ssd(range(0, k)) + ssd(range(k, len(times)))


def catalog_cut(times, counts):
    """(k*, D(k*)) for buckets sorted by time: buckets [0, k*) are fillers."""
    assert all(t > 0 for t in times) and all(c >= 1 for c in counts)
    assert all(a <= b for a, b in zip(times, times[1:])), "buckets must be sorted by time"
    n = len(times)
    if n == 1:
        return 1, 0.0
    best_k, best_d = 1, dispersion(times, counts, 1)
    for k in range(2, n):
        d = dispersion(times, counts, k)
        if d < best_d:
            best_k, best_d = k, d
    return best_k, best_d


def pack_fillers(filler_time, filler_mem, n_ranks, rank_time=None, rank_mem=None, F=0.0, M_cap=1.0):
    """Greedy placement of whole fillers: (assign, final_time, final_mem, n_overflow,
    makespan).  rank_time / rank_mem: the anchors' load per rank (default zeros)."""
    L = [float(x) for x in rank_time] if rank_time is not None else [0.0] * n_ranks
    M = [float(x) for x in rank_mem] if rank_mem is not None else [0.0] * n_ranks
    if F <= 0:
        total = 0.0
        for x in L:
            total += x
        for t in filler_time:
            total += t
        F = max(max(L), total / n_ranks)
        if not F > 0:
            F = 1.0
    order = sorted(range(len(filler_time)), key=lambda s: (-filler_time[s], s))
    assign = [None] * len(filler_time)
    overflow = 0
    for s in order:
        t, m = filler_time[s], filler_mem[s]
        scores = [min((F - L[r] - t) / F, (M_cap - M[r] - m) / M_cap) for r in range(n_ranks)]
        best = max(range(n_ranks), key=lambda r: (scores[r], -r))
        if scores[best] < -1e-9:   # negative beyond the rounding of an exact fit
            overflow += 1
        assign[s] = best
        L[best] += t
        M[best] += m
    return assign, L, M, overflow, max(L)
