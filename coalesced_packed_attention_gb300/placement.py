"""Per-rank work lists from a batch of sequences (host planning slice, no GPU).

The pages' planner ("Zellige", pith.science review, "What carries the argument") cuts
the batch's bucket catalog into anchors and fillers, places the anchors as theta=(q,h,k)
shards, and packs whole fillers into each rank's remaining time and memory.  The cut
and the packing run in the library (zl_catalog_cut, zl_pack_fillers); the anchors' own
placement (an exact CP-SAT model in the pages) is outside it, and this module stands in
for it with the plainest placement: every anchor sequence q-split evenly over all ranks
(each rank takes a contiguous block of its query rows, all heads, the whole KV range).
The result is one engine work list per rank, ready for zl_plan_worklist.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Callable, Dict, List, Sequence, Tuple

from . import zl
from .workloads import WorkItem


@dataclass
class RankPlan:
    k_star: int                      # buckets [0, k_star) are fillers
    anchor_lengths: List[int]        # sequence lengths of the anchor buckets
    assign: List[int]                # rank of each filler sequence (in filler order)
    rank_time: List[float]           # per-rank time after placement
    rank_mem: List[float]
    n_overflow: int
    makespan: float
    work: List[List[WorkItem]]       # engine work list per rank


def bucket_catalog(lengths: Sequence[int], time_of: Callable[[int], float],
                   mem_of: Callable[[int], float]) -> List[Tuple[int, int, float, float]]:
    """(seq_len, count, time, mem) per distinct length, sorted by time then length."""
    counts: Dict[int, int] = {}
    for L in lengths:
        counts[L] = counts.get(L, 0) + 1
    cat = [(L, n, float(time_of(L)), float(mem_of(L))) for L, n in counts.items()]
    return sorted(cat, key=lambda b: (b[2], b[0]))


def plan_ranks(seqs: Sequence[Tuple[int, int]], n_heads: int, n_ranks: int,
               time_of: Callable[[int], float], mem_of: Callable[[int], float],
               M_cap: float, F: float = 0.0) -> RankPlan:
    """seqs: (seq_offset, seq_len) of every sequence in the packed batch.  Anchors (the
    buckets at and above the cut) are q-split over all ranks; fillers are packed whole."""
    cat = bucket_catalog([L for _, L in seqs], time_of, mem_of)
    k_star, _ = zl.catalog_cut(cat)
    filler_lengths = {b[0] for b in cat[:k_star]}
    anchors = [(o, L) for (o, L) in seqs if L not in filler_lengths]
    fillers = [(o, L) for (o, L) in seqs if L in filler_lengths]
    work: List[List[WorkItem]] = [[] for _ in range(n_ranks)]
    rank_time = [0.0] * n_ranks
    rank_mem = [0.0] * n_ranks
    for (o, L) in anchors:
        t, m = time_of(L), mem_of(L)
        for r in range(n_ranks):
            q_lo, q_hi = (L * r) // n_ranks, (L * (r + 1)) // n_ranks
            if q_hi > q_lo:
                work[r].append(WorkItem(o, L, q_lo, q_hi, 0, n_heads, 0, L, 0))
            share = (q_hi - q_lo) / L
            rank_time[r] += t * share
            rank_mem[r] += m * share
    ft = [time_of(L) for _, L in fillers]
    fm = [mem_of(L) for _, L in fillers]
    assign, final_t, final_m, over, mk = zl.pack_fillers(ft, fm, n_ranks, rank_time, rank_mem, F, M_cap)
    for (o, L), r in zip(fillers, assign):
        work[r].append(WorkItem(o, L, 0, L, 0, n_heads, 0, L, 0))
    return RankPlan(k_star, sorted({L for _, L in anchors}), assign, final_t, final_m, over, mk, work)
