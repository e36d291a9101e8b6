"""The placement oracle's pins catch planted mistakes: a cut that ignores bucket counts
or measures raw times instead of log times; a packing that scores by the looser instead
of the tighter resource, places fillers shortest first, or breaks ties toward the
highest rank.  Each mistake is planted in the oracle on the CPU (wrapping it, or, for
the packing loop, a copy whose only change is the planted one, itself pinned to the
oracle with nothing planted), and every pin named for it must fail."""
import random

import pytest

from oracle import placement as P
from tests import test_oracle_placement as pins

CUT, PACK = P.catalog_cut, P.pack_fillers


def cut_unweighted(times, counts):
    return CUT(times, [1] * len(times))


def dispersion_raw_times(times, counts, k):
    # the oracle's within-set dispersion with the log dropped (x = T instead of ln T)
    def ssd(idx):
        n = sum(counts[b] for b in idx)
        mean = sum(counts[b] * times[b] for b in idx) / n
        return sum(counts[b] * (times[b] - mean) ** 2 for b in idx)
    return ssd(range(0, k)) + ssd(range(k, len(times)))


def pack_copy(filler_time, filler_mem, n_ranks, rank_time=None, rank_mem=None, F=0.0, M_cap=1.0,
              combine=min, shortest_first=False, ties_high=False):
    """The oracle's greedy packing with switches for the planted mistakes (all off: the
    oracle's own rules)."""
    L = [float(x) for x in rank_time] if rank_time is not None else [0.0] * n_ranks
    M = [float(x) for x in rank_mem] if rank_mem is not None else [0.0] * n_ranks
    if F <= 0:
        F = max(max(L), (sum(L) + sum(filler_time)) / n_ranks)
        if not F > 0:
            F = 1.0
    sign = 1 if shortest_first else -1
    order = sorted(range(len(filler_time)), key=lambda s: (sign * filler_time[s], s))
    assign, over = [None] * len(filler_time), 0
    for s in order:
        t, m = filler_time[s], filler_mem[s]
        sc = [combine((F - L[r] - t) / F, (M_cap - M[r] - m) / M_cap) for r in range(n_ranks)]
        best = max(range(n_ranks), key=lambda r: (sc[r], r if ties_high else -r))
        if sc[best] < -1e-9:
            over += 1
        assign[s] = best
        L[best] += t
        M[best] += m
    return assign, L, M, over, max(L)


def pack_looser(*a, **k):
    return pack_copy(*a, combine=max, **k)


def pack_shortest_first(*a, **k):
    return pack_copy(*a, shortest_first=True, **k)


def pack_ties_high(*a, **k):
    return pack_copy(*a, ties_high=True, **k)


CASES = {
    "cut ignores bucket counts": ("catalog_cut", cut_unweighted, [
        (pins.test_cut_is_the_best_of_all_two_set_splits, 0), (pins.test_cut_invariances,)]),
    "cut on raw times": ("dispersion", dispersion_raw_times, [
        (pins.test_cut_worked_example,), (pins.test_cut_invariances,)]),
    "packing scores the looser resource": ("pack_fillers", pack_looser, [(pins.test_pack_memory_binds,)]),
    "packing shortest first": ("pack_fillers", pack_shortest_first, [(pins.test_pack_places_longest_first,)]),
    "packing ties to the highest rank": ("pack_fillers", pack_ties_high, [
        (pins.test_pack_single_rank_and_one_each,)]),
}


def _fails(pin, args):
    try:
        pin(*args)
    except AssertionError:
        return True
    return False


@pytest.mark.parametrize("name", list(CASES))
def test_pins_catch_planted_mistake(name, monkeypatch):
    attr, mutant, catchers = CASES[name]
    monkeypatch.setattr(P, attr, mutant)
    caught = [_fails(pin, args) for pin, *args in catchers]
    assert all(caught), caught


def test_packing_copy_is_the_oracle_with_nothing_planted():
    rng = random.Random(7)
    for _ in range(200):
        n, N = rng.randint(0, 9), rng.randint(1, 4)
        t = [rng.choice([1.0, 2.0, 3.0, rng.uniform(0.1, 9.0)]) for _ in range(n)]
        m = [rng.choice([0.0, 1.0, rng.uniform(0.0, 3.0)]) for _ in range(n)]
        rt = [rng.uniform(0, 5) for _ in range(N)] if rng.random() < 0.5 else None
        rm = [rng.uniform(0, 2) for _ in range(N)] if rng.random() < 0.5 else None
        F = rng.choice([0.0, 6.0])
        assert pack_copy(t, m, N, rt, rm, F, 4.0) == PACK(t, m, N, rt, rm, F, 4.0)


def test_pins_pass_on_the_oracle_itself():
    for _, _, catchers in CASES.values():
        for pin, *args in catchers:
            pin(*args)
