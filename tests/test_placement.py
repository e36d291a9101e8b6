"""The host placement slice (zl_catalog_cut, zl_pack_fillers in the C++ library) against
the oracle on seeded synthetic catalogs, its argument checks, and per-rank work lists
that the engine's planner accepts and that cover every sequence once."""
import math
import random

import pytest

import oracle.placement as P
from coalesced_packed_attention_gb300 import zl
from coalesced_packed_attention_gb300.placement import plan_ranks
from coalesced_packed_attention_gb300.workloads import WorkItem
from tests._lib import ensure_library


@pytest.fixture(scope="module", autouse=True)
def lib():
    return ensure_library()


def random_catalog(rng, n):
    times = sorted(math.exp(rng.uniform(-2, 9)) for _ in range(n))
    return [(256 * (b + 1), rng.randint(1, 40), t, rng.uniform(0.1, 4.0)) for b, t in enumerate(times)]


@pytest.mark.parametrize("seed", range(20))
def test_cut_matches_oracle(seed):
    rng = random.Random(seed)
    cat = random_catalog(rng, rng.randint(1, 30))
    k, d = zl.catalog_cut(cat)
    k_ref, d_ref = P.catalog_cut([b[2] for b in cat], [b[1] for b in cat])
    assert k == k_ref
    assert abs(d - d_ref) <= 1e-9 * max(1.0, d_ref)


@pytest.mark.parametrize("seed", range(20))
def test_pack_matches_oracle(seed):
    rng = random.Random(1000 + seed)
    n, N = rng.randint(0, 300), rng.randint(1, 16)
    t = [rng.choice([1.0, 2.0, 3.5, 8.0]) * rng.randint(1, 5) for _ in range(n)]  # ties on purpose
    m = [rng.uniform(0.0, 2.0) for _ in range(n)]
    rt = [rng.uniform(0.0, 50.0) for _ in range(N)] if seed % 2 else None
    rm = [rng.uniform(0.0, 20.0) for _ in range(N)] if seed % 2 else None
    F = 0.0 if seed % 3 else rng.uniform(10.0, 200.0)
    M_cap = rng.uniform(10.0, 100.0)
    got = zl.pack_fillers(t, m, N, rt, rm, F, M_cap)
    ref = P.pack_fillers(t, m, N, rt, rm, F, M_cap)
    assert got[0] == ref[0]                      # the same rank for every filler
    assert got[3] == ref[3]                      # overflow count
    for a, b in zip(got[1] + got[2] + [got[4]], ref[1] + ref[2] + [ref[4]]):
        assert abs(a - b) <= 1e-12 * max(1.0, abs(b))


def test_placement_argument_checks():
    with pytest.raises(zl.ZlError):
        zl.catalog_cut([(256, 1, 2.0, 0.0), (512, 1, 1.0, 0.0)])     # not sorted
    with pytest.raises(zl.ZlError):
        zl.catalog_cut([(256, 0, 2.0, 0.0)])                       # empty bucket
    with pytest.raises(zl.ZlError):
        zl.catalog_cut([(256, 1, 0.0, 0.0)])                       # non-positive time
    with pytest.raises(zl.ZlError):
        zl.pack_fillers([1.0], [1.0], 0)                           # no ranks
    with pytest.raises(zl.ZlError):
        zl.pack_fillers([-1.0], [1.0], 2)                          # negative time
    with pytest.raises(zl.ZlError):
        zl.pack_fillers([1.0], [1.0], 2, M_cap=0.0)                # no memory
    assert zl.pack_fillers([], [], 3)[0] == []


def test_rank_work_lists_cover_the_batch_and_plan():
    # a mixed batch: 48 x 256 + 12 x 1024 + 4 x 4096 images, two 32760-token videos;
    # time ~ L^2 (attention), memory ~ L; 8 ranks
    H, d, R = 24, 128, 8
    lengths = [256] * 48 + [1024] * 12 + [4096] * 4 + [32760] * 2
    seqs, off = [], 0
    for L in lengths:
        seqs.append((off, L))
        off += L
    T = off
    time_of = lambda L: 3.5 * 4.0 * L * L * d * H / 1e15  # noqa: E731
    mem_of = lambda L: 10.0 * L * H * d * 2 / 1e9          # noqa: E731
    plan = plan_ranks(seqs, H, R, time_of=time_of, mem_of=mem_of, M_cap=80.0)
    # the anchors are the buckets at and above the oracle's cut of the same catalog
    distinct = sorted(set(lengths))
    k_ref, _ = P.catalog_cut([time_of(L) for L in distinct], [lengths.count(L) for L in distinct])
    assert plan.k_star == k_ref and plan.anchor_lengths == distinct[k_ref:]
    covered = {}
    for r, items in enumerate(plan.work):
        p = zl.zl_plan_worklist(items, H, d, T, flags=zl.ZL_PLAN_HOST_ONLY)
        p.check_bounds()
        for it in items:
            for h in range(it.h_lo, it.h_hi):
                key = (it.seq_offset, h)
                covered.setdefault(key, []).append((it.q_lo, it.q_hi))
            assert it.kv_lo == 0 and it.kv_hi == it.seq_len
    for (o, L) in seqs:
        for h in range(H):
            spans = sorted(covered[(o, h)])
            assert spans[0][0] == 0 and spans[-1][1] == L
            assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))   # rows tiled exactly once
    assert plan.n_overflow == 0
    # the fillers balance the ranks: within one largest filler of each other
    biggest = max(time_of(L) for L in distinct[:k_ref])
    assert max(plan.rank_time) - min(plan.rank_time) <= biggest + 1e-9
