"""Seeded random work lists through the host planner (host-only plans, no GPU): every
plan passes the bounds dry run; forward tiles cover each (item, head, query row) and
backward tiles each (item, head, KV row) exactly once, longest first; the output, LSE,
gradient and partial blocks of all items are disjoint and inside their arenas; with
ordered dQ each head's KV tiles are listed in order.  Lists whose k chunks overlap in a
group are rejected."""
import numpy as np
import pytest

from coalesced_packed_attention_gb300 import zl
from coalesced_packed_attention_gb300.workloads import WorkItem, merge_groups
from tests._lib import ensure_library

FLAG_SETS = [0, zl.ZL_PLAN_DETERMINISTIC_DQ, zl.ZL_PLAN_FUSE_LOCAL_KMERGE,
             zl.ZL_PLAN_FUSE_LOCAL_KMERGE | zl.ZL_PLAN_DETERMINISTIC_DQ]


@pytest.fixture(scope="module", autouse=True)
def lib():
    return ensure_library()


def cuts(rng, n, k):
    """k contiguous half-open ranges tiling [0, n) (some may be empty)."""
    pts = np.sort(rng.integers(0, n + 1, size=k - 1)).tolist()
    edges = [0] + pts + [n]
    return list(zip(edges[:-1], edges[1:]))


def random_list(seed):
    rng = np.random.default_rng(seed)
    H = int(rng.integers(1, 7))
    d = int(rng.choice([64, 128]))
    lens = rng.integers(1, 700, size=int(rng.integers(1, 6))).tolist()
    offs = np.concatenate([[0], np.cumsum(lens)[:-1]]).tolist()
    T = int(sum(lens))
    items = []
    for s, L in zip(offs, lens):
        kind = rng.integers(0, 5)
        if kind == 0:    # whole sequence
            items.append(WorkItem(s, L, 0, L, 0, H, 0, L, 0))
        elif kind == 1:  # q-split shards, all heads, full KV
            for (a, b) in cuts(rng, L, int(rng.integers(1, 4))):
                items.append(WorkItem(s, L, a, b, 0, H, 0, L, 0))
        elif kind == 2:  # h-split shards
            for (a, b) in cuts(rng, H, int(rng.integers(1, 3))):
                items.append(WorkItem(s, L, 0, L, a, b, 0, L, 0))
        elif kind == 3:  # a k-split group over a row/head block, chunks tiling a KV range
            q0, q1 = sorted(rng.integers(0, L + 1, size=2).tolist())
            h0, h1 = sorted(rng.integers(0, H + 1, size=2).tolist())
            for (a, b) in cuts(rng, L, int(rng.integers(2, 5))):
                items.append(WorkItem(s, L, q0, q1, h0, h1, a, b, 1))
        else:            # a k-split group with a gap between its chunks, plus a random shard
            m = int(rng.integers(0, L + 1))
            items.append(WorkItem(s, L, 0, L, 0, H, 0, m // 2, 1))
            items.append(WorkItem(s, L, 0, L, 0, H, m, L, 1))
            q0, q1 = sorted(rng.integers(0, L + 1, size=2).tolist())
            k0, k1 = sorted(rng.integers(0, L + 1, size=2).tolist())
            items.append(WorkItem(s, L, q0, q1, 0, H, k0, k1, 0))
    return H, d, T, items


def check_plan(H, d, T, items, flags):
    p = zl.zl_plan_worklist(items, H, d, T, flags=zl.ZL_PLAN_HOST_ONLY | flags)
    p.check_bounds()
    assert p.n_items == len(items)
    fused = bool(flags & zl.ZL_PLAN_FUSE_LOCAL_KMERGE)
    # backward tiles: every (user item, head, KV block) once, longest first
    bt = p.tiles(1)
    assert [t[3] for t in bt] == sorted((t[3] for t in bt), reverse=True)
    want = {(i, h, b) for i, it in enumerate(items) for h in range(it.h_lo, it.h_hi)
            for b in range(-(-it.nkv // 128))}
    got = [(i, h, b) for (i, h, b, _) in bt]
    assert len(got) == len(set(got)) and set(got) == want
    if flags & zl.ZL_PLAN_DETERMINISTIC_DQ:
        nxt = {}
        for (i, h, b) in got:
            assert nxt.get((i, h), 0) == b
            nxt[(i, h)] = b + 1
    # forward tiles: every (item, head, query block) once when nothing is fused
    ft = p.tiles(0)
    assert [t[3] for t in ft] == sorted((t[3] for t in ft), reverse=True)
    if not fused:
        fb = 256
        want = {(i, h, b) for i, it in enumerate(items) for h in range(it.h_lo, it.h_hi)
                for b in range(-(-it.nq // fb))}
        got = [(i, h, b) for (i, h, b, _) in ft]
        assert len(got) == len(set(got)) and set(got) == want
    # blocks of every arena are disjoint and inside it
    blocks = {"o": [], "op": [], "lse": [], "dq": [], "dkv": []}
    for i, it in enumerate(items):
        pl = p.item(i)
        n = it.nq * it.nh
        if pl.item.out_offset >= 0:
            blocks["op" if it.emit_lse else "o"].append((pl.item.out_offset, pl.item.out_offset + n * d))
            blocks["lse"].append((pl.item.lse_offset, pl.item.lse_offset + n))
        blocks["dq"].append((pl.dq_offset, pl.dq_offset + n * d))
        blocks["dkv"].append((pl.dkv_offset, pl.dkv_offset + it.nkv * it.nh * d))
    assert [p.group(g)[0] for g in range(p.n_groups)] == merge_groups(items)
    for g in range(p.n_groups):
        members, oo, lo = p.group(g)
        it = items[members[0]]
        blocks["o"].append((oo, oo + it.nq * it.nh * d))
        blocks["lse"].append((lo, lo + it.nq * it.nh))
    totals = {"o": p.o_elems, "op": p.o_partial_elems, "lse": p.lse_elems, "dq": p.dq_elems, "dkv": p.dkv_elems}
    for key, bl in blocks.items():
        bl = sorted(b for b in bl if b[1] > b[0])
        for a, b in zip(bl, bl[1:]):
            assert a[1] <= b[0], (key, a, b)
        assert all(b[0] >= 0 and b[1] <= totals[key] for b in bl), key


@pytest.mark.parametrize("flags", FLAG_SETS)
def test_random_lists_plan_soundly(flags):
    for seed in range(150):
        H, d, T, items = random_list(seed)
        check_plan(H, d, T, items, flags)


def test_overlapping_chunks_in_a_group_are_rejected():
    rng = np.random.default_rng(99)
    for _ in range(50):
        L = int(rng.integers(4, 500))
        a = int(rng.integers(1, L - 1))
        b = int(rng.integers(0, a))  # second chunk starts inside the first
        items = [WorkItem(0, L, 0, L, 0, 2, 0, a, 1), WorkItem(0, L, 0, L, 0, 2, b, L, 1)]
        with pytest.raises(zl.ZlError):
            zl.zl_plan_worklist(items, 2, 64, L, flags=zl.ZL_PLAN_HOST_ONLY)
