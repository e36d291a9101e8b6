"""The C-ABI library loads and exports every entry point include/zl.h declares; the
host planner's validation, placement and tiling (host-only plans, no GPU)."""
import ctypes
import os
import re

import pytest

from coalesced_packed_attention_gb300 import zl
from coalesced_packed_attention_gb300.workloads import (WorkItem, config_images, config_long_video,
                                                        config_mixed, config_tiny, merge_groups)
from tests._lib import ensure_library

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def lib():
    return ensure_library()


def declared_functions():
    txt = open(os.path.join(ROOT, "include", "zl.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(zl_[a-z_0-9]+)\s*\(", txt)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert "zl_coalesced_attn_fwd" in names and "zl_merge_partials" in names
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(zl.exported_symbols()) == sorted(n for n in names if n in zl.exported_symbols())
    # every declared entry point has a Python binding, except the allocation-free
    # forward and its status query, whose callers (and its test) use the C ABI directly
    assert set(names) - {"zl_coalesced_attn_fwd_noalloc", "zl_noalloc_get_device_status"} <= set(zl.exported_symbols())


def test_status_strings(lib):
    for s in range(7):
        assert zl.status_string(s)
    assert zl.status_string(0) == "ok"
    assert lib.zl_version() >= 100


def host_plan(work):
    return zl.zl_plan_worklist(work.items, work.n_heads, work.head_dim, work.total_tokens,
                               flags=zl.ZL_PLAN_HOST_ONLY)


@pytest.mark.parametrize("bad", [
    WorkItem(0, 100, 0, 101, 0, 4, 0, 100),        # q range past the sequence
    WorkItem(0, 100, 5, 4, 0, 4, 0, 100),          # q_lo > q_hi
    WorkItem(0, 100, 0, 100, 0, 5, 0, 100),        # head outside [0, H)
    WorkItem(0, 100, 0, 100, 0, 4, -1, 100),       # negative kv_lo
    WorkItem(950, 100, 0, 100, 0, 4, 0, 100),      # sequence past T
    WorkItem(0, 100, 0, 100, 0, 4, 0, 100, 2),     # emit_lse not 0/1
])
def test_invalid_items_are_rejected(bad):
    with pytest.raises(zl.ZlError) as e:
        zl.zl_plan_worklist([bad], 4, 64, 1000, flags=zl.ZL_PLAN_HOST_ONLY)
    assert e.value.status == zl.ZL_ERR_INVALID_ARG


@pytest.mark.parametrize("flags", [4, 32, 1 << 31])
def test_unknown_plan_flags_are_rejected(flags):
    with pytest.raises(zl.ZlError) as e:
        zl.zl_plan_worklist([WorkItem(0, 100, 0, 100, 0, 4, 0, 100)], 4, 64, 1000, flags=zl.ZL_PLAN_HOST_ONLY | flags)
    assert e.value.status == zl.ZL_ERR_INVALID_ARG


def test_unsupported_head_dim_and_alignment():
    with pytest.raises(zl.ZlError) as e:
        zl.zl_plan_worklist([WorkItem(0, 10, 0, 10, 0, 1, 0, 10)], 1, 96, 10, flags=zl.ZL_PLAN_HOST_ONLY)
    assert e.value.status == zl.ZL_ERR_UNSUPPORTED
    with pytest.raises(zl.ZlError) as e:
        zl.zl_plan_worklist([WorkItem(0, 10, 0, 10, 0, 1, 0, 10, 0, out_offset=4)], 1, 64, 10,
                            flags=zl.ZL_PLAN_HOST_ONLY)
    assert e.value.status == zl.ZL_ERR_ALIGN


def test_overlapping_k_chunks_are_rejected():
    items = [WorkItem(0, 100, 0, 100, 0, 2, 0, 60, 1), WorkItem(0, 100, 0, 100, 0, 2, 50, 100, 1)]
    with pytest.raises(zl.ZlError):
        zl.zl_plan_worklist(items, 2, 64, 100, flags=zl.ZL_PLAN_HOST_ONLY)


@pytest.mark.parametrize("make", [config_tiny, config_images, config_mixed, config_long_video])
def test_tiles_cover_every_row_head_once_longest_first(make):
    w = make()
    p = host_plan(w)
    tiles = p.tiles(0)
    seen = {}
    for (i, h, b, cost) in tiles:
        it = w.items[i]
        assert it.h_lo <= h < it.h_hi
        assert 0 <= b * 256 < max(it.nq, 1)
        assert cost == -(-it.nkv // 128)
        key = (i, h, b)
        assert key not in seen
        seen[key] = 1
    expected = sum(it.nh * -(-it.nq // 256) for it in w.items)
    assert len(tiles) == expected == p.n_fwd_tiles
    costs = [t[3] for t in tiles]
    assert costs == sorted(costs, reverse=True)
    # stable: equal costs keep work-list order
    for a, b in zip(tiles, tiles[1:]):
        if a[3] == b[3]:
            assert (a[0], a[1], a[2]) < (b[0], b[1], b[2])
    btiles = p.tiles(1)
    assert len(btiles) == sum(it.nh * -(-it.nkv // 128) for it in w.items) == p.n_bwd_tiles


@pytest.mark.parametrize("make", [config_tiny, config_images, config_mixed, config_long_video])
def test_output_blocks_are_disjoint_and_whole_sequences_packed(make):
    w = make()
    p = host_plan(w)
    H, d, T = w.n_heads, w.head_dim, w.total_tokens
    o_blocks, op_blocks, l_blocks, dq_blocks, dkv_blocks = [], [], [], [], []
    for i, it in enumerate(w.items):
        pl = p.item(i)
        r = pl.item
        n = it.nq * it.nh
        (op_blocks if it.emit_lse else o_blocks).append((r.out_offset, r.out_offset + n * d))
        l_blocks.append((r.lse_offset, r.lse_offset + n))
        dq_blocks.append((pl.dq_offset, pl.dq_offset + n * d))
        dkv_blocks.append((pl.dkv_offset, pl.dkv_offset + it.nkv * it.nh * d))
        whole = (not it.emit_lse and it.q_lo == 0 and it.q_hi == it.seq_len and it.nh == H
                 and it.kv_lo == 0 and it.kv_hi == it.seq_len)
        if whole:
            assert r.out_offset == it.seq_offset * H * d and r.lse_offset == it.seq_offset * H
            assert pl.dq_offset == it.seq_offset * H * d == pl.dkv_offset
    for g in range(p.n_groups):
        members, oo, lo = p.group(g)
        it = w.items[members[0]]
        o_blocks.append((oo, oo + it.nq * it.nh * d))
        l_blocks.append((lo, lo + it.nq * it.nh))
        for m in members:
            assert p.item(m).fin_out_offset == oo and p.item(m).fin_lse_offset == lo
    assert [p.group(g)[0] for g in range(p.n_groups)] == merge_groups(w.items)
    for blocks, total in ((o_blocks, p.o_elems), (op_blocks, p.o_partial_elems), (l_blocks, p.lse_elems),
                          (dq_blocks, p.dq_elems), (dkv_blocks, p.dkv_elems)):
        blocks = sorted(b for b in blocks if b[1] > b[0])
        for a, b in zip(blocks, blocks[1:]):
            assert a[1] <= b[0], (a, b)
        assert all(b[1] <= total for b in blocks)
    assert p.workspace_bytes >= 4 * sum(it.nq * it.nh * (d + 1) for it in w.items)


def test_whole_sequence_group_lands_packed():
    w = config_long_video()
    p = host_plan(w)
    assert p.n_groups == 1
    members, oo, lo = p.group(0)
    assert members == list(range(8))
    assert oo == 0 and lo == 0   # the video is the first packed sequence
    assert p.o_elems == w.total_tokens * w.n_heads * w.head_dim


def test_flop_counts_of_the_workloads():
    # 4 |q| |kv| d per head (non-causal forward); backward 2.5x
    assert config_tiny().fwd_flops() == 4 * 64 * 4 * (64 * 64 + 100 * 100 + 256 * 256 + 512 * 512)
    assert abs(config_images().fwd_flops() / 1e12 - 1.018) < 1e-3
    m = config_mixed()
    assert abs(m.fwd_flops() / 1e12 - 16.69) < 5e-3
    assert abs(config_mixed(with_complement=False).fwd_flops() / 1e12 - 13.39) < 5e-3
    assert abs(config_long_video().fwd_flops() / 1e12 - 269.4) < 0.1
    assert m.bwd_flops() == 5 * m.fwd_flops() // 2


def _all_lists():
    from coalesced_packed_attention_gb300.workloads import Workload, config_training, scaled
    from tests.gpu_util import tiny_edge_items
    lists = [config_tiny(), config_images(), config_mixed(), config_long_video(), config_training()]
    lists += [scaled(w, f) for w in lists[1:] for f in (4, 6, 12, 24)]
    lists += [Workload("edges", 3, d, 300, tiny_edge_items(3), d ** -0.5) for d in (64, 128)]
    return lists


@pytest.mark.parametrize("flags", [0, zl.ZL_PLAN_FUSE_LOCAL_KMERGE,
                                   zl.ZL_PLAN_DETERMINISTIC_DQ,
                                   zl.ZL_PLAN_DETERMINISTIC_DQ | zl.ZL_PLAN_FUSE_LOCAL_KMERGE])
def test_every_plan_passes_the_bounds_dry_run(flags):
    for w in _all_lists():
        p = zl.zl_plan_worklist(w.items, w.n_heads, w.head_dim, w.total_tokens,
                                flags=zl.ZL_PLAN_HOST_ONLY | flags)
        p.check_bounds()
        # the workspace holds D ([|h|,|q|] fp32) and the dQ accumulator (fp32, |q| padded
        # to whole 128-row query blocks) for every item, plus with ordered dQ adds one
        # int32 turn counter per 32 rows of the accumulator, and nothing else
        need = sum(4 * it.nh * (it.nq + -(-it.nq // 128) * 128 * w.head_dim) for it in w.items)
        if flags & zl.ZL_PLAN_DETERMINISTIC_DQ:
            need += sum(16 * it.nh * -(-it.nq // 128) for it in w.items)
        assert need <= p.workspace_bytes <= need + 16


@pytest.mark.parametrize("make", [config_tiny, config_images, config_mixed, config_long_video])
def test_deterministic_dq_plan_claims_each_heads_kv_tiles_in_order(make):
    # ZL_PLAN_DETERMINISTIC_DQ: the same backward tiles, longest first, but block-major
    # within each cost, so the KV tiles of one (item, head) are claimed in ascending
    # order (a tile's turn comes after every tile it waits on) and far apart
    w = make()
    base = host_plan(w)
    p = zl.zl_plan_worklist(w.items, w.n_heads, w.head_dim, w.total_tokens,
                            flags=zl.ZL_PLAN_HOST_ONLY | zl.ZL_PLAN_DETERMINISTIC_DQ)
    tiles = p.tiles(1)
    assert sorted(tiles) == sorted(base.tiles(1))
    assert p.tiles(0) == base.tiles(0)
    costs = [t[3] for t in tiles]
    assert costs == sorted(costs, reverse=True)
    for a, b in zip(tiles, tiles[1:]):
        if a[3] == b[3]:
            assert (a[2], a[0], a[1]) < (b[2], b[0], b[1])
    next_turn = {}
    for (i, h, b, _) in tiles:
        assert next_turn.get((i, h), 0) == b
        next_turn[(i, h)] = b + 1
    blocks = sum(it.nh * -(-it.nq // 128) for it in w.items)
    assert p.workspace_bytes == base.workspace_bytes + 16 * blocks


def _union(items):
    return min(it.kv_lo for it in items), max(it.kv_hi for it in items)


@pytest.mark.parametrize("make", [config_tiny, config_mixed, config_long_video])
def test_fused_local_kmerge_plan(make):
    # ZL_PLAN_FUSE_LOCAL_KMERGE: a merge group whose chunks tile one contiguous KV range
    # becomes one forward item over that range; members keep only their backward role
    w = make()
    flags = zl.ZL_PLAN_HOST_ONLY
    plain = zl.zl_plan_worklist(w.items, w.n_heads, w.head_dim, w.total_tokens, flags=flags)
    fused = zl.zl_plan_worklist(w.items, w.n_heads, w.head_dim, w.total_tokens,
                                flags=flags | zl.ZL_PLAN_FUSE_LOCAL_KMERGE)
    fused.check_bounds()
    groups = merge_groups(w.items)
    assert plain.n_groups == fused.n_groups == len(groups) and plain.n_merge_groups == len(groups)
    contiguous = []
    for g in groups:
        r = sorted((w.items[i].kv_lo, w.items[i].kv_hi) for i in g)
        contiguous.append(all(a[1] == b[0] for a, b in zip(r, r[1:])))
    assert fused.n_merge_groups == contiguous.count(False)
    assert any(contiguous)
    fused_members = {i for g, c in zip(groups, contiguous) if c for i in g}
    for i in range(len(w.items)):
        r = fused.item(i).item
        if i in fused_members:
            assert r.out_offset == -1 and r.lse_offset == -1
            _, oo, lo = fused.group(fused.item(i).group)
            assert (fused.item(i).fin_out_offset, fused.item(i).fin_lse_offset) == (oo, lo)
        else:
            assert r.out_offset == plain.item(i).item.out_offset
        # the O blocks in `o` and the gradient blocks do not move (LSE blocks may: fused
        # members reserve none of their own)
        for f in ("fin_out_offset", "dq_offset", "dkv_offset"):
            assert getattr(fused.item(i), f) == getattr(plain.item(i), f)
    assert fused.lse_elems <= plain.lse_elems
    # no partial blocks for fused members
    need = sum(it.nq * it.nh * w.head_dim for i, it in enumerate(w.items) if it.emit_lse and i not in fused_members)
    assert need <= fused.o_partial_elems <= need + 8 * len(w.items)
    # forward tiles: members of fused groups have none; each fused group is one item
    # (index >= n_items, in group order) tiled over its rows and heads with the union's cost
    n = fused.n_items
    tiles = fused.tiles(0)
    assert not any(t[0] in fused_members for t in tiles)
    fused_groups = [g for g, c in zip(groups, contiguous) if c]
    for k, g in enumerate(fused_groups):
        it0 = w.items[g[0]]
        lo, hi = _union([w.items[i] for i in g])
        mine = sorted((t[1], t[2]) for t in tiles if t[0] == n + k)
        assert mine == sorted((h, b) for h in range(it0.h_lo, it0.h_hi) for b in range(-(-it0.nq // 256)))
        assert {t[3] for t in tiles if t[0] == n + k} == {-(-(hi - lo) // 128)}
    plain_tiles = [t for t in plain.tiles(0) if t[0] not in fused_members]
    assert sorted(t for t in tiles if t[0] < n) == sorted(plain_tiles)
    # backward tiles are those of the plain plan
    assert fused.tiles(1) == plain.tiles(1)


def test_fused_local_kmerge_leaves_gapped_groups():
    # chunks [0,100) and [150,300) leave a gap: merged as usual
    items = [WorkItem(0, 300, 0, 300, 0, 2, 0, 100, 1), WorkItem(0, 300, 0, 300, 0, 2, 150, 300, 1)]
    p = zl.zl_plan_worklist(items, 2, 64, 300, flags=zl.ZL_PLAN_HOST_ONLY | zl.ZL_PLAN_FUSE_LOCAL_KMERGE)
    assert p.n_merge_groups == 1 and all(p.item(i).item.out_offset >= 0 for i in range(2))
    p.check_bounds()


def test_group_of_many_members_is_read_whole():
    # 100 k-chunks of one sequence form one merge group; the binding reads all of them
    items = [WorkItem(0, 1000, 0, 1000, 0, 2, 10 * c, 10 * c + 10, 1) for c in range(100)]
    p = zl.zl_plan_worklist(items, 2, 64, 1000, flags=zl.ZL_PLAN_HOST_ONLY)
    assert p.n_groups == 1
    members, _, _ = p.group(0)
    assert members == list(range(100))


def test_tensors_on_another_device_are_rejected_before_the_call():
    import torch

    class Fake:  # stands in for a tensor: only its device is looked at
        def __init__(self, index):
            self.device = torch.device("cuda", index)

    p = zl.zl_plan_worklist(config_tiny().items, 4, 64, config_tiny().total_tokens, flags=zl.ZL_PLAN_HOST_ONLY)
    p.device = 0
    zl._on_plan_device(p, Fake(0), None, Fake(0))
    with pytest.raises(ValueError):
        zl._on_plan_device(p, Fake(0), Fake(1))


@pytest.mark.parametrize("make", [config_tiny, config_mixed])
def test_o_arena_from_tokens_places_each_items_rows(make):
    # the dO layout the backward reads: every item's final block holds its rows and heads
    import torch
    w = make()
    p = host_plan(w)
    H, d, T = w.n_heads, w.head_dim, w.total_tokens
    x = torch.arange(T * H * d, dtype=torch.float64).reshape(T, H, d)
    arena = zl.o_arena_from_tokens(p, w.items, x)
    assert arena.numel() == max(p.o_elems, 8)
    for i, it in enumerate(w.items):
        pl = p.item(i)
        blk = arena[pl.fin_out_offset: pl.fin_out_offset + it.nq * it.nh * d].reshape(it.nq, it.nh, d)
        s = it.seq_offset
        assert torch.equal(blk, x[s + it.q_lo: s + it.q_hi, it.h_lo:it.h_hi])
    # whole sequences sit in place, packed like the tokens
    it = w.items[0]
    if not it.emit_lse and it.nq == it.seq_len and it.nh == H:
        s = it.seq_offset
        assert torch.equal(arena[s * H * d:(s + it.seq_len) * H * d], x[s:s + it.seq_len].reshape(-1))


def test_launches_reject_missing_and_host_only_plans(lib):
    # every launch entry point returns ZL_ERR_INVALID_ARG for a null or host-only plan
    # before it touches any pointer or the GPU (the dummy pointers are never read)
    import ctypes
    hp = host_plan(config_tiny())
    x = ctypes.c_void_p(1 << 20)
    f = ctypes.c_float(0.125)
    calls = {
        "zl_coalesced_attn_fwd": lambda p: lib.zl_coalesced_attn_fwd(p, x, x, x, x, x, x, f, None),
        "zl_merge_partials": lambda p: lib.zl_merge_partials(p, x, x, x, x, None),
        "zl_coalesced_attn_bwd": lambda p: lib.zl_coalesced_attn_bwd(p, x, x, x, x, x, x, x, x, x, x, f, None),
        "zl_bwd_preprocess": lambda p: lib.zl_bwd_preprocess(p, x, x, x, None),
        "zl_bwd_main": lambda p: lib.zl_bwd_main(p, x, x, x, x, x, x, x, x, f, None),
        "zl_bwd_finalize": lambda p: lib.zl_bwd_finalize(p, x, x, f, None),
        "zl_get_device_status": lambda p: lib.zl_get_device_status(p, None, ctypes.byref(ctypes.c_int32())),
    }
    for name, call in calls.items():
        assert call(None) == zl.ZL_ERR_INVALID_ARG, name
        assert call(hp.handle) == zl.ZL_ERR_INVALID_ARG, name


def test_plan_queries_check_their_arguments(lib):
    import ctypes
    w = config_mixed()
    p = host_plan(w)
    I64, I32 = ctypes.c_int64, ctypes.c_int32
    c = I64()
    assert lib.zl_plan_count(p.handle, 5, ctypes.byref(c)) == zl.ZL_ERR_INVALID_ARG
    assert lib.zl_plan_count(p.handle, -1, ctypes.byref(c)) == zl.ZL_ERR_INVALID_ARG
    assert lib.zl_plan_count(None, 0, ctypes.byref(c)) == zl.ZL_ERR_INVALID_ARG
    assert lib.zl_plan_item(p.handle, len(w.items), None, None, None, None, None, None) == zl.ZL_ERR_INVALID_ARG
    assert lib.zl_plan_item(p.handle, -1, None, None, None, None, None, None) == zl.ZL_ERR_INVALID_ARG
    buf = (I32 * (4 * p.n_fwd_tiles))()
    assert lib.zl_plan_tiles(p.handle, 2, buf, p.n_fwd_tiles) == zl.ZL_ERR_INVALID_ARG
    assert lib.zl_plan_tiles(p.handle, 0, buf, p.n_fwd_tiles - 1) == zl.ZL_ERR_INVALID_ARG  # buffer too small
    assert lib.zl_plan_tiles(p.handle, 0, buf, p.n_fwd_tiles) == zl.ZL_OK
    assert lib.zl_plan_group(p.handle, p.n_groups, None, 0, None, None, None) == zl.ZL_ERR_INVALID_ARG
    assert lib.zl_plan_arena_sizes(None, None, None, None, None, None, None) == zl.ZL_ERR_INVALID_ARG
    assert lib.zl_plan_check_bounds(None) == zl.ZL_ERR_INVALID_ARG
    assert lib.zl_plan_worklist(None, 0, 1, 64, 1, 0, None) == zl.ZL_ERR_INVALID_ARG


# ---------------------------------------------------------------- caller-chosen merge groups
def _kv_split_list():
    # a 512-token sequence (2 heads) as four k-split chunks, beside a whole sequence
    return [WorkItem(0, 100, 0, 100, 0, 2, 0, 100),
            WorkItem(100, 512, 0, 512, 0, 2, 0, 128, 1), WorkItem(100, 512, 0, 512, 0, 2, 128, 256, 1),
            WorkItem(100, 512, 0, 512, 0, 2, 256, 384, 1), WorkItem(100, 512, 0, 512, 0, 2, 384, 512, 1)]


def test_explicit_groups_set_membership_and_member_order():
    items = _kv_split_list()
    p = zl.zl_plan_worklist_groups(items, 2, 64, 612, [[4, 2], [1, 3]], flags=zl.ZL_PLAN_HOST_ONLY)
    assert p.n_groups == 2
    assert p.group(0)[0] == [4, 2] and p.group(1)[0] == [1, 3]
    # each group has its own final block; members read their group's
    o0, o1 = p.group(0)[1], p.group(1)[1]
    assert o0 != o1
    assert p.item(4).fin_out_offset == p.item(2).fin_out_offset == o0
    assert p.item(1).fin_out_offset == p.item(3).fin_out_offset == o1
    p.check_bounds()
    # the default grouping of the same list: one group in list order
    d = zl.zl_plan_worklist(items, 2, 64, 612, flags=zl.ZL_PLAN_HOST_ONLY)
    assert d.n_groups == 1 and d.group(0)[0] == [1, 2, 3, 4]
    same = zl.zl_plan_worklist_groups(items, 2, 64, 612, [[1, 2, 3, 4]], flags=zl.ZL_PLAN_HOST_ONLY)
    assert same.tiles(0) == d.tiles(0) and same.group(0) == d.group(0)


@pytest.mark.parametrize("groups", [
    [[1, 2], [3]],               # item 4 in no group
    [[1, 2], [3, 4], [2]],       # item 2 twice
    [[0, 1], [2, 3, 4]],         # item 0 is not a k-split item
    [[1, 2, 3, 4, 5]],           # id out of range
    [[1, 2], [], [3, 4]],        # empty group
])
def test_explicit_groups_reject_malformed_lists(groups):
    with pytest.raises(zl.ZlError) as e:
        zl.zl_plan_worklist_groups(_kv_split_list(), 2, 64, 612, groups, flags=zl.ZL_PLAN_HOST_ONLY)
    assert e.value.status == zl.ZL_ERR_INVALID_ARG


def test_explicit_groups_reject_mixed_keys_and_overlap():
    items = _kv_split_list() + [WorkItem(100, 512, 0, 256, 0, 2, 0, 512, 1)]   # other rows
    with pytest.raises(zl.ZlError):
        zl.zl_plan_worklist_groups(items, 2, 64, 612, [[1, 2, 3, 4, 5]], flags=zl.ZL_PLAN_HOST_ONLY)
    ok = zl.zl_plan_worklist_groups(items, 2, 64, 612, [[1, 2, 3, 4], [5]], flags=zl.ZL_PLAN_HOST_ONLY)
    assert ok.n_groups == 2
    over = _kv_split_list() + [WorkItem(100, 512, 0, 512, 0, 2, 64, 192, 1)]    # overlaps chunks 1, 2
    with pytest.raises(zl.ZlError):
        zl.zl_plan_worklist_groups(over, 2, 64, 612, [[1, 2, 3, 4, 5]], flags=zl.ZL_PLAN_HOST_ONLY)
    # the same chunk in a group of its own is a separate problem: accepted
    ok = zl.zl_plan_worklist_groups(over, 2, 64, 612, [[1, 2, 3, 4], [5]], flags=zl.ZL_PLAN_HOST_ONLY)
    ok.check_bounds()


def test_explicit_groups_bad_pointer_arrays(lib):
    items = zl._to_c_items(_kv_split_list())
    h = ctypes.c_void_p()
    ids = (ctypes.c_int32 * 4)(1, 2, 3, 4)
    bad_start = (ctypes.c_int32 * 2)(1, 4)
    assert lib.zl_plan_worklist_groups(items, 5, 2, 64, 612, zl.ZL_PLAN_HOST_ONLY, ids, bad_start, 1,
                                       ctypes.byref(h)) == zl.ZL_ERR_INVALID_ARG
    decreasing = (ctypes.c_int32 * 3)(0, 3, 2)
    assert lib.zl_plan_worklist_groups(items, 5, 2, 64, 612, zl.ZL_PLAN_HOST_ONLY, ids, decreasing, 2,
                                       ctypes.byref(h)) == zl.ZL_ERR_INVALID_ARG
    assert lib.zl_plan_worklist_groups(items, 5, 2, 64, 612, zl.ZL_PLAN_HOST_ONLY, None, None, 1,
                                       ctypes.byref(h)) == zl.ZL_ERR_INVALID_ARG
    assert h.value is None
