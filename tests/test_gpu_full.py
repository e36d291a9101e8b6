"""GPU parity at the full sizes of the four work lists, in the launch configuration
bench.py times (one persistent launch per stage over the whole list): every image row
of the image-only list; >= 4096 seeded random query rows per (item, head) plus tile
edges for the video shards; backward dQ on sampled rows, dK/dV on sampled KV rows of one
head per item, and the whole-item gradient sums on every head."""
import numpy as np
import pytest

import oracle
from coalesced_packed_attention_gb300.workloads import (WorkItem, config_images, config_long_video,
                                                        config_mixed, config_training, merge_groups)
from tests.gpu_util import ATOL_O, Run, check, oracle_backward_dq, oracle_forward, sample_rows

pytestmark = pytest.mark.gpu


def test_images_full_all_rows():
    Run(config_images(), seed=0).check_forward()


def test_mixed_shards_full_sampled_rows():
    Run(config_mixed(), seed=0).check_forward(sample=4096)


def test_long_video_k8_full_sampled_rows():
    Run(config_long_video(), seed=0).check_forward(sample=4096)


def test_training_full_sampled():
    w = config_training()
    r = Run(w, seed=0, backward=True)
    r.check_forward(sample=1024)
    groups = merge_groups(r.items)
    group_of = {i: g for g in groups for i in g}
    for i, it in enumerate(r.items):
        s = it.seq_offset
        rows = sample_rows(it.nq, 11 + i, 1024)
        # final O / LSE of those rows: the item's own, or its group's merge
        members = group_of.get(i, [i])
        parts = [oracle_forward(r.q, r.k, r.v, r.items[m], r.scale, rows=it.q_lo + rows) for m in members]
        O, L = oracle.merge(parts) if len(parts) > 1 else parts[0]
        do_rows = r.do[s + it.q_lo + rows][:, it.h_lo:it.h_hi]
        dQ_ref = oracle_backward_dq(r.q, r.k, r.v, do_rows, O, L, it, r.scale, it.q_lo + rows)
        check(f"item{i}.dQ", r.grad(i, "dq")[rows], dQ_ref, ATOL_O)
        # dK/dV of one head on sampled KV rows (needs every query row's final O, LSE)
        h = it.h_lo
        one = WorkItem(it.seq_offset, it.seq_len, it.q_lo, it.q_hi, h, h + 1, it.kv_lo, it.kv_hi, it.emit_lse)
        parts = [oracle.forward(r.q, r.k, r.v, WorkItem(it.seq_offset, it.seq_len, it.q_lo, it.q_hi, h, h + 1,
                                                        r.items[m].kv_lo, r.items[m].kv_hi, 1), r.scale)
                 for m in members]
        Oa, La = oracle.merge(parts) if len(parts) > 1 else parts[0]
        kv = sample_rows(it.nkv, 23 + i, 256)
        dK_ref, dV_ref = oracle.backward_dkdv(r.q, r.k, r.v, r.do[s + it.q_lo: s + it.q_hi, h:h + 1], Oa, La, one,
                                              r.scale, it.kv_lo + kv)
        check(f"item{i}.dK", r.grad(i, "dk")[kv][:, :1], dK_ref, ATOL_O)
        check(f"item{i}.dV", r.grad(i, "dv")[kv][:, :1], dV_ref, ATOL_O)
        # whole items, every head: sum_j dK_j = 0 and sum_j dV_j = sum_i dO_i
        if not it.emit_lse and it.nq == it.seq_len and it.nh == w.n_heads and it.nkv == it.seq_len:
            dv, dk = r.grad(i, "dv"), r.grad(i, "dk")
            np.testing.assert_allclose(dv.sum(axis=0), r.do[s:s + it.seq_len].sum(axis=0), atol=5e-2)
            np.testing.assert_allclose(dk.sum(axis=0), 0.0, atol=5e-2)
