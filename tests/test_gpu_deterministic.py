"""GPU checks of the ordered dQ adds (ZL_PLAN_DETERMINISTIC_DQ).  The backward still
matches the oracle, and repeated backward launches on the same inputs give bitwise
identical dQ (dK and dV are always reproducible).  The stress list is one head of an
8192-token sequence: its 64 KV tiles share one cost, so all of them are claimed at
once and each one waits for the tile before it at every query block."""
import numpy as np
import pytest

from coalesced_packed_attention_gb300 import zl
from coalesced_packed_attention_gb300.workloads import (WorkItem, Workload, config_training, make_inputs,
                                                        scaled)
from tests._lib import ensure_library
from tests.gpu_util import Run, tiny_edge_items
from tests.test_gpu_bwd import check_backward

pytestmark = pytest.mark.gpu
DET = zl.ZL_PLAN_DETERMINISTIC_DQ


def one_head_long(L=8192, d=128):
    return Workload(f"one_head_{L}", 1, d, L, [WorkItem(0, L, 0, L, 0, 1, 0, L, 0)], d ** -0.5,
                    with_backward=True)


def training_div4():
    return scaled(config_training(), 4)


def test_training_list_parity():
    r = Run(scaled(config_training(), 12), seed=4, backward=True, flags=DET)
    r.check_forward()
    check_backward(r)


@pytest.mark.parametrize("d", [64, 128])
def test_degenerate_and_ragged_shards_parity(d):
    H = 3
    w = Workload(f"edges_d{d}", H, d, 300, tiny_edge_items(H), d ** -0.5, with_backward=True)
    r = Run(w, seed=5, backward=True, flags=DET)
    check_backward(r)


def test_chained_kv_tiles_parity():
    # every KV tile of the head waits on its predecessor: the result is still the oracle's
    r = Run(one_head_long(), seed=6, backward=True, flags=DET)
    check_backward(r, kv_sample=512, q_sample=512)


def _repeat_backward(w, flags, n, seed):
    import torch
    ensure_library()
    H, d, T = w.n_heads, w.head_dim, w.total_tokens
    ins = make_inputs(T, H, d, seed, with_grad_output=True)
    plan = zl.zl_plan_worklist(w.items, H, d, T, flags)
    dev = torch.device("cuda:0")
    q, k, v = (x.to(dev) for x in ins[:3])
    bufs = zl.allocate(plan, dev, backward=True)
    zl.forward(plan, q, k, v, w.scale, bufs)
    dO = torch.zeros_like(bufs["o"])
    for i, it in enumerate(w.items):
        pl = plan.item(i)
        n_el = it.nq * it.nh * d
        blk = ins[3][it.seq_offset + it.q_lo: it.seq_offset + it.q_hi, it.h_lo:it.h_hi].reshape(-1)
        dO[pl.fin_out_offset: pl.fin_out_offset + n_el] = blk.to(dev)
    outs = []
    for _ in range(n):
        for key in ("dq", "dk", "dv"):
            bufs[key].fill_(float("nan"))
        zl.backward(plan, q, k, v, dO, w.scale, bufs)
        torch.cuda.synchronize()
        assert zl.zl_get_device_status(plan) == 0
        outs.append({key: bufs[key].view(torch.int32).cpu().numpy().copy() for key in ("dq", "dk", "dv")})
    return outs


@pytest.mark.parametrize("make", [training_div4, one_head_long])
def test_repeated_backward_is_bitwise_identical(make):
    outs = _repeat_backward(make(), DET, 4, seed=7)
    for o in outs[1:]:
        for key in ("dq", "dk", "dv"):
            np.testing.assert_array_equal(o[key], outs[0][key], err_msg=key)


def test_shards_reproduce_the_whole_gradients_bit_for_bit():
    """With ordered dQ adds every dQ element sums its KV tiles in tile order, and every
    tile walks the query blocks from the first, so a q-shard's dQ rows and an h-shard's
    dQ, dK and dV equal the whole item's bit for bit (a query row's dS and its dQ terms
    involve only that row; the shards' O and LSE equal the whole's bit for bit too)."""
    H, d, L = 4, 128, 1000
    items = [WorkItem(0, L, 0, L, 0, H, 0, L, 0),        # whole
             WorkItem(0, L, 0, 300, 0, H, 0, L, 0),      # q shards at unaligned boundaries
             WorkItem(0, L, 300, 777, 0, H, 0, L, 0),
             WorkItem(0, L, 777, L, 0, H, 0, L, 0),
             WorkItem(0, L, 0, L, 0, 1, 0, L, 0),        # h shards
             WorkItem(0, L, 0, L, 1, H, 0, L, 0)]
    w = Workload("shards_bitwise_bwd", H, d, L, items, d ** -0.5, with_backward=True)
    r = Run(w, seed=13, backward=True, flags=DET)
    dq, dk, dv = (r.grad(0, x) for x in ("dq", "dk", "dv"))
    for i in (1, 2, 3):
        it = items[i]
        assert np.array_equal(r.grad(i, "dq"), dq[it.q_lo:it.q_hi]), i
    for i in (4, 5):
        it = items[i]
        for name, whole in (("dq", dq), ("dk", dk), ("dv", dv)):
            assert np.array_equal(r.grad(i, name), whole[:, it.h_lo:it.h_hi]), (i, name)


def test_co_location_leaves_results_unchanged():
    """Co-location changes the schedule, not the result (pith.science review, "What
    carries the argument": whole sequences and shards share one launch): an image, the
    video's q shard and its k shard give the same O and LSE bit for bit whether each runs
    alone or coalesced with the other 19 items, and (with ordered dQ adds) the same dQ,
    dK and dV for the image and the q shard."""
    w = scaled(config_training(), 12)
    full = Run(w, seed=14, backward=True, flags=DET)
    picks = [0, w.labels.index("video_qsplit"), w.labels.index("video_ksplit")]
    for i in picks:
        it = w.items[i]
        alone = Run(Workload(f"alone_{i}", w.n_heads, w.head_dim, w.total_tokens, [it], w.scale,
                             with_backward=True), seed=14, backward=True, flags=DET)
        assert np.array_equal(alone.own_o(0), full.own_o(i)), i
        assert np.array_equal(alone.own_lse(0), full.own_lse(i)), i
        if not it.emit_lse:  # a k shard alone has no partner to merge with
            for name in ("dq", "dk", "dv"):
                assert np.array_equal(alone.grad(0, name), full.grad(i, name)), (i, name)
