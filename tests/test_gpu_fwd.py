"""GPU parity of the forward launch and the merge against the CPU float64 oracle,
through the C ABI, on work lists the oracle finishes in seconds (several tiles and
ragged tails), plus degenerate shards."""
import numpy as np
import pytest

from coalesced_packed_attention_gb300.workloads import (WorkItem, Workload, config_images, config_long_video,
                                                        config_mixed, config_tiny, scaled)
from tests.gpu_util import ATOL_LSE, ATOL_O, Run, check, tiny_edge_items

pytestmark = pytest.mark.gpu


def test_tiny_mixed_list_all_rows():
    r = Run(config_tiny(), seed=0)
    r.check_forward()


@pytest.mark.parametrize("seed", [1, 2])
def test_tiny_mixed_list_more_seeds(seed):
    Run(config_tiny(), seed=seed).check_forward()


def test_tiny_structured_peaky_softmax():
    Run(config_tiny(), seed=3, structured=True).check_forward()


@pytest.mark.parametrize("factor", [6])
def test_images_scaled(factor):
    Run(scaled(config_images(), factor), seed=0).check_forward()
    Run(scaled(config_images(), factor), seed=1, structured=True).check_forward()


@pytest.mark.parametrize("factor", [12])
def test_mixed_shards_scaled(factor):
    w = scaled(config_mixed(), factor)
    Run(w, seed=0).check_forward()
    Run(w, seed=1, structured=True).check_forward()


@pytest.mark.parametrize("factor", [24])
def test_long_video_k8_scaled(factor):
    Run(scaled(config_long_video(), factor), seed=0).check_forward()
    Run(scaled(config_long_video(), factor), seed=1, structured=True).check_forward()


@pytest.mark.parametrize("d", [64, 128])
def test_degenerate_and_ragged_shards(d):
    H = 3
    w = Workload(f"edges_d{d}", H, d, 300, tiny_edge_items(H), d ** -0.5)
    r = Run(w, seed=4)
    res = r.check_forward()
    # the empty-KV item: O = 0 and LSE = -inf exactly
    assert np.all(r.own_o(3) == 0.0) and np.all(np.isneginf(r.own_lse(3)))


def test_whole_sequences_land_packed_like_q():
    # the packed O of the images list reads as [T, H, d] directly
    w = scaled(config_images(), 16)
    r = Run(w, seed=5)
    r.check_forward()
    T, H, d = w.total_tokens, w.n_heads, w.head_dim
    o = r.bufs["o"][: T * H * d].reshape(T, H, d)
    assert np.isfinite(o).all()


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("n_members", [1, 3, 32, 33])
def test_merge_group_sizes(d, n_members):
    """k-split groups of 1 to 33 members (ragged chunk tails: 300 x 3 row-heads per member,
    24 KV tokens each) beside a second, smaller group and a group whose members are all
    empty (the merge's member loop in one pass up to 8 members, in batches beyond)."""
    H, nq, ck = 3, 300, 24
    L = max(nq, n_members * ck)
    items = [WorkItem(0, L, 0, nq, 0, H, c * ck, (c + 1) * ck, 1) for c in range(n_members)]
    items += [WorkItem(L, 200, 0, 150, 1, 3, 0, 90, 1), WorkItem(L, 200, 0, 150, 1, 3, 90, 200, 1)]
    items += [WorkItem(L, 200, 10, 20, 0, 1, 0, 0, 1), WorkItem(L, 200, 10, 20, 0, 1, 5, 5, 1)]
    w = Workload(f"kgroups{n_members}_d{d}", H, d, L + 200, items, d ** -0.5)
    r = Run(w, seed=7)
    r.check_forward()
    empty = len(items) - 1
    assert np.all(r.final_o(empty) == 0.0) and np.all(np.isneginf(r.final_lse(empty)))


def test_shards_reproduce_the_whole_bit_for_bit():
    """Query rows and heads are computed independently (a row's scores, weights and
    rescales involve only that row; a warp's shared rescale vote multiplies rows that
    need none by exactly 1), so q-shards at unaligned boundaries and h-shards of a
    sequence give exactly the whole item's O and LSE."""
    H, d, L = 4, 128, 1000
    items = [WorkItem(0, L, 0, L, 0, H, 0, L, 0),        # whole
             WorkItem(0, L, 0, 300, 0, H, 0, L, 0),      # q shards: [0,300) [300,777) [777,1000)
             WorkItem(0, L, 300, 777, 0, H, 0, L, 0),
             WorkItem(0, L, 777, L, 0, H, 0, L, 0),
             WorkItem(0, L, 0, L, 0, 1, 0, L, 0),        # h shards: {0}, {1, 2, 3}
             WorkItem(0, L, 0, L, 1, H, 0, L, 0)]
    w = Workload("shards_bitwise", H, d, L, items, d ** -0.5)
    r = Run(w, seed=12)
    O, lse = r.own_o(0), r.own_lse(0)
    for i, it in enumerate(items[1:], start=1):
        assert np.array_equal(r.own_o(i), O[it.q_lo:it.q_hi, it.h_lo:it.h_hi]), i
        assert np.array_equal(r.own_lse(i), lse[it.h_lo:it.h_hi, it.q_lo:it.q_hi]), i


def test_merge_with_an_empty_chunk_is_the_unsplit_item_bit_for_bit():
    """A k-split group of the full KV range and an empty chunk: the empty chunk's LSE is
    -inf, so the merge's weight is exp(0) = 1 and its LSE is the full chunk's exactly, and
    the merged O and LSE equal the unsplit item's bit for bit."""
    H, d, L = 3, 128, 500
    items = [WorkItem(0, L, 0, L, 0, H, 0, L, 0),       # unsplit
             WorkItem(0, L, 0, L, 0, H, 0, L, 1),       # full chunk, emit_lse
             WorkItem(0, L, 0, L, 0, H, L, L, 1)]       # empty chunk, same group
    w = Workload("merge_empty_chunk", H, d, L, items, d ** -0.5)
    r = Run(w, seed=15)
    assert np.array_equal(r.final_o(1), r.own_o(0))
    assert np.array_equal(r.final_lse(1), r.own_lse(0))
