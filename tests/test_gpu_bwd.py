"""GPU parity of the backward launch (row sums D, tcgen05 backward, dQ finalisation)
against the CPU float64 oracle, every item kind: whole, q-split (partial dK/dV),
h-split, k-split with the merged global LSE (partial dQ)."""
import numpy as np
import pytest

from coalesced_packed_attention_gb300.workloads import Workload, config_training, scaled
from tests.gpu_util import Run, check_gradients, oracle_pairs, tiny_edge_items

pytestmark = pytest.mark.gpu


def check_backward(r, kv_sample=None, q_sample=None, seed=0):
    _, final = oracle_pairs(r)
    check_gradients(r, final, q_sample=q_sample, kv_sample=kv_sample, seed=seed)


def test_training_list_scaled_all_rows():
    w = scaled(config_training(), 12)
    r = Run(w, seed=0, backward=True)
    r.check_forward()
    check_backward(r)


def test_training_list_scaled_structured():
    w = scaled(config_training(), 24)
    r = Run(w, seed=1, structured=True, backward=True)
    check_backward(r)


@pytest.mark.parametrize("d", [64, 128])
def test_backward_degenerate_and_ragged_shards(d):
    H = 3
    w = Workload(f"edges_d{d}", H, d, 300, tiny_edge_items(H), d ** -0.5, with_backward=True)
    r = Run(w, seed=2, backward=True)
    check_backward(r)
    # an item with no KV rows has dQ = 0; one with no query rows writes nothing
    assert np.all(r.grad(3, "dq") == 0.0)


def test_whole_item_gradient_sums():
    # for a whole item sum_j dK_j = 0 and sum_j dV_j = sum_i dO_i, per head
    w = scaled(config_training(), 12)
    r = Run(w, seed=3, backward=True)
    for i, it in enumerate(r.items):
        if it.emit_lse or it.nq != it.seq_len or it.nh != w.n_heads or it.nkv != it.seq_len:
            continue
        dk, dv = r.grad(i, "dk"), r.grad(i, "dv")
        s = it.seq_offset
        np.testing.assert_allclose(dv.sum(axis=0), r.do[s:s + it.seq_len].sum(axis=0), atol=5e-2)
        np.testing.assert_allclose(dk.sum(axis=0), 0.0, atol=5e-2)


@pytest.mark.parametrize("d,flags", [(64, 0), (128, 0), (128, "fuse"), (128, "ordered")])
def test_non_finite_tokens_outside_the_items(d, flags):
    """Tokens that belong to no item (gaps between and after the packed sequences) hold
    NaN in Q, K, V and dO.  Every ragged tile reads such tokens next to its item (an
    item's last KV block, its last query block), and the outputs must stay exactly
    those of the oracle, which never reads them; also with the k-split group fused into
    the forward and with ordered dQ adds."""
    from coalesced_packed_attention_gb300.workloads import WorkItem
    H = 3
    A, B = (0, 300), (400, 250)  # gaps [300, 400) and [650, 704)
    items = [
        WorkItem(A[0], A[1], 0, A[1], 0, H, 0, A[1], 0),     # whole A (ragged KV and query tails)
        WorkItem(B[0], B[1], 0, B[1], 0, H, 0, B[1], 0),     # whole B
        WorkItem(B[0], B[1], 0, 100, 0, H, 0, B[1], 0),      # q shard of B
        WorkItem(A[0], A[1], 0, A[1], 0, 2, 0, 130, 1),      # k split of A, heads [0, 2):
        WorkItem(A[0], A[1], 0, A[1], 0, 2, 130, A[1], 1),   # the second chunk ends at the gap
    ]
    w = Workload(f"gaps_d{d}", H, d, 704, items, d ** -0.5, with_backward=True)
    from coalesced_packed_attention_gb300 import zl
    f = {0: 0, "fuse": zl.ZL_PLAN_FUSE_LOCAL_KMERGE, "ordered": zl.ZL_PLAN_DETERMINISTIC_DQ}[flags]
    r = Run(w, seed=9, backward=True, flags=f, poison=[(300, 400), (650, 704)])
    r.check_forward()
    check_backward(r)
    for i in range(len(items)):
        for g in ("dq", "dk", "dv"):
            assert np.isfinite(r.grad(i, g)).all(), (i, g)
