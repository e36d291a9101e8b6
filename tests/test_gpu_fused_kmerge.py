"""GPU parity of the fused local k-merge (ZL_PLAN_FUSE_LOCAL_KMERGE): a k-split group
whose chunks tile one contiguous KV range is computed by the forward as one item, its
final O and LSE written straight to the group's blocks.  Checked against the oracle's
merge of the members' chunk results, against the unfused plan on the same inputs, and
through the backward (whose members read the fused final O and LSE)."""
import numpy as np
import pytest

from coalesced_packed_attention_gb300 import zl
from coalesced_packed_attention_gb300.workloads import (Workload, config_long_video, config_mixed,
                                                        config_training, scaled)
from tests.gpu_util import ATOL_LSE, ATOL_O, Run, check, tiny_edge_items
from tests.test_gpu_bwd import check_backward

pytestmark = pytest.mark.gpu
FUSE = zl.ZL_PLAN_FUSE_LOCAL_KMERGE


@pytest.mark.parametrize("d", [64, 128])
def test_fused_edges_all_rows(d):
    # a 3-way k split with an empty, unaligned middle chunk, beside whole and
    # degenerate items
    H = 3
    w = Workload(f"edges_d{d}", H, d, 300, tiny_edge_items(H), d ** -0.5)
    r = Run(w, seed=5, flags=FUSE)
    assert r.plan.n_merge_groups == 0 and r.plan.n_groups == 1
    r.check_forward()


def test_fused_long_video_sampled_rows():
    # 8 chunks of a video (lengths / 8) fused into one item of the whole KV range
    r = Run(scaled(config_long_video(), 8), seed=6, flags=FUSE)
    assert r.plan.n_merge_groups == 0
    r.check_forward(sample=1024)


def test_fused_equals_merged_on_the_same_inputs():
    w = scaled(config_mixed(), 4)
    a = Run(w, seed=7)
    b = Run(w, seed=7, flags=FUSE)
    assert a.plan.n_merge_groups == 1 and b.plan.n_merge_groups == 0
    members, _, _ = a.plan.group(0)
    check("fused vs merged O", b.final_o(members[0]), a.final_o(members[0]), 2 * ATOL_O)
    check("fused vs merged LSE", b.final_lse(members[0]), a.final_lse(members[0]), 2 * ATOL_LSE)
    # every other item's output is the same computation in both plans
    for i, it in enumerate(w.items):
        if not it.emit_lse:
            np.testing.assert_array_equal(a.own_o(i), b.own_o(i))
            np.testing.assert_array_equal(a.own_lse(i), b.own_lse(i))


def test_fused_training_list_backward():
    w = scaled(config_training(), 12)
    r = Run(w, seed=8, backward=True, flags=FUSE)
    assert r.plan.n_merge_groups == 0
    r.check_forward()
    check_backward(r)
