"""GPU parity with caller-chosen merge groups (zl_plan_worklist_groups): a sequence cut
into four k-split chunks, merged as two groups of two in a member order other than the
list order, beside a whole sequence and a second sequence whose chunks form one group.
Each group is exact attention over the union of its chunks; the backward of every member
reads its group's merged O and LSE."""
import pytest

from coalesced_packed_attention_gb300.workloads import WorkItem, Workload
from tests.gpu_util import Run, check_forward_pairs, check_gradients, oracle_pairs

pytestmark = pytest.mark.gpu


def _list(d):
    H = 3
    items = [WorkItem(0, 200, 0, 200, 0, H, 0, 200),
             WorkItem(200, 700, 0, 700, 0, H, 0, 150, 1), WorkItem(200, 700, 0, 700, 0, H, 150, 400, 1),
             WorkItem(200, 700, 0, 700, 0, H, 400, 401, 1), WorkItem(200, 700, 0, 700, 0, H, 401, 700, 1),
             WorkItem(900, 300, 10, 290, 1, 3, 0, 130, 1), WorkItem(900, 300, 10, 290, 1, 3, 130, 300, 1)]
    return Workload(f"groups_d{d}", H, d, 1200, items, d ** -0.5, with_backward=True)


@pytest.mark.parametrize("d", [64, 128])
def test_explicit_groups_forward_merge_backward(d):
    groups = [[4, 1], [3, 2], [6, 5]]
    r = Run(_list(d), seed=8, backward=True, groups=groups)
    assert [r.plan.group(g)[0] for g in range(r.plan.n_groups)] == groups
    own, final = oracle_pairs(r)
    check_forward_pairs(r, own, final)
    check_gradients(r, final)
