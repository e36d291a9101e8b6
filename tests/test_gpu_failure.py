"""Failure detection without a GPU fault: a plan built with the test flag announces
its first K tile (backward: K/V tile) but never issues the copy, so a bounded mbarrier
wait runs out; the kernel records ZL_ERR_TIMEOUT in the plan's status word, leaves its
loops, frees TMEM and returns, and the context stays usable for the next launch."""
import numpy as np
import pytest

from coalesced_packed_attention_gb300 import zl
from coalesced_packed_attention_gb300.workloads import config_tiny
from tests.gpu_util import Run
from tests._lib import ensure_library

pytestmark = pytest.mark.gpu


def test_withheld_load_reports_timeout_and_context_survives():
    import torch
    ensure_library()
    w = config_tiny()
    plan = zl.zl_plan_worklist(w.items, w.n_heads, w.head_dim, w.total_tokens, flags=zl.ZL_PLAN_TEST_WITHHOLD_LOAD)
    from coalesced_packed_attention_gb300.workloads import make_inputs
    q, k, v = (x.cuda() for x in make_inputs(w.total_tokens, w.n_heads, w.head_dim, 0))
    bufs = zl.allocate(plan, "cuda")
    zl.zl_coalesced_attn_fwd(plan, q, k, v, bufs["o"], bufs["o_partial"], bufs["lse"], w.scale)
    torch.cuda.synchronize()
    assert zl.zl_get_device_status(plan) == zl.ZL_ERR_TIMEOUT
    assert zl.zl_get_device_status(plan) == 0          # reading clears the word
    # the same context still runs a normal launch correctly
    Run(w, seed=0).check_forward()


def test_withheld_load_in_backward_reports_timeout_and_context_survives():
    import torch
    from coalesced_packed_attention_gb300.workloads import Workload, make_inputs
    from tests.gpu_util import tiny_edge_items
    ensure_library()
    H, d = 3, 128
    w = Workload("edges_d128", H, d, 300, tiny_edge_items(H), d ** -0.5, with_backward=True)
    good = zl.zl_plan_worklist(w.items, H, d, w.total_tokens)
    bad = zl.zl_plan_worklist(w.items, H, d, w.total_tokens, flags=zl.ZL_PLAN_TEST_WITHHOLD_LOAD)
    q, k, v = (x.cuda() for x in make_inputs(w.total_tokens, H, d, 0))
    bufs = zl.allocate(good, "cuda", backward=True)
    zl.forward(good, q, k, v, w.scale, bufs)
    d_o = torch.randn(bufs["o"].numel(), device="cuda").to(torch.bfloat16)
    zl.backward(bad, q, k, v, d_o, w.scale, bufs)   # same placement: the flag changes no offset
    torch.cuda.synchronize()
    assert zl.zl_get_device_status(bad) == zl.ZL_ERR_TIMEOUT
    assert zl.zl_get_device_status(bad) == 0
    assert zl.zl_get_device_status(good) == 0
    # the same context still runs a normal forward and backward correctly
    from tests.test_gpu_bwd import check_backward
    check_backward(Run(w, seed=3, backward=True))
