"""Failure detection without a GPU fault: a plan built with the test flag announces
its first K tile but never issues the copy, so the forward's bounded mbarrier wait runs
out; the kernel records ZL_ERR_TIMEOUT in the plan's status word, leaves its loops,
frees TMEM and returns, and the context stays usable for the next launch."""
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
