"""The forward entry point that allocates no device memory.

Some callers cannot call cudaMalloc: code that runs inside a host framework owning all
device memory through its own pool, or an embedding that forbids device allocation after
start-up.  zl_coalesced_attn_fwd_noalloc serves them: it takes the work list itself
(no zl_plan, whose creation allocates), keeps its tables in a fixed scratch array
compiled into the library, and launches the same forward kernel.  This test calls it
through the C ABI twice in a row and checks each result against zl_coalesced_attn_fwd
on the same inputs, with the tolerances of the other parity tests; on the tiny list it
also checks the result against the CPU float64 oracle, and after every call it reads the
array's status word through zl_noalloc_get_device_status.  It lives in a file of its own,
collected last.
"""
import ctypes

import numpy as np
import pytest

from coalesced_packed_attention_gb300 import zl
from coalesced_packed_attention_gb300.workloads import config_mixed, config_tiny, make_inputs, scaled
from tests._lib import ensure_library
from tests.gpu_util import ATOL_LSE, ATOL_O, check, oracle_forward

pytestmark = pytest.mark.gpu


def _entry(lib):
    fn = lib.zl_coalesced_attn_fwd_noalloc
    P = ctypes.c_void_p
    fn.restype = ctypes.c_int32
    fn.argtypes = [ctypes.POINTER(zl.zl_work_item), ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int64,
                   P, P, P, P, P, P, ctypes.c_float, P]
    return fn


def _status_entry(lib):
    fn = lib.zl_noalloc_get_device_status
    fn.restype = ctypes.c_int32
    fn.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32)]
    return fn


def _device_status(lib, stream):
    word = ctypes.c_int32(-1)
    st = _status_entry(lib)(stream, ctypes.byref(word))
    assert st == zl.ZL_OK, zl.status_string(st)
    return word.value


def _blocks(plan, items, bufs, d):
    """Every item's own O and LSE block, and every merge group's, as numpy arrays."""
    out = []
    o, op, lse = (bufs[k].float().cpu().numpy() for k in ("o", "o_partial", "lse"))
    for i, it in enumerate(items):
        r = plan.item(i).item
        n = it.nq * it.nh
        arena = op if it.emit_lse else o
        out.append(arena[r.out_offset: r.out_offset + n * d])
        out.append(lse[r.lse_offset: r.lse_offset + n])
    return out


def test_noalloc_status_query_before_any_forward():
    # the query sets up the array's address itself when it is the first call on a device
    import torch
    lib = ensure_library()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert _device_status(lib, stream) == zl.ZL_OK
    assert _status_entry(lib)(stream, None) == zl.ZL_ERR_INVALID_ARG


@pytest.mark.parametrize("make", [config_tiny, lambda: scaled(config_mixed(), 12)], ids=["tiny", "mixed_div12"])
def test_noalloc_forward_matches_the_plan_forward_on_two_calls(make):
    import torch
    lib = ensure_library()
    fn = _entry(lib)
    w = make()
    H, d, T = w.n_heads, w.head_dim, w.total_tokens
    q, k, v = (x.cuda() for x in make_inputs(T, H, d, seed=7))
    plan = zl.zl_plan_worklist(w.items, H, d, T)
    ref = zl.allocate(plan, "cuda")
    zl.zl_coalesced_attn_fwd(plan, q, k, v, ref["o"], ref["o_partial"], ref["lse"], w.scale)
    torch.cuda.synchronize()
    ref_blocks = _blocks(plan, w.items, ref, d)
    items = zl._to_c_items(w.items)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        out = zl.allocate(plan, "cuda")   # the caller owns the outputs; same layout as the plan's
        for key in ("o", "o_partial", "lse"):
            out[key].fill_(float("nan"))
        st = fn(items, len(w.items), H, d, T, q.data_ptr(), k.data_ptr(), v.data_ptr(), out["o"].data_ptr(),
                out["o_partial"].data_ptr(), out["lse"].data_ptr(), ctypes.c_float(w.scale), stream)
        assert st == zl.ZL_OK, zl.status_string(st)
        assert _device_status(lib, stream) == zl.ZL_OK  # no bounded wait gave up
        torch.cuda.synchronize()
        got = _blocks(plan, w.items, out, d)
        for j, (g, r) in enumerate(zip(got, ref_blocks)):
            check(f"call{call}.block{j}", g, r, ATOL_LSE if j % 2 else ATOL_O)
        if w.name.startswith("tiny"):
            # and against the oracle: every item's own O / LSE (k-split chunks: partials)
            qn, kn, vn = (x.float().cpu().numpy() for x in (q, k, v))
            for i, it in enumerate(w.items):
                O_ref, L_ref = oracle_forward(qn, kn, vn, it, w.scale)
                check(f"call{call}.item{i}.O", got[2 * i].reshape(O_ref.shape), O_ref, ATOL_O)
                check(f"call{call}.item{i}.LSE", got[2 * i + 1].reshape(L_ref.shape), L_ref, ATOL_LSE)


def test_noalloc_rejects_a_list_beyond_its_scratch():
    lib = ensure_library()
    fn = _entry(lib)
    # 600 000 one-token sequences of one head: far more tiles than the scratch holds
    from coalesced_packed_attention_gb300.workloads import WorkItem
    n = 600_000
    items = (zl.zl_work_item * n)()
    for i in range(n):
        items[i] = zl.zl_work_item(i, 1, 0, 1, 0, 1, 0, 1, 0, -1, -1)
    st = fn(items, n, 1, 64, n, 16, 16, 16, 16, 16, 16, ctypes.c_float(1.0), None)
    assert st == zl.ZL_ERR_INVALID_ARG
