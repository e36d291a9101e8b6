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


def test_training_list_scaled_all_rows_d64():
    """The same mix of item kinds (whole images; q, h and k shards of the video, merged)
    at head dim 64, forward and backward on all rows."""
    import dataclasses
    w = dataclasses.replace(scaled(config_training(), 12), head_dim=64, scale=64 ** -0.5)
    r = Run(w, seed=16, backward=True)
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


@pytest.mark.parametrize("name", ["worked_example.json", "worked_example_scale2.json"])
def test_golden_worked_example_on_the_gpu(name):
    """The hand-worked examples of tests/golden (one query over three keys, head dim 2,
    score scale 1 and 2) through the CUDA forward and backward: the head dim is padded
    with zeros to 64, which leaves every score, weight and LSE unchanged and the padded
    output columns exactly zero.  Gates: the bf16 rounding of the stored O and of the
    kernel's P and dS (at most a few 1e-3 on these O(0.1-1) values)."""
    import json
    import math
    import os
    import torch
    from coalesced_packed_attention_gb300.workloads import WorkItem
    with open(os.path.join(os.path.dirname(__file__), "golden", name)) as f:
        g = json.load(f)
    ns = {"e": math.e, "log": math.log, "exp": math.exp}
    ev = lambda a: np.array([[eval(x, {}, ns) for x in r] for r in a])  # noqa: E731
    T, d = 3, 64

    def pad(rows):
        x = torch.zeros(T, 1, d)
        x[:len(rows), 0, :2] = torch.tensor(rows, dtype=torch.float32)
        return x.to(torch.bfloat16)

    q, k, v, do = pad(g["q"]), pad(g["k"]), pad(g["v"]), pad(g["do"])
    w = Workload(f"golden_{name}", 1, d, T, [WorkItem(0, T, 0, 1, 0, 1, 0, 3, 0)], g["scale"], with_backward=True)
    r = Run(w, backward=True, inputs=(q, k, v, do))
    O, L = r.own_o(0)[:, 0, :], r.own_lse(0)[0]
    np.testing.assert_allclose(L, [eval(x, {}, ns) for x in g["expected"]["lse"]], atol=1e-5)
    np.testing.assert_allclose(O[:, :2], ev(g["expected"]["o"]), atol=5e-3)
    dq, dk, dv = (r.grad(0, x)[:, 0, :] for x in ("dq", "dk", "dv"))
    np.testing.assert_allclose(dq[:, :2], ev(g["expected"]["dq"]), atol=5e-3)
    np.testing.assert_allclose(dk[:, :2], ev(g["expected"]["dk"]), atol=5e-3)
    np.testing.assert_allclose(dv[:, :2], ev(g["expected"]["dv"]), atol=5e-3)
    for x in (O, dq, dk, dv):
        assert np.all(x[:, 2:] == 0.0)


def test_closed_forms_on_the_gpu():
    """Closed forms of exact attention through the CUDA forward and backward, with no
    oracle in between.  Three sequences, d = 128, 2 heads:
    A (300 tokens, Q = 0): P is uniform, so O = mean of V over the chunk, LSE = ln 300,
      dK = 0 exactly (every term carries a Q row) and every dV row = (sum of dO) / 300;
    B (a single key, KV [7, 8)): P = 1, so O = V_7 exactly, LSE = scale q.k_7, dS = 0
      (dQ = dK = 0 up to rounding) and dV_7 = sum of dO over the rows;
    C (V = 0.5 everywhere): O = 0.5, dS = 0 (dP = D), so dQ = dK = 0 up to rounding."""
    import torch
    from coalesced_packed_attention_gb300.workloads import WorkItem, make_inputs
    H, d = 2, 128
    A, B, C = (0, 300), (300, 256), (556, 256)
    T = 812
    q, k, v, do = make_inputs(T, H, d, seed=11, with_grad_output=True)
    q[A[0]:A[0] + A[1]] = 0
    v[C[0]:C[0] + C[1]] = 0.5
    items = [WorkItem(A[0], A[1], 0, A[1], 0, H, 0, A[1], 0),
             WorkItem(B[0], B[1], 0, B[1], 0, H, 7, 8, 0),
             WorkItem(C[0], C[1], 0, C[1], 0, H, 0, C[1], 0)]
    scale = d ** -0.5
    w = Workload("closed_forms", H, d, T, items, scale, with_backward=True)
    r = Run(w, backward=True, inputs=(q, k, v, do))
    qf, kf, vf, dof = (x.double().numpy() for x in (q, k, v, do))
    # A: uniform weights
    sa = slice(A[0], A[0] + A[1])
    np.testing.assert_allclose(r.own_lse(0), np.log(A[1]), atol=1e-5)
    np.testing.assert_allclose(r.own_o(0), np.broadcast_to(vf[sa].mean(axis=0), (A[1], H, d)), atol=2e-3)
    assert np.all(r.grad(0, "dk") == 0.0)
    np.testing.assert_allclose(r.grad(0, "dv"), np.broadcast_to(dof[sa].sum(axis=0) / A[1], (A[1], H, d)),
                               atol=2e-3)
    # B: one key
    sb = slice(B[0], B[0] + B[1])
    assert np.array_equal(r.own_o(1), np.broadcast_to(vf[B[0] + 7], (B[1], H, d)))
    s7 = scale * np.einsum("rhd,hd->hr", qf[sb], kf[B[0] + 7])
    np.testing.assert_allclose(r.own_lse(1), s7, rtol=1e-5, atol=1e-5)
    np.testing.assert_allclose(r.grad(1, "dq"), 0.0, atol=1e-3)
    np.testing.assert_allclose(r.grad(1, "dk"), 0.0, atol=1e-3)
    np.testing.assert_allclose(r.grad(1, "dv")[0], dof[sb].sum(axis=0), rtol=1e-4, atol=1e-3)
    # C: constant values
    # (the stored bf16 O may round 0.5 - 1e-3 down one step, which leaves dP - D at a
    # few 1e-3 of sum |dO| and dQ, dK at ~1e-4)
    np.testing.assert_allclose(r.own_o(2), 0.5, atol=2e-3)
    np.testing.assert_allclose(r.grad(2, "dq"), 0.0, atol=5e-3)
    np.testing.assert_allclose(r.grad(2, "dk"), 0.0, atol=5e-3)


def test_k_split_gradients_assemble_the_unsplit_item():
    """A k split of theta (pith.science review, "What carries the argument"): each chunk
    writes its contribution to dQ and the final dK, dV of its own KV rows, all with the
    group's merged LSE and O.  So the chunks' dQ sum to the unsplit item's dQ, and their
    dK, dV are the unsplit item's rows of their chunks, up to the bf16 rounding of the
    stored O that enters D (the merged O and the unsplit item's O may differ by one bf16
    step): a few 1e-3 at most, where a chunk that used its own LSE, or dropped one, would
    be off by tens of percent."""
    from coalesced_packed_attention_gb300.workloads import WorkItem
    H, d, L = 3, 128, 700
    cuts = [0, 130, 400, L]  # three uneven, unaligned chunks
    items = [WorkItem(0, L, 0, L, 0, H, 0, L, 0)]
    items += [WorkItem(0, L, 0, L, 0, H, a, b, 1) for a, b in zip(cuts, cuts[1:])]
    w = Workload("k_split_assembly", H, d, L, items, d ** -0.5, with_backward=True)
    r = Run(w, seed=17, backward=True)
    def close(got, ref):
        np.testing.assert_allclose(got, ref, rtol=0, atol=5e-3)
        assert np.linalg.norm(got - ref) <= 1e-2 * np.linalg.norm(ref)

    close(sum(r.grad(i, "dq") for i in range(1, len(items))), r.grad(0, "dq"))
    for i, (a, b) in enumerate(zip(cuts, cuts[1:]), start=1):
        for name in ("dk", "dv"):
            close(r.grad(i, name), r.grad(0, name)[a:b])


def test_q_split_partial_gradients_sum_to_the_unsplit_item():
    """A q split of theta: each shard writes dQ for its own rows and partial dK, dV (its
    rows' contribution, which a distributed run would reduce).  The shards' O and LSE are
    the whole item's bit for bit, so their partial dK, dV sum to the whole item's and their
    dQ rows are the whole item's, up to fp32 summation order only."""
    from coalesced_packed_attention_gb300.workloads import WorkItem
    H, d, L = 3, 128, 1000
    cuts = [0, 300, 777, L]
    items = [WorkItem(0, L, 0, L, 0, H, 0, L, 0)]
    items += [WorkItem(0, L, a, b, 0, H, 0, L, 0) for a, b in zip(cuts, cuts[1:])]
    w = Workload("q_split_assembly", H, d, L, items, d ** -0.5, with_backward=True)
    r = Run(w, seed=18, backward=True)
    for name in ("dk", "dv"):
        np.testing.assert_allclose(sum(r.grad(i, name) for i in range(1, len(items))), r.grad(0, name),
                                   rtol=1e-5, atol=1e-5)
    for i, (a, b) in enumerate(zip(cuts, cuts[1:]), start=1):
        np.testing.assert_allclose(r.grad(i, "dq"), r.grad(0, "dq")[a:b], rtol=1e-5, atol=1e-5)
