"""GPU parity of the backward launch (row sums D, tcgen05 backward, dQ finalisation)
against the CPU float64 oracle, every item kind: whole, q-split (partial dK/dV),
h-split, k-split with the merged global LSE (partial dQ)."""
import numpy as np
import pytest

import oracle
from coalesced_packed_attention_gb300.workloads import Workload, config_training, merge_groups, scaled
from tests.gpu_util import ATOL_GRAD_STRUCTURED, ATOL_O, Run, check, sample_rows, tiny_edge_items

pytestmark = pytest.mark.gpu


def final_reference(r, rows_of=None):
    """Oracle final O and LSE (all rows) of every item: its own, or its group's merge."""
    fin = {}
    parts = {}
    for i, it in enumerate(r.items):
        parts[i] = oracle.forward(r.q, r.k, r.v, it, r.scale)
    for g in merge_groups(r.items):
        m = oracle.merge([parts[i] for i in g])
        for i in g:
            fin[i] = m
    for i in range(len(r.items)):
        fin.setdefault(i, parts[i])
    return fin


def check_backward(r, kv_sample=None, q_sample=None, seed=0):
    fin = final_reference(r)
    tol = ATOL_GRAD_STRUCTURED if r.relative else ATOL_O
    for i, it in enumerate(r.items):
        if it.nq == 0 or it.nh == 0:
            continue
        O, L = fin[i]
        s = it.seq_offset
        do_all = r.do[s + it.q_lo: s + it.q_hi, it.h_lo:it.h_hi]
        rows = np.arange(it.nq) if q_sample is None else sample_rows(it.nq, seed + i, q_sample)
        dQ_ref = oracle.backward_dq(r.q, r.k, r.v, do_all[rows], O[rows], L[:, rows], it, r.scale, it.q_lo + rows)
        check(f"item{i}.dQ", r.grad(i, "dq")[rows], dQ_ref, tol, relative=r.relative)
        if it.nkv == 0:
            continue
        kv = np.arange(it.nkv) if kv_sample is None else sample_rows(it.nkv, seed + 7 * i, kv_sample)
        dK_ref, dV_ref = oracle.backward_dkdv(r.q, r.k, r.v, do_all, O, L, it, r.scale, it.kv_lo + kv)
        check(f"item{i}.dK", r.grad(i, "dk")[kv], dK_ref, tol, relative=r.relative)
        check(f"item{i}.dV", r.grad(i, "dv")[kv], dV_ref, tol, relative=r.relative)


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
