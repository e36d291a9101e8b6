"""Pins of the CPU float64 oracle against things other than itself.

Each test would catch a plausible mistake in the oracle: a dropped term, a wrong sign,
a wrong index or a transposed operand.  Sources:
  * brute force (scalar Python loops) on tiny inputs,
  * closed forms (single key, zero query, constant values, one dominant logit,
    hand-worked examples in tests/golden/ with score scales 1 and 2),
  * invariants (rows of P sum to 1, merge of any k split equals the unsplit result,
    q and h shards tile the whole output, KV permutation invariance,
    sum_j dS_ij = 0),
  * central finite differences of <dO, O> for every item kind,
  * torch.nn.functional.scaled_dot_product_attention in float64 on the CPU.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from coalesced_packed_attention_gb300.workloads import WorkItem, config_tiny, merge_groups

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rnd(T, H, d, seed, n=3):
    rng = np.random.default_rng(seed)
    return [rng.standard_normal((T, H, d)) for _ in range(n)]


def item(off, L, q=None, h=(0, 2), kv=None, e=0):
    q = q or (0, L)
    kv = kv or (0, L)
    return WorkItem(off, L, q[0], q[1], h[0], h[1], kv[0], kv[1], e)


# ---------------------------------------------------------------- brute force
def test_forward_matches_brute_force_tiny_mixed():
    # a scaled-down copy of the tiny mixed list: whole 6, 10, 25 and a 40-token
    # sequence as two k chunks (uneven, unaligned cut at 17)
    T, H, d = 81, 2, 8
    q, k, v = rnd(T, H, d, 1)
    items = [item(0, 6, h=(0, 2)), item(6, 10, h=(0, 2)), item(16, 25, h=(0, 2)),
             item(41, 40, kv=(0, 17), e=1), item(41, 40, kv=(17, 40), e=1),
             item(41, 40, q=(3, 31), h=(1, 2), kv=(5, 33))]
    scale = 1 / math.sqrt(d)
    for it in items:
        O, L = oracle.forward(q, k, v, it, scale)
        Ob, Lb = oracle.brute_force_forward(q, k, v, it, scale)
        np.testing.assert_allclose(O, Ob, rtol=0, atol=1e-12)
        np.testing.assert_allclose(L, Lb, rtol=0, atol=1e-12)
    # the merge of the two chunks equals the brute-force unsplit sequence
    parts = [oracle.forward(q, k, v, it, scale) for it in items[3:5]]
    O, L = oracle.merge(parts)
    Ob, Lb = oracle.brute_force_forward(q, k, v, item(41, 40), scale)
    np.testing.assert_allclose(O, Ob, rtol=0, atol=1e-12)
    np.testing.assert_allclose(L, Lb, rtol=0, atol=1e-12)


# ---------------------------------------------------------------- closed forms
@pytest.mark.parametrize("name", ["worked_example.json", "worked_example_scale2.json"])
def test_golden_worked_example(name):
    with open(os.path.join(GOLDEN, name)) as f:
        g = json.load(f)
    ns = {"e": math.e, "log": math.log, "exp": math.exp}
    ev = lambda a: np.array([[eval(x, {}, ns) for x in r] for r in a])  # noqa: E731
    q = np.array(g["q"])[:, None, :]
    k = np.array(g["k"])[:, None, :]
    v = np.array(g["v"])[:, None, :]
    do = np.array(g["do"])[:, None, :]
    # query and keys live in one packed stream: token 0 is the query's sequence row 0
    T = 3
    Q = np.zeros((T, 1, 2)); Q[0] = q[0]
    it = WorkItem(0, T, 0, 1, 0, 1, 0, 3, 0)
    O, L = oracle.forward(Q, k, v, it, g["scale"])
    np.testing.assert_allclose(L[0], [eval(x, {}, ns) for x in g["expected"]["lse"]], atol=1e-15)
    np.testing.assert_allclose(O[:, 0, :], ev(g["expected"]["o"]), atol=1e-15)
    dQ = oracle.backward_dq(Q, k, v, do, O, L, it, g["scale"], rows=[0])
    dK, dV = oracle.backward_dkdv(Q, k, v, do, O, L, it, g["scale"])
    np.testing.assert_allclose(dQ[:, 0, :], ev(g["expected"]["dq"]), atol=1e-15)
    np.testing.assert_allclose(dK[:, 0, :], ev(g["expected"]["dk"]), atol=1e-15)
    np.testing.assert_allclose(dV[:, 0, :], ev(g["expected"]["dv"]), atol=1e-15)


def test_single_key_gives_that_value():
    q, k, v = rnd(20, 2, 16, 2)
    it = item(3, 12, kv=(7, 8))
    O, L = oracle.forward(q, k, v, it, 0.3)
    for hi in range(2):
        np.testing.assert_array_equal(O[:, hi, :], np.broadcast_to(v[3 + 7, hi], O[:, hi, :].shape))
        s = 0.3 * (q[3:15, hi, :] @ k[10, hi, :])
        np.testing.assert_allclose(L[hi], s, rtol=0, atol=1e-13)


def test_zero_query_gives_mean_and_log_count():
    q, k, v = rnd(40, 2, 16, 3)
    q[:] = 0.0
    it = item(5, 30, kv=(4, 27))
    O, L = oracle.forward(q, k, v, it, 0.125)
    mean = v[5 + 4:5 + 27].mean(axis=0)
    for i in range(30):
        np.testing.assert_allclose(O[i], mean, rtol=0, atol=1e-13)
    np.testing.assert_allclose(L, math.log(23), rtol=0, atol=1e-13)


def test_constant_values():
    q, k, v = rnd(33, 2, 8, 4)
    v[:] = -1.75
    O, _ = oracle.forward(q, k, v, item(0, 33), 0.9)
    np.testing.assert_allclose(O, -1.75, rtol=0, atol=1e-13)


def test_dominant_logit_selects_its_value():
    # one key aligned with every query, 50 nats above the others
    T, d = 16, 4
    q = np.zeros((T, 1, d)); k = np.zeros((T, 1, d))
    v = np.random.default_rng(5).standard_normal((T, 1, d))
    q[:, 0, 0] = 1.0
    k[9, 0, 0] = 50.0
    it = WorkItem(0, T, 0, T, 0, 1, 0, T, 0)
    O, L = oracle.forward(q, k, v, it, 1.0)
    bound = (T - 1) * math.exp(-50) * np.abs(v - v[9]).max()
    assert np.abs(O[:, 0, :] - v[9, 0]).max() <= bound + 1e-300
    np.testing.assert_allclose(L, 50.0 + math.log1p((T - 1) * math.exp(-50)), atol=1e-13)


# ---------------------------------------------------------------- invariants
def test_probability_rows_sum_to_one():
    q, k, v = rnd(300, 3, 32, 6)
    q *= 3.0
    it = item(17, 250, q=(11, 230), h=(1, 3), kv=(40, 250))
    for h in (1, 2):
        P = oracle.probabilities(q, k, it, h, 0.2)
        assert P.min() >= 0.0
        np.testing.assert_allclose(P.sum(axis=1), 1.0, rtol=0, atol=1e-12)


@pytest.mark.parametrize("cuts", [[0, 128, 256], [0, 37, 38, 200, 256],
                                  [0, 32, 64, 96, 128, 160, 192, 224, 256],
                                  [0, 100, 100, 256], [0, 1, 255, 256]])
def test_merge_of_any_k_split_equals_unsplit(cuts):
    q, k, v = rnd(300, 2, 16, 7)
    q *= 2.0
    base = item(20, 256)
    O, L = oracle.forward(q, k, v, base, 0.25)
    parts = [oracle.forward(q, k, v, item(20, 256, kv=(a, b), e=1), 0.25)
             for a, b in zip(cuts[:-1], cuts[1:])]
    Om, Lm = oracle.merge(parts)
    np.testing.assert_allclose(Om, O, rtol=0, atol=1e-12)
    np.testing.assert_allclose(Lm, L, rtol=0, atol=1e-12)


def test_merge_of_all_empty_chunks_is_zero_and_minus_inf():
    q, k, v = rnd(64, 2, 8, 8)
    parts = [oracle.forward(q, k, v, item(0, 64, kv=(5, 5), e=1), 0.5) for _ in range(3)]
    O, L = oracle.merge(parts)
    assert np.all(O == 0.0) and np.all(np.isneginf(L))


def test_merge_is_order_independent_and_weights_chunks():
    # swapping the chunk order changes nothing; dropping a chunk changes O
    q, k, v = rnd(128, 2, 8, 9)
    p = [oracle.forward(q, k, v, item(0, 128, kv=(a, b), e=1), 0.4)
         for a, b in [(0, 50), (50, 51), (51, 128)]]
    O1, L1 = oracle.merge(p)
    O2, L2 = oracle.merge(p[::-1])
    np.testing.assert_allclose(O1, O2, atol=1e-14)
    np.testing.assert_allclose(L1, L2, atol=1e-14)
    O3, _ = oracle.merge(p[:2])
    assert np.abs(O3 - O1).max() > 1e-3


def test_q_and_h_shards_tile_the_whole_output():
    # rows and heads are independent, so the shards reproduce the whole output; BLAS
    # picks its summation blocking by matrix shape, hence 1e-14 rather than bit-exact
    # (a wrong row, head or range would be off by O(0.1))
    q, k, v = rnd(400, 4, 16, 10)
    full = item(10, 384, h=(0, 4))
    O, L = oracle.forward(q, k, v, full, 0.25)
    # q split into three uneven row ranges
    for a, b in [(0, 100), (100, 101), (101, 384)]:
        Os, Ls = oracle.forward(q, k, v, item(10, 384, q=(a, b), h=(0, 4)), 0.25)
        np.testing.assert_allclose(Os, O[a:b], rtol=0, atol=1e-14)
        np.testing.assert_allclose(Ls, L[:, a:b], rtol=0, atol=1e-14)
    # h split into two head subsets
    for a, b in [(0, 1), (1, 4)]:
        Os, Ls = oracle.forward(q, k, v, item(10, 384, h=(a, b)), 0.25)
        np.testing.assert_allclose(Os, O[:, a:b], rtol=0, atol=1e-14)
        np.testing.assert_allclose(Ls, L[a:b], rtol=0, atol=1e-14)


def test_kv_permutation_invariance():
    q, k, v = rnd(200, 2, 16, 11)
    it = item(0, 200, kv=(30, 170))
    O, L = oracle.forward(q, k, v, it, 0.25)
    perm = np.random.default_rng(0).permutation(np.arange(30, 170))
    k2, v2 = k.copy(), v.copy()
    k2[30:170] = k[perm]
    v2[30:170] = v[perm]
    O2, L2 = oracle.forward(q, k2, v2, it, 0.25)
    np.testing.assert_allclose(O2, O, rtol=0, atol=1e-12)
    np.testing.assert_allclose(L2, L, rtol=0, atol=1e-12)


def test_gradient_sums_over_whole_item():
    # for a whole item sum_j dS_ij = 0, hence sum_j dK_j = 0 and sum_j dV_j = sum_i dO_i
    q, k, v, do = rnd(160, 2, 16, 12, n=4)
    it = item(0, 160)
    O, L = oracle.forward(q, k, v, it, 0.25)
    dK, dV = oracle.backward_dkdv(q, k, v, do, O, L, it, 0.25)
    np.testing.assert_allclose(dK.sum(axis=0), 0.0, atol=1e-11)
    np.testing.assert_allclose(dV.sum(axis=0), do[:160].sum(axis=0), atol=1e-11)


# ---------------------------------------------------------------- finite differences
def _loss(q, k, v, do, items, groups, scale):
    """<dO, O> summed over the given items' outputs; grouped items are merged first."""
    tot = 0.0
    done = set()
    for g in groups:
        parts = [oracle.forward(q, k, v, items[i], scale) for i in g]
        O, _ = oracle.merge(parts)
        it = items[g[0]]
        dO = do[it.seq_offset + it.q_lo: it.seq_offset + it.q_hi, it.h_lo:it.h_hi]
        tot += float((dO * O).sum())
        done.update(g)
    for i, it in enumerate(items):
        if i in done:
            continue
        O, _ = oracle.forward(q, k, v, it, scale)
        dO = do[it.seq_offset + it.q_lo: it.seq_offset + it.q_hi, it.h_lo:it.h_hi]
        tot += float((dO * O).sum())
    return tot


def _analytic(q, k, v, do, items, groups, scale):
    """Gradient of _loss assembled from the per-item backward (global O/LSE for groups)."""
    gq, gk, gv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    final = {}
    for g in groups:
        O, L = oracle.merge([oracle.forward(q, k, v, items[i], scale) for i in g])
        for i in g:
            final[i] = (O, L)
    for i, it in enumerate(items):
        O, L = final.get(i) or oracle.forward(q, k, v, it, scale)
        s, rows = it.seq_offset, np.arange(it.q_lo, it.q_hi)
        dO = do[s + it.q_lo: s + it.q_hi, it.h_lo:it.h_hi]
        dQ = oracle.backward_dq(q, k, v, dO, O, L, it, scale, rows)
        dK, dV = oracle.backward_dkdv(q, k, v, dO, O, L, it, scale)
        gq[s + it.q_lo: s + it.q_hi, it.h_lo:it.h_hi] += dQ
        gk[s + it.kv_lo: s + it.kv_hi, it.h_lo:it.h_hi] += dK
        gv[s + it.kv_lo: s + it.kv_hi, it.h_lo:it.h_hi] += dV
    return gq, gk, gv


@pytest.mark.parametrize("kind", ["whole", "qsplit", "hsplit", "ksplit", "mixed"])
def test_gradients_match_central_differences(kind):
    T, H, d = 48, 3, 8
    q, k, v, do = rnd(T, H, d, 13, n=4)
    if kind == "whole":
        items = [item(4, 40, h=(0, 3))]
    elif kind == "qsplit":
        items = [item(4, 40, q=(5, 23), h=(0, 3))]
    elif kind == "hsplit":
        items = [item(4, 40, h=(1, 3))]
    elif kind == "ksplit":
        items = [item(4, 40, h=(0, 3), kv=(0, 13), e=1), item(4, 40, h=(0, 3), kv=(13, 40), e=1)]
    else:
        items = [item(0, 4, h=(0, 3)), item(4, 40, q=(0, 9), h=(0, 3)),
                 item(4, 40, h=(0, 2)), item(4, 40, h=(2, 3), kv=(20, 40), e=1),
                 item(4, 40, h=(2, 3), kv=(0, 20), e=1)]
    groups = merge_groups(items)
    scale = 0.35
    grads = _analytic(q, k, v, do, items, groups, scale)
    rng = np.random.default_rng(99)
    eps = 1e-6
    for which in range(3):
        X = [q, k, v][which]
        Dx = rng.standard_normal(X.shape)
        args_p = [q.copy(), k.copy(), v.copy()]
        args_m = [q.copy(), k.copy(), v.copy()]
        args_p[which] = X + eps * Dx
        args_m[which] = X - eps * Dx
        fd = (_loss(*args_p, do, items, groups, scale) - _loss(*args_m, do, items, groups, scale)) / (2 * eps)
        an = float((grads[which] * Dx).sum())
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (kind, which, fd, an)


def test_ksplit_gradients_sum_to_unsplit():
    # partial dQ of the chunks sums to the unsplit dQ; chunk dK/dV are the unsplit rows
    T, H, d = 90, 2, 16
    q, k, v, do = rnd(T, H, d, 14, n=4)
    full = item(0, 90)
    items = [item(0, 90, kv=(0, 33), e=1), item(0, 90, kv=(33, 90), e=1)]
    gq, gk, gv = _analytic(q, k, v, do, items, [[0, 1]], 0.25)
    fq, fk, fv = _analytic(q, k, v, do, [full], [], 0.25)
    np.testing.assert_allclose(gq, fq, atol=1e-12)
    np.testing.assert_allclose(gk, fk, atol=1e-12)
    np.testing.assert_allclose(gv, fv, atol=1e-12)


# ---------------------------------------------------------------- library cross-check
def test_matches_torch_sdpa_float64_with_autograd():
    torch = pytest.importorskip("torch")
    import torch.nn.functional as F
    w = config_tiny()
    # the first three (whole) sequences of the tiny mixed list, full size
    T = 420
    q, k, v, do = rnd(T, w.n_heads, w.head_dim, 15, n=4)
    for it in w.items[:3]:
        s, L = it.seq_offset, it.seq_len
        tq, tk, tv = (torch.tensor(x[s:s + L]).permute(1, 0, 2).requires_grad_(True) for x in (q, k, v))
        out = F.scaled_dot_product_attention(tq[None], tk[None], tv[None], scale=w.scale)[0]
        tdo = torch.tensor(do[s:s + L]).permute(1, 0, 2)
        (out * tdo).sum().backward()
        O, LSE = oracle.forward(q, k, v, it, w.scale)
        np.testing.assert_allclose(O, out.detach().permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)
        rows = np.arange(L)
        dQ = oracle.backward_dq(q, k, v, do[s:s + L], O, LSE, it, w.scale, rows)
        dK, dV = oracle.backward_dkdv(q, k, v, do[s:s + L], O, LSE, it, w.scale)
        np.testing.assert_allclose(dQ, tq.grad.permute(1, 0, 2).numpy(), rtol=0, atol=1e-11)
        np.testing.assert_allclose(dK, tk.grad.permute(1, 0, 2).numpy(), rtol=0, atol=1e-11)
        np.testing.assert_allclose(dV, tv.grad.permute(1, 0, 2).numpy(), rtol=0, atol=1e-11)


def test_sampled_rows_equal_full_rows():
    # the row-sampled forward/backward used for large lists equals the full computation
    q, k, v, do = rnd(300, 2, 16, 16, n=4)
    it = item(0, 300)
    O, L = oracle.forward(q, k, v, it, 0.25)
    rows = np.array([0, 5, 127, 128, 299])
    Os, Ls = oracle.forward(q, k, v, it, 0.25, rows=rows)
    np.testing.assert_allclose(Os, O[rows], atol=1e-14)
    np.testing.assert_allclose(Ls, L[:, rows], atol=1e-14)
    dQ = oracle.backward_dq(q, k, v, do[:300], O, L, it, 0.25, np.arange(300))
    dQs = oracle.backward_dq(q, k, v, do[rows], O[rows], L[:, rows], it, 0.25, rows)
    np.testing.assert_allclose(dQs, dQ[rows], atol=1e-13)
    dK, dV = oracle.backward_dkdv(q, k, v, do[:300], O, L, it, 0.25)
    dKs, dVs = oracle.backward_dkdv(q, k, v, do[:300], O, L, it, 0.25, kv_rows=rows)
    np.testing.assert_allclose(dKs, dK[rows], atol=1e-13)
    np.testing.assert_allclose(dVs, dV[rows], atol=1e-13)
