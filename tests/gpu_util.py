"""Shared helpers of the GPU parity tests: run a work list through the C ABI and
compare every item's outputs with the CPU float64 oracle."""
from __future__ import annotations

import numpy as np

import oracle
from coalesced_packed_attention_gb300 import zl
from coalesced_packed_attention_gb300.workloads import WorkItem, make_inputs
from tests._lib import ensure_library

# Tolerances: max |err| <= 1e-2 on O, dQ, dK, dV and <= 1e-3 on LSE (bf16 inputs, fp32
# accumulation), plus a normwise co-gate ||err||_F / ||ref||_F <= 2e-2 so that a long
# sequence, where |O| ~ 1/sqrt(L) is below the absolute gate, cannot pass with O = 0.
ATOL_O, ATOL_LSE, RTOL_F = 1e-2, 1e-3, 2e-2
# Structured inputs (Q x 4, V + 3): gradients are gated at 2.5% of max|ref|.  The row
# sums D_i = dO_i . O_i are formed from the stored bf16 O, whose rounding (2^-9 |O|,
# with |O| ~ 3 here) moves D by ~2^-9 * 3 * sqrt(d) and dS = P (dP - D) with it; with
# N(0,1) inputs the same effect stays far below the 1e-2 absolute gate.
ATOL_GRAD_STRUCTURED = 5e-2


def oracle_forward(q, k, v, item, scale, rows=None):
    """oracle.forward split over heads in threads (numpy releases the GIL inside BLAS and
    its ufuncs); the result is the same as one call over all heads."""
    import concurrent.futures as cf
    import os
    heads = list(range(item.h_lo, item.h_hi))
    if len(heads) <= 1:
        return oracle.forward(q, k, v, item, scale, rows=rows)

    def one(h):
        sub = WorkItem(item.seq_offset, item.seq_len, item.q_lo, item.q_hi, h, h + 1, item.kv_lo, item.kv_hi,
                       item.emit_lse)
        return oracle.forward(q, k, v, sub, scale, rows=rows)

    with cf.ThreadPoolExecutor(max_workers=min(len(heads), os.cpu_count() or 1)) as ex:
        parts = list(ex.map(one, heads))
    return np.concatenate([p[0] for p in parts], axis=1), np.concatenate([p[1] for p in parts], axis=0)


def oracle_backward_dq(q, k, v, do_rows, o_rows, lse_rows, item, scale, rows):
    """oracle.backward_dq split over heads in threads (same result as one call)."""
    import concurrent.futures as cf
    import os

    def one(hi):
        h = item.h_lo + hi
        sub = WorkItem(item.seq_offset, item.seq_len, item.q_lo, item.q_hi, h, h + 1, item.kv_lo, item.kv_hi,
                       item.emit_lse)
        return oracle.backward_dq(q, k, v, do_rows[:, hi:hi + 1], o_rows[:, hi:hi + 1], lse_rows[hi:hi + 1], sub,
                                  scale, rows)

    nh = item.h_hi - item.h_lo
    with cf.ThreadPoolExecutor(max_workers=max(1, min(nh, os.cpu_count() or 1))) as ex:
        parts = list(ex.map(one, range(nh)))
    return np.concatenate(parts, axis=1)


def check(name, got, ref, atol, rtol_f=RTOL_F, relative=False):
    """max |got - ref| <= atol (times max(1, max|ref|) when `relative`: the structured
    inputs have outputs well above 1, and bf16 operand rounding is relative), and the
    normwise co-gate."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(got), fin), f"{name}: non-finite pattern differs"
    if not fin.any():
        assert np.array_equal(got, ref), name
        return 0.0
    err = np.abs(got[fin] - ref[fin])
    mx = float(err.max()) if err.size else 0.0
    if relative:
        atol = atol * max(1.0, float(np.abs(ref[fin]).max()))
    assert mx <= atol, f"{name}: max abs err {mx:.3e} > {atol}"
    nrm = float(np.linalg.norm(ref[fin]))
    if nrm > 0 and rtol_f is not None:
        rel = float(np.linalg.norm(got[fin] - ref[fin])) / nrm
        assert rel <= rtol_f, f"{name}: normwise rel err {rel:.3e} > {rtol_f}"
    return mx


def sample_rows(n, seed, k=4096):
    """Seeded query-row sample: min(n, k) random rows plus both ends and every 128-row
    tile edge (the rows where a tile starts or ends)."""
    if n <= k:
        return np.arange(n)
    rng = np.random.default_rng(seed)
    r = set(rng.choice(n, k, replace=False).tolist())
    r.update([0, n - 1])
    for e in range(128, n, 128):
        r.update([e - 1, e])
    return np.array(sorted(r))


class Run:
    """One forward (+ merge, + backward) of a work list on cuda:0."""

    def __init__(self, work, seed=0, structured=False, backward=False, items=None, flags=0):
        import torch
        ensure_library()
        self.work = work
        self.items = list(items if items is not None else work.items)
        H, d, T = work.n_heads, work.head_dim, work.total_tokens
        self.scale = work.scale
        self.relative = structured
        ins = make_inputs(T, H, d, seed, with_grad_output=backward, structured=structured)
        self.q, self.k, self.v = (x.float().numpy() for x in ins[:3])
        self.plan = zl.zl_plan_worklist(self.items, H, d, T, flags)
        dev = torch.device("cuda:0")
        qd, kd, vd = (x.to(dev) for x in ins[:3])
        bufs = zl.allocate(self.plan, dev, backward=backward)
        # poison the outputs so unwritten blocks show up
        bufs["o"].fill_(float("nan"))
        bufs["o_partial"].fill_(float("nan"))
        bufs["lse"].fill_(float("nan"))
        zl.forward(self.plan, qd, kd, vd, self.scale, bufs)
        if backward:
            self.do = ins[3].float().numpy()
            dO = torch.zeros_like(bufs["o"])
            for i, it in enumerate(self.items):
                pl = self.plan.item(i)
                n = it.nq * it.nh * d
                blk = ins[3][it.seq_offset + it.q_lo: it.seq_offset + it.q_hi, it.h_lo:it.h_hi].reshape(-1)
                dO[pl.fin_out_offset: pl.fin_out_offset + n] = blk.to(dev)
            for key in ("dq", "dk", "dv"):
                bufs[key].fill_(float("nan"))
            zl.backward(self.plan, qd, kd, vd, dO, self.scale, bufs)
        torch.cuda.synchronize()
        self.status = zl.zl_get_device_status(self.plan)
        assert self.status == 0, f"device status {self.status}"
        self.bufs = {k: (b.float().cpu().numpy() if b.dtype != torch.uint8 else None) for k, b in bufs.items()}

    # ---- accessors of one item's blocks
    def own_o(self, i):
        it, pl = self.items[i], self.plan.item(i)
        d = self.work.head_dim
        arena = self.bufs["o_partial"] if it.emit_lse else self.bufs["o"]
        off = pl.item.out_offset
        return arena[off: off + it.nq * it.nh * d].reshape(it.nq, it.nh, d)

    def own_lse(self, i):
        it, pl = self.items[i], self.plan.item(i)
        off = pl.item.lse_offset
        return self.bufs["lse"][off: off + it.nq * it.nh].reshape(it.nh, it.nq)

    def final_o(self, i):
        it, pl = self.items[i], self.plan.item(i)
        d = self.work.head_dim
        return self.bufs["o"][pl.fin_out_offset: pl.fin_out_offset + it.nq * it.nh * d].reshape(it.nq, it.nh, d)

    def final_lse(self, i):
        it, pl = self.items[i], self.plan.item(i)
        return self.bufs["lse"][pl.fin_lse_offset: pl.fin_lse_offset + it.nq * it.nh].reshape(it.nh, it.nq)

    def grad(self, i, which):
        it, pl = self.items[i], self.plan.item(i)
        d = self.work.head_dim
        if which == "dq":
            return self.bufs["dq"][pl.dq_offset: pl.dq_offset + it.nq * it.nh * d].reshape(it.nq, it.nh, d)
        n = it.nkv * it.nh * d
        return self.bufs[which][pl.dkv_offset: pl.dkv_offset + n].reshape(it.nkv, it.nh, d)

    # ---- oracle comparisons
    def check_forward(self, sample=None, seed=0):
        """Every item's own output against the oracle (all rows, or sampled rows when
        `sample` is given), then every merge group against the oracle merge."""
        res = {}
        for i, it in enumerate(self.items):
            # members of one merge group share (sequence, rows, heads): same sample
            key = (it.seq_offset, it.q_lo, it.q_hi, it.h_lo, it.h_hi)
            rows = None if sample is None else sample_rows(it.nq, seed + hash(key) % 100003, sample)
            rel = None if rows is None else rows
            O_ref, L_ref = oracle_forward(self.q, self.k, self.v, it, self.scale,
                                          rows=None if rows is None else it.q_lo + rows)
            self._ref_cache = getattr(self, "_ref_cache", {})
            self._ref_cache[i] = (rows, O_ref, L_ref)
            if self.plan.item(i).item.out_offset < 0:
                continue  # member of a k-split group fused into the forward: no own blocks
            O, L = self.own_o(i), self.own_lse(i)
            if rel is not None:
                O, L = O[rel], L[:, rel]
            res[i] = (check(f"item{i}.O", O, O_ref, ATOL_O, relative=self.relative),
                      check(f"item{i}.LSE", L, L_ref, ATOL_LSE, relative=self.relative))
        for g in range(self.plan.n_groups):
            members, _, _ = self.plan.group(g)
            rows = self._ref_cache[members[0]][0]
            O_ref, L_ref = oracle.merge([self._ref_cache[m][1:] for m in members])
            O, L = self.final_o(members[0]), self.final_lse(members[0])
            if rows is not None:
                O, L = O[rows], L[:, rows]
            res[f"g{g}"] = (check(f"group{g}.O", O, O_ref, ATOL_O, relative=self.relative),
                            check(f"group{g}.LSE", L, L_ref, ATOL_LSE, relative=self.relative))
        return res


def tiny_edge_items(H, L=300):
    """Degenerate and ragged shards of one L-token sequence at offset 0."""
    return [
        WorkItem(0, L, 0, L, 0, H, 0, L, 0),          # whole
        WorkItem(0, L, 5, 6, 0, H, 0, L, 0),          # one query row
        WorkItem(0, L, 0, L, 1, 2, 7, 8, 0),          # one KV row, one head
        WorkItem(0, L, 3, 250, 0, H, 0, 0, 0),        # empty KV chunk -> O = 0, LSE = -inf
        WorkItem(0, L, 0, L, 0, H, 0, 129, 1),        # k split 3 ways, unaligned,
        WorkItem(0, L, 0, L, 0, H, 129, 129, 1),      # ... one chunk empty
        WorkItem(0, L, 0, L, 0, H, 129, L, 1),
        WorkItem(0, L, 100, 100, 0, H, 0, L, 0),      # empty query range (no tiles)
    ]
