"""Plain CPU float64 oracle for the coalesced attention engine.

TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and bench.py's
cpu_baseline leg may import this module.  It shares no code with the CUDA path and
imports nothing from the package.

What it computes (method: "Zellige: Moldable Sequence Placement for Mixed Image-Video
DiT Training"):
  * The engine runs whole sequences next to distributed-attention shards, each shard a
    query-row range, a head subset and a KV chunk cut by theta=(q,h,k) (pith.science
    review, "What carries the argument"; newx.sg abstract).  Sharding changes the
    schedule, not the result: each shard computes exact softmax attention over its own
    block (the cost assumption is FlashAttention's exact attention, pith.science review,
    "Assumptions", ref. [7]), bidirectional as in DiT (ref. [6]).
  * A k split yields partial outputs that are combined by log-sum-exp weights, as the
    ring-attention executor (ref. [19]) does across ranks.  The pages do not print the
    combine; the plainest reading is used (merge() below).
  * The backward is the textbook gradient of exact softmax attention with
    D_i = rowsum(dO_i * O_i).

Inputs q, k, v, do are float64 arrays [T, H, d] holding the bf16 input values exactly
upcast.  An item is any object with the attributes seq_offset, seq_len, q_lo, q_hi,
h_lo, h_hi, kv_lo, kv_hi (half-open, relative to the sequence start).

Every function here is pinned by tests/test_oracle.py (brute force, closed forms,
invariants, finite differences, torch SDPA in float64).
"""
from __future__ import annotations

import numpy as np

# Row-block size cap: rows * kv <= _BLOCK_ELEMS keeps one score block <= 256 MB.
_BLOCK_ELEMS = 1 << 25


def _rows(item, rows):
    if rows is None:
        return np.arange(item.q_lo, item.q_hi, dtype=np.int64)
    return np.asarray(rows, dtype=np.int64)


def _f64(x):
    # inputs may be float32 holding the bf16 values (exact); arithmetic is float64
    return np.asarray(x, dtype=np.float64)


def scores(q, k, item, h, rows, scale):
    """s_ij = scale * <Q[s+i, h], K[s+j, h]> for i in rows, j in the item's KV chunk."""
    s0 = item.seq_offset
    cols = np.arange(item.kv_lo, item.kv_hi, dtype=np.int64)
    return scale * (_f64(q[s0 + rows, h, :]) @ _f64(k[s0 + cols, h, :]).T)


def forward(q, k, v, item, scale, rows=None):
    """Exact attention of one work item over its own KV chunk.

    Returns (O, LSE): O [n_rows, |h|, d] with O_i = sum_j P_ij V_j and
    P_ij = exp(s_ij - LSE_i); LSE [|h|, n_rows] with LSE_i = ln sum_j exp(s_ij)
    (natural log).  An empty KV chunk gives O = 0 and LSE = -inf.
    """
    rows = _rows(item, rows)
    heads = range(item.h_lo, item.h_hi)
    d = q.shape[2]
    nkv = item.kv_hi - item.kv_lo
    O = np.zeros((len(rows), len(heads), d))
    LSE = np.full((len(heads), len(rows)), -np.inf)
    if nkv == 0 or len(rows) == 0:
        return O, LSE
    s0 = item.seq_offset
    cols = np.arange(item.kv_lo, item.kv_hi, dtype=np.int64)
    blk = max(1, _BLOCK_ELEMS // nkv)
    for hi, h in enumerate(heads):
        Vh = _f64(v[s0 + cols, h, :])
        for r0 in range(0, len(rows), blk):
            rb = rows[r0:r0 + blk]
            S = scores(q, k, item, h, rb, scale)
            m = S.max(axis=1, keepdims=True)
            lse = m[:, 0] + np.log(np.exp(S - m).sum(axis=1))
            P = np.exp(S - lse[:, None])
            O[r0:r0 + blk, hi, :] = P @ Vh
            LSE[hi, r0:r0 + blk] = lse
    return O, LSE


def probabilities(q, k, item, h, scale, rows=None):
    """P_ij = exp(s_ij - LSE_i) for one head (rows x KV chunk); used by the invariant pins."""
    rows = _rows(item, rows)
    S = scores(q, k, item, h, rows, scale)
    m = S.max(axis=1, keepdims=True)
    lse = m[:, 0] + np.log(np.exp(S - m).sum(axis=1))
    return np.exp(S - lse[:, None])


def merge(partials):
    """Combine k-split partials (O_c [n, |h|, d], LSE_c [|h|, n]) over disjoint chunks.

    LSE = ln sum_c exp(LSE_c);  O = sum_c exp(LSE_c - LSE) O_c.
    A row whose chunks are all empty (LSE_c = -inf for every c) gives O = 0, LSE = -inf.
    """
    L = np.stack([p[1] for p in partials])            # [c, h, n]
    M = L.max(axis=0)                                 # [h, n]
    finite = np.isfinite(M)
    Ms = np.where(finite, M, 0.0)
    with np.errstate(invalid="ignore"):
        tot = np.exp(L - Ms[None]).sum(axis=0)
    lse = np.where(finite, Ms + np.log(np.where(finite, tot, 1.0)), -np.inf)
    O = np.zeros_like(partials[0][0])
    for (Oc, Lc) in partials:
        w = np.where(finite, np.exp(Lc - np.where(finite, lse, 0.0)), 0.0)   # [h, n]
        O += w.T[:, :, None] * Oc
    return O, lse


def backward_dq(q, k, v, do_rows, o_rows, lse_rows, item, scale, rows):
    """dQ of one item for the given query rows.

    do_rows, o_rows [n, |h|, d] and lse_rows [|h|, n] are dO, the FINAL output and the
    FINAL (global) LSE of those rows.  With P_ij = exp(s_ij - LSE_i), dP_ij = dO_i . V_j,
    D_i = dO_i . O_i and dS_ij = P_ij (dP_ij - D_i):  dQ_i = scale * sum_j dS_ij K_j,
    the sum running over the item's own KV chunk only.
    """
    rows = np.asarray(rows, dtype=np.int64)
    s0 = item.seq_offset
    cols = np.arange(item.kv_lo, item.kv_hi, dtype=np.int64)
    d = q.shape[2]
    dQ = np.zeros((len(rows), item.h_hi - item.h_lo, d))
    if len(cols) == 0:
        return dQ
    blk = max(1, _BLOCK_ELEMS // len(cols))
    for hi, h in enumerate(range(item.h_lo, item.h_hi)):
        Kh, Vh = _f64(k[s0 + cols, h, :]), _f64(v[s0 + cols, h, :])
        for r0 in range(0, len(rows), blk):
            sl = slice(r0, r0 + blk)
            S = scores(q, k, item, h, rows[sl], scale)
            P = np.exp(S - lse_rows[hi, sl][:, None])
            dO = _f64(do_rows[sl, hi, :])
            D = (dO * _f64(o_rows[sl, hi, :])).sum(axis=1)
            dP = dO @ Vh.T
            dS = P * (dP - D[:, None])
            dQ[sl, hi, :] = scale * (dS @ Kh)
    return dQ


def backward_dkdv(q, k, v, do_all, o_all, lse_all, item, scale, kv_rows=None):
    """dK, dV of one item for the given KV rows (default: the whole chunk).

    do_all, o_all [|q|, |h|, d] and lse_all [|h|, |q|] cover ALL of the item's query
    rows (final output and global LSE).  dV_j = sum_i P_ij dO_i and
    dK_j = scale * sum_i dS_ij Q_i, the sums running over the item's own rows only.
    """
    kv_rows = (np.arange(item.kv_lo, item.kv_hi, dtype=np.int64) if kv_rows is None
               else np.asarray(kv_rows, dtype=np.int64))
    s0 = item.seq_offset
    rows = np.arange(item.q_lo, item.q_hi, dtype=np.int64)
    d = q.shape[2]
    nh = item.h_hi - item.h_lo
    dK = np.zeros((len(kv_rows), nh, d))
    dV = np.zeros((len(kv_rows), nh, d))
    if len(rows) == 0 or len(kv_rows) == 0:
        return dK, dV
    blk = max(1, _BLOCK_ELEMS // len(kv_rows))
    for hi, h in enumerate(range(item.h_lo, item.h_hi)):
        Kc, Vc = _f64(k[s0 + kv_rows, h, :]), _f64(v[s0 + kv_rows, h, :])
        for r0 in range(0, len(rows), blk):
            rb = rows[r0:r0 + blk]
            sl = slice(r0, r0 + blk)
            Qr = _f64(q[s0 + rb, h, :])
            S = scale * (Qr @ Kc.T)
            P = np.exp(S - lse_all[hi, sl][:, None])
            dO = _f64(do_all[sl, hi, :])
            D = (dO * _f64(o_all[sl, hi, :])).sum(axis=1)
            dP = dO @ Vc.T
            dS = P * (dP - D[:, None])
            dV[:, hi, :] += P.T @ dO
            dK[:, hi, :] += scale * (dS.T @ Qr)
    return dK, dV


def brute_force_forward(q, k, v, item, scale):
    """The same definition written as scalar Python loops (tiny inputs only)."""
    import math
    s0 = item.seq_offset
    d = q.shape[2]
    nq, nh = item.q_hi - item.q_lo, item.h_hi - item.h_lo
    O = [[[0.0] * d for _ in range(nh)] for _ in range(nq)]
    LSE = [[-math.inf] * nq for _ in range(nh)]
    for hi in range(nh):
        h = item.h_lo + hi
        for ii in range(nq):
            i = s0 + item.q_lo + ii
            s = []
            for j in range(s0 + item.kv_lo, s0 + item.kv_hi):
                s.append(scale * math.fsum(float(q[i, h, t]) * float(k[j, h, t]) for t in range(d)))
            if not s:
                continue
            m = max(s)
            z = math.fsum(math.exp(x - m) for x in s)
            lse = m + math.log(z)
            LSE[hi][ii] = lse
            for t in range(d):
                O[ii][hi][t] = math.fsum(math.exp(s[c] - lse) * float(v[s0 + item.kv_lo + c, h, t])
                                         for c in range(len(s)))
    return np.array(O), np.array(LSE)
