"""Seeded synthetic inputs and the five work lists of the coalesced attention engine.

This module is shared by the CUDA path's tests/bench and by the oracle's tests.  It
holds no attention arithmetic: only work-item descriptors, token packing and the
seeded random tensors (bf16 ~ N(0,1)).

The work lists follow the mixed image/video placements of "Zellige: Moldable Sequence
Placement for Mixed Image-Video DiT Training" (pith.science review, "What carries the
argument": a sequence's configuration theta=(q,h,k) splits its query rows, heads and
KV states, and whole short image sequences share a rank with shards of long videos).
The pages' datasets (OpenVid-1M, Koala-36M) are not available; N(0,1) tensors with
the same token counts stand in for them (attention FLOPs do not depend on content).

Ranges in a WorkItem are half-open and relative to the start of the item's sequence.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional, Tuple


@dataclass(frozen=True)
class WorkItem:
    """One entry of a work list: a whole sequence or a theta shard of one sequence.

    seq_offset/seq_len locate the sequence in the packed [T, H, d] token stream.
    [q_lo, q_hi) query rows, [h_lo, h_hi) heads and [kv_lo, kv_hi) key/value rows,
    all relative to the sequence start.  emit_lse=1 marks a k-split shard whose
    output is an fp32 partial O plus its LSE, to be merged with the other chunks.
    out_offset/lse_offset = -1 let the planner place the item's outputs.
    """
    seq_offset: int
    seq_len: int
    q_lo: int
    q_hi: int
    h_lo: int
    h_hi: int
    kv_lo: int
    kv_hi: int
    emit_lse: int = 0
    out_offset: int = -1
    lse_offset: int = -1

    @property
    def nq(self) -> int:
        return self.q_hi - self.q_lo

    @property
    def nh(self) -> int:
        return self.h_hi - self.h_lo

    @property
    def nkv(self) -> int:
        return self.kv_hi - self.kv_lo

    def fwd_flops(self, head_dim: int) -> int:
        """Algorithmic forward FLOPs: 4 * |q| * |kv| * d per head (non-causal)."""
        return 4 * self.nq * self.nkv * head_dim * self.nh


def whole(seq_offset: int, seq_len: int, n_heads: int) -> WorkItem:
    return WorkItem(seq_offset, seq_len, 0, seq_len, 0, n_heads, 0, seq_len, 0)


@dataclass
class Workload:
    name: str
    n_heads: int
    head_dim: int
    total_tokens: int
    items: List[WorkItem]
    scale: float
    with_backward: bool = False
    # names of items, for reports only
    labels: List[str] = field(default_factory=list)

    def fwd_flops(self) -> int:
        return sum(it.fwd_flops(self.head_dim) for it in self.items)

    def bwd_flops(self) -> int:
        # backward counted as 2.5x the forward (five matmuls instead of two)
        return (5 * self.fwd_flops()) // 2


def _pack(lengths: List[int]) -> List[Tuple[int, int]]:
    out, off = [], 0
    for L in lengths:
        out.append((off, L))
        off += L
    return out


def config_tiny() -> Workload:
    """Tiny mixed list: whole 64/100/256 + a 512-token sequence as 2 k-split chunks.
    4 heads, head_dim 64, scale 1/sqrt(64); forward only."""
    H, d = 4, 64
    seqs = _pack([64, 100, 256, 512])
    items, labels = [], []
    for (o, L) in seqs[:3]:
        items.append(whole(o, L, H)); labels.append(f"whole{L}")
    o, L = seqs[3]
    items.append(WorkItem(o, L, 0, L, 0, H, 0, 256, 1)); labels.append("kchunk0")
    items.append(WorkItem(o, L, 0, L, 0, H, 256, 512, 1)); labels.append("kchunk1")
    return Workload("tiny_mixed_h4_d64", H, d, seqs[-1][0] + seqs[-1][1], items,
                    1.0 / math.sqrt(d), labels=labels)


def config_images() -> Workload:
    """Image-only packed batch: 48x256 + 12x1024 + 4x4096 whole sequences, 24 heads, d=128."""
    H, d = 24, 128
    lens = [256] * 48 + [1024] * 12 + [4096] * 4
    seqs = _pack(lens)
    items = [whole(o, L, H) for (o, L) in seqs]
    labels = [f"img{L}" for (_, L) in seqs]
    T = seqs[-1][0] + seqs[-1][1]
    return Workload("images_48x256_12x1024_4x4096_h24_d128", H, d, T, items,
                    1.0 / math.sqrt(d), labels=labels)


def config_mixed(with_backward: bool = False, with_complement: bool = True) -> Workload:
    """16 whole 1024-token images + a 32760-token video (21x30x52) cut into a q-split
    shard (rows [0,8190), all heads), an h-split shard (heads [0,12), all rows) and a
    k-split shard (heads [12,24), KV [16380,32760), emit_lse).  The complementary
    chunk (heads [12,24), KV [0,16380)) stands in for the remote rank's share of the
    k split so that the merge has both halves."""
    H, d = 24, 128
    Lv = 21 * 30 * 52
    seqs = _pack([1024] * 16 + [Lv])
    items = [whole(o, L, H) for (o, L) in seqs[:16]]
    labels = ["img1024"] * 16
    vo, _ = seqs[16]
    items.append(WorkItem(vo, Lv, 0, 8190, 0, H, 0, Lv, 0)); labels.append("video_qsplit")
    items.append(WorkItem(vo, Lv, 0, Lv, 0, 12, 0, Lv, 0)); labels.append("video_hsplit")
    items.append(WorkItem(vo, Lv, 0, Lv, 12, 24, 16380, Lv, 1)); labels.append("video_ksplit")
    if with_complement:
        items.append(WorkItem(vo, Lv, 0, Lv, 12, 24, 0, 16380, 1)); labels.append("video_kcomplement")
    T = vo + Lv
    name = "mixed_16x1024_video32760_qhk_h24_d128" + ("_train" if with_backward else "")
    return Workload(name, H, d, T, items, 1.0 / math.sqrt(d), with_backward, labels)


def config_long_video() -> Workload:
    """A 147600-token video (41x45x80) as 8 k-split shards of 18450 KV tokens over all
    rows and heads, plus 8 whole 4096-token images, in one launch; merge of 8."""
    H, d = 24, 128
    Lv = 41 * 45 * 80
    seqs = _pack([Lv] + [4096] * 8)
    vo, _ = seqs[0]
    items, labels = [], []
    chunk = Lv // 8
    for c in range(8):
        items.append(WorkItem(vo, Lv, 0, Lv, 0, H, c * chunk, (c + 1) * chunk, 1))
        labels.append(f"video_k{c}")
    for (o, L) in seqs[1:]:
        items.append(whole(o, L, H)); labels.append("img4096")
    T = seqs[-1][0] + seqs[-1][1]
    return Workload("long_video147600_k8_8x4096_h24_d128", H, d, T, items,
                    1.0 / math.sqrt(d), labels=labels)


def config_training() -> Workload:
    """Training step of the mixed image + video-shard list: forward, merge, backward."""
    return config_mixed(with_backward=True)


CONFIGS = {
    "tiny": config_tiny,
    "images": config_images,
    "mixed": config_mixed,
    "long_video": config_long_video,
    "training": config_training,
}


def merge_groups(items: List[WorkItem]) -> List[List[int]]:
    """Group emit_lse items that cover the same sequence, rows and heads (disjoint KV
    chunks), in work-list order.  Same rule as the planner's."""
    groups, keys = [], {}
    for i, it in enumerate(items):
        if not it.emit_lse:
            continue
        key = (it.seq_offset, it.seq_len, it.q_lo, it.q_hi, it.h_lo, it.h_hi)
        if key not in keys:
            keys[key] = len(groups)
            groups.append([])
        groups[keys[key]].append(i)
    return groups


def make_inputs(total_tokens: int, n_heads: int, head_dim: int, seed: int,
                with_grad_output: bool = False, device: str = "cpu",
                structured: bool = False):
    """Seeded Q, K, V (and dO) as bf16 [T, H, d].

    Draw order Q, K, V, dO from one fp32 N(0,1) stream (torch CPU generator, or the
    device generator when device != 'cpu'), then round to nearest-even bf16.
    structured=True gives the peaky variant: Q scaled by 4 and V offset by +3, so
    that |O| is O(1) even for long sequences.
    """
    import torch
    shape = (total_tokens, n_heads, head_dim)
    if device == "cpu":
        g = torch.Generator().manual_seed(seed)
        kw = dict(generator=g, dtype=torch.float32)
    else:
        g = torch.Generator(device=device).manual_seed(seed)
        kw = dict(generator=g, dtype=torch.float32, device=device)
    out = []
    n = 4 if with_grad_output else 3
    for i in range(n):
        x = torch.randn(shape, **kw)
        if structured and i == 0:
            x = x * 4.0
        if structured and i == 2:
            x = x + 3.0
        out.append(x.to(torch.bfloat16))
    return tuple(out)


def scaled(work: Workload, factor: int, name: Optional[str] = None) -> Workload:
    """A smaller workload of the same shape family: every length divided by `factor`
    (rounded, at least 1), for parity tests the oracle finishes in seconds."""
    def sc(x):
        return max(1, int(round(x / factor))) if x > 0 else 0
    # re-pack sequences by their (offset, len) keys
    seqs = sorted({(it.seq_offset, it.seq_len) for it in work.items})
    new_off, off = {}, 0
    for (o, L) in seqs:
        new_off[(o, L)] = (off, sc(L))
        off += sc(L)
    items = []
    for it in work.items:
        o, L = new_off[(it.seq_offset, it.seq_len)]
        def rng(lo, hi):
            a, b = min(sc(lo), L), min(sc(hi), L)
            if hi == it.seq_len:
                b = L
            return a, b
        ql, qh = rng(it.q_lo, it.q_hi)
        kl, kh = rng(it.kv_lo, it.kv_hi)
        items.append(WorkItem(o, L, ql, qh, it.h_lo, it.h_hi, kl, kh, it.emit_lse))
    return Workload(name or (work.name + f"_div{factor}"), work.n_heads, work.head_dim,
                    off, items, work.scale, work.with_backward, list(work.labels))
