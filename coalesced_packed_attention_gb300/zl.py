"""Python binding of the engine's C ABI (include/zl.h), argument marshalling only.

Every entry point keeps its C name.  Tensors are torch tensors (device memory and
streams only); each call checks dtype, device, contiguity and sizes, then passes raw
pointers to libzl.so.  There is no fallback: if the library is missing the import of
this module's functions raises, and a non-OK status raises ZlError.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Dict, List, Optional, Sequence

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libzl.so")

ZL_OK, ZL_ERR_INVALID_ARG, ZL_ERR_ALIGN, ZL_ERR_CUDA, ZL_ERR_TIMEOUT, ZL_ERR_UNSUPPORTED, ZL_ERR_NO_MEMORY = range(7)
ZL_PLAN_HOST_ONLY = 1
ZL_PLAN_TEST_WITHHOLD_LOAD = 2
ZL_PLAN_FUSE_LOCAL_KMERGE = 8
ZL_PLAN_DETERMINISTIC_DQ = 16


class ZlError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


class zl_work_item(ctypes.Structure):
    _fields_ = [("seq_offset", ctypes.c_int64), ("seq_len", ctypes.c_int32),
                ("q_lo", ctypes.c_int32), ("q_hi", ctypes.c_int32),
                ("h_lo", ctypes.c_int32), ("h_hi", ctypes.c_int32),
                ("kv_lo", ctypes.c_int32), ("kv_hi", ctypes.c_int32),
                ("emit_lse", ctypes.c_int32),
                ("out_offset", ctypes.c_int64), ("lse_offset", ctypes.c_int64)]


class zl_bucket(ctypes.Structure):
    _fields_ = [("seq_len", ctypes.c_int64), ("count", ctypes.c_int32), ("time", ctypes.c_double),
                ("mem", ctypes.c_double)]


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libzl.so (built by coalesced_packed_attention_gb300.build) and declare
    the signatures.  Raises OSError when the library has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise OSError(f"{path} not found: build it with `python -m coalesced_packed_attention_gb300.build`")
    L = ctypes.CDLL(path)
    P, I32, I64, U32, F = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32, ctypes.c_float
    pI64, pI32 = ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int32)
    pD = ctypes.POINTER(ctypes.c_double)
    sig = {
        "zl_plan_worklist": (I32, [ctypes.POINTER(zl_work_item), I32, I32, I32, I64, U32, ctypes.POINTER(P)]),
        "zl_plan_worklist_groups": (I32, [ctypes.POINTER(zl_work_item), I32, I32, I32, I64, U32, pI32, pI32, I32,
                                          ctypes.POINTER(P)]),
        "zl_plan_destroy": (None, [P]),
        "zl_plan_arena_sizes": (I32, [P, pI64, pI64, pI64, pI64, pI64, pI64]),
        "zl_plan_item": (I32, [P, I32, ctypes.POINTER(zl_work_item), pI64, pI64, pI64, pI64, pI32]),
        "zl_plan_count": (I32, [P, I32, pI64]),
        "zl_plan_check_bounds": (I32, [P]),
        "zl_plan_tiles": (I32, [P, I32, pI32, I64]),
        "zl_plan_group": (I32, [P, I32, pI32, I32, pI32, pI64, pI64]),
        "zl_coalesced_attn_fwd": (I32, [P, P, P, P, P, P, P, F, P]),
        "zl_merge_partials": (I32, [P, P, P, P, P, P]),
        "zl_coalesced_attn_bwd": (I32, [P, P, P, P, P, P, P, P, P, P, P, F, P]),
        "zl_bwd_preprocess": (I32, [P, P, P, P, P]),
        "zl_bwd_main": (I32, [P, P, P, P, P, P, P, P, P, F, P]),
        "zl_bwd_finalize": (I32, [P, P, P, F, P]),
        "zl_get_device_status": (I32, [P, P, pI32]),
        "zl_status_string": (ctypes.c_char_p, [I32]),
        "zl_version": (I32, []),
        "zl_catalog_cut": (I32, [ctypes.POINTER(zl_bucket), I32, pI32, ctypes.POINTER(ctypes.c_double)]),
        "zl_pack_fillers": (I32, [pD, pD, I32, I32, pD, pD, ctypes.c_double, ctypes.c_double, pI32, pD, pD, pI32, pD]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L


def status_string(status: int) -> str:
    return load_library().zl_status_string(status).decode()


def _check(status: int, what: str):
    if status != ZL_OK:
        raise ZlError(status, what)


@dataclass
class ItemPlacement:
    item: zl_work_item
    fin_out_offset: int
    fin_lse_offset: int
    dq_offset: int
    dkv_offset: int
    group: int


class Plan:
    """Owner of one zl_plan*.  Created by zl_plan_worklist()."""

    def __init__(self, handle: int, n_heads: int, head_dim: int, total_tokens: int, host_only: bool,
                 device: Optional[int] = None):
        self.handle = ctypes.c_void_p(handle)
        self.n_heads, self.head_dim, self.total_tokens, self.host_only = n_heads, head_dim, total_tokens, host_only
        self.device = device  # CUDA device index the plan was built on (None: host-only plan)
        L = load_library()
        v = [ctypes.c_int64() for _ in range(6)]
        _check(L.zl_plan_arena_sizes(self.handle, *[ctypes.byref(x) for x in v]), "zl_plan_arena_sizes")
        (self.o_elems, self.o_partial_elems, self.lse_elems, self.dq_elems, self.dkv_elems,
         self.workspace_bytes) = (x.value for x in v)
        self.n_fwd_tiles = self._count(0)
        self.n_bwd_tiles = self._count(1)
        self.n_groups = self._count(2)
        self.n_items = self._count(3)
        self.n_merge_groups = self._count(4)  # groups the merge launch combines (unfused)

    def _count(self, which: int) -> int:
        c = ctypes.c_int64()
        _check(load_library().zl_plan_count(self.handle, which, ctypes.byref(c)), "zl_plan_count")
        return c.value

    def item(self, i: int) -> ItemPlacement:
        it = zl_work_item()
        vals = [ctypes.c_int64() for _ in range(4)]
        g = ctypes.c_int32()
        _check(load_library().zl_plan_item(self.handle, i, ctypes.byref(it), *[ctypes.byref(x) for x in vals],
                                           ctypes.byref(g)), "zl_plan_item")
        return ItemPlacement(it, vals[0].value, vals[1].value, vals[2].value, vals[3].value, g.value)

    def check_bounds(self):
        """Host dry run: every access a launch would make stays inside the arenas."""
        _check(load_library().zl_plan_check_bounds(self.handle), "zl_plan_check_bounds")

    def tiles(self, which: int = 0):
        """Tile list in scheduler order as a list of (item, head, block, cost)."""
        n = self.n_fwd_tiles if which == 0 else self.n_bwd_tiles
        buf = (ctypes.c_int32 * (4 * max(n, 1)))()
        _check(load_library().zl_plan_tiles(self.handle, which, buf, n), "zl_plan_tiles")
        return [tuple(buf[4 * i:4 * i + 4]) for i in range(n)]

    def group(self, g: int):
        """(member item ids, final O offset, final LSE offset) of merge group g."""
        n = ctypes.c_int32()
        oo, lo = ctypes.c_int64(), ctypes.c_int64()
        cap = 64
        while True:
            buf = (ctypes.c_int32 * cap)()
            _check(load_library().zl_plan_group(self.handle, g, buf, cap, ctypes.byref(n), ctypes.byref(oo),
                                                ctypes.byref(lo)), "zl_plan_group")
            if n.value <= cap:
                return list(buf[:n.value]), oo.value, lo.value
            cap = n.value

    def destroy(self):
        if self.handle is not None and self.handle.value:
            load_library().zl_plan_destroy(self.handle)
        self.handle = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


def _to_c_items(items: Sequence) -> ctypes.Array:
    arr = (zl_work_item * max(1, len(items)))()
    for i, it in enumerate(items):
        arr[i] = zl_work_item(it.seq_offset, it.seq_len, it.q_lo, it.q_hi, it.h_lo, it.h_hi, it.kv_lo, it.kv_hi,
                              it.emit_lse, getattr(it, "out_offset", -1), getattr(it, "lse_offset", -1))
    return arr


def _plan_device(flags: int):
    if flags & ZL_PLAN_HOST_ONLY:
        return None
    import torch
    return torch.cuda.current_device() if torch.cuda.is_available() else None  # else the library reports it


def zl_plan_worklist(items: Sequence, n_heads: int, head_dim: int, total_tokens: int, flags: int = 0) -> Plan:
    L = load_library()
    h = ctypes.c_void_p()
    device = _plan_device(flags)
    _check(L.zl_plan_worklist(_to_c_items(items), len(items), n_heads, head_dim, total_tokens, flags,
                              ctypes.byref(h)), "zl_plan_worklist")
    return Plan(h.value, n_heads, head_dim, total_tokens, bool(flags & ZL_PLAN_HOST_ONLY), device)


def zl_plan_worklist_groups(items: Sequence, n_heads: int, head_dim: int, total_tokens: int,
                            groups: Sequence[Sequence[int]], flags: int = 0) -> Plan:
    """zl_plan_worklist with caller-chosen merge groups: groups[g] lists the work-list
    indices of group g's emit_lse items in member order (passed as group_item_ids /
    group_ptr)."""
    L = load_library()
    h = ctypes.c_void_p()
    ids = [int(i) for g in groups for i in g]
    ptr = [0]
    for g in groups:
        ptr.append(ptr[-1] + len(g))
    c_ids = (ctypes.c_int32 * max(1, len(ids)))(*ids)
    c_ptr = (ctypes.c_int32 * len(ptr))(*ptr)
    device = _plan_device(flags)
    _check(L.zl_plan_worklist_groups(_to_c_items(items), len(items), n_heads, head_dim, total_tokens, flags, c_ids,
                                     c_ptr, len(groups), ctypes.byref(h)), "zl_plan_worklist_groups")
    return Plan(h.value, n_heads, head_dim, total_tokens, bool(flags & ZL_PLAN_HOST_ONLY), device)


# ---------------------------------------------------------------- launches
def _ptr(t, dtype, what, numel=None):
    import torch
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or t.device.type != "cuda":
        raise TypeError(f"{what}: expected a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{what}: expected {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{what}: must be contiguous")
    if numel is not None and t.numel() < numel:
        raise ValueError(f"{what}: needs at least {numel} elements, has {t.numel()}")
    return t.data_ptr()


def _on_plan_device(plan: Plan, *tensors):
    """Every tensor lives on the plan's device (the library checks the current device)."""
    for t in tensors:
        if t is not None and getattr(t, "device", None) is not None and t.device.type == "cuda" \
                and t.device.index != plan.device:
            raise ValueError(f"tensor on cuda:{t.device.index}, plan built on cuda:{plan.device}")


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _qkv(plan: Plan, q, k, v):
    import torch
    shape = (plan.total_tokens, plan.n_heads, plan.head_dim)
    for name, t in (("q", q), ("k", k), ("v", v)):
        if tuple(t.shape) != shape:
            raise ValueError(f"{name}: expected shape {shape}, got {tuple(t.shape)}")
    return [_ptr(t, torch.bfloat16, n) for t, n in ((q, "q"), (k, "k"), (v, "v"))]


def zl_coalesced_attn_fwd(plan: Plan, q, k, v, o, o_partial, lse, scale: float, stream=None):
    import torch
    _on_plan_device(plan, q, k, v, o, o_partial, lse)
    pq, pk, pv = _qkv(plan, q, k, v)
    st = load_library().zl_coalesced_attn_fwd(
        plan.handle, pq, pk, pv,
        _ptr(o, torch.bfloat16, "o", plan.o_elems) if o is not None else None,
        _ptr(o_partial, torch.float32, "o_partial", plan.o_partial_elems) if o_partial is not None else None,
        _ptr(lse, torch.float32, "lse", plan.lse_elems), ctypes.c_float(scale), _stream(stream))
    _check(st, "zl_coalesced_attn_fwd")


def zl_merge_partials(plan: Plan, o_partial, lse_partial, o, lse_out, stream=None):
    import torch
    _on_plan_device(plan, o_partial, lse_partial, o, lse_out)
    st = load_library().zl_merge_partials(
        plan.handle, _ptr(o_partial, torch.float32, "o_partial", plan.o_partial_elems),
        _ptr(lse_partial, torch.float32, "lse_partial", plan.lse_elems),
        _ptr(o, torch.bfloat16, "o", plan.o_elems), _ptr(lse_out, torch.float32, "lse_out", plan.lse_elems),
        _stream(stream))
    _check(st, "zl_merge_partials")


def zl_coalesced_attn_bwd(plan: Plan, q, k, v, o, d_o, lse, dq, dk, dv, workspace, scale: float, stream=None):
    import torch
    _on_plan_device(plan, q, k, v, o, d_o, lse, dq, dk, dv, workspace)
    pq, pk, pv = _qkv(plan, q, k, v)
    st = load_library().zl_coalesced_attn_bwd(
        plan.handle, pq, pk, pv, _ptr(o, torch.bfloat16, "o", plan.o_elems),
        _ptr(d_o, torch.bfloat16, "d_o", plan.o_elems), _ptr(lse, torch.float32, "lse", plan.lse_elems),
        _ptr(dq, torch.float32, "dq", plan.dq_elems), _ptr(dk, torch.float32, "dk", plan.dkv_elems),
        _ptr(dv, torch.float32, "dv", plan.dkv_elems),
        _ptr(workspace, torch.uint8, "workspace", plan.workspace_bytes), ctypes.c_float(scale), _stream(stream))
    _check(st, "zl_coalesced_attn_bwd")


def zl_bwd_preprocess(plan: Plan, o, d_o, workspace, stream=None):
    import torch
    _on_plan_device(plan, o, d_o, workspace)
    _check(load_library().zl_bwd_preprocess(
        plan.handle, _ptr(o, torch.bfloat16, "o", plan.o_elems), _ptr(d_o, torch.bfloat16, "d_o", plan.o_elems),
        _ptr(workspace, torch.uint8, "workspace", plan.workspace_bytes), _stream(stream)), "zl_bwd_preprocess")


def zl_bwd_main(plan: Plan, q, k, v, d_o, lse, dk, dv, workspace, scale: float, stream=None):
    import torch
    _on_plan_device(plan, q, k, v, d_o, lse, dk, dv, workspace)
    pq, pk, pv = _qkv(plan, q, k, v)
    _check(load_library().zl_bwd_main(
        plan.handle, pq, pk, pv, _ptr(d_o, torch.bfloat16, "d_o", plan.o_elems),
        _ptr(lse, torch.float32, "lse", plan.lse_elems), _ptr(dk, torch.float32, "dk", plan.dkv_elems),
        _ptr(dv, torch.float32, "dv", plan.dkv_elems), _ptr(workspace, torch.uint8, "workspace", plan.workspace_bytes),
        ctypes.c_float(scale), _stream(stream)), "zl_bwd_main")


def zl_bwd_finalize(plan: Plan, dq, workspace, scale: float, stream=None):
    import torch
    _on_plan_device(plan, dq, workspace)
    _check(load_library().zl_bwd_finalize(
        plan.handle, _ptr(dq, torch.float32, "dq", plan.dq_elems),
        _ptr(workspace, torch.uint8, "workspace", plan.workspace_bytes), ctypes.c_float(scale), _stream(stream)),
        "zl_bwd_finalize")


def zl_get_device_status(plan: Plan, stream=None) -> int:
    s = ctypes.c_int32()
    _check(load_library().zl_get_device_status(plan.handle, _stream(stream), ctypes.byref(s)),
           "zl_get_device_status")
    return s.value


# ---------------------------------------------------------------- conveniences
def allocate(plan: Plan, device="cuda", backward: bool = False) -> Dict[str, "object"]:
    """Device arenas sized for the plan (fresh torch allocations, uninitialised)."""
    import torch
    out = {
        "o": torch.empty(max(plan.o_elems, 8), dtype=torch.bfloat16, device=device),
        "o_partial": torch.empty(max(plan.o_partial_elems, 8), dtype=torch.float32, device=device),
        "lse": torch.empty(max(plan.lse_elems, 4), dtype=torch.float32, device=device),
    }
    if backward:
        out["dq"] = torch.empty(max(plan.dq_elems, 4), dtype=torch.float32, device=device)
        out["dk"] = torch.empty(max(plan.dkv_elems, 4), dtype=torch.float32, device=device)
        out["dv"] = torch.empty(max(plan.dkv_elems, 4), dtype=torch.float32, device=device)
        out["workspace"] = torch.empty(max(plan.workspace_bytes, 16), dtype=torch.uint8, device=device)
    return out


def o_arena_from_tokens(plan: Plan, items: Sequence, x):
    """A [T, H, d] token tensor laid out like the `o` arena: each work item's final block
    (its own, or its merge group's) holds that item's query rows and heads of x.  This is
    the layout in which the backward reads the output gradient dO."""
    import torch
    d = plan.head_dim
    arena = torch.zeros(max(plan.o_elems, 8), dtype=x.dtype, device=x.device)
    for i, it in enumerate(items):
        pl = plan.item(i)
        n = (it.q_hi - it.q_lo) * (it.h_hi - it.h_lo) * d
        arena[pl.fin_out_offset: pl.fin_out_offset + n] = \
            x[it.seq_offset + it.q_lo: it.seq_offset + it.q_hi, it.h_lo:it.h_hi].reshape(-1)
    return arena


def forward(plan: Plan, q, k, v, scale: float, bufs: Optional[dict] = None, stream=None) -> dict:
    """Forward of every item, then the merge of every k-split group."""
    bufs = bufs if bufs is not None else allocate(plan, q.device)
    zl_coalesced_attn_fwd(plan, q, k, v, bufs["o"], bufs["o_partial"], bufs["lse"], scale, stream)
    if plan.n_merge_groups:
        zl_merge_partials(plan, bufs["o_partial"], bufs["lse"], bufs["o"], bufs["lse"], stream)
    return bufs


def backward(plan: Plan, q, k, v, d_o, scale: float, bufs: dict, stream=None) -> dict:
    zl_coalesced_attn_bwd(plan, q, k, v, bufs["o"], d_o, bufs["lse"], bufs["dq"], bufs["dk"], bufs["dv"],
                          bufs["workspace"], scale, stream)
    return bufs


def exported_symbols() -> List[str]:
    """Names of the entry points declared in include/zl.h."""
    return ["zl_plan_worklist", "zl_plan_worklist_groups", "zl_plan_destroy", "zl_plan_arena_sizes", "zl_plan_item", "zl_plan_check_bounds",
            "zl_plan_count",
            "zl_plan_tiles", "zl_plan_group", "zl_coalesced_attn_fwd", "zl_merge_partials",
            "zl_coalesced_attn_bwd", "zl_bwd_preprocess", "zl_bwd_main", "zl_bwd_finalize",
            "zl_get_device_status", "zl_status_string", "zl_version", "zl_catalog_cut", "zl_pack_fillers"]


# ---------------------------------------------------------------- host placement slice
def catalog_cut(buckets):
    """zl_catalog_cut over [(seq_len, count, time, mem), ...] sorted by time: returns
    (k_star, dispersion); buckets[:k_star] are fillers, the rest anchors."""
    arr = (zl_bucket * len(buckets))(*[zl_bucket(int(L), int(n), float(t), float(m)) for (L, n, t, m) in buckets])
    k = ctypes.c_int32()
    disp = ctypes.c_double()
    _check(load_library().zl_catalog_cut(arr, len(buckets), ctypes.byref(k), ctypes.byref(disp)), "zl_catalog_cut")
    return k.value, disp.value


def pack_fillers(filler_time, filler_mem, n_ranks, rank_time=None, rank_mem=None, F=0.0, M_cap=1.0):
    """zl_pack_fillers: returns (assign, final_time, final_mem, n_overflow, makespan)."""
    D = ctypes.c_double
    n = len(filler_time)
    ft = (D * max(n, 1))(*map(float, filler_time))
    fm = (D * max(n, 1))(*map(float, filler_mem))
    rt = (D * n_ranks)(*map(float, rank_time)) if rank_time is not None else None
    rm = (D * n_ranks)(*map(float, rank_mem)) if rank_mem is not None else None
    assign = (ctypes.c_int32 * max(n, 1))()
    out_t, out_m = (D * n_ranks)(), (D * n_ranks)()
    over, mk = ctypes.c_int32(), D()
    _check(load_library().zl_pack_fillers(ft, fm, n, n_ranks, rt, rm, float(F), float(M_cap), assign, out_t, out_m,
                                          ctypes.byref(over), ctypes.byref(mk)), "zl_pack_fillers")
    return list(assign[:n]), list(out_t), list(out_m), over.value, mk.value

