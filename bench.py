"""Benchmark of the coalesced attention engine: one training step of the mixed image +
video-shard work list (16 whole 1024-token images plus q-, h- and k-split shards of a
32760-token video, 24 heads, d=128), through the C ABI.

A step is the whole hot path: forward launch over every tile, LSE merge of the k-split
group, backward (row sums D, tcgen05 backward, dQ finalisation).  The plan is built once
outside the timed region.  Metric: algorithmic TFLOP/s of forward + backward
(4 |q| |kv| d per head forward, 2.5x that backward).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Under torchrun (N > 1) every rank runs its own replica of the step on its own GPU (the
path has no exchange step on one GPU); the time is the max over ranks and the value is
the work of all ranks over that time.  --impl reference times the CPU float64 oracle
on the host cores instead (bounded row samples of the same workload).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "coalesced attn TFLOP/s (fwd+bwd training step)"
UNIT = "TFLOP/s"
KERNEL_SOURCES = {"zl_bwd_main": "coalesced_packed_attention_gb300/csrc/zl_bwd.cu",
                  "zl_coalesced_attn_fwd": "coalesced_packed_attention_gb300/csrc/zl_fwd2.cu"}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def aggregate(total_ms, ws: int, flops_per_rank: float, steps: int):
    """Whole-job value over replicas: the slowest rank's time (max over ranks of the
    timed region) and the work of all ranks.  Returns (TFLOP/s, ms per step)."""
    import torch
    t = total_ms.clone() if hasattr(total_ms, "clone") else torch.tensor([float(total_ms)])
    if ws > 1 and torch.distributed.is_available() and torch.distributed.is_initialized():
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    ms_step = float(t.reshape(-1)[0].item()) / steps
    return ws * flops_per_rank / (ms_step * 1e-3) / 1e12, ms_step


def sample_clocks(stop: threading.Event, out: list):
    # power.draw.instant: power.draw is a windowed average that blends in the idle time
    # around a timed region shorter than its window
    q = ("--query-gpu=index,clocks.sm,clocks.max.sm,power.draw.instant,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    try:
        p = subprocess.Popen(["nvidia-smi", q, "--format=csv,noheader,nounits", "-lms", "200"],
                             stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
    except OSError:
        return
    try:
        while not stop.is_set():
            line = p.stdout.readline()
            if not line:
                break
            out.append(line.strip())
    finally:
        p.terminate()


def summarize_clocks(lines, gpu_index):
    """Median SM clock and instantaneous board power over the samples, the maximum SM
    clock, and every throttle reason seen active."""
    sm, pw, mx, reasons = [], [], None, set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for ln in lines:
        f = [x.strip() for x in ln.split(",")]
        if len(f) < 9 or f[0] != str(gpu_index):
            continue
        try:
            sm.append(float(f[1]))
            mx = float(f[2])
        except ValueError:
            continue
        try:
            pw.append(float(f[3]))
        except ValueError:
            pass
        for n, v in zip(names, f[5:9]):
            if v.lower() == "active":
                reasons.add(n)
    if not sm:
        return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": 0}
    return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm),
            "power_w": float(np.median(pw)) if pw else None}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def kernel_source_sha256(kernel: str) -> str:
    """Hash of a kernel's device code: its source file up to the host launcher (the
    first `cudaError_t launch_` definition), with comments and blank lines removed, so
    that neither a host-only change to the launch nor a comment voids counters taken on
    the kernel."""
    text = open(os.path.join(ROOT, KERNEL_SOURCES[kernel]), "rb").read()
    cut = text.find(b"\ncudaError_t launch_")
    text = text[:cut] if cut > 0 else text
    text = re.sub(rb"/\*.*?\*/", b"", text, flags=re.S)
    text = re.sub(rb"//[^\n]*", b"", text)
    text = b"\n".join(ln.rstrip() for ln in text.split(b"\n") if ln.strip())
    return hashlib.sha256(text).hexdigest()


def recorded_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the
    current device code of that kernel (else None)."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_training_traffic.txt")
    if not os.path.exists(path):
        return None
    sha = kernel_source_sha256(kernel)
    vals = {}
    for ln in open(path):
        if ":" in ln:
            k, v = ln.split(":", 1)
            vals[k.strip()] = v.strip()
    if vals.get("source_sha256") != sha:
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def dO_arena(plan, work, do_tok, device):
    """dO laid out like the `o` arena: each item's final block gets the matching rows and
    heads of the [T, H, d] gradient."""
    from coalesced_packed_attention_gb300 import zl
    return zl.o_arena_from_tokens(plan, work.items, do_tok.to(device))


def oracle_inputs(work, seed=0):
    from coalesced_packed_attention_gb300.workloads import make_inputs
    return tuple(x.float().numpy() for x in make_inputs(work.total_tokens, work.n_heads, work.head_dim, seed,
                                                        with_grad_output=True))


def cpu_oracle_sample(work, seed=0, rows_per_item=2048, heads_per_item=2, inputs=None):
    """Time the oracle (as it stands) on a bounded sample of the workload: for every item,
    `rows_per_item` query rows x `heads_per_item` heads, forward + dQ backward.  Returns
    (TFLOP/s over the sampled algorithmic FLOPs, seconds, description)."""
    import oracle
    from coalesced_packed_attention_gb300.workloads import WorkItem
    q, k, v, do = inputs if inputs is not None else oracle_inputs(work, seed)
    rng = np.random.default_rng(seed)
    flops = 0
    t0 = time.perf_counter()
    for it in work.items:
        if it.nq == 0 or it.nkv == 0:
            continue
        sub = WorkItem(it.seq_offset, it.seq_len, it.q_lo, it.q_hi, it.h_lo, min(it.h_hi, it.h_lo + heads_per_item),
                       it.kv_lo, it.kv_hi, it.emit_lse)
        rows = it.q_lo + np.sort(rng.choice(it.nq, min(rows_per_item, it.nq), replace=False))
        O, L = oracle.forward(q, k, v, sub, work.scale, rows=rows)
        dO = do[it.seq_offset + rows][:, sub.h_lo:sub.h_hi]
        oracle.backward_dq(q, k, v, dO, O, L, sub, work.scale, rows)
        flops += int(3.5 * 4 * len(rows) * it.nkv * work.head_dim * sub.nh)
    dt = time.perf_counter() - t0
    desc = (f"{rows_per_item} random query rows x {heads_per_item} heads of every item: forward + dQ backward "
            f"in float64 ({flops / 1e9:.1f} GFLOP algorithmic)")
    return flops / dt / 1e12, dt, desc


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    from coalesced_packed_attention_gb300.workloads import config_training
    work = config_training()
    inputs = oracle_inputs(work, 0)
    for _ in range(args.warmup):
        cpu_oracle_sample(work, rows_per_item=4, inputs=inputs)
    vals, secs = [], []
    for s in range(args.steps):
        v, dt, desc = cpu_oracle_sample(work, seed=s, inputs=inputs)
        vals.append(v)
        secs.append(dt)
    value = float(np.median(vals))
    cores = os.cpu_count()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * float(np.median(secs)), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": work.name, "n_heads": work.n_heads, "head_dim": work.head_dim,
                   "total_tokens": work.total_tokens, "items": len(work.items)},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_gpu(args):
    import torch
    from coalesced_packed_attention_gb300 import zl
    from coalesced_packed_attention_gb300.workloads import config_training, make_inputs

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(dev)
    zl.load_library()

    work = config_training()
    if args.scale > 1:  # smaller case of the same list, for profiler captures
        from coalesced_packed_attention_gb300.workloads import scaled
        work = scaled(work, args.scale)
    H, d, T, scale = work.n_heads, work.head_dim, work.total_tokens, work.scale
    F_fwd = work.fwd_flops()
    F_bwd = work.bwd_flops()
    F_step = F_fwd + F_bwd

    t_plan = time.perf_counter()
    plan = zl.zl_plan_worklist(work.items, H, d, T,
                               (zl.ZL_PLAN_FUSE_LOCAL_KMERGE if args.fuse_kmerge else 0)
                               | (zl.ZL_PLAN_DETERMINISTIC_DQ if args.deterministic else 0))
    t_plan = time.perf_counter() - t_plan

    q, k, v, do_tok = make_inputs(T, H, d, seed=rank, with_grad_output=True, device=str(dev))
    d_o = dO_arena(plan, work, do_tok, dev)
    bufs = zl.allocate(plan, dev, backward=True)
    stream = torch.cuda.current_stream(dev)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        zl.zl_coalesced_attn_fwd(plan, q, k, v, bufs["o"], bufs["o_partial"], bufs["lse"], scale, stream)
        if ev is not None:
            ev[1].record(stream)
        zl.zl_merge_partials(plan, bufs["o_partial"], bufs["lse"], bufs["o"], bufs["lse"], stream)
        if ev is not None:
            ev[2].record(stream)
        zl.zl_bwd_preprocess(plan, bufs["o"], d_o, bufs["workspace"], stream)
        if ev is not None:
            ev[3].record(stream)
        zl.zl_bwd_main(plan, q, k, v, d_o, bufs["lse"], bufs["dk"], bufs["dv"], bufs["workspace"], scale, stream)
        if ev is not None:
            ev[4].record(stream)
        zl.zl_bwd_finalize(plan, bufs["dq"], bufs["workspace"], scale, stream)
        if ev is not None:
            ev[5].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    status = zl.zl_get_device_status(plan, stream)
    if status != 0:
        raise RuntimeError(f"device status {status} after warm-up")

    clock_lines, stop = [], threading.Event()
    th = threading.Thread(target=sample_clocks, args=(stop, clock_lines), daemon=True)
    th.start()
    time.sleep(0.3)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(args.steps)]
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for s in range(args.steps):
        step(evs[s])
    t1.record(stream)
    torch.cuda.synchronize(dev)
    if ws > 1:
        torch.distributed.barrier()
    stop.set()
    th.join(timeout=2)
    total_ms = t0.elapsed_time(t1)
    parts = np.array([[e[i].elapsed_time(e[i + 1]) for i in range(5)] for e in evs])  # ms per stage per step
    status = zl.zl_get_device_status(plan, stream)
    if status != 0:
        raise RuntimeError(f"device status {status} in the timed region")
    value, ms_step = aggregate(torch.tensor([total_ms], device=dev), ws, F_step, args.steps)

    # ---- end to end through host buffers (pinned), every step's copies inside the timed
    # region: each input's H2D and each output's D2H on a copy stream of its own (several
    # copy engines in flight at once), the step on the compute stream; two device buffer
    # sets let step i+1's uploads and step i-1's downloads run under step i's kernels
    # (whole-job throughput of a stream of steps)
    e2e = None
    if not args.no_e2e:
        hq, hk, hv, hdo = (x.cpu().pin_memory() for x in (q, k, v, d_o))
        out_names = ("o", "lse", "dq", "dk", "dv")
        sets = []
        for _ in range(2):
            din = [torch.empty_like(x) for x in (q, k, v, d_o)]
            dbufs = zl.allocate(plan, dev, backward=True)
            hout = {n: torch.empty(dbufs[n].shape, dtype=dbufs[n].dtype, pin_memory=True) for n in out_names}
            sets.append((din, dbufs, hout))
        h2d = sum(x.numel() * x.element_size() for x in (hq, hk, hv, hdo))
        d2h = sum(x.numel() * x.element_size() for x in sets[0][2].values())
        s_comp = stream
        s_in = [torch.cuda.Stream(dev) for _ in range(4)]                # one per input tensor
        s_out = [torch.cuda.Stream(dev) for _ in range(len(out_names))]  # one per output arena
        ev_in = [[torch.cuda.Event() for _ in s_in] for _ in range(2)]
        ev_comp = [torch.cuda.Event() for _ in range(2)]
        ev_out = [[torch.cuda.Event() for _ in s_out] for _ in range(2)]

        def e2e_step(i):
            din, dbufs, hout = sets[i % 2]
            for j, (st, dst, src) in enumerate(zip(s_in, din, (hq, hk, hv, hdo))):
                if i >= 2:
                    st.wait_event(ev_comp[i % 2])   # step i-2 has finished reading this input set
                with torch.cuda.stream(st):
                    dst.copy_(src, non_blocking=True)
                ev_in[i % 2][j].record(st)
                s_comp.wait_event(ev_in[i % 2][j])
            if i >= 2:
                for ev in ev_out[i % 2]:
                    s_comp.wait_event(ev)           # step i-2's outputs have left this set
            dq_, dk_, dv_, ddo = din
            zl.zl_coalesced_attn_fwd(plan, dq_, dk_, dv_, dbufs["o"], dbufs["o_partial"], dbufs["lse"], scale, s_comp)
            zl.zl_merge_partials(plan, dbufs["o_partial"], dbufs["lse"], dbufs["o"], dbufs["lse"], s_comp)
            zl.zl_coalesced_attn_bwd(plan, dq_, dk_, dv_, dbufs["o"], ddo, dbufs["lse"], dbufs["dq"], dbufs["dk"],
                                     dbufs["dv"], dbufs["workspace"], scale, s_comp)
            ev_comp[i % 2].record(s_comp)
            for j, (st, (n, hb)) in enumerate(zip(s_out, hout.items())):
                st.wait_event(ev_comp[i % 2])
                with torch.cuda.stream(st):
                    hb.copy_(dbufs[n], non_blocking=True)
                ev_out[i % 2][j].record(st)

        for i in range(2):
            e2e_step(i)
        torch.cuda.synchronize(dev)
        n_e2e = max(4, args.steps)  # as many steps as the device-timed region
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s_comp)
        for st in s_in + s_out:
            st.wait_event(a)
        for i in range(n_e2e):
            e2e_step(i)
        for evs in ev_out:
            for ev in evs:
                s_comp.wait_event(ev)
        b.record(s_comp)
        torch.cuda.synchronize(dev)
        e_val, e_ms = aggregate(torch.tensor([a.elapsed_time(b)], device=dev), ws, F_step, n_e2e)
        # one call at a time: a step's uploads, its launches and its downloads, then the
        # host waits for the results before the next call (host clock, host to host)
        single = []
        for _ in range(max(3, min(args.steps, 6))):
            t_a = time.perf_counter()
            e2e_step(0)
            torch.cuda.synchronize(dev)
            single.append(time.perf_counter() - t_a)
        s_ms = 1e3 * float(np.median(single))
        e2e = {"value": e_val, "unit": UNIT, "ms_per_step": e_ms,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "pipelined": ("throughput of a stream of steps: 2 device buffer sets, so one step's uploads and "
                             "the previous step's downloads run under the current step's kernels; every "
                             "input's H2D and every output's D2H on its own stream"),
               "single_call": {"value": F_step / (s_ms * 1e-3) / 1e12, "unit": UNIT, "ms_per_step": s_ms,
                               "note": "one call's host-to-host time (uploads, step, downloads, host sync)"}}
        del sets

    peaks, peak_kind = measured_peaks()
    med = np.median(parts, axis=0)
    fwd_ms, merge_ms, pre_ms, bwd_ms, fin_ms = (float(x) for x in med)
    step_each = parts.sum(axis=1)  # device time of each timed step (its five stages)
    # dominant kernel: the tcgen05 backward (largest share of the step)
    bwd_tf = F_bwd / (bwd_ms * 1e-3) / 1e12
    fwd_tf = F_fwd / (fwd_ms * 1e-3) / 1e12
    # both kernels are event-timed inside a step of ~50 ms (under a second of timed steps):
    # the burst figure of the measured cuBLAS bf16 GEMM is the matching denominator
    peak = float(peaks["bf16_tflops"])
    clocks = summarize_clocks(clock_lines, dev.index or 0)
    # the same rates at the maximum SM clock, from the clocks sampled in the timed region
    clk = (clocks["sm_max_mhz"] / clocks["sm_mhz"]) if clocks.get("sm_mhz") and clocks.get("sm_max_mhz") else None
    traffic = recorded_traffic("zl_bwd_main")
    # algorithmic bytes of the HBM-bound kernels
    merge_bytes = 0
    for g in range(plan.n_groups):
        members, _, _ = plan.group(g)
        it = work.items[members[0]]
        merge_bytes += len(members) * it.nq * it.nh * (4 * d + 4) + it.nq * it.nh * (2 * d + 4)
    pre_bytes = sum(it.nq * it.nh * (2 * d + 2 * d + 4 + 4 * d) for it in work.items)
    fin_bytes = sum(it.nq * it.nh * 8 * d for it in work.items)
    hbm = float(peaks["hbm_gbs"])
    extra = {}
    if rank == 0 and not args.no_extras:
        # the co-location check and the forward-only lists, after the timed region
        extra["additivity"] = additivity_numbers(work, q, k, v, do_tok, dev, stream, 3)
        del bufs, d_o
        torch.cuda.empty_cache()
        extra["forward_configs"] = forward_config_numbers(dev, stream, 5, 2, peak)
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": work.name, "n_heads": H, "head_dim": d, "total_tokens": T,
                       "items": len(work.items), "fwd_tflop": F_fwd / 1e12, "bwd_tflop": F_bwd / 1e12,
                       "l2": "inputs larger than L2 (Q, K, V, dO 302 MB each)",
                       "parallelism": f"replicas x{ws}", "fused_kmerge": bool(args.fuse_kmerge),
                       "deterministic_dq": bool(args.deterministic)},
            "fwd_tflops": fwd_tf, "bwd_tflops": bwd_tf,
            "stage_ms": {"fwd": fwd_ms, "merge": merge_ms, "bwd_preprocess": pre_ms, "bwd_main": bwd_ms,
                         "bwd_finalize": fin_ms},
            "step_ms": {"median": float(np.median(step_each)), "min": float(step_each.min()),
                        "max": float(step_each.max())},
            "merge_gbs": merge_bytes / (merge_ms * 1e-3) / 1e9 if merge_ms > 0 and plan.n_merge_groups else None,
            "bwd_preprocess_gbs": pre_bytes / (pre_ms * 1e-3) / 1e9 if pre_ms > 0 else None,
            "bwd_finalize_gbs": fin_bytes / (fin_ms * 1e-3) / 1e9 if fin_ms > 0 else None,
            "hbm_peak_gbs": hbm,
            "plan_ms": t_plan * 1e3,
            "roofline": {"kernel": "zl_bwd_main (tcgen05 backward)", "bound": "tensor", "achieved": bwd_tf,
                         "peak": peak, "peak_kind": f"{peak_kind} bf16 burst", "unit": "TFLOP/s",
                         "frac": bwd_tf / peak, "traffic": traffic,
                         "clock_adjusted": ({"achieved": bwd_tf * clk, "frac": bwd_tf * clk / peak,
                                             "sm_mhz": clocks["sm_mhz"], "sm_max_mhz": clocks["sm_max_mhz"]}
                                            if clk else None),
                         "fwd": {"achieved": fwd_tf, "frac": fwd_tf / peak,
                                 "clock_adjusted_frac": fwd_tf * clk / peak if clk else None}},
            # forward, merge (unless every group is fused), row sums, backward, finalize
            "gpu_launches": (4 + (1 if plan.n_merge_groups else 0)) * args.steps,
            "clocks": clocks,
        }
        line.update(extra)
        if e2e is not None:
            line["e2e"] = e2e
        if ws == 1 and not args.no_cpu_baseline:
            v_cpu, dt, desc = cpu_oracle_sample(work)
            line["cpu_baseline"] = {"value": v_cpu, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                                    "sample": desc, "seconds": dt}
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


def additivity_numbers(work, q, k, v, do_tok, dev, stream, reps):
    """Co-location check of the additive time model: every work item timed alone (a plan
    holding only that item, same inputs) against the coalesced launch of the whole list,
    forward + merge + backward.  The pages' profiler prices each (bucket, configuration)
    pair separately and takes a rank's time as their sum, assuming that co-locating whole
    sequences with shards costs nothing extra (pith.science review, "Load-bearing premise").
    ratio = coalesced / sum of solo times: 1.0 means additive, < 1 means co-location helps
    (the persistent launch fills SMs that a lone item would leave idle).  Each plan runs
    one untimed step, then `reps` steps between two events; the median of three such
    rounds is kept."""
    import torch
    from coalesced_packed_attention_gb300 import zl
    H, d, T, scale = work.n_heads, work.head_dim, work.total_tokens, work.scale

    def timed(items):
        plan = zl.zl_plan_worklist(items, H, d, T)
        d_o = dO_arena(plan, type(work)(work.name, H, d, T, list(items), scale), do_tok, dev)
        bufs = zl.allocate(plan, dev, backward=True)

        def step():
            zl.zl_coalesced_attn_fwd(plan, q, k, v, bufs["o"], bufs["o_partial"], bufs["lse"], scale, stream)
            zl.zl_merge_partials(plan, bufs["o_partial"], bufs["lse"], bufs["o"], bufs["lse"], stream)
            zl.zl_coalesced_attn_bwd(plan, q, k, v, bufs["o"], d_o, bufs["lse"], bufs["dq"], bufs["dk"], bufs["dv"],
                                     bufs["workspace"], scale, stream)
        step()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        rounds = []
        for _ in range(3):
            torch.cuda.synchronize(dev)
            a.record(stream)
            for _ in range(reps):
                step()
            b.record(stream)
            torch.cuda.synchronize(dev)
            rounds.append(a.elapsed_time(b) / reps)
        if zl.zl_get_device_status(plan, stream) != 0:
            raise RuntimeError("device status in the co-location check")
        del bufs, d_o
        plan.destroy()
        return float(np.median(rounds))

    coalesced = timed(work.items)
    solo = [timed([it]) for it in work.items]
    return {"workload": work.name, "coalesced_ms": coalesced, "sum_solo_ms": float(sum(solo)),
            "ratio": coalesced / float(sum(solo)), "reps": reps,
            "items": [{"label": lab, "solo_ms": s, "fwd_tflop": it.fwd_flops(d) / 1e12}
                      for lab, s, it in zip(work.labels, solo, work.items)]}


def run_additivity(args):
    """--additivity: the co-location check alone (its own JSON line)."""
    import torch
    from coalesced_packed_attention_gb300 import zl
    from coalesced_packed_attention_gb300.workloads import config_training, make_inputs

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    zl.load_library()
    work = config_training()
    if args.scale > 1:
        from coalesced_packed_attention_gb300.workloads import scaled
        work = scaled(work, args.scale)
    q, k, v, do_tok = make_inputs(work.total_tokens, work.n_heads, work.head_dim, seed=0, with_grad_output=True,
                                  device=str(dev))
    stream = torch.cuda.current_stream(dev)
    print(json.dumps({"additivity": additivity_numbers(work, q, k, v, do_tok, dev, stream, max(2, args.steps))}),
          flush=True)


def forward_config_numbers(dev, stream, steps, warmup, peak):
    """Forward (+ merge) TFLOP/s of the forward-only work lists: 64 whole images
    (48 x 256, 12 x 1024, 4 x 4096 tokens), and the 147600-token video as 8 k chunks
    beside 8 x 4096-token images, merged (fp32 partials + merge launch) and with the
    k-split group fused into the forward (ZL_PLAN_FUSE_LOCAL_KMERGE).  After the warm-up,
    `steps` iterations or as many as fill ~50 ms (at most 200) run back to back, each
    bracketed by events, with one synchronize at the end; median of them.  The merge's
    GB/s from its algorithmic bytes."""
    import torch
    from coalesced_packed_attention_gb300 import zl
    from coalesced_packed_attention_gb300.workloads import config_images, config_long_video, make_inputs

    out = []
    for work, flags, tag in ((config_images(), 0, "merged"), (config_long_video(), 0, "merged"),
                             (config_long_video(), zl.ZL_PLAN_FUSE_LOCAL_KMERGE, "fused")):
        H, d, T, scale = work.n_heads, work.head_dim, work.total_tokens, work.scale
        q, k, v = make_inputs(T, H, d, seed=0, device=str(dev))[:3]
        plan = zl.zl_plan_worklist(work.items, H, d, T, flags)
        bufs = zl.allocate(plan, dev)
        def launch(evs):
            evs[0].record(stream)
            zl.zl_coalesced_attn_fwd(plan, q, k, v, bufs["o"], bufs["o_partial"], bufs["lse"], scale, stream)
            evs[1].record(stream)
            zl.zl_merge_partials(plan, bufs["o_partial"], bufs["lse"], bufs["o"], bufs["lse"], stream)
            evs[2].record(stream)

        warm = []
        for _ in range(max(2, warmup)):
            evs = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            launch(evs)
            torch.cuda.synchronize(dev)
            warm.append(evs[0].elapsed_time(evs[2]))
        n = max(steps, min(200, int(50.0 / max(min(warm), 1e-3))))
        evs_all = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]
        for evs in evs_all:
            launch(evs)
        torch.cuda.synchronize(dev)
        times = [(e[0].elapsed_time(e[1]), e[1].elapsed_time(e[2])) for e in evs_all]
        if zl.zl_get_device_status(plan, stream) != 0:
            raise RuntimeError(f"device status after {work.name}")
        f_ms = float(np.median([a for a, _ in times]))
        m_ms = float(np.median([b for _, b in times]))
        F = work.fwd_flops()
        merge_bytes = 0
        for g in range(plan.n_groups):
            members, _, _ = plan.group(g)
            it = work.items[members[0]]
            if plan.n_merge_groups:
                merge_bytes += len(members) * it.nq * it.nh * (4 * d + 4) + it.nq * it.nh * (2 * d + 4)
        tf = F / ((f_ms + m_ms) * 1e-3) / 1e12
        out.append({"workload": work.name, "kmerge": tag if plan.n_groups else None, "fwd_tflop": F / 1e12,
                    "iterations": n, "fwd_ms": f_ms, "merge_ms": m_ms, "tflops_fwd_plus_merge": tf,
                    "tflops_fwd": F / (f_ms * 1e-3) / 1e12, "frac_fwd_plus_merge": tf / peak,
                    "merge_gbs": merge_bytes / (m_ms * 1e-3) / 1e9 if merge_bytes and m_ms > 0 else None,
                    "fwd_tiles": plan.n_fwd_tiles})
        del bufs, q, k, v
        plan.destroy()
        torch.cuda.empty_cache()
    return out


def run_forward_configs(args):
    """--forward-configs: the forward-only lists alone (one JSON line)."""
    import torch
    from coalesced_packed_attention_gb300 import zl
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    zl.load_library()
    peaks, _ = measured_peaks()
    print(json.dumps({"forward_configs": forward_config_numbers(dev, torch.cuda.current_stream(dev), args.steps,
                                                                args.warmup, float(peaks["bf16_tflops"]))}),
          flush=True)


def run_kmerge_compare(args):
    """Forward of the long-video list (a 147600-token video as 8 k-split chunks of
    18450 KV tokens over all rows and heads, plus 8 whole 4096-token images), timed with
    the chunks' fp32 partials and the merge launch, and with the group fused into the
    forward (ZL_PLAN_FUSE_LOCAL_KMERGE: one item over the whole KV range, final O and LSE
    written directly).  Same algorithmic FLOPs; the fused step skips writing and
    re-reading the partials."""
    import torch
    from coalesced_packed_attention_gb300 import zl
    from coalesced_packed_attention_gb300.workloads import config_long_video, make_inputs, scaled

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    work = config_long_video()
    if args.scale > 1:
        work = scaled(work, args.scale)
    H, d, T, scale = work.n_heads, work.head_dim, work.total_tokens, work.scale
    q, k, v = make_inputs(T, H, d, seed=0, device=str(dev))[:3]
    stream = torch.cuda.current_stream(dev)
    F = work.fwd_flops()
    out = {"workload": work.name, "fwd_tflop": F / 1e12}
    for name, flags in (("merged", 0), ("fused", zl.ZL_PLAN_FUSE_LOCAL_KMERGE)):
        plan = zl.zl_plan_worklist(work.items, H, d, T, flags)
        bufs = zl.allocate(plan, dev)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]

        def step(record=False):
            if record:
                ev[0].record(stream)
            zl.zl_coalesced_attn_fwd(plan, q, k, v, bufs["o"], bufs["o_partial"], bufs["lse"], scale, stream)
            if record:
                ev[1].record(stream)
            zl.zl_merge_partials(plan, bufs["o_partial"], bufs["lse"], bufs["o"], bufs["lse"], stream)
            if record:
                ev[2].record(stream)
        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize(dev)
        fwd, mrg = [], []
        for _ in range(args.steps):
            step(True)
            torch.cuda.synchronize(dev)
            fwd.append(ev[0].elapsed_time(ev[1]))
            mrg.append(ev[1].elapsed_time(ev[2]))
        if zl.zl_get_device_status(plan, stream) != 0:
            raise RuntimeError("device status after the k-merge comparison")
        ms = float(np.median(np.array(fwd) + np.array(mrg)))
        out[name] = {"ms_per_step": ms, "fwd_ms": float(np.median(fwd)), "merge_ms": float(np.median(mrg)),
                     "tflops": F / (ms * 1e-3) / 1e12, "o_partial_bytes": 4 * plan.o_partial_elems}
        del bufs
        plan.destroy()
    out["speedup"] = out["merged"]["ms_per_step"] / out["fused"]["ms_per_step"]
    print(json.dumps({"kmerge_compare": out}), flush=True)


def run_planner(args):
    """Host placement slice (no GPU): catalog cut and filler packing of a synthetic
    batch of 10 000 sequences (images of 256-4096 tokens, videos of 8k-147k tokens,
    time ~ L^2, memory ~ L) over 32 ranks, the anchors q-split evenly over all ranks
    (parity with the oracle is checked by the tests, not here)."""
    import random
    from coalesced_packed_attention_gb300 import zl

    rng = random.Random(0)
    img = [256, 512, 1024, 2048, 4096]
    vid = [8190, 16380, 32760, 65520, 147600]
    lengths = [rng.choice(img) for _ in range(9600)] + [rng.choice(vid) for _ in range(400)]
    N, H, d = 32, 24, 128
    t_of = lambda L: 3.5 * 4.0 * L * L * d * H / 1.3e15   # noqa: E731  seconds at ~1.3 PFLOP/s
    m_of = lambda L: 10.0 * L * H * d * 2 / 1e9          # noqa: E731  GB, ten [L, H, d] bf16 tensors
    counts = {}
    for L in lengths:
        counts[L] = counts.get(L, 0) + 1
    cat = sorted(((L, n, t_of(L), m_of(L)) for L, n in counts.items()), key=lambda b: (b[2], b[0]))

    # inputs of the packing: the anchors' per-rank load (q-split evenly) and the fillers
    k, _ = zl.catalog_cut(cat)
    fl = {b[0] for b in cat[:k]}
    anchor_t = sum(t_of(L) for L in lengths if L not in fl) / N
    anchor_m = sum(m_of(L) for L in lengths if L not in fl) / N
    rt, rm = [anchor_t] * N, [anchor_m] * N
    ft = [t_of(L) for L in lengths if L in fl]
    fm = [m_of(L) for L in lengths if L in fl]

    def lib_run():  # the two library calls, argument marshalling included
        kk, _ = zl.catalog_cut(cat)
        return kk, zl.pack_fillers(ft, fm, N, rt, rm, 0.0, 180.0)

    for _ in range(3):
        lib_run()
    reps = 50
    t0 = time.perf_counter()
    for _ in range(reps):
        k, res = lib_run()
    lib_ms = (time.perf_counter() - t0) * 1e3 / reps
    lb = max(max(rt), (sum(rt) + sum(ft)) / N)
    print(json.dumps({"planner": {
        "sequences": len(lengths), "ranks": N, "buckets": len(cat), "k_star": k, "fillers": len(ft),
        "library_ms": lib_ms, "makespan_s": res[4], "lower_bound_s": lb,
        "makespan_over_lower_bound": res[4] / lb, "overflow": res[3]}}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the co-location check and the forward-only lists after the timed region")
    ap.add_argument("--scale", type=int, default=1,
                    help="divide every length of the list by this factor (profiler captures only)")
    ap.add_argument("--additivity", action="store_true",
                    help="time every work item alone and the coalesced list (co-location check)")
    ap.add_argument("--fuse-kmerge", action="store_true",
                    help="plan with ZL_PLAN_FUSE_LOCAL_KMERGE (k-split groups fused into the forward)")
    ap.add_argument("--deterministic", action="store_true",
                    help="plan with ZL_PLAN_DETERMINISTIC_DQ (ordered, bitwise reproducible dQ adds)")
    ap.add_argument("--kmerge-compare", action="store_true",
                    help="time the long-video forward list merged and fused")
    ap.add_argument("--forward-configs", action="store_true",
                    help="forward (+ merge) TFLOP/s of the images, mixed and long-video lists")
    ap.add_argument("--planner", action="store_true",
                    help="time the host placement slice (catalog cut, filler packing) on a synthetic batch")
    args = ap.parse_args()
    if args.planner:
        run_planner(args)
    elif args.forward_configs:
        run_forward_configs(args)
    elif args.kmerge_compare:
        run_kmerge_compare(args)
    elif args.additivity:
        run_additivity(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
