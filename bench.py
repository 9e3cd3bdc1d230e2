"""Benchmark: descriptor-guided masked attention, forward + backward, on one GB300.

One step = the whole hot path on one batch of synthetic input already resident in HBM:
Execution Descriptor build (preprocess kernels, forward and backward halves), attention forward,
attention backward (D prologue, main kernel, dQ conversion).

Metric: effective TFLOP/s over visible pairs only: sum_b 14 * d * V_b * H / step time, where
V_b is the number of visible (query, key) pairs of sample b (4 d V for the forward's two
matmuls, 10 d V for the backward's five).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config 3] [--impl reference]

Prints one JSON line (rank 0).  ``--impl reference`` times the fp64 CPU oracle on the host cores
on a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "masked attn fwd+bwd effective TFLOP/s (visible FLOPs) at 32K; % BF16 peak"
UNIT = "TFLOP/s"
FLOPS_PER_PAIR_PER_D = 14  # 4 (forward) + 10 (backward)
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------------------------------------
# clocks sampled during the timed region
# ------------------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[5 + k] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------------------------------------
# distributed helpers (replicas: every rank runs the whole workload on its own GPU)
# ------------------------------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def aggregate(seconds: float, units: float, world: int):
    """Max time over ranks and total units over ranks (weak scaling: each rank has its own)."""
    if world == 1:
        return seconds, units
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([seconds], dtype=torch.float64, device=dev)
    u = torch.tensor([units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


# ------------------------------------------------------------------------------------------------
# reference arm / CPU baseline: the fp64 oracle on a bounded sample
# ------------------------------------------------------------------------------------------------
def oracle_sample(wid: int, rows: int):
    """Time the oracle's forward + backward on `rows` query rows of head (0, 0) of the workload.

    Returns (seconds, visible pairs in the sample, cores used, description)."""
    import numpy as np
    import torch

    from masked_flashattention_gb300 import workloads as W
    from oracle import attention as A
    from oracle import masks as M

    cores = len(os.sched_getaffinity(0))
    torch.set_num_threads(cores)
    w = W.WORKLOADS[wid]
    seg, nseg = W.segments(wid, w.B, w.S)
    q, k, v, do = W.head_tensors(wid, 0, 0, w.S, w.d, w.H)
    r1 = w.S
    r0 = max(0, r1 - rows)  # the last rows see the most keys
    idx = np.arange(r0, r1)
    mask = M.dense_mask(wid, seg[0], int(nseg[0]), w.S, rows=idx)
    t0 = time.perf_counter()
    A.attention_forward(q[r0:r1], k, v, mask, block_rows=1024)
    A.attention_backward(q[r0:r1], k, v, do[r0:r1], mask, block_rows=1024)
    dt = time.perf_counter() - t0
    pairs = int(mask.sum())
    desc = (f"{w.name}: fp64 oracle forward+backward of query rows [{r0}, {r1}) of head (0, 0) "
            f"against all {w.S} keys ({pairs} visible pairs)")
    return dt, pairs, torch.get_num_threads(), desc


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    from masked_flashattention_gb300 import workloads as W
    w = W.WORKLOADS[args.config]
    # each step is a bounded sample: about 8192 rows x 33 steps of CPU work in total (a few
    # minutes on the GB300 host), whatever K and W are
    rows = args.ref_rows or max(256, min(w.S, (8192 * 33) // max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample(args.config, rows)
    times, pairs, cores, desc = [], 0, 0, ""
    for _ in range(args.steps):
        dt, pairs, cores, desc = oracle_sample(args.config, rows)
        times.append(dt)
    total = sum(times)
    flops = FLOPS_PER_PAIR_PER_D * w.d * pairs * args.steps
    value = flops / total / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": w.name, "B": w.B, "H": w.H, "S": w.S, "d": w.d,
                                        "sample_rows": rows},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line))
    return 0


# ------------------------------------------------------------------------------------------------
# GPU arm
# ------------------------------------------------------------------------------------------------
def visible_pairs(desc, B: int, S: int):
    """Visible pairs per sample from the device Interval Table (union of each row's slots)."""
    import torch
    t = desc.itab_f.view(B, desc.ni_f, S, 2).long()
    s, e = t[..., 0], t[..., 1]
    order = torch.argsort(s, dim=1)
    s = torch.gather(s, 1, order)
    e = torch.gather(e, 1, order)
    run_end = torch.zeros(B, S, dtype=torch.long, device=t.device)
    total = torch.zeros(B, S, dtype=torch.long, device=t.device)
    for n in range(desc.ni_f):
        sn, en = s[:, n], e[:, n]
        valid = en > sn
        start = torch.maximum(sn, run_end)
        total += torch.where(valid, (en - start).clamp(min=0), torch.zeros_like(total))
        run_end = torch.where(valid, torch.maximum(run_end, en), run_end)
    return [int(x) for x in total.sum(dim=1).tolist()]


def preprocess_sweep(Bd, fwd, bwd, seg_np, nseg_np, S, dev, target_mb=64.0, reps=20):
    """Descriptor build replicated over a batch large enough that the descriptor (>= 64 MB)
    exceeds what launch latency hides: achieved HBM GB/s of the preprocess kernels."""
    import numpy as np
    import torch
    per_sample = sum(Bd.cm_descriptor_sizes(fwd, bwd, 1, S))
    nt = S // 128
    Bs = max(1, min(32768 // nt, math.ceil(target_mb * 2**20 / per_sample)))
    rep = math.ceil(Bs / seg_np.shape[0])
    seg = torch.from_numpy(np.tile(seg_np, (rep, 1))[:Bs].copy()).to(dev)
    nseg = torch.from_numpy(np.tile(nseg_np, rep)[:Bs].copy()).to(dev)
    desc = Bd.Descriptor(fwd, bwd, Bs, S, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(3):
        Bd.cm_build_descriptor(fwd, bwd, seg, nseg, desc, stream)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(reps):
        Bd.cm_build_descriptor(fwd, bwd, seg, nseg, desc, stream)
    b.record(stream)
    torch.cuda.synchronize(dev)
    us = a.elapsed_time(b) * 1e3 / reps
    nbytes = seg.numel() * 4 + nseg.numel() * 4 + desc.nbytes()
    return {"B": Bs, "MB": nbytes / 2**20, "us": us, "gbs": nbytes / (us * 1e-6) / 1e9}


def run_gpu(args):
    import torch
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)

    from masked_flashattention_gb300 import binding as Bd
    from masked_flashattention_gb300 import specs
    from masked_flashattention_gb300 import workloads as W

    Bd.lib()
    w = W.WORKLOADS[args.config]
    if args.heads:
        w = W.Workload(w.id, f"{w.name}@H{args.heads}", w.B, args.heads, w.S, w.d)
    Bn, H, S, d = w.B, w.H, w.S, w.d
    scale = 1.0 / math.sqrt(d)
    seg_np, nseg_np = W.segments(w.id, Bn, S)
    fwd, bwd = Bd.cm_compile_spec(specs.FWD[w.id]), Bd.cm_compile_spec(specs.BWD[w.id])
    desc = Bd.Descriptor(fwd, bwd, Bn, S, device=dev)
    seg = torch.from_numpy(seg_np).to(dev)
    nseg = torch.from_numpy(nseg_np).to(dev)

    g = torch.Generator(device=dev)
    g.manual_seed(2000 + w.id + 97 * rank)
    shape = (Bn, H, S, d)
    q, k, v, do = (torch.randn(shape, generator=g, device=dev, dtype=torch.float32)
                   .to(torch.bfloat16) for _ in range(4))
    o = torch.empty_like(q)
    lse = torch.empty(Bn, H, S, dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(Bd.cm_attn_bwd_workspace_size(Bn, H, S, d), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        Bd.cm_build_descriptor(fwd, bwd, seg, nseg, desc, stream)
        if ev is not None:
            ev[1].record(stream)
        Bd.cm_attn_fwd(desc, q, k, v, o, lse, scale, stream)
        if ev is not None:
            ev[2].record(stream)
        Bd.cm_attn_bwd(desc, q, k, v, o, lse, do, dq, dk, dv, ws, scale, stream)
        if ev is not None:
            ev[3].record(stream)

    step()
    torch.cuda.synchronize(dev)
    st = Bd.cm_get_status(desc)
    if st != 0:
        raise RuntimeError(f"device status {st}: {Bd.cm_error_string(st)}")
    pairs = visible_pairs(desc, Bn, S)
    flops = FLOPS_PER_PAIR_PER_D * d * H * sum(pairs)
    fwd_flops = 4 * d * H * sum(pairs)
    bwd_flops = 10 * d * H * sum(pairs)

    for _ in range(args.warmup):
        step()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    clocks = ClockSampler(local)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    clocks.start()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for s in range(args.steps):
        step(evs[s])
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    if world > 1:
        torch.distributed.barrier()
    elapsed = t_start.elapsed_time(t_end) / 1e3
    build_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    fwd_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
    bwd_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in evs)
    st = Bd.cm_get_status(desc)
    if st != 0:
        raise RuntimeError(f"device status {st}: {Bd.cm_error_string(st)}")

    t_max, units = aggregate(elapsed, flops * args.steps, world)
    value = units / t_max / 1e12

    # ---- optional: the partial-tile check forms of the paper's section 4.4 ablation ----
    ablation = None
    if args.ablation:
        ablation = {}
        names = {Bd.CM_CHECK_UNSIGNED: "unsigned_visible", Bd.CM_CHECK_TWO_COMPARE: "two_compare_visible",
                 Bd.CM_CHECK_MASKED: "masked_intervals"}
        for mode in (Bd.CM_CHECK_UNSIGNED, Bd.CM_CHECK_TWO_COMPARE, Bd.CM_CHECK_MASKED):
            Bd.cm_set_interval_check(mode)
            for _ in range(max(3, args.warmup)):
                step()
            aevs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
            torch.cuda.synchronize(dev)
            for s_ in range(args.steps):
                step(aevs[s_])
            torch.cuda.synchronize(dev)
            f_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in aevs)
            b_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in aevs)
            ablation[names[mode]] = {"fwd_ms": f_ms, "bwd_ms": b_ms, "fwd_bwd_ms": f_ms + b_ms}
        Bd.cm_set_interval_check(Bd.CM_CHECK_UNSIGNED)
        st = Bd.cm_get_status(desc)
        if st != 0:
            raise RuntimeError(f"device status {st}: {Bd.cm_error_string(st)}")
        base = ablation["unsigned_visible"]["fwd_bwd_ms"]
        for v_ in ablation.values():
            v_["vs_unsigned"] = v_["fwd_bwd_ms"] / base

    # ---- end to end through the public API with pinned host buffers ----
    hq, hk, hv, hdo = (t.cpu().pin_memory() for t in (q, k, v, do))
    hseg, hnseg = seg.cpu().pin_memory(), nseg.cpu().pin_memory()
    ho, hdq, hdk, hdv = (torch.empty(shape, dtype=torch.bfloat16).pin_memory() for _ in range(4))
    hlse = torch.empty(Bn, H, S, dtype=torch.float32).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hdo, hseg, hnseg))
    d2h = sum(t.numel() * t.element_size() for t in (ho, hlse, hdq, hdk, hdv))

    def e2e_step():
        for dst, src in ((q, hq), (k, hk), (v, hv), (do, hdo), (seg, hseg), (nseg, hnseg)):
            dst.copy_(src, non_blocking=True)
        step()
        for dst, src in ((ho, o), (hlse, lse), (hdq, dq), (hdk, dk), (hdv, dv)):
            dst.copy_(src, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize(dev)
    e2e_steps = max(1, min(args.steps, 5))
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    b_.record(stream)
    torch.cuda.synchronize(dev)
    e2e_t, e2e_units = aggregate(a.elapsed_time(b_) / 1e3, flops * e2e_steps, world)
    e2e_value = e2e_units / e2e_t / 1e12

    # ---- roofline of the dominant kernel (the backward pass) ----
    peaks, peak_src = load_peaks()
    peak = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    bwd_tf = bwd_flops / (bwd_ms / 1e3) / 1e12
    fwd_tf = fwd_flops / (fwd_ms / 1e3) / 1e12
    meta_bytes = seg.numel() * 4 + nseg.numel() * 4
    prep_bytes = meta_bytes + desc.nbytes()
    sweep = preprocess_sweep(Bd, fwd, bwd, seg_np, nseg_np, S, dev)
    if sweep is not None:
        sweep["pct_hbm"] = 100.0 * sweep["gbs"] / float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    traffic = None
    tp = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tp):
        import hashlib
        with open(tp) as f:
            rec = json.load(f).get(f"attn_bwd@{w.name}")
        def sha1(name):
            with open(os.path.join(ROOT, "masked_flashattention_gb300", "csrc", name), "rb") as f:
                return hashlib.sha1(f.read()).hexdigest()
        # counters only count for the kernel sources they were measured on
        if rec and all(sha1(n) == h for n, h in rec.get("source_sha1", {}).items()):
            traffic = rec["bytes"]

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t_max / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": w.name, "B": Bn, "H": H, "S": S, "d": d,
                       "visible_pairs_per_head": pairs, "parallelism": f"replicas{world}",
                       "l2": "inputs larger than L2 (each of Q, K, V, dO is "
                             f"{q.numel() * 2 / 2**20:.0f} MiB); no flush",
                       "pct_bf16_peak": 100.0 * value / peak,
                       "fwd_ms": fwd_ms, "bwd_ms": bwd_ms, "build_ms": build_ms,
                       "fwd_tflops": fwd_tf, "bwd_tflops": bwd_tf,
                       "preprocess_gbs": prep_bytes / (build_ms / 1e3) / 1e9,
                       "preprocess_sweep": sweep,
                       "peak_source": f"{peak_src} bf16_tflops_sustained"},
            "roofline": {"bound": "tensor", "kernel": "attention backward (prologue + dK/dV kernel + dQ kernel)",
                         "achieved": bwd_tf, "peak": peak, "unit": "TFLOP/s",
                         "frac": bwd_tf / peak, "traffic": traffic},
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            # per step: descriptor (2 generated kernels + schedule), forward, backward (prologue,
            # dK/dV, dQ)
            "gpu_launches": 7 * args.steps,
            "clocks": clk,
        }
        if ablation is not None:
            line["ablation"] = ablation
        if world == 1 and not args.no_cpu_baseline:
            dt, pr, cores, sdesc = oracle_sample(args.config, args.ref_rows or 8192)
            line["cpu_baseline"] = {"value": FLOPS_PER_PAIR_PER_D * d * pr / dt / 1e12,
                                    "unit": UNIT, "cores": cores, "kind": "oracle",
                                    "sample": sdesc}
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--config", type=int, default=3, help="workload 1..6 (default: 3, RM 32K)")
    ap.add_argument("--impl", default="cm", choices=["cm", "reference"])
    ap.add_argument("--ref-rows", type=int, default=0,
                    help="query rows of the oracle sample (default: sized to the run length)")
    ap.add_argument("--heads", type=int, default=0,
                    help="override the head count (small cases for profiler captures)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ablation", action="store_true",
                    help="also time the three partial-tile check forms (section 4.4); use with --config 4")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
