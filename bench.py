"""Reshard executor benchmark: destination GB/s on one GB300 (device-timed) and % of HBM roofline.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--mode direct|packed] [--suite FILE]

A step is one reshard of the whole workload (every tensor, one batched plan, one execute) with
inputs resident in HBM. The plan is built once before timing (the descriptor cache a refit
reuses every step). The default workload is the largest single-GPU configuration, the MoE
expert refit EP16 -> EP8 (8 layers x 128 experts, 38.65 GB each way). The line's ``targets`` key
times, in the same run and the same way, the dense FFN refit (direct), the MoE refit into TP4
with MXFP8 on receive (direct), and the fused MXFP8 unpack pass alone (its own event pairs), each
against its fraction of the measured copy rate. Multi-GPU runs (torchrun, one rank per GPU) run
independent replicas of the same workload (weak scaling): with every shard of a workload on one
GPU there is no exchange step; the multi-process exchange (``exchange``) is exercised by the
tests. Prints ONE JSON line on rank 0.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "reshard GB/s (dst bytes, device-timed) on 1 GB300; % of HBM roofline"
DEFAULT_WORKLOAD = "moe_8x128x1536x4096_ep16_to_ep8"
NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e nominal, context only
FALLBACK_HBM_GBS = 6800.0


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def copy_rate_same_run(dev, nbytes: int = 4 << 30, reps: int = 10) -> float:
    """The box's device-to-device copy rate, re-measured in this run: read + write bytes per
    second of a torch copy between two 4 GiB buffers (far above the 129 MB L2), CUDA events."""
    import torch
    a = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    b = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    a.fill_(1)
    s = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(s):
        for _ in range(3):
            b.copy_(a)
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(s)
        for _ in range(reps):
            b.copy_(a)
        t1.record(s)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / reps
    del a, b
    torch.cuda.empty_cache()
    return 2 * nbytes / (ms / 1e3) / 1e9


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in ("execute.cu", "plan.h"):
        with open(os.path.join(ROOT, "dtensor_resharding_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str, mode: str):
    """DRAM bytes per launch from a committed ncu summary, if taken on the current kernel source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        recs = json.load(f)
    for r in recs:
        if (r.get("kernel") == kernel and r.get("workload") == workload and r.get("mode") == mode
                and r.get("source_hash") == kernel_source_hash()):
            return r.get("traffic_bytes_per_launch")
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while the bench runs."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,utilization.gpu,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.proc = None
        self.path = os.path.join("/tmp", f"reshard_clocks_{os.getpid()}.csv")
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        self.proc.wait()
        self.fh.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) == 8:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        busy = [r for r in rows if (num(r[3]) or 0) > 0] or rows
        sm = [num(r[0]) for r in busy if num(r[0]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in busy for i in range(4) if r[4 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": num(rows[0][1]),
                "power_w_max": max((num(r[2]) or 0) for r in rows), "reasons": reasons, "samples": len(busy)}


# ----------------------------------------------------------------------------- ranks

def max_over_ranks(value: float, world: int, device=None) -> float:
    """The largest of every rank's `value` (the slowest replica sets the job's time)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(bytes_per_step_per_rank: int, steps: int, world: int, max_ms: float) -> float:
    """Whole-job GB/s: every rank's bytes over the slowest rank's time (weak scaling)."""
    return world * bytes_per_step_per_rank * steps / (max_ms / 1e3) / 1e9


# ----------------------------------------------------------------------------- oracle timing

def time_oracle_sample(wl, src_host, src_off, budget_s: float, max_tensors: int):
    """Run the C oracle over the first tensors of the workload until ~budget_s of host time.

    Returns (dst bytes produced, seconds, tensors used). Single thread."""
    import numpy as np
    from oracle import coracle
    es_of = {"u8": 1, "bf16": 2, "f16": 2, "f32": 4, "i32": 4, "i64": 8}
    done_bytes, spent, used = 0, 0.0, 0
    for ti, t in enumerate(wl.tensors[:max_tensors]):
        es = es_of[t.dtype]
        dst = []
        for v in t.dst_views:
            n = wl.dst_buffer_numel[v.buffer] * (1 if wl.quant == "mxfp8" else es)
            dst.append(np.empty(n, np.uint8))
        sc = [np.empty(wl.dst_buffer_numel[v.buffer] // 32, np.uint8) for v in t.dst_views] if wl.quant == "mxfp8" else None
        sb = [src_host[src_off[v.buffer]: src_off[v.buffer] + wl.src_buffer_numel[v.buffer] * es] for v in t.src_views]
        t0 = time.perf_counter()
        coracle.reshard_tensor(t, sb, dst, wl.quant, sc)
        spent += time.perf_counter() - t0
        done_bytes += sum(d.size for d in dst) + (sum(s.size for s in sc) if sc else 0)
        used += 1
        if spent >= budget_s:
            break
    return done_bytes, spent, used


def time_oracle_parallel(wl, src_host, src_off, n_tensors: int):
    """The same oracle, unchanged, run on the first n_tensors tensors at once: one tensor per
    task on a pool of as many threads as host cores (the C oracle releases the GIL)."""
    from concurrent.futures import ThreadPoolExecutor
    cores = os.cpu_count() or 1
    ts = list(range(min(n_tensors, len(wl.tensors))))
    out_bytes = [0]

    def one(ti):
        sub = type(wl)(wl.name, [wl.tensors[ti]], wl.quant, wl.values, wl.src_buffer_numel, wl.src_buffer_dtype,
                       wl.dst_buffer_numel, wl.dst_buffer_dtype)
        b, _, _ = time_oracle_sample(sub, src_host, src_off, 1e30, 1)
        return b

    t0 = time.perf_counter()
    with ThreadPoolExecutor(cores) as ex:
        done = sum(ex.map(one, ts))
    secs = time.perf_counter() - t0
    out_bytes[0] = done
    return {"value": round(done / secs / 1e9, 4), "unit": "GB/s", "cores": cores, "seconds": round(secs, 2),
            "sample": f"the same {len(ts)} tensors, one per task on {cores} threads"}


def _scaled_first_tensor(wl, frac: float):
    """The workload's first tensor with one dim cut to about `frac` of its length (dense views):
    the outermost dim with room for that cut in whole multiples of the shard counts that split
    it (source times destination), else the dim with the most such room."""
    import numpy as np
    import synthetic as S
    t = wl.tensors[0]
    nd_ = len(t.global_shape)

    def splits(d):
        g = 1
        for mesh, pls in ((t.src_mesh, t.src_placements), (t.dst_mesh, t.dst_placements)):
            g *= int(np.prod([m for m, p in zip(mesh, pls) if p == f"S{d}"] or [1]))
        return g

    room = [t.global_shape[d] // splits(d) for d in range(nd_)]
    need = 1.0 / max(frac, 1e-9)
    cut = next((d for d in range(nd_) if room[d] >= need), int(np.argmax(room)))
    g = splits(cut)
    shape = list(t.global_shape)
    shape[cut] = max(g, int(t.global_shape[cut] * frac) // g * g)
    shape = tuple(shape)
    ns, nd = int(np.prod(t.src_mesh)), int(np.prod(t.dst_mesh))
    d = S.TensorDesc(t.name, shape, t.dtype, t.src_mesh, t.src_placements, t.dst_mesh, t.dst_placements,
                     [S.View(i) for i in range(ns)], [S.View(i) for i in range(nd)], t.seed, t.std)
    return S.workloads._size_buffers(S.Workload(wl.name, [d], wl.quant, wl.values), ns, nd)


def reference_arm(args, rank: int) -> None:
    """The oracle as it stands, timed on the host cores over a bounded sample per step."""
    if rank != 0:
        return
    import synthetic as S
    from oracle import coracle
    coracle.build()
    wl = S.workload_by_name(args.workload)
    steps_total = args.steps + args.warmup
    budget = 150.0  # seconds of oracle time for the whole run
    probe = S.Workload(wl.name, wl.tensors[:1], wl.quant, wl.values)
    probe = S.workloads._size_buffers(probe, len(wl.src_buffer_numel), len(wl.dst_buffer_numel))
    lay = S.allocate(probe, "cpu")
    S.fill_sources(probe, lay)
    _, t_one, _ = time_oracle_sample(probe, lay.src_slab.numpy(), lay.src_off, 0.0, 1)
    if t_one * steps_total <= budget:
        n = max(1, min(len(wl.tensors), int(budget / steps_total / max(t_one, 1e-6))))
        sample = S.Workload(wl.name, wl.tensors[:n], wl.quant, wl.values)
        sample = S.workloads._size_buffers(sample, len(wl.src_buffer_numel), len(wl.dst_buffer_numel))
        what = f"first {n} of {len(wl.tensors)} tensors per step"
    else:
        sample = _scaled_first_tensor(wl, budget / steps_total / t_one)
        n = 1
        what = (f"first tensor cut to {sample.tensors[0].global_shape} (of {wl.tensors[0].global_shape}) per step, "
                "same meshes and placements")
    lay = S.allocate(sample, "cpu")
    S.fill_sources(sample, lay)
    src = lay.src_slab.numpy()
    times, nbytes = [], 0
    for i in range(steps_total):
        b, sec, _ = time_oracle_sample(sample, src, lay.src_off, 1e30, n)
        if i >= args.warmup:
            times.append(sec)
            nbytes = b
    total = sum(times)
    value = nbytes * len(times) / total / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * total / len(times), 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": wl.name, "mode": "oracle (full broadcast then slice)", "sample_dst_bytes": nbytes},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": what + ", host buffers, one thread"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------------- our arm

def launches_per_execute(R, plan, mode: str) -> int:
    """Kernel launches the last execute enqueued (the library counts them)."""
    return R.reshard_plan_stats(plan)["last_launches"]


def dominant_kernel(R, plan, mode: str, quant: str) -> str:
    """The kernel that moves most of the bytes of the (last) pass of the last execute."""
    p = 0 if mode == "direct" else 2
    copy_items = R.reshard_plan_items(plan, p)[0]
    t_items = R.reshard_plan_items(plan, p + 3)[0]
    copy_elems = int((copy_items["rows"].astype("int64") * copy_items["run"]).sum()) if len(copy_items) else 0
    t_elems = int((t_items["rows"].astype("int64") * t_items["cols"]).sum()) if len(t_items) else 0
    if t_elems > copy_elems:
        return "reshard_transpose_kernel"
    if quant == "mxfp8":
        return "reshard_mxfp8_kernel"
    st = R.reshard_plan_stats(plan)
    counts = {"reshard_copy_aligned_kernel": st["last_aligned_items"],
              "reshard_copy_staged_kernel": st["last_staged_items"],
              "reshard_copy_gather_kernel": st["last_gather_items"],
              ("reshard_copy_rows_kernel" if st["last_rows_kernel"] else "reshard_copy_kernel"): st["last_general_items"]}
    return max(counts, key=counts.get)


# page-locked host copies of one rank's slabs may take at most this share of the host's memory,
# split over the ranks on the host; past it the end-to-end leg runs on a prefix of the tensors
E2E_HOST_FRACTION = 0.45


def host_ram_bytes():
    """Physical memory of this host in bytes, or None where sysconf does not say."""
    try:
        return os.sysconf("SC_PAGE_SIZE") * os.sysconf("SC_PHYS_PAGES")
    except (ValueError, OSError, AttributeError):
        return None


def e2e_prefix(wl, budget: int):
    """(workload, k): `wl` cut to its longest prefix of k tensors whose page-locked host copies
    (source, destination and scale slabs, laid out as for the device) fit in `budget` bytes;
    `wl` itself when all of it fits, (None, 0) when not even the first tensor does."""
    import synthetic as S

    def sub(k):
        w = S.Workload(wl.name, wl.tensors[:k], wl.quant, wl.values)
        return S.workloads._size_buffers(w, len(wl.src_buffer_numel), len(wl.dst_buffer_numel))

    def host_bytes(w):
        lay = S.allocate(w, "meta")
        return lay.src_slab.numel() + lay.dst_slab.numel() + (lay.scale_slab.numel() if lay.scale_slab is not None else 0)

    if host_bytes(wl) <= budget:
        return wl, len(wl.tensors)
    lo, hi = 0, len(wl.tensors) - 1  # the largest k that fits lies in [lo, hi]
    while lo < hi:
        mid = (lo + hi + 1) // 2
        if host_bytes(sub(mid)) <= budget:
            lo = mid
        else:
            hi = mid - 1
    return (sub(lo), lo) if lo else (None, 0)


def e2e_run(R, wl, plan, sp, dp, lay, args, quant, world, dev, dst_bytes, barrier, st):
    """End to end through the public call with host buffers.

    The headline figure passes page-locked host pointers straight to reshard_execute: every step
    the kernels read the step's sources from host memory and write its destinations to host
    memory over the host link, inside the timed region, with no staging copy in device memory
    (the bytes crossing the link are the step's source bytes in, once per destination replica
    group, and its destination bytes out). For context, `staged` runs the same step through
    device memory: copy-engine H2D of the source slab, the device-to-device reshard, D2H of the
    destination slab, on three streams with step k+1's H2D overlapping step k's D2H."""
    import dataclasses

    import torch
    hsrc = torch.empty(lay.src_slab.numel(), dtype=torch.uint8, pin_memory=True)
    hdst = torch.empty(lay.dst_slab.numel(), dtype=torch.uint8, pin_memory=True)
    hsc = (torch.empty(lay.scale_slab.numel(), dtype=torch.uint8, pin_memory=True)
           if lay.scale_slab is not None else None)
    hsrc.copy_(lay.src_slab)
    ek = args.e2e_steps

    # --- in place: the kernels stream host memory
    hl = dataclasses.replace(lay, src_slab=hsrc, dst_slab=hdst, scale_slab=hsc)
    hsp, hdp = R.workload_pointers(wl, hl)
    s = torch.cuda.Stream(device=dev)
    R.reshard_execute(plan, hsp, hdp, mode=args.mode, quant=quant, stream=s.cuda_stream)   # warm-up
    torch.cuda.synchronize()
    barrier()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(s)
    for _ in range(ek):
        R.reshard_execute(plan, hsp, hdp, mode=args.mode, quant=quant, stream=s.cuda_stream)
    t1.record(s)
    torch.cuda.synchronize()
    e_ms = max_over_ranks(t0.elapsed_time(t1), world, dev)
    # the host result must equal the device-resident run's (same plan, same sources)
    n_chk = min(hdst.numel(), 1 << 28)
    same = bool(torch.equal(hdst[:n_chk], lay.dst_slab[:n_chk].cpu()))
    out = {"value": round(job_throughput(dst_bytes, ek, world, e_ms), 3), "unit": "GB/s",
           "h2d_bytes_per_step": st["bytes_read"], "d2h_bytes_per_step": dst_bytes,
           "steps": ek, "ms_per_step": round(e_ms / ek, 3), "matches_device_result": same,
           "path": "reshard_execute on page-locked host sources and destinations: the kernels read "
                   "and write host memory over the host link inside the timed region"}

    # --- the host link's ceiling in this run: copy-engine H2D and D2H at the same time (the
    # same pinned buffers and device slabs; the H2D rewrites the device sources with their own
    # bytes), against which the in-place step's bytes in and out are set
    nb = min(hsrc.numel(), hdst.numel(), lay.dst_slab.numel(), 1 << 31)
    s_a, s_b = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def both():
        with torch.cuda.stream(s_a):
            lay.src_slab[:nb].copy_(hsrc[:nb], non_blocking=True)
        with torch.cuda.stream(s_b):
            hdst[:nb].copy_(lay.dst_slab[:nb], non_blocking=True)

    both()
    torch.cuda.synchronize()
    start, end_a, end_b = (torch.cuda.Event(enable_timing=True) for _ in range(3))
    start.record(s_a)
    s_b.wait_event(start)
    reps = 3
    for _ in range(reps):
        both()
    end_a.record(s_a)
    end_b.record(s_b)
    torch.cuda.synchronize()
    l_ms = max(start.elapsed_time(end_a), start.elapsed_time(end_b))
    link_each = nb * reps / (l_ms / 1e3) / 1e9
    in_place_each = (st["bytes_read"] + dst_bytes) / 2 * ek / (e_ms / 1e3) / 1e9
    out["link"] = {"copy_engines_each_way_GBps": round(link_each, 1), "in_place_each_way_GBps": round(in_place_each, 1),
                   "frac_of_link": round(in_place_each / link_each, 3),
                   "what": "copy-engine H2D and D2H of 2 GiB pinned buffers at the same time, this run; the "
                           "in-place step's source bytes in and destination bytes out per second, averaged"}

    # --- staged through device memory with copy-engine transfers
    s_in, s_run, s_out = (torch.cuda.Stream(device=dev) for _ in range(3))

    def step(prev_out_done, prev_run_done):
        in_done, run_done, out_done = (torch.cuda.Event() for _ in range(3))
        with torch.cuda.stream(s_in):
            if prev_run_done is not None:
                s_in.wait_event(prev_run_done)        # the previous reshard has read the sources
            lay.src_slab.copy_(hsrc, non_blocking=True)
            in_done.record(s_in)
        s_run.wait_event(in_done)
        if prev_out_done is not None:
            s_run.wait_event(prev_out_done)           # the previous destinations have left
        R.reshard_execute(plan, sp, dp, mode=args.mode, quant=quant, stream=s_run.cuda_stream)
        run_done.record(s_run)
        with torch.cuda.stream(s_out):
            s_out.wait_event(run_done)
            hdst.copy_(lay.dst_slab, non_blocking=True)
            if hsc is not None:
                hsc.copy_(lay.scale_slab, non_blocking=True)
            out_done.record(s_out)
        return out_done, run_done

    step(None, None)                                  # warm-up step
    torch.cuda.synchronize()
    barrier()
    t0.record(s_in)
    o, r = None, None
    for _ in range(ek):
        o, r = step(o, r)
    s_in.wait_event(o)
    t1.record(s_in)
    torch.cuda.synchronize()
    g_ms = max_over_ranks(t0.elapsed_time(t1), world, dev)
    out["staged"] = {"value": round(job_throughput(dst_bytes, ek, world, g_ms), 3), "unit": "GB/s",
                     "ms_per_step": round(g_ms / ek, 3), "h2d_bytes_per_step": lay.src_slab.numel(),
                     "d2h_bytes_per_step": lay.dst_slab.numel() + (hsc.numel() if hsc is not None else 0)}
    del hsrc, hdst, hsc
    return out


# spec targets, as fractions of the measured copy rate
TARGETS = [
    ("dense_ffn_32x14336x4096_tp8_to_dp2tp2", "direct", 0.80),
    ("moe_8x128x1536x4096_ep16_to_tp4_mxfp8", "direct", None),
    ("moe_8x128x1536x4096_ep16_to_tp4_mxfp8", "fused_unpack", 0.70),
]


def time_calls(call, stream, k, warm, world, dev, barrier):
    """k calls back to back between one event pair, then k more each in its own event pair.
    Returns (max-over-ranks ms of the k back-to-back calls, per-call ms list)."""
    import torch
    for _ in range(warm):
        call()
    stream.synchronize()
    barrier()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(k):
        call()
    end.record(stream)
    torch.cuda.synchronize()
    barrier()
    total = max_over_ranks(start.elapsed_time(end), world, dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(k)]
    for a, b in ev:
        a.record(stream)
        call()
        b.record(stream)
    torch.cuda.synchronize()
    return total, [a.elapsed_time(b) for a, b in ev]


def measure_target(name, how, goal, steps, warm, world, dev, barrier, peak):
    """One spec target on its full-size workload, timed like the headline."""
    import torch

    import dtensor_resharding_gb300 as R
    import synthetic as S
    wl = S.workload_by_name(name)
    lay = S.allocate(wl, dev)
    S.fill_sources(wl, lay)
    plan = R.plan_workload(wl)
    st = R.reshard_plan_stats(plan)
    sp, dp = R.workload_pointers(wl, lay)
    stream = torch.cuda.Stream(device=dev)
    sh = stream.cuda_stream
    dst_bytes = wl.dst_bytes()
    out = {"workload": name, "mode": how}
    msg = None
    if how == "fused_unpack":
        # messages packed once (unquantized BF16 regions, 16-byte aligned); the timed call is the
        # unpack pass alone: messages in, E4M3 bytes and E8M0 scales out, fanned out to replicas
        msg = torch.empty(st["message_bytes"], dtype=torch.uint8, device=dev)
        R.reshard_execute_pack(plan, sp, None, msg, stream=sh)

        def call():
            R.reshard_execute_unpack(plan, msg, dp, quant=wl.quant, stream=sh)
        algo = st["bytes_read"] + dst_bytes
        out["read"] = "packed messages (the region bytes, 16-byte aligned)"
    else:
        def call():
            R.reshard_execute(plan, sp, dp, mode="direct", quant=wl.quant, stream=sh)
        algo = st["bytes_read"] + (st["bytes_written"] if wl.quant == "none" else dst_bytes)
    total, per = time_calls(call, stream, steps, warm, world, dev, barrier)
    ms = total / steps
    achieved = algo / (ms / 1e3) / 1e9
    out.update({"ms_per_step": round(ms, 4), "dst_GBps": round(job_throughput(dst_bytes, steps, world, total), 2),
                "algorithmic_bytes": algo, "achieved_GBps": round(achieved, 1), "frac": round(achieved / peak, 4),
                "launch_ms_median": round(statistics.median(per), 4), "launches": R.reshard_plan_stats(plan)["last_launches"],
                "kernel": "reshard_mxfp8_kernel" if wl.quant == "mxfp8" else dominant_kernel(R, plan, "direct", "none"),
                "target_frac": goal, "meets_target": None if goal is None else bool(achieved / peak >= goal)})
    R.reshard_plan_destroy(plan)
    del lay, msg
    torch.cuda.empty_cache()
    return out


def our_arm(args, rank: int, world: int, local_rank: int) -> None:
    import torch
    import torch.distributed as dist

    import dtensor_resharding_gb300 as R
    import synthetic as S

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    wl = S.workload_by_name(args.workload)
    lay = S.allocate(wl, dev)
    S.fill_sources(wl, lay)
    S.fill_canary(lay)
    t0 = time.perf_counter()
    plan = R.plan_workload(wl)
    plan_s = time.perf_counter() - t0
    st = R.reshard_plan_stats(plan)
    sp, dp = R.workload_pointers(wl, lay)
    quant = wl.quant
    dst_bytes = wl.dst_bytes()
    stream = torch.cuda.Stream(device=dev)
    sh = stream.cuda_stream

    def barrier():
        if world > 1:
            dist.barrier()

    def run_steps(mode, k, warm):
        """Time k executes back to back (events only around the whole run, so consecutive launches
        overlap as they would for a caller); then time k more, each bracketed by its own event
        pair, for the per-launch durations the roofline uses (an event between two launches is a
        stream operation of its own and keeps them from overlapping)."""
        for _ in range(warm):
            R.reshard_execute(plan, sp, dp, mode=mode, quant=quant, stream=sh)
        stream.synchronize()
        barrier()
        torch.cuda.synchronize()
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for _ in range(k):
            R.reshard_execute(plan, sp, dp, mode=mode, quant=quant, stream=sh)
        end.record(stream)
        torch.cuda.synchronize()
        barrier()
        total_ms = max_over_ranks(start.elapsed_time(end), world, dev)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(k)]
        for a, b in ev:
            a.record(stream)
            R.reshard_execute(plan, sp, dp, mode=mode, quant=quant, stream=sh)
            b.record(stream)
        torch.cuda.synchronize()
        per = [a.elapsed_time(b) for a, b in ev]
        return total_ms, per

    clocks = ClockSampler(local_rank)
    total_ms, per = run_steps(args.mode, args.steps, args.warmup)
    clk = clocks.stop()
    ms_per_step = total_ms / args.steps
    value = job_throughput(dst_bytes, args.steps, world, total_ms)

    # roofline of the dominant kernel (direct: the one copy kernel per execute)
    peak, peak_kind = peaks()
    launches = launches_per_execute(R, plan, args.mode)
    if args.mode == "direct":
        algo = st["bytes_read"] + (st["bytes_written"] if quant == "none" else dst_bytes)
    else:  # pack (sources in, messages out) + unpack (messages in, destinations out)
        algo = (st["bytes_read"] + 2 * st["message_bytes"] + (st["bytes_written"] if quant == "none" else dst_bytes))
    kernel = dominant_kernel(R, plan, args.mode, quant)
    # average launch duration over the timed region: one execute per step, timed back to back
    launch_ms = total_ms / args.steps
    achieved = algo / (launch_ms / 1e3) / 1e9
    roofline = {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": recorded_traffic(kernel, args.workload, args.mode),
                "kernel": kernel, "algorithmic_bytes_per_launch": algo, "peak_source": peak_kind,
                "launch_ms_mean": round(launch_ms, 4),
                # each launch alone, bracketed by an event pair (no overlap with its neighbours)
                "launch_ms_median": round(statistics.median(per), 4),
                "launch_ms_min": round(min(per), 4), "launch_ms_max": round(max(per), 4)}
    if args.mode == "packed":
        roofline["note"] = "packed mode: the step is the pack and unpack launches; achieved counts both passes' bytes"
    elif launches > 1:
        roofline["note"] = (f"the step is {launches} launches (aligned walker, bulk-staged kernel, general "
                            "walker, gather kernel and/or transposing kernel, back to back on one stream): achieved and "
                            "frac cover the whole step; the kernel named is the one with the most items")
    same = copy_rate_same_run(dev)
    roofline["copy_rate_same_run"] = round(same, 1)
    roofline["frac_of_same_run_copy"] = round(achieved / same, 4)
    roofline["frac_of_nominal"] = round(achieved / NOMINAL_HBM_GBS, 4)
    roofline["nominal_gbs"] = NOMINAL_HBM_GBS

    # the other mode on the same inputs, for context
    other = "packed" if args.mode == "direct" else "direct"
    o_ms, _ = run_steps(other, max(3, args.steps // 4), 2)
    modes = {other: {"ms_per_step": round(o_ms / max(3, args.steps // 4), 4),
                     "value": round(job_throughput(dst_bytes, max(3, args.steps // 4), world, o_ms), 2)}}

    # end to end through the public call with host buffers: the step's sources come from and its
    # destinations go to page-locked host memory inside the timed region
    e2e = None
    if not args.no_e2e:
        ranks_here = max(1, int(os.environ.get("LOCAL_WORLD_SIZE", str(world))))
        ram = host_ram_bytes()
        frac = args.e2e_host_fraction
        budget = int(frac * ram / ranks_here) if ram else None
        try:
            ew, k = (wl, len(wl.tensors)) if budget is None else e2e_prefix(wl, budget)
            if ew is wl:
                e2e = e2e_run(R, wl, plan, sp, dp, lay, args, quant, world, dev, dst_bytes, barrier, st)
            elif k == 0:
                e2e = {"value": None, "unit": "GB/s",
                       "skipped": f"one tensor's page-locked copies exceed {budget / 1e9:.1f} GB per rank"}
            else:
                lay_e = S.allocate(ew, dev)
                S.fill_sources(ew, lay_e)
                S.fill_canary(lay_e)
                plan_e = R.plan_workload(ew)
                sp_e, dp_e = R.workload_pointers(ew, lay_e)
                # the device-resident result the host one is compared with
                R.reshard_execute(plan_e, sp_e, dp_e, mode=args.mode, quant=quant, stream=sh)
                torch.cuda.synchronize()
                e2e = e2e_run(R, ew, plan_e, sp_e, dp_e, lay_e, args, quant, world, dev, ew.dst_bytes(), barrier,
                              R.reshard_plan_stats(plan_e))
                e2e["sample"] = (f"first {k} of {len(wl.tensors)} tensors per rank: page-locked copies of the whole "
                                 f"workload for {ranks_here} rank(s) would pass {frac:.0%} of this "
                                 f"host's {ram / 1e9:.0f} GB")
                del lay_e, plan_e
        except RuntimeError as e:
            e2e = {"value": None, "unit": "GB/s", "error": str(e)[:200]}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import numpy as np  # noqa: F401
        from oracle import coracle
        coracle.build()
        # host copy of the slab prefix that the first tensors' sources occupy (buffers are laid
        # out in tensor order), at most ~12 GB or one tensor, not of the whole slab
        es_of = {"u8": 1, "bf16": 2, "f16": 2, "f32": 4, "i32": 4, "i64": 8}
        first, end = [], 0
        for t in wl.tensors:
            e = max(lay.src_off[v.buffer] + wl.src_buffer_numel[v.buffer] * es_of[t.dtype] for v in t.src_views)
            if first and (max(end, e) > 12 << 30 or len(first) >= 64):
                break
            first.append(t)
            end = max(end, e)
        src_host = lay.src_slab[:end].cpu().numpy()
        nb, secs, used = time_oracle_sample(wl, src_host, lay.src_off, args.cpu_budget, len(first))
        cpu = {"value": round(nb / secs / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": f"first {used} of {len(wl.tensors)} tensors ({nb} destination bytes), host copies, one thread",
               "seconds": round(secs, 2)}
        cpu["all_cores"] = time_oracle_parallel(wl, src_host, lay.src_off, used)

    R.reshard_plan_destroy(plan)
    del lay, sp, dp
    torch.cuda.empty_cache()
    targets = None
    if not args.no_targets:
        targets = [measure_target(n, how, goal, max(5, args.steps // 4), 3, world, dev, barrier, peak)
                   for n, how, goal in TARGETS]
        # the headline workload is the MoE target of the direct executor
        if args.workload == DEFAULT_WORKLOAD and args.mode == "direct":
            targets.insert(0, {"workload": args.workload, "mode": "direct", "ms_per_step": round(ms_per_step, 4),
                               "achieved_GBps": roofline["achieved"], "frac": roofline["frac"], "target_frac": 0.80,
                               "meets_target": bool(roofline["frac"] >= 0.80), "kernel": kernel,
                               "note": "the headline measurement above"})

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 3), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": args.workload, "mode": args.mode, "quant": quant, "tensors": len(wl.tensors),
                       "src_bytes": st["bytes_read"], "dst_bytes": dst_bytes,
                       "regions": st["regions"], "items": st["items"],
                       "l2": "inputs larger than L2 (every step streams all sources and destinations)",
                       "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
                       "plan_build_s": round(plan_s, 3)},
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "clocks": clk,
            "gpu_launches": args.steps * launches,
            "modes": modes,
            "targets": targets,
        }
        print(json.dumps(line), flush=True)
        if args.suite:
            with open(args.suite, "a") as f:
                f.write(json.dumps(line) + "\n")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--mode", default="direct", choices=["direct", "packed"])
    ap.add_argument("--e2e-steps", type=int, default=4)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-targets", action="store_true", help="skip the other north-star workloads")
    ap.add_argument("--suite", default=None, help="also append the JSON line to this file")
    ap.add_argument("--e2e-host-fraction", type=float, default=E2E_HOST_FRACTION,
                    help="share of host memory the end-to-end leg's page-locked copies may take, split over "
                         "the ranks on the host; past it the leg runs on the longest prefix of tensors that fits")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        reference_arm(args, rank)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    try:
        our_arm(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
