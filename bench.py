#!/usr/bin/env python
"""Benchmark of the GB300 mHC sublayer boundary.

One step = one boundary call (stage-1 sum, post-mix, prenorm GEMV, mixes,
Sinkhorn, collapse + RMSNorm, MXFP8 copy) over the workload's tokens, inputs
already resident in HBM.  Prints one JSON line (rank 0):

  value      tokens/s of the whole job (N GPUs run independent replicas)
  roofline   the stage kernel's algorithmic bytes per launch / its average
             device time (CUDA events around it inside the timed region)
             against the measured HBM copy bandwidth
  e2e        the same metric through mhc_boundary_run_host (host buffers,
             host<->device copies inside the timed region)
  cpu_baseline  the CPU oracle on the host cores (rank 0, N = 1)

--impl reference times the oracle itself (the reference arm of this method:
no other implementation of it exists to run).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                       [--workload large_mxfp8|glm|decode|moe|tiny] [--m M]
"""
import argparse
import concurrent.futures
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "mHC boundary tokens/s and achieved HBM GB/s (% of GB300 peak) vs token count"
L2_BYTES_FALLBACK = 126 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="large_mxfp8")
    ap.add_argument("--m", type=int, default=None, help="token count (default: the workload's largest)")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle CPU baseline")
    ap.add_argument("--no-per-config", action="store_true", help="skip the other workloads' rows")
    ap.add_argument("--no-static-weight", action="store_true",
                    help="read the prenorm weight only after the preceding kernel (not as a layer weight)")
    ap.add_argument("--sweep", action="store_true",
                    help="one line per workload and token count (call time, GB/s, kernel times)")
    return ap.parse_args()


# ---------------------------------------------------------------- workload
def workload(name, m):
    from mhc_residual_boundary_gb300 import synth
    cands = synth.WORKLOADS[name]
    w = cands[-1] if m is None else next((c for c in cands if c.m == m), None)
    if w is None:
        base = cands[-1]
        w = synth.Workload(base.name, base.hidden, base.tp, m, base.top_k, base.moe, base.mxfp8, base.bf16_fn,
                           base.consume, base.residual_only, base.owner)
    return w


def call_bytes(w):
    """Algorithmic HBM bytes of one call, split by kernel (each tensor read
    or written once; scratch traffic excluded)."""
    H, tp, M, K = w.hidden, w.tp, w.m, w.top_k
    if w.moe:
        stage1 = tp * K * 2 * H + tp * 2 * H + tp * K * 4 + K * 4
    else:
        stage1 = 2 * tp * H
    if w.owner:
        stage1 += 4 * H   # the owners' sums, written and read back
    if w.consume:
        # the delayed-mHC consumer: no weight, no mixes; pre read, layer input written
        stage = M * (stage1 + 8 * H + 8 * H + 16 + 64)
        finish = 0 if w.residual_only else 2 * H + M * (16 + 2 * H)
        return {"stage": stage, "finish": finish, "mixes": 0, "total": stage + finish}
    stage = M * (stage1 + 8 * H + 8 * H + 16 + 64) + 4 * H * 24 * (2 if w.bf16_fn else 4)
    finish = 2 * H + M * 2 * H
    if w.mxfp8:
        padded = (M + 127) // 128 * 128
        finish += M * H + padded * (H // 32)
    mixes = M * (16 + 64) + 12 + 96
    return {"stage": stage, "finish": finish, "mixes": mixes, "total": stage + finish + mixes}


# The prenorm weight is a layer weight (MHC_FLAG_STATIC_WEIGHT): each call's
# stage kernel stages and splits it while the kernel before it finishes.
STATIC_WEIGHT = True


def describe(w):
    return {"workload": w.name, "tokens": w.m, "hidden": w.hidden, "tp": w.tp, "hc": 4,
            "top_k": w.top_k, "moe": w.moe, "mxfp8": w.mxfp8,
            "weight": "none (carried pre)" if w.consume else "bf16 [24][4H]" if w.bf16_fn else "f32 [4H][24]",
            "weight_staging": ("layer weight: staged while the preceding kernel ends" if STATIC_WEIGHT
                               else "after the preceding kernel"),
            "reduction": "MoE fold" if w.moe else "two-shot (owner reduce)" if w.owner else "direct",
            "residual_only": w.residual_only}


# ------------------------------------------------------------------ ranks
def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, local):
    """One process per GPU over NCCL (replicas: NCCL carries only the timing
    barrier and the max over ranks); gloo on a host without a GPU, where the
    same rank logic runs in the tests."""
    import torch
    import torch.distributed as dist
    if world > 1:
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group("gloo")
    return dist if world > 1 else None


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(dist, value):
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(world, tokens_per_rank, steps, seconds):
    """Whole-job throughput: the tokens all ranks processed (each rank a full
    replica of the workload) over the slowest rank's time."""
    return world * tokens_per_rank * steps / seconds


# ----------------------------------------------------------------- peaks etc
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, b.copy_ of 1 Gi bf16)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback (6.8 TB/s, an earlier GB300 copy measurement)"


def kernel_traffic(w):
    """dram bytes per launch of the stage kernel from the committed ncu
    summary, only if it was taken on this workload with the current source."""
    src = os.path.join(ROOT, "mhc_residual_boundary_gb300", "csrc", "k_stage_tc.cu")
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:12]
    pat = re.compile(r"traffic: workload=(\S+) tokens=(\d+) kernel=k_stage_tc source_sha=(\w+) "
                     r"bytes_per_launch=(\d+)")
    pdir = os.path.join(ROOT, "profiles")
    for name in sorted(os.listdir(pdir)) if os.path.isdir(pdir) else []:
        if not name.endswith((".md", ".txt")):
            continue
        for mt in pat.finditer(open(os.path.join(pdir, name)).read()):
            if mt.group(1) == w.name and int(mt.group(2)) == w.m and mt.group(3) == sha:
                return int(mt.group(4))
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons every 50 ms while running."""
    FIELDS = ("index,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid):
        self.uuid = uuid
        self.proc = None
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None:
            return None
        self.file.flush()
        rows = []
        with open(self.file.name) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                if self.uuid and parts[1] != self.uuid:
                    continue
                rows.append(parts)
        os.unlink(self.file.name)
        if not rows:
            return None
        sm = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        smax = max(float(r[3]) for r in rows if r[3].replace(".", "").isdigit())
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({n for r in rows for n, v in zip(names, r[6:10]) if v.lower() == "active"})
        power = [float(r[4]) for r in rows if re.match(r"^[\d.]+$", r[4])]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax, "reasons": reasons,
                "samples": len(rows), "power_w_max": max(power) if power else None}


# -------------------------------------------------------------- CPU oracle
def oracle_tokens_per_s(w, inputs, tokens, threads):
    """The oracle over `tokens` tokens of the workload, split in token ranges
    over `threads` host threads (the C code releases the GIL)."""
    import numpy as np
    import oracle
    p = oracle.Problem(w.hidden, w.tp, w.m, top_k=w.top_k, rows_per_rank=w.m * w.top_k if w.moe else 0)
    outs = {
        "residual_out": np.zeros((w.m, 4, w.hidden), np.uint16),
        "layer_input": np.zeros((w.m, w.hidden), np.uint16),
        "post_out": np.zeros((w.m, 4), np.float32), "comb_out": np.zeros((w.m, 4, 4), np.float32),
        "mixes": np.zeros((w.m, 24), np.float32), "pre": np.zeros((w.m, 4), np.float32),
    }
    if w.mxfp8:
        outs["mx_values"] = np.zeros((w.m, w.hidden), np.uint8)
        outs["mx_scales"] = np.zeros((oracle.mxfp8_scale_bytes(w.m, w.hidden),), np.uint8)
    chunk = max(1, math.ceil(tokens / threads))
    ranges = [(s, min(s + chunk, tokens)) for s in range(0, tokens, chunk)]
    t0 = time.perf_counter()
    with concurrent.futures.ThreadPoolExecutor(max_workers=threads) as pool:
        list(pool.map(lambda r: oracle.boundary(p, inputs, moe=w.moe, mxfp8_out=w.mxfp8,
                                                t0=r[0], t1=r[1], outputs=outs), ranges))
    return tokens / (time.perf_counter() - t0)


def cpu_baseline(w, inputs):
    """The oracle as it stands, timed on the host cores: every token of the
    workload once over all cores, and up to 512 tokens on one thread."""
    import oracle
    oracle.build()
    threads = os.cpu_count() or 1
    sample = w.m
    one = min(sample, 512)
    return {"value": oracle_tokens_per_s(w, inputs, sample, threads), "unit": "tokens/s",
            "cores": threads, "kind": "oracle",
            "sample": f"all {sample} tokens of the workload once, token ranges over {threads} threads",
            "single_thread_value": oracle_tokens_per_s(w, inputs, one, 1),
            "single_thread_sample": f"the first {one} tokens on one thread"}


def run_reference(args, w):
    world, rank, _ = dist_info()
    if rank != 0:
        return
    from mhc_residual_boundary_gb300 import synth
    import oracle
    oracle.build()
    inputs = synth.inputs_for(w)
    threads = os.cpu_count() or 1
    sample = min(w.m, 512)
    for _ in range(max(args.warmup, 0)):
        oracle_tokens_per_s(w, inputs, sample, threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_tokens_per_s(w, inputs, sample, threads)
    elapsed = time.perf_counter() - t0
    value = sample * args.steps / elapsed
    sample_desc = f"{sample} of the workload's {w.m} tokens per step, {threads} threads"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": elapsed / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded)", "config": describe(w),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": sample_desc},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


# -------------------------------------------------------------- GPU path
def run_ours(args, w):
    import numpy as np
    import torch

    world, rank, local = dist_info()
    dist = init_dist(world, local)
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    from __graft_entry__ import build
    build()
    from mhc_residual_boundary_gb300 import Boundary, synth

    inputs = synth.inputs_for(w, seed=0)

    def to_dev(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)
        return torch.from_numpy(a).to(device)

    dev_in = {("norm_weight" if k == "gamma" else k): to_dev(v) for k, v in inputs.items()}
    b = Boundary(hidden=w.hidden, tp=w.tp, max_num_tokens=w.m, top_k=w.top_k, mxfp8=w.mxfp8,
                 host_staging=not w.moe, static_weight=STATIC_WEIGHT, owner_reduce=w.owner, device=local)
    props = torch.cuda.get_device_properties(device)
    l2 = getattr(props, "L2_cache_size", 0) or L2_BYTES_FALLBACK
    nbytes = call_bytes(w)
    # rotate buffer sets until one pass over them is >= 3x L2, so every call
    # reads and writes HBM (the large workload alone is already > L2)
    nsets = 1 if nbytes["total"] >= 3 * l2 else math.ceil(3 * l2 / nbytes["total"]) + 1
    sets = []
    for s in range(nsets):
        ins = dev_in if s == 0 else {k: v.clone() for k, v in dev_in.items()}
        outs = b.empty_outputs(w.m, mxfp8=w.mxfp8)
        sets.append((ins, outs))
    call = b.finalize_moe if w.moe else b.run
    stream = torch.cuda.current_stream()

    uuid = None
    try:
        uuid = str(props.uuid)
        uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        pass
    with ClockSampler(uuid) as clocks:
        for i in range(args.warmup):
            call(*sets[i % nsets], stream=stream)
        b.join(stream)
        torch.cuda.synchronize()
        barrier(dist)
        torch.cuda.synchronize()
        # timed region: K calls with nothing between them (events between the
        # kernels would break the programmatic overlap of consecutive kernels)
        start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for i in range(args.steps):
            call(*sets[i % nsets], stream=stream)
        b.join(stream)
        stop.record(stream)
        torch.cuda.synchronize()
        barrier(dist)
        # the same K calls again with CUDA events around every kernel, on the
        # stream each is launched on: the per-kernel times of the roofline
        b.profile_begin(args.steps)
        for i in range(args.steps):
            call(*sets[i % nsets], stream=stream)
        b.join(stream)
        torch.cuda.synchronize()
        barrier(dist)
        prof = b.profile_end()
    b.check_errors()   # a device-side timeout or bad argument fails the run here
    clock = clocks.summary()
    elapsed_ms = max_over_ranks(dist, start.elapsed_time(stop))
    value = job_value(world, w.m, args.steps, elapsed_ms / 1e3)
    ms_per_step = elapsed_ms / args.steps

    peak, peak_src = measured_peaks()
    stage_ms = prof["stage_ms"] / max(prof["calls"], 1)
    achieved = nbytes["stage"] / (stage_ms * 1e-3) / 1e9
    call_gbs = nbytes["total"] / (ms_per_step * 1e-3) / 1e9
    roofline = {"bound": "hbm", "kernel": "k_stage_tc", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": kernel_traffic(w),
                "algorithmic_bytes_per_launch": nbytes["stage"], "avg_launch_ms": stage_ms,
                "peak_source": peak_src,
                "kernel_ms_per_call": {"stage": stage_ms, "finish": prof["finish_ms"] / max(prof["calls"], 1),
                                       "mixes": prof["mixes_ms"] / max(prof["calls"], 1)},
                "call_gbs": call_gbs, "call_frac": call_gbs / peak, "call_frac_8tbs": call_gbs / 8000.0,
                "call_algorithmic_bytes": nbytes["total"]}

    # end to end through the host-buffer entry point
    e2e = None
    if not w.moe and args.e2e_steps > 0:
        host_in = {k: v.cpu().pin_memory() for k, v in dev_in.items() if k in (
            "partials", "residual", "post", "comb", "hc_fn", "hc_fn_bf16", "scale", "base", "norm_weight")}
        host_out = b.empty_outputs(w.m, mxfp8=w.mxfp8, device="cpu", pin_memory=True)
        h2d = sum(t.numel() * t.element_size() for t in host_in.values())
        d2h = sum(t.numel() * t.element_size() for t in host_out.values())
        b.run_host(host_in, host_out, stream=stream)
        barrier(dist)
        t0 = time.perf_counter()
        for _ in range(args.e2e_steps):
            b.run_host(host_in, host_out, stream=stream)
        barrier(dist)
        e2e_s = max_over_ranks(dist, time.perf_counter() - t0)
        # the host link's bound: the same byte counts copied with no kernels,
        # one pinned buffer up while another comes down
        import torch
        flat_up = torch.empty(h2d, dtype=torch.uint8).pin_memory()
        flat_down = torch.empty(d2h, dtype=torch.uint8).pin_memory()
        dev_up = torch.empty(h2d, dtype=torch.uint8, device=device)
        dev_down = torch.empty(d2h, dtype=torch.uint8, device=device)
        up, down = torch.cuda.Stream(device), torch.cuda.Stream(device)

        def copies_only():
            with torch.cuda.stream(up):
                dev_up.copy_(flat_up, non_blocking=True)
            with torch.cuda.stream(down):
                flat_down.copy_(dev_down, non_blocking=True)
            torch.cuda.synchronize(device)

        copies_only()
        t0 = time.perf_counter()
        for _ in range(args.e2e_steps):
            copies_only()
        link_s = max_over_ranks(dist, time.perf_counter() - t0)
        del flat_up, flat_down, dev_up, dev_down
        e2e = {"value": job_value(world, w.m, args.e2e_steps, e2e_s), "unit": "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": args.e2e_steps,
               "copies_only_tokens_per_s": job_value(world, w.m, args.e2e_steps, link_s),
               "copies_only": "the same byte counts as one pinned copy each way, both at once, no kernels"}

    cpu = cpu_baseline(w, inputs) if rank == 0 and world == 1 and not args.no_cpu else None
    pc = per_config(device, peak, l2) if rank == 0 and not args.no_per_config else None

    launches = b.launches_per_call() + (1 if w.moe else 0)
    b.close()
    if rank == 0:
        print(json.dumps({
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded: numpy default_rng, distributions of the named workload)",
            "config": dict(describe(w), l2=(f"inputs larger than L2: {nbytes['total'] / 1e6:.1f} MB per call, "
                                            f"{nsets} buffer set(s) rotated, L2 {l2 / 1e6:.0f} MB"),
                           parallelism=f"replicas x{world}"),
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "per_config": pc,
            "gpu_launches": args.steps * launches, "clocks": clock,
        }), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def measure_workload(w, steps, warmup, device, peak, l2, profile=True, latency=False):
    """One workload: per-call device time over back-to-back calls (buffer sets
    rotated so that each call reads HBM), from Python stream launches and from
    a CUDA graph replaying the calls; achieved algorithmic GB/s against the
    measured and the nominal 8 TB/s peak; per-kernel times of a profiled pass;
    a hot-L2 replay (labelled as such); with `latency`, the device time of one
    call on its own (events around a single call after the stream drained)."""
    import numpy as np
    import torch
    from mhc_residual_boundary_gb300 import Boundary, synth
    stream = torch.cuda.current_stream()
    inputs = synth.inputs_for(w, seed=0)
    dev_in = {("norm_weight" if k == "gamma" else k):
              (torch.from_numpy(v.view(np.int16)).view(torch.bfloat16) if v.dtype == np.uint16
               else torch.from_numpy(v)).to(device) for k, v in inputs.items()}
    b = Boundary(hidden=w.hidden, tp=w.tp, max_num_tokens=w.m, top_k=w.top_k, mxfp8=w.mxfp8,
                 static_weight=STATIC_WEIGHT, owner_reduce=w.owner, device=device.index)
    nbytes = call_bytes(w)
    nsets = 1 if nbytes["total"] >= 3 * l2 else math.ceil(3 * l2 / nbytes["total"]) + 1

    def outputs():
        o = b.empty_outputs(w.m, mxfp8=w.mxfp8)
        if w.consume:
            o = {k: v for k, v in o.items()
                 if k == "residual_out" or (k == "layer_input" and not w.residual_only)}
        return o
    if w.residual_only:
        dev_in.pop("norm_weight", None)
    sets = [(dev_in if s == 0 else {k: v.clone() for k, v in dev_in.items()}, outputs())
            for s in range(nsets)]
    call = b.consume if w.consume else b.finalize_moe if w.moe else b.run
    steps = max(steps, nsets)
    for i in range(max(warmup, 3)):
        call(*sets[i % nsets], stream=stream)
    b.join(stream)
    torch.cuda.synchronize()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(steps):
        call(*sets[i % nsets], stream=stream)
    b.join(stream)
    stop.record(stream)
    torch.cuda.synchronize()
    us = start.elapsed_time(stop) * 1e3 / steps
    prof = None
    if profile:
        b.profile_begin(steps)
        for i in range(steps):
            call(*sets[i % nsets], stream=stream)
        b.join(stream)
        torch.cuda.synchronize()
        prof = b.profile_end()
    # the same calls replayed from a CUDA graph: device time without the
    # Python binding's per-call host cost
    graph_us = None
    if nsets <= 512:
        cap = torch.cuda.Stream(device)
        cap.wait_stream(stream)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            for i in range(nsets):
                call(*sets[i], stream=cap)
            b.join(cap)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        reps = max(1, steps // nsets)
        start.record(stream)
        for _ in range(reps):
            g.replay()
        stop.record(stream)
        torch.cuda.synchronize()
        graph_us = start.elapsed_time(stop) * 1e3 / (reps * nsets)
        del g
    # hot L2 (labelled as such): the same graph replay on one buffer set, so
    # that a workload smaller than L2 reads it from L2
    hot_us = None
    if nsets > 1:
        cap = torch.cuda.Stream(device)
        cap.wait_stream(stream)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            for _ in range(16):
                call(*sets[0], stream=cap)
            b.join(cap)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        reps = max(1, steps // 16)
        start.record(stream)
        for _ in range(reps):
            g.replay()
        stop.record(stream)
        torch.cuda.synchronize()
        hot_us = start.elapsed_time(stop) * 1e3 / (reps * 16)
        del g
    # one call on its own: the stream drained before it, events around it
    isolated_us = None
    if latency:
        times = []
        for i in range(200):
            torch.cuda.synchronize()
            start.record(stream)
            call(*sets[i % nsets], stream=stream)
            b.join(stream)
            stop.record(stream)
            torch.cuda.synchronize()
            times.append(start.elapsed_time(stop) * 1e3)
        isolated_us = statistics.median(times)
    b.check_errors()
    b.close()
    best = graph_us if graph_us else us
    gbs = nbytes["total"] / (best * 1e-6) / 1e9
    res = {"config": describe(w), "us_per_call": best, "tokens_per_s": w.m / (best * 1e-6),
           "algorithmic_bytes": nbytes["total"], "gbs": gbs, "frac_measured": gbs / peak,
           "frac_8tbs": gbs / 8000.0, "buffer_sets": nsets, "steps": steps,
           "timing": "CUDA graph replay of back-to-back calls" if graph_us else "stream launches",
           "stream_us_per_call": us, "hot_l2_graph_us_per_call": hot_us}
    if isolated_us is not None:
        res["isolated_call_us"] = isolated_us
    if prof:
        n = max(prof["calls"], 1)
        res["kernel_us"] = {"stage": prof["stage_ms"] / n * 1e3, "finish": prof["finish_ms"] / n * 1e3,
                            "mixes": prof["mixes_ms"] / n * 1e3}
    return res


# Workloads reported beside the headline one in every bench line: (name, M)
PER_CONFIG = [("tiny", 4), ("decode", 64), ("glm", 1), ("glm", 8), ("glm", 12), ("glm", 256), ("glm", 512),
              ("moe", 256)]


def per_config(device, peak, l2, steps=2000):
    out = {}
    for name, m in PER_CONFIG:
        w = workload(name, m)
        r = measure_workload(w, steps, 20, device, peak, l2, profile=False, latency=(name == "glm" and m == 1))
        out[f"{name}_m{m}"] = {k: r[k] for k in ("us_per_call", "tokens_per_s", "gbs", "frac_measured", "frac_8tbs",
                                                 "algorithmic_bytes", "buffer_sets", "timing")
                               } | ({"isolated_call_us": r["isolated_call_us"]} if "isolated_call_us" in r else {})
    return out


def run_sweep(args):
    """Every workload at every token count (one JSON line each)."""
    import torch
    from __graft_entry__ import build
    build()
    from mhc_residual_boundary_gb300 import synth
    device = torch.device("cuda", 0)
    peak, _ = measured_peaks()
    props = torch.cuda.get_device_properties(device)
    l2 = getattr(props, "L2_cache_size", 0) or L2_BYTES_FALLBACK
    for name, cands in synth.WORKLOADS.items():
        for w in cands:
            r = measure_workload(w, args.steps, args.warmup, device, peak, l2,
                                 latency=(w.m == 1))
            print(json.dumps(dict(r, sweep=True)), flush=True)


def main():
    global STATIC_WEIGHT
    args = parse_args()
    STATIC_WEIGHT = not args.no_static_weight
    if args.sweep:
        run_sweep(args)
        return
    w = workload(args.workload, args.m)
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
