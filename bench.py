"""Benchmark of the ragged BF16 grouped GEMM on GB300: one step = forward +
data gradient + weight gradient over one batch of synthetic inputs.

Default workload: MoE gate_up, E=8 experts, M=131072 routed rows split evenly,
K=4096 hidden, N=3072, BF16 inputs (X~N(0,1), W~N(0,1/K), G~N(0,1)), BF16
output, deterministic mode.  Operands (2.1 GB per step) are larger than the
129 MB L2, so no flush is needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--out-dtype bf16|fp32] [--det 0|1]

Prints one JSON line (rank 0).  ``--impl reference`` times the FP64 CPU
oracle on the host cores instead (a bounded sample of the same workload per
step).  Under torchrun each rank runs an independent replica (weak scaling).

    python bench.py --grid pages [--grid-filter TEXT] [--grid-reps R]
    python bench.py --workload router     (FP32 router GEMM, BF16x3 emulation)

times the GB300 rows of flashinfer PR #8269's per-row latency table (weight
gradient, checkpointed forward + backward, and the same with early stop) the
way that table was measured: one call, cold L2, median over repetitions.  It
prints one JSON line per row and a summary line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "grouped-GEMM TFLOP/s (fwd/dgrad/wgrad) and % of GB300 dense BF16 peak"
UNIT = "TFLOP/s"


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="moe_gate_up")
    ap.add_argument("--out-dtype", default="bf16", choices=["bf16", "fp32"])
    ap.add_argument("--det", type=int, default=1)
    ap.add_argument("--passes", default="fwd,dgrad,wgrad")
    ap.add_argument("--e2e-steps", type=int, default=6)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--pass-events", type=int, default=1,
                    help="1: per-pass CUDA events inside the timed region; 0: none there (kernels back to "
                         "back), per-pass times from a separate loop")
    ap.add_argument("--graph", action="store_true",
                    help="replay each pass from a captured CUDA graph (removes host launch overhead)")
    ap.add_argument("--corun", default="8,16,32",
                    help="comma list of SM counts (default 8,16,32; empty = skip): after the timed region, "
                         "time the same steps again while a spinner on another stream holds that many SMs")
    ap.add_argument("--no-pages-sample", action="store_true",
                    help="skip the pages' grid sample (dW, ckpt, ckpt ES of gate_up E8 M131072 bal)")
    ap.add_argument("--grid", default="", choices=["", "pages"],
                    help="pages: time the GB300 rows of the pages' per-row latency table")
    ap.add_argument("--grid-filter", default="", help="only rows whose 'shape op' contains this text")
    ap.add_argument("--grid-reps", type=int, default=7)
    ap.add_argument("--no-thin", action="store_true",
                    help="skip the dense projection records (thin 4096->48 passes, mid-size 4096->512 wgrad)")
    ap.add_argument("--sustained-seconds", type=float, default=1.2,
                    help="length of the second, longer timing of the step (0 = skip)")
    ap.add_argument("--decide", default="", choices=["", "tail", "streamk", "split", "wide", "csplit"],
                    help="run the planner decision protocol for one plan rule (candidate vs baseline)")
    ap.add_argument("--decide-points", default="", help="comma list of points (workload names) to test")
    ap.add_argument("--decide-runs", type=int, default=2)
    ap.add_argument("--decide-groups", type=int, default=9)
    ap.add_argument("--decide-steps", type=int, default=5)
    return ap.parse_args()


def get_workload(name):
    from moe_ragged_grouped_gb300 import workloads as wl
    if name == "moe_gate_up":
        return wl.moe_gate_up()
    if name == "moe_gate_up_m16k":
        return wl.Workload("moe_gate_up_E8_M16384_K4096_N3072", 8, 3072, 4096, wl.balanced_sizes(8, 16384))
    if name == "moe_gate_up_e2":
        # two gate_up experts of 16384 rows: the per-expert working set of the full
        # step (above the L2) at a quarter of its device memory, for profiling
        return wl.Workload("moe_gate_up_E2_M32768_K4096_N3072", 2, 3072, 4096, wl.balanced_sizes(2, 32768))
    if name == "moe_down":
        return wl.moe_down()
    if name == "moe_skew":
        return wl.moe_skewed(False)
    if name == "moe_skew_t":
        return wl.moe_skewed(True)
    if name == "tiny":
        return wl.tiny()
    if name.startswith("dense_"):
        spec, _, t = name[len("dense_"):].partition("_T")
        d_in, d_out = (int(v) for v in spec.split("to"))
        return wl.dense_projection(d_in, d_out, int(t) if t else 16384)
    raise SystemExit(f"unknown workload {name}")


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value, dist, device):
    """The largest value over the ranks (a timing is the slowest rank's); `dist` None = one rank."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"bf16_tflops": float(d["bf16_tflops"]), "hbm_gbs": float(d["hbm_gbs"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"bf16_tflops": 1900.0, "hbm_gbs": 6800.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def kernel_source_digest():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "moe_ragged_grouped_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_for(workload_name, pass_, out_dtype, det):
    """DRAM bytes per launch from a committed ncu summary, if taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    if d.get("kernel_source_digest") != kernel_source_digest():
        return None
    key = f"{workload_name}|{pass_}|{out_dtype}|det{int(det)}"
    return d.get("per_launch_bytes", {}).get(key)


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.gpu = gpu_index
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        self.t_start = self.t_end = None

    def mark_start(self):
        self.t_start = time.time()

    def mark_end(self):
        self.t_end = time.time()

    def finish(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        rows = []
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                ts += float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                rows.append((ts, float(parts[2]), float(parts[3]), parts[6:10]))
            except Exception:
                continue
        if not rows:
            return None
        inside = [r for r in rows if self.t_start - 0.15 <= r[0] <= self.t_end + 0.15] or rows
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in inside:
            for n, v in zip(names, r[3]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": sorted(reasons), "samples": len(inside)}


# ---------------------------------------------------------------------------- GPU arm


def run_ours(args, wk):
    import torch
    from moe_ragged_grouped_gb300 import build as gg_build
    from moe_ragged_grouped_gb300 import cake_gg as gg

    ws, rank, local = dist_env()
    dist = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        gg_build.build()
    if dist is not None:
        dist.barrier()
    gg.load_library()

    passes = [p for p in args.passes.split(",") if p]
    od, det = args.out_dtype, args.det
    X, W, G = wk.make_torch(seed=0, device=dev)
    offs = torch.from_numpy(wk.offsets).to(dev)
    M, E, N, K = wk.M, wk.E, wk.N, wk.K
    tdt = torch.float32 if od == "fp32" else torch.bfloat16
    Y = torch.empty((M, N), dtype=tdt, device=dev)
    dX = torch.empty((M, K), dtype=tdt, device=dev)
    dW = torch.empty((E, N, K), dtype=tdt, device=dev)
    plans = {p: gg.cake_gg_plan(p, E, M, N, K, od, det) for p in passes}
    wss = {p: gg.make_workspace(plans[p], dev) for p in passes}
    stream = torch.cuda.current_stream(dev)
    s = stream.cuda_stream

    def launch(p):
        s = torch.cuda.current_stream(dev).cuda_stream
        if p == "fwd":
            rc = gg.cake_gg_fwd(plans[p], X, W, Y, offs, od, det, wss[p], stream=s)
        elif p == "dgrad":
            rc = gg.cake_gg_dgrad(plans[p], G, W, dX, offs, od, det, wss[p], stream=s)
        else:
            rc = gg.cake_gg_wgrad(plans[p], G, X, dW, offs, od, det, wss[p], stream=s)
        if rc != 0:
            raise gg.CakeGGError(rc, p)

    for _ in range(args.warmup):
        for p in passes:
            launch(p)
    torch.cuda.synchronize(dev)
    run_pass = launch
    if args.graph:
        graphs = {}
        cap = torch.cuda.Stream(dev)
        for p in passes:
            g_ = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_, stream=cap):
                launch(p)
            graphs[p] = g_
        torch.cuda.synchronize(dev)
        run_pass = lambda p: graphs[p].replay()
        for _ in range(2):
            for p in passes:
                run_pass(p)
        torch.cuda.synchronize(dev)
    for p in passes:
        st = gg.cake_gg_check_status(wss[p], s)
        if st != 0:
            raise gg.CakeGGError(st, f"{p} device status")

    sampler = ClockSampler(local) if rank == 0 else None
    time.sleep(0.3 if sampler else 0.0)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(passes) + 1)] for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    if sampler:
        sampler.mark_start()
    # one pass per step: the whole timed region is that kernel's launches, back
    # to back; several passes: events between them (inside the timed region)
    pass_events = args.pass_events and len(passes) > 1
    start.record(stream)
    for i in range(args.steps):
        if pass_events:
            evs[i][0].record(stream)
        for j, p in enumerate(passes):
            run_pass(p)
            if pass_events:
                evs[i][j + 1].record(stream)
    end.record(stream)
    torch.cuda.synchronize(dev)
    if sampler:
        sampler.mark_end()
    elapsed_ms = start.elapsed_time(end)
    if len(passes) == 1:
        per_pass_ms = {passes[0]: elapsed_ms / args.steps}
    elif not pass_events:
        # per-pass breakdown from a separate loop
        for i in range(args.steps):
            evs[i][0].record(stream)
            for j, p in enumerate(passes):
                run_pass(p)
                evs[i][j + 1].record(stream)
        torch.cuda.synchronize(dev)
    if len(passes) > 1:
        per_pass_ms = {p: statistics.mean(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(args.steps))
                       for j, p in enumerate(passes)}
    if dist is not None:
        dist.barrier()
    elapsed_ms = max_over_ranks(elapsed_ms, dist, dev)
    clocks = sampler.finish() if sampler else None

    flop_step = wk.flops(len(passes))
    value = flop_step * args.steps * ws / (elapsed_ms * 1e-3) / 1e12
    ms_per_step = elapsed_ms / args.steps

    # ---- the same step timed again for >= 1 s (the sustained, power-capped regime) ----
    sustained = None
    if args.sustained_seconds > 0:
        n_sus = max(args.steps, int(math.ceil(args.sustained_seconds * 1e3 / ms_per_step)))
        sampler2 = ClockSampler(local) if rank == 0 else None
        time.sleep(0.3 if sampler2 else 0.0)
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)
        if sampler2:
            sampler2.mark_start()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(n_sus):
            for p in passes:
                run_pass(p)
        b.record(stream)
        torch.cuda.synchronize(dev)
        if sampler2:
            sampler2.mark_end()
        sus_ms = max_over_ranks(a.elapsed_time(b), dist, dev)
        sus_value = flop_step * n_sus * ws / (sus_ms * 1e-3) / 1e12
        pk = measured_peaks()
        sustained = {"steps": n_sus, "seconds": round(sus_ms / 1e3, 3), "value": round(sus_value, 2),
                     "unit": UNIT, "ms_per_step": round(sus_ms / n_sus, 4),
                     "frac_of_sustained_peak": round(sus_value / ws / pk["bf16_tflops_sustained"], 4),
                     "peak_source": f"{pk['source']} bf16_tflops_sustained",
                     "clocks": sampler2.finish() if sampler2 else None}

    # ---- end to end through the public API with host buffers ----
    # Every step copies its inputs in from pinned host memory and all of its
    # outputs back out.  The copies run on their own streams and two device
    # buffer sets alternate, so step i+1's inputs stream in and step i's
    # outputs stream out while the kernels of the steps run: host->device,
    # device->host and compute overlap, as a training loop that prefetches its
    # next batch would run them.  The kernels stay on one stream (the
    # workspaces' ordering rule).
    e2e = None
    if args.e2e_steps > 0:
        hX = torch.empty(X.shape, dtype=X.dtype, pin_memory=True)
        hW = torch.empty(W.shape, dtype=W.dtype, pin_memory=True)
        hG = torch.empty(G.shape, dtype=G.dtype, pin_memory=True)
        hX.copy_(X)
        hW.copy_(W)
        hG.copy_(G)
        outs0 = {"fwd": Y, "dgrad": dX, "wgrad": dW}
        ins = [(X, W, G), tuple(torch.empty_like(t) for t in (X, W, G))]
        outs = [outs0, {p: torch.empty_like(outs0[p]) for p in passes}]
        houts = [{p: torch.empty(outs0[p].shape, dtype=tdt, pin_memory=True) for p in passes} for _ in range(2)]
        h2d = sum(t.numel() * t.element_size() for t in (hX, hW, hG))
        d2h = sum(houts[0][p].numel() * houts[0][p].element_size() for p in passes)
        h2d_s, d2h_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        free_in, free_out = [None, None], [None, None]

        def launch_set(p, k):
            x, w, g = ins[k]
            o = outs[k][p]
            if p == "fwd":
                rc = gg.cake_gg_fwd(plans[p], x, w, o, offs, od, det, wss[p], stream=s)
            elif p == "dgrad":
                rc = gg.cake_gg_dgrad(plans[p], g, w, o, offs, od, det, wss[p], stream=s)
            else:
                rc = gg.cake_gg_wgrad(plans[p], g, x, o, offs, od, det, wss[p], stream=s)
            if rc != 0:
                raise gg.CakeGGError(rc, p)

        def e2e_step(i):
            k = i % 2
            x, w, g = ins[k]
            # inputs of set k: free once the step two back has computed
            if free_in[k] is not None:
                h2d_s.wait_event(free_in[k])
            with torch.cuda.stream(h2d_s):
                x.copy_(hX, non_blocking=True)
                w.copy_(hW, non_blocking=True)
                ev_xw = torch.cuda.Event()
                ev_xw.record(h2d_s)
                g.copy_(hG, non_blocking=True)
                ev_g = torch.cuda.Event()
                ev_g.record(h2d_s)
            # outputs of set k: free once the step two back has copied them out
            if free_out[k] is not None:
                stream.wait_event(free_out[k])
            stream.wait_event(ev_xw)
            done = {}
            for p in passes:
                if p != "fwd":
                    stream.wait_event(ev_g)
                launch_set(p, k)
                done[p] = torch.cuda.Event()
                done[p].record(stream)
            free_in[k] = done[passes[-1]]
            with torch.cuda.stream(d2h_s):
                for p in passes:
                    d2h_s.wait_event(done[p])
                    houts[k][p].copy_(outs[k][p], non_blocking=True)
                free_out[k] = torch.cuda.Event()
                free_out[k].record(d2h_s)

        for i in range(2):
            e2e_step(i)
        torch.cuda.synchronize(dev)
        if dist is not None:
            dist.barrier()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        h2d_s.wait_event(a)
        d2h_s.wait_event(a)
        for i in range(args.e2e_steps):
            e2e_step(2 + i)
        stream.wait_event(free_out[(1 + args.e2e_steps) % 2])
        b.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = max_over_ranks(a.elapsed_time(b), dist, dev)
        # both buffer sets' copied-out results equal the device-resident loop's
        # (same inputs; deterministic mode: bitwise; sampled rows of Y and dX)
        e2e_ok = None
        if det:
            rows = torch.arange(0, M, max(1, M // 64))
            ref = {p: (outs0[p][rows.to(dev)] if p != "wgrad" else outs0[p]).cpu() for p in passes}
            e2e_ok = all(torch.equal(houts[k][p][rows] if p != "wgrad" else houts[k][p], ref[p])
                         for k in range(2) for p in passes)
        e2e = {"value": flop_step * args.e2e_steps * ws / (e2e_ms * 1e-3) / 1e12, "unit": UNIT,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": e2e_ms / args.e2e_steps,
               "overlap": "host->device, kernels and device->host on three streams, two device buffer sets",
               "copied_out_equals_device": e2e_ok}

    # ---- roofline of the dominant kernel ----
    peaks = measured_peaks()
    dom = max(per_pass_ms, key=per_pass_ms.get)
    obytes = 4 if od == "fp32" else 2
    dom_s = per_pass_ms[dom] * 1e-3
    flop_pass, bytes_pass = wk.flops(1), wk.algorithmic_bytes(dom, obytes)
    # the pass is memory-bound when its arithmetic intensity is below the measured ridge point
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    traffic = traffic_for(wk.name, dom, od, det)
    if flop_pass / bytes_pass < ridge:
        achieved, peak = bytes_pass / dom_s / 1e9, peaks["hbm_gbs"]
        roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                    "peak_source": f"{peaks['source']} hbm_gbs (copy)"}
    else:
        achieved, peak = flop_pass / dom_s / 1e12, peaks["bf16_tflops"]
        roofline = {"bound": "tensor", "achieved": round(achieved, 1), "peak": peak, "unit": "TFLOP/s",
                    "peak_source": f"{peaks['source']} bf16_tflops (burst)"}
    roofline.update({"frac": round(achieved / peak, 4), "traffic": traffic,
                     "algorithmic_bytes": int(bytes_pass), "flop": int(flop_pass),
                     "kernel": f"cake_gg_kernel<{dom}>",
                     "per_pass_ms": {p: round(v, 4) for p, v in per_pass_ms.items()},
                     "per_pass_tflops": {p: round(flop_pass / (v * 1e-3) / 1e12, 1)
                                         for p, v in per_pass_ms.items()},
                     "per_pass_gbs": {p: round(wk.algorithmic_bytes(p, obytes) / (v * 1e-3) / 1e9, 1)
                                      for p, v in per_pass_ms.items()}})

    corun = None
    if args.corun:
        # co-run robustness: a bounded spinner holds n SMs for 60 % of the
        # plain timed region; ideal extra time = the SM-time it takes away
        corun = {"sms": [], "ms_per_step": [], "slowdown": [], "ideal_slowdown": [], "spin_ms": []}
        side = torch.cuda.Stream(dev)
        nsm = torch.cuda.get_device_properties(dev).multi_processor_count
        spin_ms = 0.6 * elapsed_ms
        for n in (int(v) for v in args.corun.split(",") if v):
            torch.cuda.synchronize(dev)
            rc = gg.cake_gg_corun_spinner(n, int(spin_ms * 1e6), side.cuda_stream)
            if rc != 0:
                raise gg.CakeGGError(rc, "corun spinner")
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(args.steps):
                for p in passes:
                    run_pass(p)
            b.record(stream)
            torch.cuda.synchronize(dev)
            t = a.elapsed_time(b)
            corun["sms"].append(n)
            corun["ms_per_step"].append(round(t / args.steps, 4))
            corun["slowdown"].append(round(t / elapsed_ms - 1.0, 4))
            corun["ideal_slowdown"].append(round(n * spin_ms / nsm / elapsed_ms, 4))
            corun["spin_ms"].append(round(spin_ms, 3))

    projection = {}
    if not args.no_thin and args.workload == "moe_gate_up":
        # the HBM-bound half of the target (thin projection) and the mid-size
        # dense weight gradient, each timed in this process on its own inputs
        if e2e is not None:
            del ins, outs, houts
        torch.cuda.empty_cache()
        projection["thin"] = projection_record(gg, dev, local, rank, 4096, 48, ("wgrad", "fwd", "dgrad"))
        projection["mid"] = projection_record(gg, dev, local, rank, 4096, 512, ("wgrad",))

    if not args.no_pages_sample and args.workload == "moe_gate_up" and ws == 1:
        # a sample of the pages' latency table, ckpt / ckpt ES through the autograd API
        projection["pages_sample"] = {
            "rows": pages_rows(PAGES_SAMPLE, 5, dev),
            "note": "one call per repetition, cold L2, median of 5; the pages' latencies are their GB300 "
                    "table's, measured on their machine with their kernels (context, not a target)"}

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wk, X, W, G, passes, args.cpu_seconds)

    line = {"metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": wk.name, "E": E, "M": M, "N": N, "K": K,
                       "group_sizes": sizes_desc(wk), "passes": passes, "out_dtype": od,
                       "deterministic": bool(det), "accumulate": "fp32",
                       "l2": "no flush: operands per step (%.2f GB) exceed the 129 MB L2" % (
                           (X.numel() + W.numel() + G.numel()) * 2 / 1e9),
                       "parallelism": f"replicas x{ws}",
                       "launch": "cuda-graph replay per pass" if args.graph else "eager",
                       "plans": {p: {k: v for k, v in plans[p].as_dict().items()
                                     if k in ("tile_n", "tile_k", "stages", "pair", "swap_ab", "split_chunk",
                                              "staging_bufs", "cluster_splits", "tail_units", "tail_splits",
                                              "epi_groups")} for p in passes}},
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            **({"corun": corun} if corun else {}),
            "gpu_launches": len(passes) * args.steps, "clocks": clocks,
            "sustained": sustained, **projection}
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def projection_record(gg, dev, local, rank, d_in, d_out, passes, seconds=0.4, per_graph=60, sets=3):
    """Dense projection (T = 16384, E = 1) passes timed back to back: `per_graph` calls captured
    once in a CUDA graph (no host launch gaps), rotating over `sets` input sets so that no call
    finds its operands in L2 from the call before (each set is larger than the L2), replayed for
    about `seconds` per pass with clocks sampled.  Weight gradient FP32 output, forward and data
    gradient BF16 output (the dense configuration), deterministic."""
    import torch
    from moe_ragged_grouped_gb300 import workloads as wl
    wk = wl.dense_projection(d_in, d_out)
    M, E, N, K = wk.M, wk.E, wk.N, wk.K
    data = [wk.make_torch(seed=s, device=dev) for s in range(sets)]
    offs = torch.from_numpy(wk.offsets).to(dev)
    peaks = measured_peaks()
    stream = torch.cuda.Stream(dev)
    out_rec = {"workload": wk.name, "T": M, "d_in": K, "d_out": N, "deterministic": True, "passes": {}}
    for p in passes:
        od = "fp32" if p == "wgrad" else "bf16"
        plan = gg.cake_gg_plan(p, E, M, N, K, od, 1)
        wsp = gg.make_workspace(plan, dev)
        tdt = torch.float32 if od == "fp32" else torch.bfloat16
        shape = {"fwd": (M, N), "dgrad": (M, K), "wgrad": (E, N, K)}[p]
        out = torch.empty(shape, dtype=tdt, device=dev)
        fn = {"fwd": gg.cake_gg_fwd, "dgrad": gg.cake_gg_dgrad, "wgrad": gg.cake_gg_wgrad}[p]

        def launch(i):
            X, W, G = data[i % sets]
            a, b = {"fwd": (X, W), "dgrad": (G, W), "wgrad": (G, X)}[p]
            rc = fn(plan, a, b, out, offs, od, 1, wsp, stream=stream.cuda_stream)
            if rc != 0:
                raise gg.CakeGGError(rc, f"{wk.name} {p}")

        with torch.cuda.stream(stream):
            for i in range(3 * sets):
                launch(i)
            torch.cuda.synchronize(dev)
            st = gg.cake_gg_check_status(wsp, stream.cuda_stream)
            if st != 0:
                raise gg.CakeGGError(st, f"{wk.name} {p} device status")
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                for i in range(per_graph):
                    launch(i)
            for _ in range(3):
                graph.replay()
            torch.cuda.synchronize(dev)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            graph.replay()
            b.record(stream)
            torch.cuda.synchronize(dev)
            reps = max(3, int(seconds / max(a.elapsed_time(b) * 1e-3, 1e-6)))
            sampler = ClockSampler(local) if rank == 0 else None
            time.sleep(0.3 if sampler else 0.0)
            torch.cuda.synchronize(dev)
            if sampler:
                sampler.mark_start()
            a.record(stream)
            for _ in range(reps):
                graph.replay()
            b.record(stream)
            torch.cuda.synchronize(dev)
            if sampler:
                sampler.mark_end()
            st = gg.cake_gg_check_status(wsp, stream.cuda_stream)
            if st != 0:
                raise gg.CakeGGError(st, f"{wk.name} {p} device status")
        n = reps * per_graph
        sec = a.elapsed_time(b) * 1e-3 / n
        ob = 4 if od == "fp32" else 2
        alg = wk.algorithmic_bytes(p, ob)
        flop = wk.flops(1)
        ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
        if flop / alg < ridge:
            ach, peak = alg / sec / 1e9, peaks["hbm_gbs"]
            roof = {"bound": "hbm", "achieved": round(ach, 1), "peak": peak, "unit": "GB/s",
                    "peak_source": f"{peaks['source']} hbm_gbs (copy)"}
        else:
            ach, peak = flop / sec / 1e12, peaks["bf16_tflops"]
            roof = {"bound": "tensor", "achieved": round(ach, 1), "peak": peak, "unit": "TFLOP/s",
                    "peak_source": f"{peaks['source']} bf16_tflops (burst)"}
        roof.update({"frac": round(ach / peak, 4), "traffic": traffic_for(wk.name, p, od, 1),
                     "algorithmic_bytes": int(alg), "flop": int(flop)})
        out_rec["passes"][p] = {
            "out_dtype": od, "us_per_launch": round(sec * 1e6, 3), "launches": n,
            "tflops": round(flop / sec / 1e12, 1), "gbs": round(alg / sec / 1e9, 1),
            "plan": {k: v for k, v in plan.as_dict().items()
                     if k in ("tile_n", "tile_k", "stages", "pair", "swap_ab", "split_chunk", "cluster_splits",
                              "tail_units", "tail_splits", "staging_bufs", "epi_groups")},
            "roofline": roof, "clocks": sampler.finish() if sampler else None}
        del wsp, out, graph
    out_rec["launch"] = (f"CUDA graph of {per_graph} back-to-back calls, replayed; {sets} input sets "
                         f"rotated ({sets * wk.M * wk.K * 2 / 1e6:.0f} MB of X) so no call's operands "
                         "are in L2 from the call before")
    del data
    torch.cuda.empty_cache()
    return out_rec


def sizes_desc(wk):
    s = wk.sizes
    if len(set(s)) == 1:
        return f"balanced {s[0]} x {len(s)}"
    return s


# ---------------------------------------------------------------------------- oracle timing


def _sample_plan(wk, passes, rng, n_per_pass):
    import numpy as np
    off = wk.offsets
    M = int(off[-1])
    sizes = np.diff(off)
    out = {}
    for p in passes:
        n = n_per_pass[p]
        if p in ("fwd", "dgrad"):
            rows = rng.integers(0, M, n)
            cols = rng.integers(0, wk.N if p == "fwd" else wk.K, n)
            L = np.full(n, wk.K if p == "fwd" else wk.N, np.float64)
            out[p] = (rows, cols, L)
        else:
            nonempty = np.nonzero(sizes)[0]
            es = nonempty[rng.integers(0, len(nonempty), n)]
            ns = rng.integers(0, wk.N, n)
            ks = rng.integers(0, wk.K, n)
            out[p] = (es, ns, ks, sizes[es].astype(np.float64))
    return out


def _run_oracle_sample(oracle, wk, Xb, Wb, Gb, samp):
    off = wk.offsets
    flop = 0.0
    t0 = time.perf_counter()
    for p, s in samp.items():
        if p == "fwd":
            oracle.fwd_at(Xb, Wb, off, s[0], s[1])
            flop += 2.0 * s[2].sum()
        elif p == "dgrad":
            oracle.dgrad_at(Gb, Wb, off, s[0], s[1])
            flop += 2.0 * s[2].sum()
        else:
            oracle.wgrad_at(Gb, Xb, off, wk.E, s[0], s[1], s[2])
            flop += 2.0 * s[3].sum()
    return flop, time.perf_counter() - t0


def _calibrate(oracle, wk, Xb, Wb, Gb, passes, seconds):
    """Sample sizes per pass so that one oracle sample of all passes takes about `seconds`."""
    import numpy as np
    rng = np.random.default_rng(1234)
    n = {}
    for p in passes:
        k = 64
        while True:
            samp = _sample_plan(wk, [p], rng, {p: k})
            _, dt = _run_oracle_sample(oracle, wk, Xb, Wb, Gb, samp)
            if dt >= 0.1 or k >= 1 << 22:
                break
            k *= 4
        per = max(dt / k, 1e-9)
        n[p] = max(16, int(seconds / len(passes) / per))
    return n


def host_bits(wk, X, W, G):
    from moe_ragged_grouped_gb300 import workloads as wl
    return wl.torch_bf16_to_bits(X), wl.torch_bf16_to_bits(W), wl.torch_bf16_to_bits(G)


def cpu_baseline(wk, X, W, G, passes, seconds):
    import numpy as np
    import oracle
    Xb, Wb, Gb = host_bits(wk, X, W, G)
    n = _calibrate(oracle, wk, Xb, Wb, Gb, passes, seconds / 4)
    n = {p: int(v * 4) for p, v in n.items()}
    samp = _sample_plan(wk, passes, np.random.default_rng(99), n)
    flop, dt = _run_oracle_sample(oracle, wk, Xb, Wb, Gb, samp)
    return {"value": flop / dt / 1e12, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": ("%s output elements sampled uniformly (each a full FP64 dot product over its "
                       "reduction length), %.1f s of CPU work" % (
                           ", ".join(f"{n[p]} {p}" for p in passes), dt)),
            "seconds": round(dt, 2)}


def run_reference(args, wk):
    import numpy as np
    ws, rank, local = dist_env()
    if rank != 0:
        return
    import oracle
    passes = [p for p in args.passes.split(",") if p]
    try:
        import torch
        dev = "cuda" if torch.cuda.is_available() else "cpu"
    except Exception:
        dev = "cpu"
    X, W, G = wk.make_torch(seed=0, device=dev)
    Xb, Wb, Gb = host_bits(wk, X, W, G)
    del X, W, G
    per_step = 1.5
    n = _calibrate(oracle, wk, Xb, Wb, Gb, passes, per_step)
    rng = np.random.default_rng(7)
    for _ in range(args.warmup):
        _run_oracle_sample(oracle, wk, Xb, Wb, Gb, _sample_plan(wk, passes, rng, n))
    flop = dt = 0.0
    for _ in range(args.steps):
        f, t = _run_oracle_sample(oracle, wk, Xb, Wb, Gb, _sample_plan(wk, passes, rng, n))
        flop += f
        dt += t
    value = flop / dt / 1e12
    sample = ("per step: %s output elements sampled uniformly (FP64 dot products over the full "
              "reduction length)" % ", ".join(f"{n[p]} {p}" for p in passes))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": wk.name, "E": wk.E, "M": wk.M, "N": wk.N, "K": wk.K,
                       "group_sizes": sizes_desc(wk), "passes": passes, "out_dtype": args.out_dtype,
                       "deterministic": bool(args.det)},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


PAGES_SAMPLE = [("gate_up E8 M131072 bal", "dW"), ("gate_up E8 M131072 bal", "ckpt"),
                ("gate_up E8 M131072 bal", "ckpt ES")]


def pages_rows(rows, reps, dev):
    """Time rows of the pages' GB300 latency table (PR #8269) the way it was measured: one call
    per repetition, L2 flushed (256 MB written) before it, CUDA events around it, median over
    `reps`.  "dW" is one cake_gg_wgrad call.  "ckpt" and "ckpt ES" go through the autograd API:
    checkpointed_grouped_linear (grouped_linear in a non-reentrant torch checkpoint, early stop
    off / on) forward, then backward with the upstream gradient G.  Before the start event a GPU
    sleep of a few milliseconds is queued so that the host's enqueueing (autograd and checkpoint
    bookkeeping) runs while the GPU sleeps: the events then bracket the device work alone.
    Returns one dict per row."""
    import torch
    from moe_ragged_grouped_gb300 import cake_gg as gg
    from moe_ragged_grouped_gb300 import workloads as wl
    from moe_ragged_grouped_gb300.autograd import checkpointed_grouped_linear
    gg.load_library()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)   # twice the L2
    stream = torch.cuda.current_stream(dev)
    table = {(r[0], r[1]): r for r in wl.PAGES_GB300_ROWS}
    cur_shape, tensors = None, None
    out_rows = []
    for shape, op in rows:
        _, _, det_ms, sota_ms, sota_key, nd_ms = table[(shape, op)]
        wk, od_dw = wl.pages_workload(shape)
        if shape != cur_shape:
            tensors = None
            torch.cuda.empty_cache()
            X, W, G = wk.make_torch(seed=0, device=dev)
            offs = torch.from_numpy(wk.offsets).to(dev)
            tensors = (X, W, G, offs)
            cur_shape = shape
        X, W, G, offs = tensors
        passes = wl.PAGES_OPS[op]
        od = od_dw if op == "dW" else "bf16"
        tdt = torch.float32 if od == "fp32" else torch.bfloat16
        outs = {"wgrad": torch.empty((wk.E, wk.N, wk.K), dtype=tdt, device=dev)} if op == "dW" else {}
        plans = {p: gg.cake_gg_plan(p, wk.E, wk.M, wk.N, wk.K, od, 1) for p in set(passes)} if op == "dW" else {}
        wss = {p: gg.make_workspace(plans[p], dev) for p in plans}
        Xl, Wl = X.detach().requires_grad_(), W.detach().requires_grad_()

        def call():
            if op == "dW":
                rc = gg.cake_gg_wgrad(plans["wgrad"], G, X, outs["wgrad"], offs, od, 1, wss["wgrad"],
                                      stream=stream.cuda_stream)
                if rc != 0:
                    raise gg.CakeGGError(rc, "wgrad")
            else:
                Xl.grad = Wl.grad = None
                Y = checkpointed_grouped_linear(Xl, Wl, offs, early_stop=(op == "ckpt ES"))
                Y.backward(G)

        for _ in range(2):
            call()
        torch.cuda.synchronize(dev)
        for p in plans:
            st = gg.cake_gg_check_status(wss[p], stream.cuda_stream)
            if st != 0:
                raise gg.CakeGGError(st, f"{shape} {p} device status")
        times = []
        for _ in range(reps):
            flush.zero_()
            torch.cuda._sleep(6_000_000)   # ~3 ms at 2 GHz: the host enqueues meanwhile
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            call()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            times.append(e0.elapsed_time(e1))
        ms = statistics.median(times)
        out_rows.append({"grid": "pages_gb300", "shape": shape, "op": op, "out_dtype": od, "deterministic": True,
                         "path": "cake_gg_wgrad" if op == "dW" else "checkpointed_grouped_linear (autograd)",
                         "ms": round(ms, 4), "tflops": round(wk.flops(len(passes)) / (ms * 1e-3) / 1e12, 1),
                         "ms_min_max": [round(min(times), 4), round(max(times), 4)],
                         "pages_det_ms": det_ms, "vs_pages_det": round(det_ms / ms, 4),
                         "pages_nondet_ms": nd_ms, "vs_pages_nondet": round(nd_ms / ms, 4),
                         "pages_sota_ms": sota_ms, "pages_sota": sota_key, "vs_pages_sota": round(sota_ms / ms, 4)})
        del outs, wss, Xl, Wl
    del tensors, flush
    torch.cuda.empty_cache()
    return out_rows


def run_pages_grid(args):
    """The 100 GB300 rows of the pages' latency table (or those matching --grid-filter)."""
    import torch
    from moe_ragged_grouped_gb300 import workloads as wl
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    rows = [(r[0], r[1]) for r in wl.PAGES_GB300_ROWS if args.grid_filter in f"{r[0]} {r[1]}"]
    ratios = {}
    lines = pages_rows(rows, args.grid_reps, dev)
    for line in lines:
        print(json.dumps(line), flush=True)
        for k in ("det", "nondet", "sota"):
            ratios.setdefault((line["op"], k), []).append(line[f"vs_pages_{k}"])
    summary = {"grid": "pages_gb300", "summary": "geomean of (pages' latency / ours) per operation", "rows": len(rows)}
    for (op, k), v in sorted(ratios.items()):
        summary[f"{op} vs {k}"] = round(math.exp(sum(math.log(x) for x in v) / len(v)), 4)
    print(json.dumps(summary), flush=True)


# ---------------------------------------------------------------------------- planner decisions

# Plan rules under test: (candidate plan environment, baseline plan environment, default points).
# The environment is read by cake_gg_plan only; each arm plans under its own.
DECIDE_RULES = {
    # the weight gradient's split tail (last partial wave of equal units as pieces) vs whole units
    "tail": ({"CAKE_GG_TAIL": "1"}, {"CAKE_GG_TAIL": "0"},
             ["moe_gate_up", "dense_5120to1024", "pages:gate_up E8 M131072 bal", "pages:down E8 M131072 bal",
              "pages:gate_up E4 M112576 bal", "pages:down E4 M136064 bal fp32"]),
    # the stream-K walk of a one-expert weight gradient vs the split / split-tail plan
    "streamk": ({"CAKE_GG_STREAMK": "1"}, {"CAKE_GG_STREAMK": "0"},
                ["dense_4096to512", "dense_5120to512", "dense_4096to1024", "dense_5120to1024"]),
    # the global split of few-tile weight gradients vs one unit per tile
    "split": ({}, {"CAKE_GG_SPLIT_CHUNK": "0", "CAKE_GG_TAIL": "0"},
              ["dense_4096to512", "dense_5120to512", "dense_4096to64"]),
    # 256 x 512 weight-gradient tiles vs 256 x 256
    "wide": ({}, {"CAKE_GG_WIDE": "0"}, ["moe_gate_up", "pages:gate_up E4 M112576 bal", "dense_4096to4096"]),
    # a split tile reduced on chip by its cluster vs the same splits through workspace slots
    "csplit": ({}, {"CAKE_GG_CSPLIT": "0"}, ["dense_4096to512", "dense_4096to48", "dense_4096to64"]),
}


def _sign_test_p(wins, n):
    """One-sided sign test: P(X >= wins) for X ~ Binomial(n, 1/2)."""
    return sum(math.comb(n, i) for i in range(wins, n + 1)) / 2.0 ** n


def run_decide(args):
    """The pages' rule for keeping a plan choice (flashinfer PR #8363 and its follow-up, "Summary"
    and "Definitions"): at a point the candidate is kept only if (a) at the op (the weight gradient)
    it is faster in every run -- a one-sided paired sign test over the groups with p < 0.05 and a
    median paired ratio below 0.99 -- in eager launches and in CUDA graph replays; (b) next to a
    kernel holding 8, 16 or 32 SMs on another stream it is at most 3 % slower than the baseline, in
    both launch orders; (c) the backward (data + weight gradient) and the checkpointed step
    (2 x forward + backward) are at most 1.3 % slower, as the ratio of the medians over the runs,
    eager and graph.  Every iteration runs with a cold L2 (256 MB written before it); the two
    arms alternate inside each group, in an order that flips from group to group; a GPU sleep
    queued before each iteration's start event keeps host launch overhead out of the device
    interval."""
    import torch
    from moe_ragged_grouped_gb300 import cake_gg as gg
    from moe_ragged_grouped_gb300 import workloads as wl
    cand_env, base_env, default_points = DECIDE_RULES[args.decide]
    points = [p for p in args.decide_points.split(",") if p] or default_points
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    gg.load_library()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    side = torch.cuda.Stream(dev)
    det = 1 if args.det else 0
    summary = {"decide": args.decide, "deterministic": bool(det), "candidate_env": cand_env,
               "baseline_env": base_env, "points": {}}

    def plan_under(env, *a):
        # (the planner's own per-point decisions are switched off: both arms plan by their rule)
        env = dict(env, CAKE_GG_DECIDED="0")
        old = {k: os.environ.get(k) for k in env}
        os.environ.update(env)
        try:
            return gg.cake_gg_plan(*a)
        finally:
            for k, v in old.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v

    for point in points:
        if point.startswith("pages:"):
            wk, od_w = wl.pages_workload(point[len("pages:"):])
        else:
            wk, od_w = get_workload(point), "bf16"
            if point.startswith("dense_"):
                od_w = "fp32"
        X, W, G = wk.make_torch(seed=0, device=dev)
        offs = torch.from_numpy(wk.offsets).to(dev)
        M, E, N, K = wk.M, wk.E, wk.N, wk.K
        outs = {"fwd": torch.empty((M, N), dtype=torch.bfloat16, device=dev),
                "dgrad": torch.empty((M, K), dtype=torch.bfloat16, device=dev),
                "wgrad": torch.empty((E, N, K), dtype=torch.float32 if od_w == "fp32" else torch.bfloat16,
                                     device=dev)}
        arms = {}
        for arm, env in (("cand", cand_env), ("base", base_env)):
            pl = {"fwd": plan_under(env, "fwd", E, M, N, K, "bf16", det),
                  "dgrad": plan_under(env, "dgrad", E, M, N, K, "bf16", det),
                  "wgrad": plan_under(env, "wgrad", E, M, N, K, od_w, det)}
            arms[arm] = (pl, {p: gg.make_workspace(pl[p], dev) for p in pl})
        pc, pb = arms["cand"][0]["wgrad"].as_dict(), arms["base"][0]["wgrad"].as_dict()
        rec = {"workload": wk.name, "wgrad_out": od_w, "deterministic": bool(det),
               "cand_plan": {k: pc[k] for k in ("tile_n", "split_chunk", "tail_units", "tail_splits",
                                                "streamk_kblocks")},
               "base_plan": {k: pb[k] for k in ("tile_n", "split_chunk", "tail_units", "tail_splits",
                                                "streamk_kblocks")}}
        if pc == pb:
            rec["verdict"] = "rule does not apply (same plan)"
            print(json.dumps(rec), flush=True)
            summary["points"][point] = rec["verdict"]
            continue
        calls = {"fwd": (gg.cake_gg_fwd, X, W, "bf16"), "dgrad": (gg.cake_gg_dgrad, G, W, "bf16"),
                 "wgrad": (gg.cake_gg_wgrad, G, X, od_w)}
        ops = {"wgrad": ("wgrad",), "bwd": ("dgrad", "wgrad"), "ckpt": ("fwd", "fwd", "dgrad", "wgrad")}

        def run_op(arm, op, s):
            pl, wsp = arms[arm]
            for p in ops[op]:
                fn, a, b, od = calls[p]
                rc = fn(pl[p], a, b, outs[p], offs, od, det, wsp[p], stream=s.cuda_stream)
                if rc != 0:
                    raise gg.CakeGGError(rc, f"{point} {arm} {p}")

        for arm in arms:
            for op in ops:
                run_op(arm, op, stream)
        torch.cuda.synchronize(dev)
        for arm in arms:
            for p, wsp in arms[arm][1].items():
                st = gg.cake_gg_check_status(wsp, stream.cuda_stream)
                if st != 0:
                    raise gg.CakeGGError(st, f"{point} {arm} {p} device status")
        graphs = {}
        cap = torch.cuda.Stream(dev)
        for arm in arms:
            for op in ops:
                g_ = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g_, stream=cap):
                    run_op(arm, op, cap)
                graphs[(arm, op)] = g_
        torch.cuda.synchronize(dev)

        def one(arm, op, mode):
            flush.zero_()
            torch.cuda._sleep(4_000_000)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            if mode == "graph":
                graphs[(arm, op)].replay()
            else:
                run_op(arm, op, stream)
            e1.record(stream)
            return e0, e1

        def measure(op, mode, groups, steps):
            """Per group: the median over `steps` iterations of each arm; arms alternate."""
            per = {"cand": [], "base": []}
            for gi in range(groups):
                order = ("cand", "base") if gi % 2 == 0 else ("base", "cand")
                evs = {a: [] for a in order}
                for _ in range(steps):
                    for a in order:
                        evs[a].append(one(a, op, mode))
                torch.cuda.synchronize(dev)
                for a in order:
                    per[a].append(statistics.median(x.elapsed_time(y) for x, y in evs[a]))
            return per

        crit_a, crit_c = True, True
        rec["a"], rec["c"] = [], []
        for mode in ("eager", "graph"):
            med = {op: {"cand": [], "base": []} for op in ops}
            for run in range(args.decide_runs):
                for op in ops:
                    per = measure(op, mode, args.decide_groups, args.decide_steps if op == "wgrad" else 3)
                    med[op]["cand"].append(statistics.median(per["cand"]))
                    med[op]["base"].append(statistics.median(per["base"]))
                    if op == "wgrad":
                        ratios = [c / b for c, b in zip(per["cand"], per["base"])]
                        wins = sum(r < 1.0 for r in ratios)
                        p = _sign_test_p(wins, len(ratios))
                        mr = statistics.median(ratios)
                        ok = p < 0.05 and mr < 0.99
                        crit_a &= ok
                        rec["a"].append({"mode": mode, "run": run, "wins": wins, "groups": len(ratios),
                                         "p": round(p, 4), "median_ratio": round(mr, 4), "pass": ok,
                                         "cand_ms": round(statistics.median(per["cand"]), 4),
                                         "base_ms": round(statistics.median(per["base"]), 4)})
            for op in ("bwd", "ckpt"):
                r = statistics.median(med[op]["cand"]) / statistics.median(med[op]["base"])
                ok = r <= 1.013
                crit_c &= ok
                rec["c"].append({"mode": mode, "op": op, "ratio": round(r, 4), "pass": ok})
        # (b) co-run: a spinner holds n SMs on another stream for about three baseline op times
        crit_b = True
        rec["b"] = []
        base_ms = statistics.median(x["base_ms"] for x in rec["a"])
        spin_ns = int(max(3 * base_ms, 0.05) * 1e6)
        for n in (8, 16, 32):
            for order in ("spinner first", "op first"):
                t = {}
                for arm in ("cand", "base"):
                    ts = []
                    for _ in range(5):
                        flush.zero_()
                        torch.cuda.synchronize(dev)
                        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                        if order == "spinner first":
                            gg.cake_gg_corun_spinner(n, spin_ns, side.cuda_stream)
                        e0.record(stream)
                        run_op(arm, "wgrad", stream)
                        e1.record(stream)
                        if order == "op first":
                            gg.cake_gg_corun_spinner(n, spin_ns, side.cuda_stream)
                        torch.cuda.synchronize(dev)
                        ts.append(e0.elapsed_time(e1))
                    t[arm] = statistics.median(ts)
                r = t["cand"] / t["base"]
                ok = r <= 1.03
                crit_b &= ok
                rec["b"].append({"sms": n, "order": order, "ratio": round(r, 4), "pass": ok})
        rec["verdict"] = "keep" if (crit_a and crit_b and crit_c) else "drop"
        rec["criteria"] = {"a": crit_a, "b": crit_b, "c": crit_c}
        print(json.dumps(rec), flush=True)
        summary["points"][point] = rec["verdict"]
        del graphs, arms, outs, X, W, G
        torch.cuda.empty_cache()
    print(json.dumps(summary), flush=True)


def run_router(args):
    """The dense projection family's FP32 router GEMM (BF16x3 emulation): T = 16384 tokens,
    K = 4096, R = 256 experts, FP32 X and W (flashinfer PR #8438, "Summary").  A step is one
    router call: W split into BF16 high / low parts, then the router kernel (FP32 X tiles split
    on chip, three BF16 products per k).  value = 2 T R K per step / time."""
    import torch
    from moe_ragged_grouped_gb300 import cake_gg as gg
    from moe_ragged_grouped_gb300 import workloads as wl
    gg.load_library()
    T, K, R = wl.ROUTER_T, wl.ROUTER_K, wl.ROUTER_R
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    X, W = wl.router_inputs_torch(T, K, R, seed=0, device="cuda")
    rp = gg.cake_gg_router_plan(T, R, K)
    ws = torch.zeros(int(rp.workspace_bytes), dtype=torch.uint8, device=dev)
    Y = torch.empty((T, R), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        rc = gg.cake_gg_router_fp32(rp, X, W, Y, ws)
        if rc != gg.CAKE_GG_OK:
            raise gg.CakeGGError(rc, "router")

    for _ in range(max(3, args.warmup)):
        step()
    st = gg.cake_gg_check_status(ws)
    if st != gg.CAKE_GG_OK:
        raise gg.CakeGGError(st, "router (device status)")
    sampler = ClockSampler(0)
    torch.cuda.synchronize()
    sampler.mark_start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    sampler.mark_end()
    ms = e0.elapsed_time(e1) / args.steps
    clocks = sampler.finish()
    peaks = measured_peaks()
    flop = 2.0 * T * R * K
    mma_flop = 3.0 * flop                                   # three BF16 products per FP32 product
    alg_bytes = 4.0 * (T + R) * K + 4.0 * T * R             # FP32 X, W read once, FP32 logits written
    mma_tf = mma_flop / (ms * 1e-3) / 1e12
    line = {"metric": METRIC, "value": round(flop / (ms * 1e-3) / 1e12, 1), "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32 via bf16x3", "data": "synthetic",
            "config": {"workload": f"router_T{T}_K{K}_R{R}", "T": T, "K": K, "R": R,
                       "inputs": "X~N(0,1), W~N(0,1/K), float32",
                       "emulation": "bf16x3: x_hi w_hi + x_hi w_lo + x_lo w_hi, FP32 accumulation",
                       "value_flop": "2 T R K per step (the FP32 GEMM)",
                       "l2": "no flush: X (268 MB) exceeds the 129 MB L2",
                       "plan": {"tile_n": rp.gemm.tile_n, "tile_k": rp.gemm.tile_k, "stages": rp.gemm.stages,
                                "pair": rp.gemm.pair}},
            "roofline": {"bound": "tensor", "achieved": round(mma_tf, 1), "peak": peaks["bf16_tflops"],
                         "unit": "TFLOP/s", "frac": round(mma_tf / peaks["bf16_tflops"], 4), "traffic": None,
                         "kernel": "cake_gg_kernel<router>: FP32 X tiles split on chip, 3 bf16 products",
                         "flop_per_step": mma_flop, "algorithmic_bytes": alg_bytes,
                         "achieved_gbs": round(alg_bytes / (ms * 1e-3) / 1e9, 1),
                         "memory_roof_ms": round(alg_bytes / (peaks["hbm_gbs"] * 1e9) * 1e3, 4),
                         "tensor_roof_ms": round(mma_flop / (peaks["bf16_tflops"] * 1e12) * 1e3, 4)},
            "gpu_launches": 2 * args.steps, "clocks": clocks}
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.grid == "pages":
        run_pages_grid(args)
        return
    if args.decide:
        run_decide(args)
        return
    if args.workload == "router":
        run_router(args)
        return
    wk = get_workload(args.workload)
    if args.workload != "moe_gate_up" and "wgrad" in args.passes and wk.passes == ("wgrad",):
        args.passes = "wgrad"
    if args.impl == "reference":
        run_reference(args, wk)
    else:
        run_ours(args, wk)


if __name__ == "__main__":
    main()
