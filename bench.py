#!/usr/bin/env python
"""Benchmark of the deterministic attention backward (DASH schedules) on one GB300.

One step = one whole backward through the C ABI: preprocess (D = rowsum(dO*O)), the main
kernel (compute + ordered dQ reduction) and, for the non-deterministic variant, the dQ
convert. Default workload: full mask, batch 2, 16 heads, seqlen 8192, headdim 128, BF16
N(0,1) inputs, Shift Scheduling (the best DASH order for a full mask). Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--schedule NAME]

Under torchrun (N > 1) every rank runs the same workload on its own GPU (replicas: the
path has no exchange between heads); value = total FLOPs of all ranks / max time.
--impl reference times the fp64 CPU oracle on the host cores instead.
"""

import os

# BLAS threads for the CPU oracle legs: all cores this process may use (set before numpy).
_CORES = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
os.environ.setdefault("OPENBLAS_NUM_THREADS", str(_CORES))
os.environ.setdefault("OMP_NUM_THREADS", str(_CORES))

import argparse  # noqa: E402
import hashlib  # noqa: E402
import json  # noqa: E402
import math  # noqa: E402
import statistics  # noqa: E402
import subprocess  # noqa: E402
import sys  # noqa: E402
import time  # noqa: E402

import numpy as np  # noqa: E402
import torch  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "deterministic attn-bwd TFLOPS (BF16, 1×GB300) and % of tensor peak vs non-det"

WORKLOADS = {
    "full-1x256x1x64": dict(mask="full", B=1, S=256, H=1, D=64),
    "causal-4x2048x16x64": dict(mask="causal", B=4, S=2048, H=16, D=64),
    "full-2x8192x16x128": dict(mask="full", B=2, S=8192, H=16, D=128),
    "causal-1x16384x32x128": dict(mask="causal", B=1, S=16384, H=32, D=128),
    # smaller full-mask case for kernel profiles (inputs still larger than L2)
    "full-2x4096x16x128": dict(mask="full", B=2, S=4096, H=16, D=128),
    # the same with a last partial round of 16 units on 152 CTAs, whose KV tiles the
    # dealing splits over two CTAs (the kernel instance with the split-tile epilogue)
    "full-3x4096x16x128": dict(mask="full", B=3, S=4096, H=16, D=128),
    # long full-mask sequence: where the pages see Shift fall behind the baseline order
    "full-1x16384x16x128": dict(mask="full", B=1, S=16384, H=16, D=128),
}
# the transformer-block sweep: causal, 16384 tokens (B * S), 32 heads, D = 64 and 128
for _s in (1024, 2048, 4096, 8192, 16384):
    for _d in (64, 128):
        WORKLOADS.setdefault(f"causal-{16384 // _s}x{_s}x32x{_d}",
                             dict(mask="causal", B=16384 // _s, S=_s, H=32, D=_d))
DEFAULT_WORKLOAD = "full-2x8192x16x128"
BEST_DASH = {"full": "shift", "causal": "symmetric_shift"}   # reference arm's naming only
# Cost model of the run-time selector (dash_sched_select), cycles per 128 x 128 task measured
# on GB300 with the head-dim-128 kernel: compute step, hold of a dQ block's turn, hand-off
# between SMs; two-engine SM.
SELECT_COSTS = {"c": 6900.0, "r": 5600.0, "h": 3000.0, "overlapped": 1}
L2_BYTES = 129 * 1024 * 1024


def bwd_flops(w) -> float:
    """Algorithmic backward FLOPs: 10*B*H*S^2*D (5 GEMM-shaped products), halved when causal."""
    f = 10.0 * w["B"] * w["H"] * w["S"] ** 2 * w["D"]
    return f / 2 if w["mask"] == "causal" else f


def slice_flops(w) -> float:
    return bwd_flops(w) / (w["B"] * w["H"])


def input_bytes(w) -> int:
    t = w["B"] * w["S"] * w["H"] * w["D"] * 2
    return 5 * t + w["B"] * w["H"] * w["S"] * 4


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The largest of every rank's value (the timing rule: max over ranks)."""
    if world <= 1:
        return value
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flops_per_rank: float, world: int, ms_per_step: float) -> float:
    """Whole-job throughput: the FLOPs of all ranks over the slowest rank's step time."""
    return flops_per_rank * world / (ms_per_step / 1e3) / 1e12


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["bf16_tflops"]), float(p["hbm_gbs"]), "measured"
    return 1900.0, 6800.0, "fallback"


# ---------------------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "100"]
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            cmd += ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
        except Exception:
            pass
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except Exception:
            self.proc = None
        self.first = ""
        if self.proc is not None:
            # nvidia-smi's start-up must not overlap the timed region: wait for its first
            # sample (it is kept and counted with the rest)
            import select

            ready, _, _ = select.select([self.proc.stdout], [], [], 10.0)
            if ready:
                self.first = self.proc.stdout.readline()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        out = self.first + out
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[3:7]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------------------
# the fp64 CPU oracle (reported baseline / reference arm)
# ---------------------------------------------------------------------------------------
def oracle_slices(w, budget_s: float, max_slices: int, seed: int = 0):
    """Time the oracle backward on (b, h) slices of the workload until budget_s is used.

    Returns (seconds per slice, slices timed). Inputs are the workload's own seeded bf16
    tensors; O and LSE come from the oracle forward (untimed)."""
    from oracle.attention import attn_bwd_slice, attn_fwd_slice
    from reproducible_deterministic_attn_gb300.inputs import make_inputs

    x = make_inputs(w["B"], w["S"], w["H"], w["D"], seed)
    f = lambda t, b, h: t[b, :, h].float().double().numpy()
    causal = w["mask"] == "causal"
    scale = 1.0 / math.sqrt(w["D"])
    times = []
    for idx in range(min(max_slices, w["B"] * w["H"])):
        b, h = divmod(idx, w["H"])
        q, k, v, do = (f(x[n], b, h) for n in ("q", "k", "v", "do"))
        o, lse = attn_fwd_slice(q, k, v, scale, causal, row_block=1024)
        t0 = time.perf_counter()
        attn_bwd_slice(q, k, v, o, do, lse, scale, causal, row_block=1024)
        times.append(time.perf_counter() - t0)
        if sum(times) >= budget_s:
            break
    return statistics.median(times), len(times)


def cpu_baseline(w, budget_s=12.0):
    per_slice, n = oracle_slices(w, budget_s, max_slices=64)
    tflops = slice_flops(w) / per_slice / 1e12
    return {"value": tflops, "unit": "TFLOPS", "cores": int(os.environ["OPENBLAS_NUM_THREADS"]),
            "kind": "oracle",
            "sample": f"{n} (batch, head) slice(s) of the workload (seqlen {w['S']}, headdim "
                      f"{w['D']}, {w['mask']} mask), fp64 NumPy/OpenBLAS, median time per slice "
                      f"scaled to the slice's FLOPs"}


def run_reference(args, w, rank):
    if rank != 0:
        return
    per = []
    steps = args.steps if args.steps else 3
    warm = args.warmup if args.warmup is not None else 1
    # each step: one (b, h) slice of the backward (bounded sample of the workload)
    from oracle.attention import attn_bwd_slice, attn_fwd_slice
    from reproducible_deterministic_attn_gb300.inputs import make_inputs

    x = make_inputs(1, w["S"], 1, w["D"], 0)
    f = lambda t: t[0, :, 0].float().double().numpy()
    q, k, v, do = (f(x[n]) for n in ("q", "k", "v", "do"))
    causal = w["mask"] == "causal"
    scale = 1.0 / math.sqrt(w["D"])
    o, lse = attn_fwd_slice(q, k, v, scale, causal, row_block=1024)
    for it in range(warm + steps):
        t0 = time.perf_counter()
        attn_bwd_slice(q, k, v, o, do, lse, scale, causal, row_block=1024)
        dt = time.perf_counter() - t0
        if it >= warm:
            per.append(dt)
    ms = statistics.median(per) * 1e3
    value = slice_flops(w) / (ms / 1e3) / 1e12
    cores = int(os.environ["OPENBLAS_NUM_THREADS"])
    sample = (f"one (batch, head) slice per step (seqlen {w['S']}, headdim {w['D']}, "
              f"{w['mask']} mask), fp64 NumPy/OpenBLAS oracle")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOPS",
        "n_gpus": args.gpus, "steps": steps, "warmup": warm, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(args, w),
        "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(args, w):
    return {"workload": args.workload, "mask": w["mask"], "batch": w["B"], "heads": w["H"],
            "seqlen": w["S"], "headdim": w["D"], "schedule": args.schedule,
            "deterministic": True,
            "l2": ("inputs larger than L2 (%.0f MB read per step vs 129 MB L2)"
                   % (input_bytes(w) / 2**20)) if input_bytes(w) > L2_BYTES else
                  "L2 flushed before every step (256 MB write, outside the step's own CUDA events)"}


# ---------------------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------------------
def traffic_from_profile(w, sched):
    """Per-launch DRAM bytes of the main kernel from the committed ncu summary, if it was
    taken on the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", "bwd_main_traffic.json")
    if not os.path.exists(path):
        return None
    try:
        with open(path) as f:
            rec = json.load(f)
    except Exception:
        return None
    if rec.get("source_hash") != kernel_source_hash():
        return None
    key = f"{w['mask']}-{w['B']}x{w['S']}x{w['H']}x{w['D']}-{sched}"
    ent = rec.get("per_launch_bytes", {}).get(key)
    return float(ent) if ent is not None else None


# the sources the main kernel is compiled from (the file and its includes) and the
# dealing that spreads its work over the CTAs: the traffic record stays valid while none
# of them changes
MAIN_KERNEL_SOURCES = ("common.cuh", "tc_shared.cuh", "bwd_main.cuh", "tc_ptx.cuh",
                       "sched.h", "sched.cpp")


def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "reproducible_deterministic_attn_gb300", "csrc")
    for name in MAIN_KERNEL_SOURCES:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def run_gpu(args, w, rank, world, local_rank):
    import torch.distributed as dist

    import reproducible_deterministic_attn_gb300 as da
    from reproducible_deterministic_attn_gb300 import build as _build
    from reproducible_deterministic_attn_gb300.inputs import make_inputs

    _build.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    B, S, H, D = w["B"], w["S"], w["H"], w["D"]
    causal = w["mask"] == "causal"
    mask = da.MASK_CAUSAL if causal else da.MASK_FULL
    scale = 1.0 / math.sqrt(D)
    selected_by = "command line"
    if args.schedule == "auto":
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        choice, _ = da.dash_sched_select(mask, S // 128, B * H, sms, SELECT_COSTS["c"],
                                         SELECT_COSTS["r"], SELECT_COSTS["h"],
                                         SELECT_COSTS["overlapped"], head_dim=D)
        args.schedule = {v: k for k, v in da.SCHEDULES.items()}[choice]
        selected_by = "dash_sched_select, costs " + json.dumps(SELECT_COSTS)
    sched = da.SCHEDULES[args.schedule]
    # deterministic mode: 1 = one fixed chain per dQ block (the pages' order as one serial
    # chain), 2 = the same order as two interleaved chains. Measured on GB300 (TF/s, two
    # chains vs one) the second pays at head dimension 128 from S = 4096 on (full
    # 2x8192x16x128: 998 vs 948; causal 4x4096x32x128: 809 vs 776; causal 1x16384x32x128:
    # 1004 vs 940) and not below (causal 8x2048x32x128: 638 vs 645; 16x1024x32x128: 442 vs
    # 482), nor at head dimension 64 (causal 4x4096x32x64: 499 vs 532; 1x16384x32x64: 637
    # vs 633), where the dealing's balanced pieces already keep the waits short and zeroing
    # and summing the second fp32 copy costs more than they save.
    DET = ((2 if D == 128 and S >= 4096 else 1) if args.dq_chains == "auto"
           else int(args.dq_chains))

    x = make_inputs(B, S, H, D, seed=rank)
    q, k, v, do = (x[nm].to(dev) for nm in ("q", "k", "v", "do"))
    o, lse = da.attn_forward(q, k, v, scale, causal)
    ws = da.new_workspace(B, S, H, D, dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    flush = None
    if input_bytes(w) <= L2_BYTES:
        flush = torch.empty(256 * 2**20, dtype=torch.uint8, device=dev)

    def step(det=DET, s=sched):
        if flush is not None:
            flush.fill_(1)
        da.dash_attn_bwd(q, k, v, o, do, lse, dq, dk, dv, ws, scale, mask, s, det)

    def timed_steps(n_steps, det, s):
        """Device time of n_steps backward calls in ms. With the L2 flush, each call is
        bracketed by its own event pair after its flush, so the flush is not timed."""
        if flush is None:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(n_steps):
                step(det, s)
            e1.record()
            torch.cuda.synchronize()
            return e0.elapsed_time(e1)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(n_steps)]
        for a, b in ev:
            flush.fill_(1)
            a.record()
            da.dash_attn_bwd(q, k, v, o, do, lse, dq, dk, dv, ws, scale, mask, s, det)
            b.record()
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in ev)

    def barrier():
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()

    def timed(n_steps, det=DET, s=sched, profile=False):
        barrier()
        if profile:
            da.dash_profile_enable(True)
            da.dash_profile_read()
        ms = timed_steps(n_steps, det, s)
        barrier()
        main = None
        if profile:
            tot, cnt = da.dash_profile_read()
            da.dash_profile_enable(False)
            main = tot / max(cnt, 1)
        return max_over_ranks(ms, world, dev) / n_steps, main

    sampler = ClockSampler(local_rank) if rank == 0 else None
    warm = args.warmup if args.warmup is not None else 3
    for _ in range(warm):
        step()
    st = da.dash_attn_get_status(ws)
    if st != da.DASH_OK:
        raise da.DashError(st, "warm-up backward")
    if args.steps:
        steps = args.steps
    else:
        t0 = time.perf_counter()
        step()
        torch.cuda.synchronize()
        one = time.perf_counter() - t0
        steps = int(min(500, max(10, math.ceil(2.0 / max(one, 1e-4)))))

    ms_step, main_ms = timed(steps, profile=True)
    clocks = sampler.stop() if sampler else None
    st = da.dash_attn_get_status(ws)
    if st != da.DASH_OK:
        raise da.DashError(st, "timed backward")

    value = job_tflops(bwd_flops(w), world, ms_step)
    peak_tf, _, peak_kind = load_peaks()

    # the other variants of the same run: non-deterministic with the same schedule and
    # dealing (the speed reference: the same work with unordered adds, so the ratio is the
    # cost of the fixed order alone), and the FA3-baseline ascending order
    side = {}
    n_side = max(3, steps // 4)
    variants = [("nondet", 0, sched), ("ascending", DET, da.SCHED_ASCENDING),
                ("descending", DET, da.SCHED_DESCENDING)]
    if DET != 1:
        variants.append(("single_chain", 1, sched))
    for name, det, s in variants:
        if name == args.schedule:
            continue
        for _ in range(2):
            step(det, s)
        ms_s, _ = timed(n_side, det, s)
        side[name] = job_tflops(bwd_flops(w), world, ms_s)

    # The ordered reduction's waits, from the kernel's own wait-cycle trace in one extra,
    # untimed launch of the timed mode: cycles per 128 x 128 task (summed over CTAs,
    # divided by the tasks) spent waiting for a dQ block's turn and adding + handing it on.
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    trace = torch.zeros(sms * da.TRACE_SITES, dtype=torch.int64, device=dev)
    da.dash_debug_set_trace(trace)
    step()
    torch.cuda.synchronize()
    da.dash_debug_set_trace(None)
    st = da.dash_attn_get_status(ws)
    if st != da.DASH_OK:
        raise da.DashError(st, "traced backward")
    n_t = S // 128
    tasks = B * H * (n_t * (n_t + 1) // 2 if causal else n_t * n_t)
    tr = trace.view(sms, da.TRACE_SITES).sum(dim=0).double().cpu()
    dq_sem = {"turn_wait_cycles_per_task": float(tr[da.TRACE_DQ_TURN_WAIT]) / tasks,
              "add_and_handoff_cycles_per_task": float(tr[da.TRACE_DQ_ADD]) / tasks,
              "cycles_per_task": float(tr[da.TRACE_TOTAL]) / tasks,
              "source": "in-kernel clock64 wait trace (dash_debug_set_trace), one untimed launch"}

    # End to end through the public API with host buffers: every step uploads its inputs
    # from pinned host memory, runs the backward and downloads dQ/dK/dV. Two device buffer
    # sets and two copy streams let step i+1's upload and step i-1's download run while
    # step i computes (every step's copies stay inside the timed region).
    host = {nm: t.cpu().pin_memory() for nm, t in
            (("q", q), ("k", k), ("v", v), ("o", o), ("do", do), ("lse", lse))}
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    sets = [dict(q=q, k=k, v=v, o=o, do=do, lse=lse, dq=dq, dk=dk, dv=dv)]
    sets.append({nm: torch.empty_like(t) for nm, t in sets[0].items()})
    host_out = [{nm: torch.empty(q.shape, dtype=q.dtype).pin_memory() for nm in ("dq", "dk", "dv")}
                for _ in range(2)]
    d2h = sum(t.numel() * t.element_size() for t in host_out[0].values())
    n_e2e = max(3, steps // 4)
    comp = torch.cuda.current_stream(dev)
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def run_e2e(n):
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        h2d_done = [torch.cuda.Event() for _ in range(n)]
        comp_done = [torch.cuda.Event() for _ in range(n)]
        d2h_done = [torch.cuda.Event() for _ in range(n)]
        start.record(comp)
        up.wait_event(start)
        down.wait_event(start)

        def upload(i):
            st = sets[i % 2]
            with torch.cuda.stream(up):
                if i >= 2:
                    up.wait_event(comp_done[i - 2])          # that compute read this set
                for nm in ("q", "k", "v", "o", "do", "lse"):
                    st[nm].copy_(host[nm], non_blocking=True)
                h2d_done[i].record(up)

        upload(0)
        for i in range(n):
            if i + 1 < n:
                upload(i + 1)
            st = sets[i % 2]
            comp.wait_event(h2d_done[i])
            if i >= 2:
                comp.wait_event(d2h_done[i - 2])              # its gradients have been read
            da.dash_attn_bwd(st["q"], st["k"], st["v"], st["o"], st["do"], st["lse"], st["dq"],
                             st["dk"], st["dv"], ws, scale, mask, sched, DET)
            comp_done[i].record(comp)
            with torch.cuda.stream(down):
                down.wait_event(comp_done[i])
                for nm in ("dq", "dk", "dv"):
                    host_out[i % 2][nm].copy_(st[nm], non_blocking=True)
                d2h_done[i].record(down)
        comp.wait_event(d2h_done[n - 1])
        end.record(comp)
        return start, end

    run_e2e(2)
    barrier()
    e0, e1 = run_e2e(n_e2e)
    barrier()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / n_e2e, world, dev)

    if rank != 0:
        return
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w)
    achieved = bwd_flops(w) / (main_ms / 1e3) / 1e12 if main_ms else None
    launches_per_step = 3          # preprocess, main backward, dQ convert
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world, "steps": steps,
        "warmup": warm, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {**workload_config(args, w), "schedule_selected_by": selected_by,
                   "dq_chains": DET},
        "pct_of_peak": 100.0 * value / world / peak_tf,
        "nondet_tflops": side.get("nondet"),
        "det_vs_nondet": value / side["nondet"] if side.get("nondet") else None,
        "schedules": {args.schedule: value,
                      **{kk: vv for kk, vv in side.items() if kk not in ("nondet", "single_chain")}},
        "det_single_chain_tflops": side.get("single_chain", value if DET == 1 else None),
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak_tf,
                     "unit": "TFLOP/s", "frac": (achieved / peak_tf) if achieved else None,
                     "traffic": traffic_from_profile(w, args.schedule),
                     "kernel": "bwd main (compute + ordered dQ reduction)",
                     "peak_kind": f"{peak_kind} bf16 dense (burst)"},
        "cpu_baseline": cpu,
        "e2e": {"value": job_tflops(bwd_flops(w), world, e2e_ms), "unit": "TFLOPS",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "overlap": "two device buffer sets: step i+1's upload and step i-1's download "
                           "run on copy streams while step i computes"},
        "gpu_launches": launches_per_step * steps,
        "clocks": clocks,
        "dq_semaphore": dq_sem,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=0)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--schedule", default="auto",
                    choices=["auto", "ascending", "descending", "shift", "symmetric_shift"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--dq-chains", default="auto", choices=["auto", "1", "2"],
                    help="deterministic dQ order as 1 chain or 2 interleaved chains")
    args = ap.parse_args()
    w = WORKLOADS[args.workload]
    if args.schedule == "auto" and args.impl == "reference":
        args.schedule = BEST_DASH[w["mask"]]
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, w, rank)
        return
    if world > 1:
        import torch.distributed as dist

        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", rank=rank, world_size=world)
    try:
        run_gpu(args, w, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()


if __name__ == "__main__":
    main()
