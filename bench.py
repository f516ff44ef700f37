"""Benchmark of the sparse-MoE layer forward on B300 (one JSON line).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload large_prefill] [--no-decode] [--no-training] [--no-cpu-baseline]

A step is one forward of the whole layer (router -> top-k -> capacity
dispatch -> grouped expert FFNs (+ shared expert) -> combine -> statistics)
over one batch of the workload, through the public C ABI.  The timed region
runs K steps through the single moe_layer_fwd call (`value`,
`ms_per_step`), then the same K steps through the stage entry points
(moe_route, moe_dispatch, moe_expert_ffn, moe_combine) with a CUDA event
before each step and after every stage, on the launching stream: those give
each kernel's time (`components_ms`, the roofline's GEMM time), and a
step-start event that fires after the previous stage's end shows the GPU
waiting on the host (`host_gap`).  End to end (pinned host input in, output
back to the host) is `e2e`.  Inputs and weights are resident in HBM.  The headline workload is the
E=64 top-2 bf16 prefill layer (T=16384, d=4096, SwiGLU h=14336, capacity
factor 1.25, Zipf(1.1) logit bias); its weights (22.5 GB) and activations are
far larger than the 126 MB L2, so no flush is needed between steps.

Multi-GPU: the layer does not shard in this build; with torchrun every rank
runs an independent replica ("replicas only"), value = all ranks' tokens /
the slowest rank's time.

--impl reference times the fp64 CPU oracle (the checker) on the host cores
on a bounded sample of the same workload.
"""

from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s at E=64 top-2 bf16; grouped-GEMM % peak; decode % HBM BW"
WEIGHTS = ("Wr", "W1", "W3", "W2", "b1", "b2", "Ws1", "Ws3", "Ws2", "bs1", "bs2", "expert_bias")
# DRAM bytes (read + write) of one moe_expert_ffn call -- its GEMM-1 and
# GEMM-2 launches together -- at the large-prefill shapes, from an ncu
# capture of the four-expert slice scaled to the 64 experts by the kept
# rows, keyed by the sha256 of the kernel source it was taken on (the figure
# is reported only while that source is unchanged)
GEMM_TRAFFIC = {
    # 1.5740 GB (GEMM-1 1.0415 GB + GEMM-2 0.5325 GB) x 32607 / 2048 kept rows
    "6a2928a03c1e43faf19c3305852226cfcad480c7488ba6149452f6feffc6befa": 25.059e9,
}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return dict(hbm_gbs=d["hbm_gbs"], bf16=d["bf16_tflops"], bf16_sus=d["bf16_tflops_sustained"],
                    source="measured")
    except Exception:
        return dict(hbm_gbs=6400.0, bf16=1800.0, bf16_sus=1400.0, source="fallback")


class ClockSampler:
    """SM clock / throttle-reason samples while running, each stamped with
    the host time, so a summary can cover one timed region.  NVML is read
    every 5 ms from a thread (read-only queries); without NVML, nvidia-smi
    every 50 ms."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.rows = []
        self.proc = None
        self.stop = threading.Event()
        self.thread = None
        self.source = None

    def __enter__(self):
        try:
            self.thread = threading.Thread(target=self._nvml, args=(self._nvml_open(),), daemon=True)
            self.thread.start()
            self.source = "nvml"
            return self
        except Exception as e:
            self.nvml_error = repr(e)[:120]
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            self.source = "nvidia-smi"
        except OSError:
            self.proc = None
        return self

    def _nvml_open(self):
        """The driver's NVML library through ctypes (read-only queries):
        (lib, device handle, max SM clock, the clock-event reasons call)."""
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit_v2")
        h = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.index), ctypes.byref(h)) != 0:
            raise RuntimeError("nvmlDeviceGetHandleByIndex_v2")
        mx = ctypes.c_uint()
        if lib.nvmlDeviceGetMaxClockInfo(h, self.NVML_CLOCK_SM, ctypes.byref(mx)) != 0:
            raise RuntimeError("nvmlDeviceGetMaxClockInfo")
        try:
            reasons = lib.nvmlDeviceGetCurrentClocksEventReasons
        except AttributeError:
            reasons = lib.nvmlDeviceGetCurrentClocksThrottleReasons
        return lib, h, mx.value, reasons

    # NVML_CLOCK_SM, and the clock-event reason bits in the order of FIELDS[3:]:
    # hardware slowdown, hardware thermal, software thermal, software power cap
    NVML_CLOCK_SM = 1
    NVML_REASONS = (0x8, 0x40, 0x20, 0x4)

    def _nvml(self, opened):
        lib, h, mx, get_reasons = opened
        sm, mw, bits = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        while not self.stop.is_set():
            if (lib.nvmlDeviceGetClockInfo(h, self.NVML_CLOCK_SM, ctypes.byref(sm)) != 0 or
                    lib.nvmlDeviceGetPowerUsage(h, ctypes.byref(mw)) != 0 or get_reasons(h, ctypes.byref(bits)) != 0):
                break
            act = ["Active" if bits.value & b else "Not Active" for b in self.NVML_REASONS]
            self.rows.append((time.time(), [str(sm.value), str(mx), f"{mw.value / 1000.0:.1f}", *act]))
            self.stop.wait(0.005)
        lib.nvmlShutdown()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == 7:
                self.rows.append((time.time(), parts))

    def __exit__(self, *a):
        self.stop.set()
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        elif self.thread:
            self.thread.join(timeout=5)

    def summary(self, t_from=None, t_to=None):
        """Median SM clock, max clock and the throttle reasons seen, over the
        samples taken between host times t_from and t_to (all if None)."""
        rows = [r for ts, r in self.rows if (t_from is None or ts >= t_from) and (t_to is None or ts <= t_to)]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({names[i] for r in rows for i in range(4) if r[3 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "source": self.source}


def percentiles(ms):
    """Median and the p10-p90 range of per-step times (ms)."""
    import numpy as np
    a = np.asarray(ms, dtype=np.float64)
    return {"median": float(np.median(a)), "p10": float(np.percentile(a, 10)), "p90": float(np.percentile(a, 90))}


def gemm_bytes(r):
    """Algorithmic DRAM bytes of one moe_expert_ffn call: the touched expert
    weights once, and per kept row its input row read, its hidden row written
    by GEMM-1 and read by GEMM-2, its output row written (bf16)."""
    wl = r["wl"]
    return r["touched_weight_bytes"] + r["stats"]["kept_slots"] * 2 * (2 * wl.d + 2 * wl.h)


def gemm_traffic():
    import hashlib
    src = os.path.join(ROOT, "sparse_mixture_experts_sum_b300", "csrc", "gemm_tc.cu")
    try:
        h = hashlib.sha256(open(src, "rb").read()).hexdigest()
    except OSError:
        return None
    return GEMM_TRAFFIC.get(h)


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(ms, world, device):
    """The job's time for a region every rank times between two barriers:
    the slowest rank's (replicas do no collective in their own steps)."""
    if world <= 1:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank, world, ms_max):
    """Whole-job rate: the units all ranks processed over the slowest
    rank's time (units per second)."""
    return units_per_rank * world / (ms_max * 1e-3)


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------


def expert_ffn_flops(wl, kept):
    return 2.0 * kept * wl.d * wl.h * (3 if wl.act == "swiglu" else 2)


def shared_flops(wl):
    return 2.0 * wl.T * wl.d * wl.h * (3 if wl.act == "swiglu" else 2) if wl.has_shared else 0.0


def run_gpu(args, wl_name, world, rank, local, main=True):
    import torch
    import moe_synth as S
    import sparse_mixture_experts_sum_b300 as M

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wl = S.WORKLOADS[wl_name]
    t = S.make_inputs(wl, dev)
    cfg = M.config_of(wl)
    weights = {n: t.get(n) for n in WEIGHTS}
    x, noise = t["x"], t.get("noise")
    sdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    y = torch.empty(wl.T, wl.d, dtype=sdt, device=dev)
    st = M.moe.stats_buffer(dev)
    saved = M.moe.alloc_saved(cfg, dev)
    ws = M.moe.workspace(cfg, training=True, device=dev)
    stream = torch.cuda.current_stream(dev)

    Hs = torch.empty(wl.T, wl.h, dtype=sdt, device=dev) if wl.has_shared else None
    sv = saved

    # one step = the layer's C-ABI stages in the order moe_layer_fwd runs them
    stages = [
        ("route", lambda: M.moe_route(cfg, x, weights["Wr"], weights.get("expert_bias"), noise, sv["idx"], sv["w"],
                                      sv["counts"], ws)),
        ("dispatch", lambda: M.moe_dispatch(cfg, sv["idx"], x, sv["kept"], sv["offsets"], sv["pos"], sv["Xp"], st,
                                            ws)),
        ("expert_ffn", lambda: M.moe_expert_ffn(cfg, sv["Xp"], sv["offsets"], weights["W1"], weights.get("W3"),
                                                weights.get("b1"), weights["W2"], weights.get("b2"), sv["H"],
                                                sv["Yp"], ws)),
    ]
    if wl.has_shared:
        # routed experts and the shared expert in the same two launches
        stages[-1] = ("expert_ffn", lambda: M.moe.moe_expert_ffn_shared(cfg, sv["Xp"], sv["offsets"], weights,
                                                                         sv["H"], sv["Yp"], x, Hs, sv["Sx"], ws))
    stages.append(("combine", lambda: M.moe_combine(cfg, sv["Yp"], sv["pos"], sv["w"], sv.get("Sx"), y)))

    def step():
        for _, fn in stages:
            fn()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    assert M.moe_check_error(ws) == 0, "a kernel gave up a bounded wait"
    stats = M.moe.read_stats(st)
    kept = stats["kept_slots"]

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)

    steps = args.steps
    sampler = ClockSampler(local)
    with sampler:
        # --- timed region 1: K forwards through the single moe_layer_fwd call
        # (the value), an event after each step for the per-step spread ---
        barrier()
        h0 = time.time()
        fe = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
        fe[0].record(stream)
        for i in range(steps):
            M.moe_layer_fwd(cfg, weights, x, noise, y, saved, st, ws)
            fe[i + 1].record(stream)
        barrier()
        h1 = time.time()
        # --- timed region 2: the same steps through the stage entry points, an
        # event before each step and after every stage (the per-kernel times;
        # a step-start event that fires late marks the GPU waiting on the host) ---
        pre = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(stages))] for _ in range(steps)]
        e0 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(steps):
            pre[i].record(stream)
            for j, (_, fn) in enumerate(stages):
                fn()
                evs[i][j].record(stream)
        barrier()
        h2 = time.time()
    # the clocks of each region side by side: the stage path's kernel times
    # (the GEMM figure of the roofline) come from region 2
    clocks = sampler.summary(h0, h1)
    stage_clocks = sampler.summary(h1, h2)
    ms_total = fe[0].elapsed_time(fe[-1])
    step_ms = [fe[i].elapsed_time(fe[i + 1]) for i in range(steps)]
    stage_ms_total = e0.elapsed_time(evs[-1][-1])
    stage_step_ms = [(pre[i].elapsed_time(evs[i][-1])) for i in range(steps)]
    comp = {name: 0.0 for name, _ in stages}
    comp["host_gap"] = 0.0
    prev = e0
    for i in range(steps):
        comp["host_gap"] += prev.elapsed_time(pre[i]) / steps
        prev = pre[i]
        for j, (name, _) in enumerate(stages):
            comp[name] += prev.elapsed_time(evs[i][j]) / steps
            prev = evs[i][j]
    ms_total = max_over_ranks(ms_total, world, dev)
    ms_step = ms_total / steps
    layer_fwd_ms = ms_step
    assert M.moe_check_error(ws) == 0, "a kernel gave up a bounded wait"

    peaks = load_peaks()
    # router: one launch (fp32, or the bf16 logits GEMM with its top-k
    # epilogue up to 64 experts), else the logits GEMM and a top-k kernel;
    # dispatch: one fused kernel + the permute for up to 4096 slots and 128
    # experts, else histogram, scan, assignment + the permute
    small = wl.T * wl.k <= 4096 and wl.E <= 128
    layer_launches = 1 + (2 if wl.dtype == "bf16" and wl.E > 64 else 1) + (2 if small else 4) + 2 + 1
    out = {
        "ms_per_step": ms_step,
        "step_ms": percentiles(step_ms),
        "layer_fwd_ms": layer_fwd_ms,
        "stage_path_ms": stage_ms_total / steps,
        "stage_step_ms": percentiles(stage_step_ms),
        "stage_clocks": stage_clocks,
        # our kernels per step of both regions: moe_layer_fwd = zeroing,
        # router and dispatch (above)
        # (the entropy mean rides in the capacity scan), 2 grouped GEMMs,
        # combine; the stage path = the same plus moe_expert_ffn's zeroing of
        # the error word
        "layer_launches": layer_launches,
        "launches_per_step": 2 * layer_launches + 1,
        "tokens_per_s": job_throughput(wl.T, world, ms_step),
        "stats": stats,
        "components_ms": comp,
        "clocks": clocks,
        "wl": wl,
    }
    gemm_flops = expert_ffn_flops(wl, kept)
    gemm_ms = comp["expert_ffn"]
    out["gemm"] = {"flops": gemm_flops, "ms": gemm_ms, "tflops": gemm_flops / (gemm_ms * 1e-3) / 1e12}
    # touched expert weights (bytes): experts with >= 1 kept row, plus the shared expert
    kept_per_e = saved["kept"].cpu()
    n_touched = int((kept_per_e > 0).sum().item())
    per_expert_bytes = wl.d * wl.h * (3 if wl.act == "swiglu" else 2) * 2
    out["touched_weight_bytes"] = (n_touched + (1 if wl.has_shared else 0)) * per_expert_bytes
    out["n_touched"] = n_touched
    out["weight_bytes"] = wl.E * per_expert_bytes

    # --- e2e: pinned host input -> device, forward, device -> pinned host output ---
    # Every step copies its input up and its output down inside the timed
    # region; the copies run on their own stream with two device buffers,
    # so step i+1's upload and step i's download overlap step i+1's / i's
    # neighbours' compute (events order each buffer's reuse).
    xh = x.cpu().pin_memory()
    nh = noise.cpu().pin_memory() if noise is not None else None
    yh = [torch.empty(wl.T, wl.d, dtype=sdt).pin_memory() for _ in range(2)]
    xd = [torch.empty_like(x) for _ in range(2)]
    nd = [torch.empty_like(noise) if noise is not None else None for _ in range(2)]
    yd = [torch.empty_like(y) for _ in range(2)]
    cstream = torch.cuda.Stream(dev)
    n_e2e = args.steps

    def e2e_run(n):
        h2d_done = [torch.cuda.Event() for _ in range(n)]
        fwd_done = [torch.cuda.Event() for _ in range(n)]

        def upload(i):
            b = i % 2
            with torch.cuda.stream(cstream):
                if i >= 2:
                    cstream.wait_event(fwd_done[i - 2])  # buffer b was step i-2's input
                xd[b].copy_(xh, non_blocking=True)
                if nh is not None:
                    nd[b].copy_(nh, non_blocking=True)
                h2d_done[i].record(cstream)

        upload(0)
        for i in range(n):
            b = i % 2
            if i + 1 < n:
                upload(i + 1)
            stream.wait_event(h2d_done[i])  # also orders after step i-2's download (same stream, earlier)
            M.moe_layer_fwd(cfg, weights, xd[b], nd[b], yd[b], saved, st, ws)
            fwd_done[i].record(stream)
            with torch.cuda.stream(cstream):
                cstream.wait_event(fwd_done[i])
                yh[b].copy_(yd[b], non_blocking=True)

    e2e_run(2)
    torch.cuda.synchronize(dev)
    barrier()
    e2e0, e2e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e0.record(stream)
    cstream.wait_event(e2e0)
    e2e_run(n_e2e)
    e2e1.record(cstream)
    barrier()
    e2e_ms = e2e0.elapsed_time(e2e1) / n_e2e
    e2e_ms = max_over_ranks(e2e_ms, world, dev)
    yh = yh[0]
    h2d = xh.numel() * xh.element_size() + (nh.numel() * nh.element_size() if nh is not None else 0)
    out["e2e"] = {"value": job_throughput(wl.T, world, e2e_ms), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                  "d2h_bytes_per_step": yh.numel() * yh.element_size()}
    out["peaks"] = peaks
    out["tensors"] = dict(t=t, saved=saved)
    return out


def run_training(args, world, rank, local):
    """Training-shaped step (forward with saved activations + backward) of
    the training workload through moe_layer_fwd / moe_layer_bwd, with an
    event between the two halves.  Returns timings and algorithmic FLOPs."""
    import torch
    import moe_synth as S
    import sparse_mixture_experts_sum_b300 as M

    dev = torch.device("cuda", local)
    wl = S.WORKLOADS["training"]
    t = S.make_inputs(wl, dev)
    cfg = M.config_of(wl)
    weights = {n: t.get(n) for n in WEIGHTS}
    x, noise, dY = t["x"], t.get("noise"), t["dY"]
    y = torch.empty(wl.T, wl.d, dtype=torch.bfloat16, device=dev)
    st = M.moe.stats_buffer(dev)
    saved = M.moe.alloc_saved(cfg, dev, backward=True)
    grads = M.moe.alloc_grads(cfg, dev)
    ws_f = M.moe.workspace(cfg, 1, device=dev)
    ws_b = M.moe.workspace(cfg, 2, device=dev)
    stream = torch.cuda.current_stream(dev)

    def fwd():
        M.moe_layer_fwd(cfg, weights, x, noise, y, saved, st, ws_f)

    def bwd():
        M.moe_layer_bwd(cfg, weights, x, saved, dY, grads, ws_b)

    for _ in range(max(3, args.warmup)):
        fwd()
        bwd()
    torch.cuda.synchronize(dev)
    assert M.moe_check_error(ws_f) == 0 and M.moe_check_error(ws_b) == 0
    stats = M.moe.read_stats(st)
    steps = max(3, min(args.steps, 10))
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    sampler = ClockSampler(local)
    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)

    with sampler:
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(steps):
            fwd()
            ev[i][0].record(stream)
            bwd()
            ev[i][1].record(stream)
        barrier()
    assert M.moe_check_error(ws_b) == 0
    f_ms = b_ms = 0.0
    prev = e0
    for a, b in ev:
        f_ms += prev.elapsed_time(a) / steps
        b_ms += a.elapsed_time(b) / steps
        prev = b
    # the job's step is the slowest rank's; the halves are reported as this rank measured them
    step_ms = max_over_ranks(f_ms + b_ms, world, dev)
    kept = stats["kept_slots"]
    per = 2.0 * wl.d * wl.h * (3 if wl.act == "swiglu" else 2)
    fwd_flops = per * (kept + (wl.T if wl.has_shared else 0)) + 2.0 * wl.T * wl.d * wl.E
    bwd_flops = 2.0 * per * (kept + (wl.T if wl.has_shared else 0)) + 4.0 * wl.T * wl.d * wl.E
    return {"workload": f"training: T={wl.T} d={wl.d} h={wl.h} E={wl.E}+1 shared top-{wl.k} {wl.act} "
                        f"cf={wl.capacity_factor} gumbel bf16, fp32 grads",
            "steps": steps, "ms_per_step": step_ms, "fwd_ms": f_ms, "bwd_ms": b_ms,
            "tokens_per_s": job_throughput(wl.T, world, step_ms),
            "tflops": (fwd_flops + bwd_flops) * world / (step_ms * 1e-3) / 1e12,
            "bwd_tflops": bwd_flops / (b_ms * 1e-3) / 1e12, "kept_slots": kept,
            "clocks": sampler.summary()}


def _cpu_model():
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


# How the oracle is timed per workload.  The forward runs on the C++ fp64
# oracle (oracle/moe_oracle.cpp: plain single-threaded loops, inputs read as
# the stored bf16/fp32 bits): the whole layer where that takes seconds;
# else the router, top-k, capacity and dispatch of the whole batch plus the
# expert rows of the two busiest experts (at most the given rows each),
# extrapolated per token by the measured cost of an expert row.  The
# training step runs the same routing plus the C++ oracle's forward and
# backward of the sampled rows.
CPU_PLAN = {"tiny_fp32": ("whole", None), "small_prefill": ("experts", 256), "decode": ("experts", None),
            "large_prefill": ("experts", 32), "training": ("train", 4)}


def cpu_baseline(wl_name, gpu_tensors=None, mode=None, max_rows=None, tokens=None):
    """The oracle as it stands, on ONE host core, on the workload's inputs
    (from the GPU run when given, else drawn on the host at T <= 2048 for
    the expert-sampling modes):
      whole   -- the C++ oracle's layer forward over the whole batch;
      experts -- the C++ oracle's router, top-k, capacity and dispatch of the
                 whole batch, then its expert FFN on the kept rows of the two
                 busiest experts (at most max_rows each); tokens/s
                 extrapolated: routing share + expert rows per token (kept
                 slots / T, + 1 with a shared expert) x cost per row;
      train   -- the same routing, then the C++ oracle's forward and
                 backward of the sampled rows (expert_ffn_backward),
                 extrapolated alike.
    tokens: route only the batch's first `tokens` tokens (a bounded sample
    per step for the reference arm); the rates are per token either way."""
    import numpy as np
    import torch
    import moe_synth as S

    wl = S.WORKLOADS[wl_name]
    plan, rows_cap = CPU_PLAN.get(wl_name, ("experts", None))
    mode = mode or plan
    max_rows = max_rows if max_rows is not None else rows_cap
    if gpu_tensors is not None:
        t, T = gpu_tensors, wl.T
    elif mode == "whole":
        T = wl.T
        t = S.make_inputs(wl, "cpu")
    else:
        # a 2048-token batch on the host; expert weights are drawn below for
        # the two experts that are timed only
        T = min(wl.T, 2048)
        t = S.make_inputs(wl.replace(T=T), "cpu", parts=["x", "Wr", "expert_bias", "noise", "dY"])
    if tokens is not None and tokens < T:
        T = tokens
        t = dict(t, x=t["x"][:T], **({"noise": t["noise"][:T]} if t.get("noise") is not None else {}),
                 **({"dY": t["dY"][:T]} if t.get("dY") is not None else {}))
    cfg = dict(T=T, d=wl.d, h=wl.h, E=wl.E, k=wl.k, act=wl.act,
               capacity_factor=float(np.float32(wl.capacity_factor)), min_capacity=wl.min_capacity,
               lam=float(np.float32(wl.lam)), has_shared=wl.has_shared)
    host = os.cpu_count() or 1
    cores = 1
    common = {"unit": "tokens/s", "cores": cores, "kind": "oracle", "host_cores": host, "cpu_model": _cpu_model(),
              "threads": f"{cores} core{'s' if cores != 1 else ''} of {host}"}
    cpu = lambda a: None if a is None else a.detach().to("cpu")
    if mode == "whole":
        from oracle import cpp
        hw = {n: cpu(v) for n, v in t.items()}
        t0 = time.perf_counter()
        cpp.layer_forward(cfg, hw, hw["x"], hw.get("expert_bias"), hw.get("noise"))
        dt = time.perf_counter() - t0
        return dict(common, value=T / dt, seconds=dt, extrapolated=False, impl="C++ fp64 oracle, single thread",
                    sample=f"C++ fp64 oracle layer forward of the whole batch ({T} tokens) in {dt:.2f} s")
    x, Wr = cpu(t["x"]), cpu(t["Wr"])
    bias, noise = cpu(t.get("expert_bias")), cpu(t.get("noise"))
    from oracle import cpp
    t0 = time.perf_counter()
    l = cpp.router_logits(x, Wr, bias, noise)
    idx, w_, _ = cpp.top_k(l, wl.k)
    cpp.usage_counts(idx, wl.E)
    C = cpp.capacity(T, wl.k, wl.E, cfg["capacity_factor"], wl.min_capacity)
    rank, kept_e = cpp.assign_capacity(idx, wl.E, C)
    _, pos = cpp.dispatch_positions(idx, rank, kept_e)
    t_route = time.perf_counter() - t0
    impl = "C++ fp64 oracle, single thread"
    experts = [int(e) for e in np.argsort(-kept_e, kind="stable")[:2]]
    if "W1" not in t:
        t = dict(t)
        for name, (rows_, cols, fan) in dict(W1=(wl.h, wl.d, wl.d), W3=(wl.h, wl.d, wl.d),
                                             W2=(wl.d, wl.h, wl.h)).items():
            if name == "W3" and wl.act != "swiglu":
                continue
            t[name] = {e: S.tensor("normal", wl.seed, S.TID[name], (rows_, cols), wl.dtype, wl.std(fan), "cpu",
                                   start=e * rows_ * cols) for e in experts}
    slots, t_ffn = 0, 0.0
    for e in experts:
        rows, sl = np.nonzero((idx == e) & (pos >= 0))
        if max_rows is not None:
            rows, sl = rows[:max_rows], sl[:max_rows]
        if rows.size == 0:
            continue
        v = x[torch.as_tensor(rows)]
        p = {n: cpu(t[n][e]) if t.get(n) is not None else None for n in ("W1", "W3", "W2", "b1", "b2")}
        if wl.act != "swiglu":
            p["W3"] = None
        if mode == "train":
            dy = cpu(t["dY"])[torch.as_tensor(rows)].double().numpy()
            t1 = time.perf_counter()
            cpp.expert_ffn_backward(v, w_[rows, sl][:, None] * dy, wl.act, p["W1"], p["W2"], W3=p["W3"], b1=p["b1"],
                                    b2=p["b2"])
        else:
            t1 = time.perf_counter()
            cpp.expert_ffn(v, wl.act, p["W1"], p["W2"], W3=p["W3"], b1=p["b1"], b2=p["b2"])
        t_ffn += time.perf_counter() - t1
        slots += rows.size
    per_row = t_ffn / max(slots, 1)
    rows_per_token = float(kept_e.sum()) / T + (1 if wl.has_shared else 0)
    per_token = t_route / T + per_row * rows_per_token
    what = "forward and backward of" if mode == "train" else "expert FFN of"
    return dict(common, value=1.0 / per_token, seconds=t_route + t_ffn, extrapolated=True, impl=impl,
                sample=f"{impl}: router+top-k+capacity+dispatch of all {T} tokens ({t_route:.2f} s), "
                       f"{what} {slots} kept rows of experts {experts} ({t_ffn:.2f} s); whole-layer tokens/s "
                       f"extrapolated per token at {rows_per_token:.3f} expert rows/token")


ONE_THREAD = {v: "1" for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS")}


def cpu_baselines(local):
    """cpu_baseline of every workload of the plan, each in a child process
    whose BLAS is held to one thread by the thread-count variables (set
    before numpy loads); the child draws its inputs on the GPU."""
    out = {}
    for name in ("tiny_fp32", "small_prefill", "decode", "large_prefill", "training"):
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-baseline-child", name,
                            "--local-rank", str(local)], env=dict(os.environ, **ONE_THREAD),
                           capture_output=True, text=True, timeout=900)
        lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
        out[name] = json.loads(lines[-1]) if r.returncode == 0 and lines else {
            "unavailable": (r.stderr.strip().splitlines() or ["no output"])[-1]}
    return out


def layer_section(r, peaks, peak):
    """Throughput and roofline of one workload's layer forward (run_gpu's
    result): tokens/s, the per-step spread, algorithmic FLOPs (expert rows,
    the shared expert's T rows, the router's 2*T*d*E) and bytes (the touched
    weights once, x read, y written), and the roofline fraction
    max(FLOPs / tensor peak, bytes / HBM) / measured step time."""
    wl = r["wl"]
    es = 2 if wl.dtype == "bf16" else 4
    flops = r["gemm"]["flops"] + shared_flops(wl) + 2.0 * wl.T * wl.d * wl.E
    bytes_ = r["touched_weight_bytes"] * es // 2 + 2 * wl.T * wl.d * es
    t_tensor, t_hbm = flops / (peak * 1e12), bytes_ / (peaks["hbm_gbs"] * 1e9)
    ms = r["ms_per_step"]
    bias = "" if wl.zipf_s is None else f" zipf_bias={'ln pmf ' if wl.zipf_log else ''}{wl.zipf_s}"
    out = {"workload": f"{wl.name}: T={wl.T} d={wl.d} h={wl.h} E={wl.E}{'+1 shared' if wl.has_shared else ''} "
                       f"top-{wl.k} {wl.act} cf={wl.capacity_factor}{bias} {wl.dtype}",
           "ms_per_step": ms, "step_ms": r["step_ms"], "tokens_per_s": r["tokens_per_s"],
           "tflops": flops / (ms * 1e-3) / 1e12, "algorithmic_flops": flops, "algorithmic_bytes": bytes_,
           "bound": "tensor" if t_tensor >= t_hbm else "hbm",
           "roofline_ms": max(t_tensor, t_hbm) * 1e3, "roofline_frac": max(t_tensor, t_hbm) / (ms * 1e-3),
           "kept_slots": r["stats"]["kept_slots"], "drop_rate": r["stats"]["drop_rate"],
           "balance_stat": r["stats"]["balance_stat"], "e2e": r["e2e"],
           "components_ms": {k: round(v, 4) for k, v in r["components_ms"].items()}, "clocks": r["clocks"]}
    if wl.dtype != "bf16":
        # fp32 runs on the CUDA cores, not the bf16 tensor path; at this size
        # the layer is launch-latency bound and the fraction is only a figure
        out["bound"] = "latency"
        out["launches_per_step"] = r["layer_launches"]
        out["us_per_launch"] = ms * 1e3 / out["launches_per_step"]
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="large_prefill")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-training", action="store_true")
    ap.add_argument("--no-fine-grained", action="store_true")
    ap.add_argument("--no-small-prefill", action="store_true")
    ap.add_argument("--no-tiny-fp32", action="store_true")
    ap.add_argument("--no-large-prefill-3z", action="store_true")
    ap.add_argument("--cpu-baseline-child", default=None, help=argparse.SUPPRESS)
    ap.add_argument("--local-rank", type=int, default=0, help=argparse.SUPPRESS)
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    world, rank, local = dist_setup()

    if args.cpu_baseline_child:
        # one workload's oracle timing (run by cpu_baselines with one BLAS thread)
        import torch
        import moe_synth as S
        dev = torch.device("cuda", args.local_rank)
        torch.cuda.set_device(dev)
        t = S.make_inputs(S.WORKLOADS[args.cpu_baseline_child], dev)
        print(json.dumps(cpu_baseline(args.cpu_baseline_child, t)))
        return 0

    if args.impl == "reference":
        if rank != 0:
            return 0
        # the oracle on one host core: the BLAS reads these before numpy loads
        os.environ.update(ONE_THREAD)
        import torch
        dev_ok = torch.cuda.is_available()
        t0 = time.time()
        vals = []
        cb = None
        gt = None
        if dev_ok:
            import moe_synth as S
            torch.cuda.set_device(local)
            gt = S.make_inputs(S.WORKLOADS[args.workload], torch.device("cuda", local))
        for i in range(args.warmup + args.steps):
            # each step a bounded sample on one core: the routing of the
            # batch's first 512 tokens plus up to 8 rows (the training
            # step's forward and backward: 1 row, ~0.8 s) of each of the two
            # busiest experts among them
            train = args.workload == "training"
            cb = cpu_baseline(args.workload, gt, mode="train" if train else None, max_rows=1 if train else 8,
                              tokens=512)
            if i >= args.warmup:
                vals.append(cb["value"])
        v = statistics.median(vals)
        cb["value"] = v
        print(json.dumps({"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": args.gpus,
                          "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
                          "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                          "config": {"workload": args.workload}, "cpu_baseline": cb,
                          "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                                  "d2h_bytes_per_step": 0},
                          "wall_s": time.time() - t0}))
        return 0

    import torch
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    r = run_gpu(args, args.workload, world, rank, local)
    wl = r["wl"]
    peaks = r["peaks"]
    gemm = r["gemm"]
    peak = peaks["bf16_sus"]
    line = {
        "metric": METRIC,
        "value": r["tokens_per_s"],
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": r["ms_per_step"],
        "stage_path_ms_per_step": r["stage_path_ms"],
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": f"{wl.name}: T={wl.T} d={wl.d} h={wl.h} E={wl.E} top-{wl.k} {wl.act} "
                               f"cf={wl.capacity_factor} zipf_bias={wl.zipf_s} {wl.dtype}",
                   "global_batch_tokens": wl.T * world, "parallelism": "replicas" if world > 1 else "single",
                   "l2": f"inputs larger than L2 (expert weights {r['weight_bytes'] / 1e9:.2f} GB, "
                         f"x {wl.T * wl.d * 2 / 1e6:.0f} MB vs 126 MB L2), no flush"},
        "roofline": {"bound": "tensor", "achieved": gemm["tflops"], "peak": peak, "unit": "TFLOP/s",
                     "frac": gemm["tflops"] / peak, "traffic": gemm_traffic(),
                     "traffic_per": "one moe_expert_ffn call (its GEMM-1 and GEMM-2 launches), DRAM bytes",
                     "algorithmic_bytes": gemm_bytes(r),
                     "kernel": "grouped_gemm_tc_kernel (GEMM-1 SwiGLU + GEMM-2, one moe_expert_ffn call)",
                     "peak_kind": f"bf16 sustained ({peaks['source']})",
                     "frac_of_burst": gemm["tflops"] / peaks["bf16"],
                     "gemm_ms": gemm["ms"], "gemm_ms_from": "stage-path region (clocks: stage_clocks)"},
        "step_ms": r["step_ms"],
        "clocks": r["clocks"],
        "stage_clocks": r["stage_clocks"],
        "stage_step_ms": r["stage_step_ms"],
        "e2e": r["e2e"],
        # our kernels in the value's timed region (K moe_layer_fwd calls); the
        # stage-path region that times the kernels one by one launches
        # gpu_launches_stage_path more
        "gpu_launches": r["layer_launches"] * args.steps,
        "gpu_launches_stage_path": (r["launches_per_step"] - r["layer_launches"]) * args.steps,
        "components_ms": {k: round(v, 4) for k, v in r["components_ms"].items()},
        "layer_stats": {k: r["stats"][k] for k in ("kept_slots", "dropped_slots", "capacity", "drop_rate",
                                                    "balance_stat")},
    }
    # whole-layer roofline: max(flops / tensor peak, bytes / HBM) vs measured step time
    flops = gemm["flops"] + 2.0 * wl.T * wl.d * wl.E
    bytes_ = r["touched_weight_bytes"] + 2 * wl.T * wl.d * 2
    t_roof = max(flops / (peak * 1e12), bytes_ / (peaks["hbm_gbs"] * 1e9))
    line["layer_roofline_frac"] = t_roof / (r["ms_per_step"] * 1e-3)

    del r["tensors"]
    # the small prefill and the tiny fp32 layer: throughput and roofline
    for name, n_min in (("small_prefill", 100), ("tiny_fp32", 200), ("large_prefill_3z", 40)):
        if getattr(args, "no_" + name):
            continue
        sargs = argparse.Namespace(**vars(args))
        sargs.steps = max(args.steps, n_min)  # >= 0.25 s timed for the clock sampler (small prefill)
        sr = run_gpu(sargs, name, world, rank, local)
        line[name] = layer_section(sr, peaks, peak)
        del sr["tensors"]
    if not args.no_decode:
        dargs = argparse.Namespace(**vars(args))
        dargs.steps = max(args.steps, 100)  # >= 0.25 s timed, so the clock sampler sees it
        d = run_gpu(dargs, "decode", world, rank, local)
        dwl = d["wl"]
        ffn_ms = d["components_ms"]["expert_ffn"]
        gbs = d["touched_weight_bytes"] / (ffn_ms * 1e-3) / 1e9
        line["decode"] = {"workload": f"decode: T={dwl.T} d={dwl.d} h={dwl.h} E={dwl.E}+1 shared top-{dwl.k}",
                          "ms_per_step": d["ms_per_step"], "tokens_per_s": d["tokens_per_s"],
                          "touched_experts": d["n_touched"] + 1,
                          "touched_weight_gb": d["touched_weight_bytes"] / 1e9,
                          "expert_ffn_ms": ffn_ms, "hbm_gbs": gbs, "hbm_frac": gbs / peaks["hbm_gbs"],
                          "layer_hbm_frac": d["touched_weight_bytes"] / (d["ms_per_step"] * 1e-3) / 1e9
                          / peaks["hbm_gbs"],
                          "components_ms": {k: round(v, 4) for k, v in d["components_ms"].items()},
                          "clocks": d["clocks"]}
        del d["tensors"]
    if not args.no_fine_grained:
        # fine-grained routing: E=384 top-6 + shared, ~128 rows per expert;
        # its expert weights (9.7 GB) take longer to stream than its FLOPs
        # take on the tensor cores, so both fractions are reported
        fargs = argparse.Namespace(**vars(args))
        fargs.steps = max(args.steps, 40)
        f = run_gpu(fargs, "fine_grained", world, rank, local)
        fwl = f["wl"]
        ffn_ms = f["components_ms"]["expert_ffn"]
        fflops = expert_ffn_flops(fwl, f["stats"]["kept_slots"]) + shared_flops(fwl)
        # algorithmic bytes of the two grouped GEMMs: the touched weights once,
        # plus per row (kept slots and the shared expert's T rows) its input
        # row read, its hidden row written and read back, its output row written
        rows = f["stats"]["kept_slots"] + (fwl.T if fwl.has_shared else 0)
        act_bytes = rows * 2 * (2 * fwl.d + 2 * fwl.h)
        fbytes = f["touched_weight_bytes"] + act_bytes
        gbs = fbytes / (ffn_ms * 1e-3) / 1e9
        t_roof = max(fflops / (peak * 1e12), fbytes / (peaks["hbm_gbs"] * 1e9))
        line["fine_grained"] = {
            "workload": f"fine_grained: T={fwl.T} d={fwl.d} h={fwl.h} E={fwl.E}+1 shared top-{fwl.k} "
                        f"cf={fwl.capacity_factor} {fwl.dtype}",
            "ms_per_step": f["ms_per_step"], "tokens_per_s": f["tokens_per_s"], "e2e": f["e2e"],
            "kept_slots": f["stats"]["kept_slots"], "touched_experts": f["n_touched"] + 1,
            "touched_weight_gb": f["touched_weight_bytes"] / 1e9, "activation_gb": act_bytes / 1e9,
            "expert_ffn_ms": ffn_ms,
            "gemm_tflops": fflops / (ffn_ms * 1e-3) / 1e12,
            "gemm_frac_of_sustained": fflops / (ffn_ms * 1e-3) / 1e12 / peak,
            "hbm_gbs": gbs, "hbm_frac": gbs / peaks["hbm_gbs"],
            "expert_ffn_roofline_frac": t_roof / (ffn_ms * 1e-3),
            "components_ms": {k: round(v, 4) for k, v in f["components_ms"].items()},
            "clocks": f["clocks"]}
        del f["tensors"]
    if not args.no_training:
        tr = run_training(args, world, rank, local)
        tr["frac_of_sustained"] = tr["tflops"] / (peaks["bf16_sus"] * world)  # per GPU
        line["training"] = tr
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cb = cpu_baselines(local)
        line["cpu_baseline"] = cb[args.workload] if args.workload in cb else None
        line["cpu_baselines"] = cb
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
