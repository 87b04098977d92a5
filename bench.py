#!/usr/bin/env python3
"""Benchmark of the FORGE fused backward step on Llama-3.1-8B-shaped linears.

One step = the backward of the seven linear layers of one decoder layer
(down, up, gate, o, v, k, q; T = 16384 tokens): for each layer one launch
computes dX = dY W from the pre-update weights and the fused weight-gradient
+ AdamW step (bf16 weights with stochastic rounding, fp32 moments).  Inputs are seeded synthetic
tensors resident in HBM; one step streams ~8 GB (activations >= 134 MB, the
k/v output gradients 34 MB, 1.7 GB of states) through the 129 MB L2, so no
input is still resident when it is read again and no L2 flush is needed.

Printed: one JSON line (rank 0).  ``value`` = (2NKT for dW + 2NKT for dX,
summed over the layers and ranks) / step time, in TFLOP/s; the timed region of
``--steps`` steps is repeated back to back until it has run for at least 3 s
(``timed_region``) and ``ms_per_step`` is the median region, so the clock
samples cover the number.  ``roofline`` is the step kernel's own rate (CUDA
events around its launches) against the measured dense-bf16 peak that applies
to the region's length: the sustained peak for a region of 3 s or more, else
the burst peak.  ``fused_wgrad_opt`` is the rate of the fused weight-gradient
+ optimizer launches alone (2NKT, dX launched separately and not counted).
``two_launch`` times the same step with dX and the fused step as separate
launches (and each kernel's rate).  ``configs`` measures the other
configurations in the same run (the Llama set with INT8 moments, the
4096x4096 optimizer sweep, the 40-layer Qwen3-14B sweep at T = 4096, the
fp32-master 256x256 layer), one key each.  ``e2e`` repeats the step with the
inputs copied from pinned host memory inside the timed region (on a copy
stream, overlapping the previous step's compute) and the status word read
back every step.  ``unfused``
times the two-pass schedule (fp32 dW for every layer, then the optimizer).
``fp8`` times the same step with the weight gradient from E4M3 copies of X
and dY (token-contiguous, one power-of-two scale per tensor; dX stays a bf16
launch) against the bf16 peak times the nominal FP8/BF16 tensor-rate ratio 2.

``--impl reference`` times the CPU oracle on a bounded sample of the same
workload instead (no GPU work).  ``--workload KEY`` prints one line for another
measured configuration instead of the headline one (marked ``"secondary"``):
the fp32-master 256x256 layer, the Llama set with INT8 moments, the 4096x4096
optimizer sweep, or the 40-layer Qwen3-14B sweep at T = 4096.
"""

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from optimizer_tcgen05_dw_gb300 import inputs  # noqa: E402

METRIC = "fused wgrad+optimizer TFLOP/s and % of roofline at Llama-8B linear shapes"
WORKLOAD_KEY = "llama8b_bf16_fp32state"
# backward order through the decoder layer, and which activation feeds each linear
ORDER = ["down_proj", "up_proj", "gate_proj", "o_proj", "v_proj", "k_proj", "q_proj"]
ACT = {"q_proj": "x_attn", "k_proj": "x_attn", "v_proj": "x_attn", "o_proj": "x_o",
       "gate_proj": "x_mlp", "up_proj": "x_mlp", "down_proj": "x_down"}


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return p["hbm_gbs"], p["bf16_tflops"], p["bf16_tflops_sustained"], "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


TRAFFIC_PROFILE = os.path.join(ROOT, "profiles", "fused_traffic_llama8b_step.md")


def _profiled_traffic():
    """DRAM bytes per fused launch from the committed ncu summary, or None when
    the library sources changed since those counters were taken."""
    try:
        from optimizer_tcgen05_dw_gb300 import build as B
        fields = {}
        with open(TRAFFIC_PROFILE) as f:
            for ln in f:
                if ":" in ln and ln.split(":", 1)[0].strip() in ("source_digest", "traffic_bytes_per_launch"):
                    k, v = ln.split(":", 1)
                    fields[k.strip()] = v.strip().strip("`")
        if fields.get("source_digest") != B._digest(B.LIBS["libforge.so"]):
            return None
        return float(fields["traffic_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


# A timed region at least this long runs at the clocks a seconds-long GEMM
# loop settles to under the power cap, the conditions of the sustained peak;
# a shorter one is compared with the burst peak.
SUSTAINED_REGION_S = 3.0
SECONDARY_REGION_S = 0.5  # a secondary configuration's timed regions run at least this long


def applicable_peak(region_s: float, burst: float, sustained: float, src: str):
    """(peak, description) for a kernel timed over a region of region_s seconds."""
    if region_s >= SUSTAINED_REGION_S:
        return sustained, (f"bf16 sustained ({src}): the timed region ran {region_s:.2f} s, "
                           f">= {SUSTAINED_REGION_S:.0f} s")
    return burst, (f"bf16 burst ({src}): the timed region ran {region_s:.2f} s, "
                   f"< {SUSTAINED_REGION_S:.0f} s")


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo), or "unknown"."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.lower().startswith(("model name", "cpu model", "hardware")):
                    return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def host_cores() -> int:
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()


def max_over_ranks(x: float, dist=None, device=None) -> float:
    """The slowest rank's value (replicas report the max time).  Works with
    NCCL (device tensor) and gloo (CPU tensor)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


THROTTLE_REASONS = {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"}


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for nm, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------
# Reference arm: the CPU oracle
# ----------------------------------------------------------------------------

def oracle_sample(layer="k_proj", T=16384, seed=7):
    """One oracle step (dX + dW + AdamW, bf16 SR) on one Llama linear.  Returns
    (seconds, flops counted like the GPU metric)."""
    from oracle import linear_step as ls
    from oracle import optimizers as opt
    from oracle import rounding
    w = inputs.WORKLOADS[WORKLOAD_KEY]
    N, K = {n: (a, b) for n, a, b in inputs.LLAMA31_8B_LINEARS}[layer]
    X = inputs.bf16_to_bits(inputs.normal((T, K), 1.0, seed))
    dY = inputs.bf16_to_bits(inputs.normal((T, N), w.dy_std, seed + 1))
    W = rounding.bf16_bits_rne(inputs.normal((N, K), 0.02, seed + 2, torch.float32).numpy())
    st = {"W": W, "w_dtype": "bf16", "s_dtype": "fp32", "s1": np.zeros((N, K), np.float32),
          "s2": np.zeros((N, K), np.float32)}
    t0 = time.perf_counter()
    ls.linear_bwd_step(X, dY, st, opt.ADAMW, opt.Hparams(**w.hparams), 1, seed, want_dx=True)
    dt = time.perf_counter() - t0
    return dt, 4.0 * N * K * T


def oracle_sample_workload(key, seed=7):
    """The oracle as it stands on a bounded sample of a secondary workload:
    the whole fp32-master layer (its 3 steps), else one step of one
    representative linear (the smallest of the set, with that workload's
    state dtype and rule; the first optimizer of a sweep).  Returns (seconds,
    flops counted like that workload's GPU line, a description)."""
    from oracle import linear_step as ls
    from oracle import optimizers as opt
    from oracle import quant, rounding
    w = inputs.WORKLOADS[key]
    name, N, K = min(w.linears, key=lambda x: x[1] * x[2])
    T = w.T
    opt_name = list(inputs.SWEEP_HPARAMS)[0] if key == "sweep_4096" else w.opt
    hp = inputs.SWEEP_HPARAMS[opt_name] if key == "sweep_4096" else w.hparams
    kind = opt.NAMES.index(opt_name)
    want_dx = key != "sweep_4096"
    steps = w.steps if key == "single_256" else 1
    W = inputs.normal((N, K), w.w_std, seed + 2, torch.float32).numpy()
    st = {"w_dtype": w.w_dtype, "s_dtype": w.s_dtype,
          "W": W if w.w_dtype == "fp32" else rounding.bf16_bits_rne(W)}
    if w.s_dtype == "int8":
        st["s1"], st["s1_scale"] = quant.quantize_blocks(
            inputs.normal((N, K), max(w.m_init_std, 1e-30), seed + 3, torch.float32).numpy(), True)
        st["s2"], st["s2_scale"] = quant.quantize_blocks(
            inputs.abs_normal((N, K), max(w.v_init_std, 1e-30), seed + 4).numpy(), False)
    else:
        st["s1"] = np.zeros((N, K), np.float32)
        st["s2"] = np.zeros((N, K), np.float32)
    dt = 0.0
    for s in range(steps):
        X = inputs.bf16_to_bits(inputs.normal((T, K), w.x_std, seed + 10 * s + 5))
        dY = inputs.bf16_to_bits(inputs.normal((T, N), w.dy_std, seed + 10 * s + 6))
        t0 = time.perf_counter()
        out = ls.linear_bwd_step(X, dY, st, kind, opt.Hparams(**hp), s + 1, seed, want_dx=want_dx)
        dt += time.perf_counter() - t0
        st.update({k: out[k] for k in ("W", "s1", "s2", "s1_scale", "s2_scale") if k in out})
    flops = steps * (4.0 if want_dx else 2.0) * N * K * T
    desc = (f"{steps} step(s) of the {name} ({N}x{K}, T={T}): "
            f"{'dX + ' if want_dx else ''}dW + {opt_name} with {w.w_dtype} weights, {w.s_dtype} states")
    return dt, flops, desc


def run_reference(args):
    world, rank, _ = _dist()
    if rank != 0:
        return
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    for _ in range(args.warmup):
        oracle_sample()
    times, flops = [], 0.0
    for _ in range(args.steps):
        dt, f = oracle_sample()
        times.append(dt)
        flops = f
    tot = sum(times)
    val = flops * len(times) / tot / 1e12
    sample = ("one k_proj linear (1024x4096, T=16384) per step: dX + dW + AdamW with bf16 "
              "stochastic rounding, numpy float64 GEMMs on all host cores")
    print(json.dumps({
        "metric": METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "impl": "reference",
        "config": {"workload": inputs.WORKLOADS[WORKLOAD_KEY].name, "sample": "k_proj per step"},
        "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": cores, "cpu_model": cpu_model(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


# ----------------------------------------------------------------------------
# Our arm
# ----------------------------------------------------------------------------

class Layer:
    def __init__(self, name, N, K, T, dev, seed, host=False):
        self.name, self.N, self.K, self.T = name, N, K, T
        self.W = inputs.normal((N, K), 0.02, seed, torch.bfloat16, dev)
        self.m = torch.zeros((N, K), dtype=torch.float32, device=dev)
        self.v = torch.zeros((N, K), dtype=torch.float32, device=dev)
        self.dY = inputs.normal((T, N), 1e-3, seed + 1, torch.bfloat16, dev)
        self.dX = torch.empty((T, K), dtype=torch.bfloat16, device=dev)
        self.seed = seed


def build_workload(dev, T, only=None):
    names = [n for n in ORDER if not only or n in only]
    acts = {"x_attn": 4096, "x_o": 4096, "x_mlp": 4096, "x_down": 14336}
    used = {ACT[n] for n in names}
    X = {a: inputs.normal((T, k), 1.0, 100 + i, torch.bfloat16, dev)
         for i, (a, k) in enumerate(acts.items()) if a in used}
    shapes = {n: (N, K) for n, N, K in inputs.LLAMA31_8B_LINEARS}
    layers = [Layer(n, *shapes[n], T, dev, 1000 + 17 * ORDER.index(n)) for n in names]
    return X, layers


def run_ours(args):
    from optimizer_tcgen05_dw_gb300 import api
    from optimizer_tcgen05_dw_gb300.build import build

    world, rank, local = _dist()
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist_mod
        dist_mod.init_process_group("nccl", device_id=torch.device("cuda", local))
        dist = dist_mod
    build()
    api.lib()
    dev = torch.device("cuda", local)
    w = inputs.WORKLOADS[WORKLOAD_KEY]
    T = w.T
    hp = w.hparams
    X, layers = build_workload(dev, T, args.layers)
    stream = torch.cuda.current_stream()
    flops_dw = sum(2.0 * L.N * L.K * T for L in layers)
    flops_step = 2.0 * flops_dw  # dW + dX

    ev = {L.name: [] for L in layers}

    def step(s, record=False):
        """One backward step: per linear, dX and the FORGE step in one launch."""
        for L in layers:
            if record:
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record(stream)
            api.forge_linear_bwd_step(X[ACT[L.name]], L.dY, L.W, "adamw", hp, s, L.seed, L.m, L.v,
                                      dX=L.dX)
            if record:
                b.record(stream)
                ev[L.name].append((a, b))

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    s_no = 1
    for _ in range(args.warmup):
        step(s_no)
        s_no += 1
    api.forge_get_device_status()
    barrier()

    def timed_region():
        """R back-to-back regions of exactly args.steps steps each, R chosen so
        that together they run for at least SUSTAINED_REGION_S seconds (the
        nvidia-smi samples, 200 ms apart, then cover the number they qualify).
        Returns the per-region step times (ms), the total seconds and the clocks."""
        nonlocal s_no
        for v in ev.values():
            v.clear()
        region_ms = []
        with ClockSampler(local) as clk:
            barrier()
            t_start = time.perf_counter()
            while True:
                start = torch.cuda.Event(enable_timing=True)
                end = torch.cuda.Event(enable_timing=True)
                start.record(stream)
                for _ in range(args.steps):
                    step(s_no, record=True)
                    s_no += 1
                end.record(stream)
                end.synchronize()
                region_ms.append(start.elapsed_time(end) / args.steps)
                # every rank runs the same number of regions
                go_on = time.perf_counter() - t_start < args.min_region_s
                if max_over_ranks(1.0 if go_on else 0.0, dist, dev) == 0.0:
                    break
            torch.cuda.synchronize()
            total_s = time.perf_counter() - t_start
        barrier()
        api.forge_get_device_status()
        return region_ms, total_s, clk

    region_ms, region_s, clk = timed_region()
    # A region whose clock samples saw a hardware or thermal slowdown on any
    # rank is measured once more (sw_power_cap is normal under load and kept).
    first_reasons = clk.summary()["reasons"]
    throttled = max_over_ranks(1.0 if THROTTLE_REASONS & set(first_reasons) else 0.0, dist, dev)
    remeasured_after = None
    if throttled > 0:
        remeasured_after = first_reasons
        region_ms, region_s, clk = timed_region()
    ms = statistics.median(region_ms)
    ms = max_over_ranks(ms, dist, dev)
    kern_ms = sum(a.elapsed_time(b) for L in layers for (a, b) in ev[L.name])
    launches = sum(len(v) for v in ev.values())
    kern_tflops = flops_step * launches / len(layers) / (kern_ms * 1e-3) / 1e12
    hbm_gbs, peak_burst, peak_sust, peak_src = _peaks()
    peak, peak_kind = applicable_peak(region_s, peak_burst, peak_sust, peak_src)
    value = flops_step * world / (ms * 1e-3) / 1e12
    per_layer = {L.name: round(4.0 * L.N * L.K * T / (np.mean([a.elapsed_time(b) for a, b in ev[L.name]]) * 1e-3) / 1e12, 1)
                 for L in layers}
    # algorithmic bytes of the step launches: X, dY and W read once, W and the
    # fp32 m, v read and written, dX written
    params = sum(L.N * L.K for L in layers)
    bytes_step = sum(2 * (2 * L.T * L.K + L.T * L.N) for L in layers) + params * (4 + 16)

    if args.no_extras:
        if rank == 0:
            print(json.dumps({"metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s",
                              "ms_per_step": round(ms, 4), "layers": [L.name for L in layers],
                              "roofline_achieved": round(kern_tflops, 2),
                              "note": "partial run (--no-extras): not a bench result"}), flush=True)
        if dist is not None:
            dist.destroy_process_group()
        return

    # ---- e2e: every step's X and dY copied from pinned host memory through the
    # public API's buffers (a copy stream, two device buffer sets, so the copy
    # of step i+1 overlaps the compute of step i), and the step's status word
    # read back to the host.
    hostX = {k: v.cpu().pin_memory() for k, v in X.items()}
    hostdY = {L.name: L.dY.cpu().pin_memory() for L in layers}
    h2d = sum(t.numel() * 2 for t in hostX.values()) + sum(t.numel() * 2 for t in hostdY.values())
    bufX = [X, {k: torch.empty_like(v) for k, v in X.items()}]
    bufdY = [{L.name: L.dY for L in layers}, {L.name: torch.empty_like(L.dY) for L in layers}]
    copy_stream = torch.cuda.Stream(device=dev)
    copied = [torch.cuda.Event() for _ in range(2)]
    used = [torch.cuda.Event() for _ in range(2)]

    def enqueue_copy(i):
        b = i % 2
        copy_stream.wait_event(used[b])  # the step that last read this buffer set is done
        with torch.cuda.stream(copy_stream):
            for k in hostX:
                bufX[b][k].copy_(hostX[k], non_blocking=True)
            for L in layers:
                bufdY[b][L.name].copy_(hostdY[L.name], non_blocking=True)
        copied[b].record(copy_stream)

    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e2e_steps = max(4, args.steps // 4)
    e0.record(stream)
    copy_stream.wait_event(e0)
    enqueue_copy(0)
    for i in range(e2e_steps):
        if i + 1 < e2e_steps:
            enqueue_copy(i + 1)
        b = i % 2
        stream.wait_event(copied[b])
        for L in layers:
            api.forge_linear_bwd_step(bufX[b][ACT[L.name]], bufdY[b][L.name], L.W, "adamw", hp, s_no,
                                      L.seed, L.m, L.v, dX=L.dX)
        used[b].record(stream)
        s_no += 1
        api.forge_get_device_status()  # device -> host read of the step's status word
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, dist, dev)
    e2e_val = flops_step * world / (e2e_ms * 1e-3) / 1e12
    del hostX, hostdY, bufX, bufdY

    # ---- the same step as two launches per linear (dX, then the fused step)
    ev2 = {L.name: [] for L in layers}
    ev2_dx = {L.name: [] for L in layers}

    def two_launch_step(s, record=False):
        for L in layers:
            if record:
                z = torch.cuda.Event(enable_timing=True)
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                z.record(stream)
            api.forge_linear_dgrad(L.dY, L.W, L.dX)
            if record:
                a.record(stream)
            api.forge_linear_bwd_step(X[ACT[L.name]], L.dY, L.W, "adamw", hp, s, L.seed, L.m, L.v)
            if record:
                b.record(stream)
                ev2_dx[L.name].append((z, a))
                ev2[L.name].append((a, b))

    for _ in range(2):
        two_launch_step(s_no)
        s_no += 1
    barrier()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t_steps = args.steps
    t0.record(stream)
    for _ in range(t_steps):
        two_launch_step(s_no, record=True)
        s_no += 1
    t1.record(stream)
    torch.cuda.synchronize()
    api.forge_get_device_status()
    two_ms = max_over_ranks(t0.elapsed_time(t1) / t_steps, dist, dev)
    fused_peak, fused_peak_kind = applicable_peak(t0.elapsed_time(t1) * 1e-3, peak_burst, peak_sust,
                                                  peak_src)
    fused_ms = sum(a.elapsed_time(b) for L in layers for (a, b) in ev2[L.name])
    fused_tflops = flops_dw * t_steps / (fused_ms * 1e-3) / 1e12
    fused_per_layer = {L.name: round(2.0 * L.N * L.K * T / (np.mean([a.elapsed_time(b) for a, b in ev2[L.name]]) * 1e-3) / 1e12, 1)
                       for L in layers}
    dx_per_layer = {L.name: round(2.0 * L.N * L.K * T / (np.mean([a.elapsed_time(b) for a, b in ev2_dx[L.name]]) * 1e-3) / 1e12, 1)
                    for L in layers}

    # ---- unfused two-pass schedule on the same layers: all dW alive before the optimizer
    torch.cuda.reset_peak_memory_stats(dev)
    base_alloc = torch.cuda.memory_allocated(dev)
    dW = {L.name: torch.empty((L.N, L.K), dtype=torch.float32, device=dev) for L in layers}
    unf_peak = torch.cuda.max_memory_allocated(dev)

    def unfused_step(s):
        for L in layers:
            api.forge_linear_dgrad(L.dY, L.W, L.dX)
            api.forge_unfused_wgrad(X[ACT[L.name]], L.dY, dW[L.name])
        for L in layers:
            api.forge_unfused_opt_step(dW[L.name], L.W, "adamw", hp, s, L.seed, L.m, L.v)

    for _ in range(2):
        unfused_step(s_no)
        s_no += 1
    barrier()
    # The two schedules alternate in short regions of u_steps steps (three of
    # each, the fastest kept), so that both see the same clocks: the headline
    # region above runs for seconds under the power cap, these do not.
    u_steps = max(3, args.steps // 4)

    def short_region(fn):
        nonlocal s_no
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(u_steps):
            fn(s_no)
            s_no += 1
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / u_steps

    unf_runs, fused_runs = [], []
    for _ in range(3):
        fused_runs.append(short_region(step))
        unf_runs.append(short_region(unfused_step))
    api.forge_get_device_status()
    unf_ms = max_over_ranks(min(unf_runs), dist, dev)
    fused_short_ms = max_over_ranks(min(fused_runs), dist, dev)
    del dW
    torch.cuda.synchronize()

    # ---- E4M3 operands: the FORGE step from FP8 X^T and dY^T (dX from bf16 dY)
    def to_e4m3(t):
        """[T x C] bf16 -> ([C x T] E4M3 codes, power-of-two scale bringing the
        largest magnitude to at most 448)."""
        amax = float(t.abs().max().float())
        sc = 2.0 ** int(np.ceil(np.log2(amax / 448.0))) if amax > 0 else 1.0
        return (t.t().float() / sc).to(torch.float8_e4m3fn).contiguous(), sc

    X8 = {a: to_e4m3(x) for a, x in X.items()}
    dY8 = {L.name: to_e4m3(L.dY) for L in layers}
    ev8 = {L.name: [] for L in layers}

    def fp8_step(s, record=False):
        for L in layers:
            api.forge_linear_dgrad(L.dY, L.W, L.dX)
            if record:
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record(stream)
            (xt, sx), (dyt, sdy) = X8[ACT[L.name]], dY8[L.name]
            api.forge_linear_bwd_step_fp8(xt, dyt, sx, sdy, L.W, "adamw", hp, s, L.seed, L.m, L.v)
            if record:
                b.record(stream)
                ev8[L.name].append((a, b))

    for _ in range(2):
        fp8_step(s_no)
        s_no += 1
    barrier()
    f0 = torch.cuda.Event(enable_timing=True)
    f1 = torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for _ in range(t_steps):
        fp8_step(s_no, record=True)
        s_no += 1
    f1.record(stream)
    torch.cuda.synchronize()
    api.forge_get_device_status()
    fp8_ms = max_over_ranks(f0.elapsed_time(f1) / t_steps, dist, dev)
    fp8_peak, fp8_peak_kind = applicable_peak(f0.elapsed_time(f1) * 1e-3, peak_burst, peak_sust, peak_src)
    fp8_kern_ms = sum(a.elapsed_time(b) for L in layers for (a, b) in ev8[L.name])
    fp8_tflops = flops_dw * t_steps / (fp8_kern_ms * 1e-3) / 1e12
    fp8_per_layer = {L.name: round(2.0 * L.N * L.K * T / (np.mean([a.elapsed_time(b) for a, b in ev8[L.name]]) * 1e-3) / 1e12, 1)
                     for L in layers}
    del X8, dY8
    torch.cuda.synchronize()

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return
    ck = clk.summary()
    if remeasured_after is not None:
        ck["remeasured_after"] = remeasured_after
    out = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": w.name, "T": T, "layers": ORDER, "optimizer": "adamw",
                   "hparams": hp, "weights": "bf16, stochastic rounding",
                   "states": "fp32 m, v", "flops_per_step": flops_step,
                   "flops_counted": "2NKT (dW) + 2NKT (dX) per linear",
                   "l2": "no flush: a step streams ~8 GB (X >= 134 MB, dY 34-470 MB, 1.7 GB of "
                         "states) through the 129 MB L2 between two reads of any input",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "tensor",
                     "kernel": "one-launch FORGE step (tc_kernel mode 3: dX tiles, then dW tiles "
                               "with the AdamW epilogue), 4NKT flops per launch",
                     "achieved": round(kern_tflops, 2),
                     "peak": peak, "unit": "TFLOP/s",
                     "frac": round(kern_tflops / peak, 4),
                     "peak_kind": peak_kind,
                     "frac_of_burst_peak": round(kern_tflops / peak_burst, 4),
                     "frac_of_sustained_peak": round(kern_tflops / peak_sust, 4),
                     "traffic": _profiled_traffic(),
                     "traffic_unit": "DRAM bytes per step launch (mean of the 7 layers, ncu)",
                     "algorithmic_bytes_per_launch": round(bytes_step / len(layers)),
                     "algorithmic_bytes_per_step": bytes_step,
                     "launches_timed": launches,
                     "per_layer_tflops": per_layer},
        "timed_region": {"regions": len(region_ms), "steps_per_region": args.steps,
                         "seconds": round(region_s, 3),
                         "ms_per_step_min": round(min(region_ms), 4),
                         "ms_per_step_max": round(max(region_ms), 4),
                         "ms_per_step_x_median_sm_mhz": (None if ck["sm_mhz"] is None
                                                         else round(ms * ck["sm_mhz"], 1))},
        "fused_wgrad_opt": {
            "definition": "2NKT per linear / the fused weight-gradient + optimizer launches' own "
                          "time, dX launched separately and not counted (the two-launch form)",
            "tflops": round(fused_tflops, 2), "peak": fused_peak,
            "frac": round(fused_tflops / fused_peak, 4), "peak_kind": fused_peak_kind,
            "frac_of_burst_peak": round(fused_tflops / peak_burst, 4),
            "per_layer_tflops": fused_per_layer},
        "two_launch": {"ms_per_step": round(two_ms, 4),
                       "value": round(flops_step * world / (two_ms * 1e-3) / 1e12, 2),
                       "fused_wgrad_opt_tflops": round(fused_tflops, 2),
                       "fused_per_layer_tflops": fused_per_layer,
                       "dgrad_per_layer_tflops": dx_per_layer},
        "e2e": {"value": round(e2e_val, 2), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": 4, "ms_per_step": round(e2e_ms, 4)},
        "unfused": {"ms_per_step": round(unf_ms, 4),
                    "value": round(flops_step * world / (unf_ms * 1e-3) / 1e12, 2),
                    "fused_ms_per_step_same_regions": round(fused_short_ms, 4),
                    "speedup_fused_vs_unfused": round(unf_ms / fused_short_ms, 3),
                    "regions": f"3 x {u_steps} steps of each schedule, alternating; fastest of each",
                    "dW_pool_bytes": params * 4,
                    "peak_alloc_bytes_fused": base_alloc,
                    "peak_alloc_bytes_unfused": unf_peak},
        "fp8": {"ms_per_step": round(fp8_ms, 4),
                "value": round(flops_step * world / (fp8_ms * 1e-3) / 1e12, 2),
                "operands": "E4M3 X^T and dY^T, one power-of-two scale per tensor; dX from bf16 dY",
                "fused_wgrad_opt_tflops": round(fp8_tflops, 2),
                "peak": round(2 * fp8_peak, 1),
                "peak_kind": "2 x " + fp8_peak_kind + " (nominal FP8/BF16 tensor-rate ratio)",
                "frac": round(fp8_tflops / (2 * fp8_peak), 4),
                "fused_per_layer_tflops": fp8_per_layer},
        "hbm_bytes_per_param_algorithmic": round(bytes_step / params, 3),
        "hbm_bytes_per_param_measured": (None if _profiled_traffic() is None else
                                         round(_profiled_traffic() * len(layers) / params, 3)),
        "gpu_launches": launches,
        "clocks": ck,
    }
    # ---- the other measured configurations, in the same run, one key each
    # (the headline's tensors are freed first: the Qwen3-14B sweep holds ~99 GB)
    X.clear()
    layers.clear()
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    if not args.no_configs:
        out["configs"] = {}
        for key in CONFIG_KEYS:
            r = measure_workload(api, key, args.steps, args.warmup, local, cpu=not args.no_cpu_baseline)
            out["configs"][key] = r
            torch.cuda.empty_cache()
    if not args.no_configs:
        out["int8_block_sizes"] = measure_int8_blocks(api, args.steps, args.warmup, local)
        torch.cuda.empty_cache()
    if not args.no_cpu_baseline:
        dt, f = oracle_sample()
        out["cpu_baseline"] = {"value": round(f / dt / 1e12, 6), "unit": "TFLOP/s", "cores": host_cores(),
                               "cpu_model": cpu_model(), "kind": "oracle",
                               "sample": "one k_proj linear (1024x4096, T=16384): dX + dW + AdamW "
                                         "with bf16 stochastic rounding, one step"}
    print(json.dumps(out), flush=True)
    if dist is not None:
        dist.destroy_process_group()


# ----------------------------------------------------------------------------
# Secondary workloads (`--workload`): the other measured configurations
# ----------------------------------------------------------------------------

SECONDARY = ("single_256", "llama8b_bf16_int8state", "sweep_4096", "qwen14b_int8")
QWEN_ACT = {"q_proj": "x_attn", "k_proj": "x_attn", "v_proj": "x_attn", "o_proj": "x_o",
            "gate_proj": "x_mlp", "up_proj": "x_mlp", "down_proj": "x_down"}


class _SLayer:
    """One linear of a secondary workload: bf16 or fp32 W, fp32 or INT8 AdamW-
    style states (INT8 codes made by the library's own quantiser), its dY and dX."""

    def __init__(self, api, name, N, K, T, dev, seed, w, want_dx=True):
        self.name, self.N, self.K, self.T, self.seed = name, N, K, T, seed
        wdt = torch.float32 if w.w_dtype == "fp32" else torch.bfloat16
        self.W = inputs.normal((N, K), w.w_std, seed, wdt, dev)
        self.dY = inputs.normal((T, N), w.dy_std, seed + 1, torch.bfloat16, dev)
        self.dX = torch.empty((T, K), dtype=torch.bfloat16, device=dev) if want_dx else None
        if w.s_dtype == "int8":
            self.m = torch.empty((N, K), dtype=torch.int8, device=dev)
            self.v = torch.empty((N, K), dtype=torch.uint8, device=dev)
            self.ms = torch.empty((N, K // 64), dtype=torch.float32, device=dev)
            self.vs = torch.empty((N, K // 64), dtype=torch.float32, device=dev)
            api.forge_quantize_state(inputs.normal((N, K), w.m_init_std, seed + 2, torch.float32, dev),
                                     self.m, self.ms, True)
            api.forge_quantize_state(inputs.abs_normal((N, K), w.v_init_std, seed + 3, torch.float32, dev),
                                     self.v, self.vs, False)
        else:
            self.m = torch.zeros((N, K), dtype=torch.float32, device=dev)
            self.v = torch.zeros((N, K), dtype=torch.float32, device=dev)
            self.ms = self.vs = None
        self.state_bytes = 2 * N * K * (1 if w.s_dtype == "int8" else 4) + \
            (2 * 4 * N * (K // 64) if w.s_dtype == "int8" else 0)


CONFIG_KEYS = ("llama8b_bf16_int8state", "sweep_4096", "qwen14b_int8", "single_256")


def measure_workload(api, key, steps, warmup, local=0, only_layers=None, num_layers=None,
                     no_dx=False, cpu=True, tokens=None, optimizers=None):
    """One secondary workload: its step timed with CUDA events between
    synchronisations (warmup steps, then `steps`), the step launches' own rate
    against the dense-bf16 peak that applies to the region's length, the
    slower-roofline fraction, per-linear rates, peak device memory and the
    algorithmic HBM bytes per parameter; with `cpu`, the oracle timed on a
    bounded sample of the same configuration.  Returns a dict."""
    dev = torch.device("cuda", local)
    w = inputs.WORKLOADS[key]
    T = w.T if tokens is None else tokens
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats(dev)
    hbm_gbs, peak_burst, peak_sust, peak_src = _peaks()
    sweep = key == "sweep_4096"
    opts = list(inputs.SWEEP_HPARAMS) if sweep else [w.opt]
    if sweep and optimizers:
        opts = [o for o in opts if o in optimizers]
    # layers: (layer index, name, N, K); activations per layer
    if key == "qwen14b_int8":
        n_layers = w.layers if num_layers is None else num_layers
        shapes = [(li, n, N, K) for li in range(n_layers) for n, N, K in inputs.QWEN3_14B_LINEARS
                  if not only_layers or n in only_layers]
        acts = {"x_attn": 5120, "x_o": 5120, "x_mlp": 5120, "x_down": 17408}
        act_of = QWEN_ACT
    elif key == "llama8b_bf16_int8state":
        shapes = [(0, n, N, K) for n, N, K in sorted(inputs.LLAMA31_8B_LINEARS, key=lambda x: ORDER.index(x[0]))
                  if not only_layers or n in only_layers]
        acts = {"x_attn": 4096, "x_o": 4096, "x_mlp": 4096, "x_down": 14336}
        act_of = ACT
    else:  # one linear
        (n0, N0, K0), = w.linears
        shapes = [(0, n0, N0, K0)]
        acts = {"x": K0}
        act_of = {n0: "x"}
    want_dx = not sweep and not no_dx
    X = {(li, a): inputs.normal((T, k), w.x_std, inputs.layer_seed(7, li, 0, 50 + j), torch.bfloat16, dev)
         for li in sorted({s[0] for s in shapes}) for j, (a, k) in enumerate(acts.items())}
    layers = [(li, _SLayer(api, n, N, K, T, dev, inputs.layer_seed(7, li, 0, 10 * (1 + i)), w, want_dx))
              for i, (li, n, N, K) in enumerate(shapes)]
    torch.cuda.synchronize()
    flops_dw = sum(2.0 * L.N * L.K * T for _, L in layers)
    flops_step = flops_dw * (2.0 if want_dx else 1.0)
    params = sum(L.N * L.K for _, L in layers)
    w_bytes = 2 * (4 if w.w_dtype == "fp32" else 2)
    bytes_step = sum(2 * (L.T * L.K + L.T * L.N) + (2 * L.T * L.K if want_dx else 0) for _, L in layers) + \
        params * w_bytes + sum(L.state_bytes for _, L in layers)
    results = {}
    per_linear_ms = {}
    s_no = 1
    # events around each call give the per-linear rates; with one linear the
    # region's own events give them, and per-call events would only add gaps
    per_call = len(layers) > 1
    for opt_name in opts:
        hp = inputs.SWEEP_HPARAMS[opt_name] if sweep else w.hparams
        ev = []

        def step(s, record=False):
            for li, L in layers:
                if record:
                    a = torch.cuda.Event(enable_timing=True)
                    b = torch.cuda.Event(enable_timing=True)
                    a.record(stream)
                s1 = L.m if opt_name in api.USES_S1 else None
                s2 = L.v if opt_name in api.USES_S2 else None
                api.forge_linear_bwd_step(X[(li, act_of[L.name])], L.dY, L.W, opt_name, hp, s, L.seed,
                                          s1, s2, L.ms if s1 is not None else None,
                                          L.vs if s2 is not None else None, dX=L.dX)
                if record:
                    b.record(stream)
                    ev.append((L.name, a, b))

        for _ in range(warmup):
            step(s_no)
            s_no += 1
        api.forge_get_device_status()
        torch.cuda.synchronize()
        region_ms = []
        with ClockSampler(local) as clk:
            step(s_no)  # the GPU idled while the sampler started: one untimed step first
            s_no += 1
            torch.cuda.synchronize()
            t_start = time.perf_counter()
            while True:  # regions of `steps` steps, back to back, for SECONDARY_REGION_S
                start = torch.cuda.Event(enable_timing=True)
                end = torch.cuda.Event(enable_timing=True)
                start.record(stream)
                for _ in range(steps):
                    step(s_no, record=per_call)
                    s_no += 1
                end.record(stream)
                end.synchronize()
                region_ms.append(start.elapsed_time(end) / steps)
                if time.perf_counter() - t_start >= SECONDARY_REGION_S:
                    break
            total_s = time.perf_counter() - t_start
        api.forge_get_device_status()
        ms = statistics.median(region_ms)
        if per_call:
            kern_ms = sum(a.elapsed_time(b) for _, a, b in ev)
            for name, a, b in ev:
                per_linear_ms.setdefault(name, []).append(a.elapsed_time(b))
        else:  # one linear: its launches are the whole region
            kern_ms = sum(region_ms) * steps
            per_linear_ms.setdefault(layers[0][1].name, []).extend(region_ms)
        results[opt_name] = {"ms_per_step": round(ms, 4),
                             "value": round(flops_step / (ms * 1e-3) / 1e12, 2),
                             "kernel_tflops": round(flops_step * steps * len(region_ms) /
                                                    (kern_ms * 1e-3) / 1e12, 2),
                             "region_s": round(total_s, 4), "regions": len(region_ms),
                             "clocks": clk.summary()}
    tot_ms = sum(r["ms_per_step"] for r in results.values())
    value = flops_step * len(opts) / (tot_ms * 1e-3) / 1e12
    kern = statistics.mean(r["kernel_tflops"] for r in results.values())
    region_s = max(r["region_s"] for r in results.values())
    peak, peak_kind = applicable_peak(region_s, peak_burst, peak_sust, peak_src)
    t_flop = flops_step / (peak * 1e12)
    t_byte = bytes_step / (hbm_gbs * 1e9)
    bound = "tensor" if t_flop >= t_byte else "hbm"
    # per distinct linear shape: 2NKT (+ 2NKT for dX) over its mean launch time
    shape_of = {L.name: (L.N, L.K) for _, L in layers}
    per_linear = {n: round((4.0 if want_dx else 2.0) * shape_of[n][0] * shape_of[n][1] * T /
                           (statistics.mean(v) * 1e-3) / 1e12, 1) for n, v in per_linear_ms.items()}
    out = {
        "value": round(value, 2), "unit": "TFLOP/s", "ms_per_step": round(tot_ms / len(opts), 4),
        "steps": steps, "warmup": warmup,
        "timed_region": {"steps_per_region": steps,
                         "regions": sum(r["regions"] for r in results.values()),
                         "seconds": round(sum(r["region_s"] for r in results.values()), 3),
                         "ms_per_step": "median region"},
        "dtype": "bf16" if w.w_dtype == "bf16" else "fp32",
        "config": {"workload": w.name, "key": key, "T": T, "linears": len(layers),
                   "flops_counted": "2NKT (dW)" + (" + 2NKT (dX)" if want_dx else "") + " per linear",
                   "w_dtype": w.w_dtype, "s_dtype": w.s_dtype, "optimizers": opts,
                   "partial": bool(only_layers or num_layers is not None or no_dx or tokens is not None
                                   or (sweep and optimizers))},
        "roofline": {"bound": bound, "achieved": round(kern, 2), "unit": "TFLOP/s",
                     "peak": peak, "peak_kind": peak_kind,
                     "frac": round(kern / peak, 4),
                     "frac_of_burst_peak": round(kern / peak_burst, 4),
                     "frac_of_slower_roofline": round(max(t_flop, t_byte) * 1e3 / (tot_ms / len(opts)), 4),
                     "algorithmic_bytes_per_step": bytes_step},
        "per_linear_tflops": per_linear,
        "hbm_bytes_per_param_algorithmic": round(bytes_step / params, 3),
        "params": params,
        "peak_device_memory_bytes": torch.cuda.max_memory_allocated(dev),
        "per_optimizer": results if sweep else None,
        "clocks": results[opts[-1]]["clocks"],
        "cpu_baseline": None,
        "gpu_launches": sum(1 if (not want_dx or (w.w_dtype == "bf16" and L.N % 64 == 0 and L.K % 64 == 0))
                            else 2 for _, L in layers) * steps * sum(r["regions"] for r in results.values()),
        "note": "inputs are drawn once per linear and reused by every timed step (timing does "
                "not depend on their values); parity for this configuration is in the tests",
    }
    del layers, X
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    if cpu and not out["config"]["partial"]:
        dt, f, desc = oracle_sample_workload(key)
        out["cpu_baseline"] = {"value": round(f / dt / 1e12, 6), "unit": "TFLOP/s", "cores": host_cores(),
                               "cpu_model": cpu_model(), "kind": "oracle", "sample": desc}
    return out


INT8_BLOCKS = (32, 64, 128, 256)


def measure_int8_blocks(api, steps, warmup, local=0, moment_steps=10):
    """The INT8-moment Llama step (dX + FORGE step, T = 16384, AdamW) with each
    absmax block width the kernels support, and the quantisation error each
    width leaves in the moments: one q_proj (4096 x 4096) stepped
    `moment_steps` times with INT8 moments and, from the same dequantised
    start and the same inputs, with fp32 moments (the moments of AdamW do not
    depend on the weights, so the fp32 run is the INT8 run's exact reference);
    reported as ||dequant(m_B) - m|| / ||m||, and likewise for v."""
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    w = inputs.WORKLOADS["llama8b_bf16_int8state"]
    T, hp = w.T, w.hparams
    _, peak_burst, _, _ = _peaks()
    acts = {"x_attn": 4096, "x_o": 4096, "x_mlp": 4096, "x_down": 14336}
    X = {a: inputs.normal((T, k), 1.0, 200 + i, torch.bfloat16, dev) for i, (a, k) in enumerate(acts.items())}
    shapes = {n: (N, K) for n, N, K in inputs.LLAMA31_8B_LINEARS}
    res = {}
    for qb in INT8_BLOCKS:
        layers = []
        for i, n in enumerate(ORDER):
            N, K = shapes[n]
            L = {"name": n, "N": N, "K": K, "seed": 3000 + 17 * i,
                 "W": inputs.normal((N, K), 0.02, 3000 + 17 * i, torch.bfloat16, dev),
                 "dY": inputs.normal((T, N), 1e-3, 3001 + 17 * i, torch.bfloat16, dev),
                 "dX": torch.empty((T, K), dtype=torch.bfloat16, device=dev),
                 "m": torch.empty((N, K), dtype=torch.int8, device=dev),
                 "v": torch.empty((N, K), dtype=torch.uint8, device=dev),
                 "ms": torch.empty((N, K // qb), dtype=torch.float32, device=dev),
                 "vs": torch.empty((N, K // qb), dtype=torch.float32, device=dev)}
            api.forge_quantize_state(inputs.normal((N, K), w.m_init_std, 3002 + 17 * i, torch.float32, dev),
                                     L["m"], L["ms"], True, block=qb)
            api.forge_quantize_state(inputs.abs_normal((N, K), w.v_init_std, 3003 + 17 * i, torch.float32, dev),
                                     L["v"], L["vs"], False, block=qb)
            layers.append(L)

        def step(s):
            for L in layers:
                api.forge_linear_bwd_step(X[ACT[L["name"]]], L["dY"], L["W"], "adamw", hp, s, L["seed"],
                                          L["m"], L["v"], L["ms"], L["vs"], dX=L["dX"])

        for s in range(warmup):
            step(s + 1)
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for s in range(steps):
            step(warmup + s + 1)
        b.record(stream)
        torch.cuda.synchronize()
        api.forge_get_device_status()
        step_ms = a.elapsed_time(b) / steps
        flops = sum(4.0 * L["N"] * L["K"] * T for L in layers)
        del layers
        torch.cuda.empty_cache()
        # moment error after moment_steps steps of one q_proj
        N = K = 4096
        W8 = inputs.normal((N, K), 0.02, 4000, torch.bfloat16, dev)
        W32 = W8.clone()
        m8 = torch.empty((N, K), dtype=torch.int8, device=dev)
        v8 = torch.empty((N, K), dtype=torch.uint8, device=dev)
        sm8 = torch.empty((N, K // qb), dtype=torch.float32, device=dev)
        sv8 = torch.empty((N, K // qb), dtype=torch.float32, device=dev)
        api.forge_quantize_state(inputs.normal((N, K), w.m_init_std, 4001, torch.float32, dev), m8, sm8, True, block=qb)
        api.forge_quantize_state(inputs.abs_normal((N, K), w.v_init_std, 4002, torch.float32, dev), v8, sv8, False,
                                 block=qb)
        m32 = torch.empty((N, K), dtype=torch.float32, device=dev)
        v32 = torch.empty((N, K), dtype=torch.float32, device=dev)
        api.forge_dequantize_state(m8, sm8, m32, True, block=qb)
        api.forge_dequantize_state(v8, sv8, v32, False, block=qb)
        for s in range(moment_steps):
            Xs = inputs.normal((T, K), 1.0, 4100 + s, torch.bfloat16, dev)
            dYs = inputs.normal((T, N), 1e-3, 4200 + s, torch.bfloat16, dev)
            api.forge_linear_bwd_step(Xs, dYs, W8, "adamw", hp, s + 1, 4003, m8, v8, sm8, sv8)
            api.forge_linear_bwd_step(Xs, dYs, W32, "adamw", hp, s + 1, 4003, m32, v32)
        mq = torch.empty_like(m32)
        vq = torch.empty_like(v32)
        api.forge_dequantize_state(m8, sm8, mq, True, block=qb)
        api.forge_dequantize_state(v8, sv8, vq, False, block=qb)
        api.forge_get_device_status()
        rel = lambda a, r: float((a.double() - r.double()).norm() / r.double().norm())  # noqa: E731
        res[str(qb)] = {"ms_per_step": round(step_ms, 4), "tflops": round(flops / (step_ms * 1e-3) / 1e12, 1),
                        "frac_of_burst_peak": round(flops / (step_ms * 1e-3) / 1e12 / peak_burst, 4),
                        "m_rel_error": rel(mq, m32), "v_rel_error": rel(vq, v32),
                        "scale_bytes_per_param": 2 * 4.0 / qb}
        del W8, W32, m8, v8, sm8, sv8, m32, v32, mq, vq
        torch.cuda.empty_cache()
    return {"workload": "Llama-3.1-8B layer linears, T=16384, dX + FORGE step, bf16 W (SR), INT8 AdamW "
                        "moments with one fp32 absmax per block of B row elements",
            "moment_error": f"q_proj 4096x4096 after 10 steps against fp32 moments from the same start",
            "per_block": res}


def run_workload(args):
    """One JSON line for a secondary workload (marked "secondary")."""
    from optimizer_tcgen05_dw_gb300 import api
    from optimizer_tcgen05_dw_gb300.build import build

    world, rank, local = _dist()
    if rank != 0:
        return
    torch.cuda.set_device(local)
    build()
    api.lib()
    r = measure_workload(api, args.workload, args.steps, args.warmup, local, args.layers,
                         args.num_layers, args.no_dx, cpu=not args.no_cpu_baseline,
                         tokens=args.tokens, optimizers=args.optimizers)
    out = {"metric": METRIC, "value": r.pop("value"), "unit": r.pop("unit"), "n_gpus": 1,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": r.pop("ms_per_step"),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
           "dtype": r.pop("dtype"), "data": "synthetic", "secondary": True}
    r.pop("steps")
    r.pop("warmup")
    out.update(r)
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--min-region-s", type=float, default=None,
                    help="repeat the timed region of --steps steps until this many seconds have "
                         "run (the value is the median region); 0 = one region; default "
                         f"{SUSTAINED_REGION_S:.0f}, or 0 with --no-extras")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other measured configurations in the headline line")
    ap.add_argument("--layers", nargs="*", default=None, choices=ORDER,
                    help="restrict to some linears (profiling); the bench line uses all seven")
    ap.add_argument("--no-extras", action="store_true",
                    help="time the step only (profiling runs): no e2e, unfused or CPU legs")
    ap.add_argument("--num-layers", type=int, default=None,
                    help="with --workload qwen14b_int8: decoder layers to sweep (profiling; default 40)")
    ap.add_argument("--tokens", type=int, default=None,
                    help="with --workload: another token count T (profiling; the line is marked partial)")
    ap.add_argument("--optimizers", nargs="*", default=None, choices=list(inputs.SWEEP_HPARAMS),
                    help="with --workload sweep_4096: only these rules (profiling)")
    ap.add_argument("--no-dx", action="store_true",
                    help="with --workload: the weight step alone, without dX (profiling)")
    ap.add_argument("--workload", default=WORKLOAD_KEY, choices=(WORKLOAD_KEY,) + SECONDARY,
                    help="a secondary measured configuration instead of the headline one "
                         "(its own JSON line, marked \"secondary\")")
    args = ap.parse_args()
    if args.min_region_s is None:
        args.min_region_s = 0.0 if args.no_extras else SUSTAINED_REGION_S
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.workload != WORKLOAD_KEY:
        run_workload(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
