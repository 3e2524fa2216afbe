"""Benchmark of the FSDP FlatParameter step on GB300.

One step = one pass of the whole hot path over one unit: the fused
reduce-scatter + AdamW + cast over all N emulated ranks' blocks, then the
all-gather(s) of the updated compute-dtype shards into the N full buffers
(twice for the 70B unit: before forward and before backward). Flatten/pad and
the unflatten views are set-up (once per unit) and are not in the step.

Default workload: the Llama-70B-style block unit (855,654,400 parameters, N=8,
bf16 gradients ~N(0, 1e-4), AdamW lr 3e-5, wd 0.1, two all-gathers per step),
the largest unit of the set, on which the fused kernel's HBM-bandwidth target
is stated. Inputs are synthetic (seeded), resident in HBM, and far larger
than L2; for the small units (--config gpt2_small, gpt2_large, tiny) L2 is
flushed before every timed step, outside that step's CUDA events.

Printed (rank 0, one JSON line): value = algorithmic bytes of the step / step
time (GB/s, whole job over all ranks); roofline of the fused kernel (its own
CUDA-event time inside the timed region; mean and median); e2e with the
gradients in pinned host memory, the faster of the binding's copy pipeline
and the C ABI call reading the host buffers in place (the other beside it);
the CPU oracle timed on the host cores; clocks sampled during the timed
region. Beside them, on the same unit: the fused-gather and no-reshard steps
on their own byte models (`variants`), the variant optimizers' kernels
(`variant_kernels`), the fused kernel with its state in pinned host memory
(`offload_state_on_host`), the per-unit driver on a 12-unit GPT-2 small model
(`driver_gpt2_small_model_12_units`) and on a model of 200 units of 50,000
parameters (`driver_model_200_units_of_50k`, batched launches: a model
validated once, validated every call, and captured); then, with that unit
freed, the fused kernel alone on the GPT-3 13B, GPT-2 Large and GPT-2 small
block units (`per_config`, each with its own clocks). The last four run on
one GPU only; --no-variants, --no-offload, --no-driver and --no-per-config
skip them.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

Under torchrun each rank runs its own unit on its own GPU (independent
units: weak scaling, no data-path collective); rank 0 prints the MAX step
time over ranks.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
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

METRIC = "fused RS+AdamW+cast GB/s and params/s per FSDP unit vs HBM roofline, 1 GB300"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0  # GB300 HBM3e, the ~8 TB/s nominal figure
WORKLOAD_NAMES = {
    "tiny": "tiny_unit_4099_n2",
    "gpt2_small": "gpt2_small_block_unit_n8",
    "gpt2_large": "gpt2_large_block_unit_n2_fp16",
    "gpt3_13b": "gpt3_13b_block_unit_n8",
    "llama70b": "llama70b_block_unit_n8",
}
RSA_SOURCES = ("sharded_fsdp_reduce_gb300/csrc/rsa_impl.cuh", "sharded_fsdp_reduce_gb300/csrc/common.cuh")


# ---------------------------------------------------------------- helpers

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def step_bytes(P_pad: int, world: int, gsize: int, osize: int, gathers: int, n_dst: int):
    """Algorithmic bytes: fused kernel per launch, all-gathers per step."""
    rsa = P_pad * (world * gsize + 3 * (4 + 4) + osize)
    ag = gathers * P_pad * osize * (1 + n_dst)
    return rsa, ag


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def host_info() -> dict:
    """Host name and CPU model of the machine the oracle is timed on."""
    import platform
    import socket
    import subprocess

    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    if model is None:
        try:
            with open("/proc/cpuinfo") as f:
                for line in f:
                    if line.lower().startswith("model name"):
                        model = line.split(":", 1)[1].strip()
                        break
        except OSError:
            pass
    return {"host": socket.gethostname(), "cpu_model": model or platform.machine(),
            "host_cpus": os.cpu_count()}


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for rel in RSA_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


# The committed ncu summary that holds each workload's fused-kernel DRAM
# traffic. The 13B unit runs the same kernel build as the 70B unit (N = 8,
# bf16 gradients and output), so both take the small-case captures of that
# build; the GPT-2 units are small enough to be captured whole.
TRAFFIC_SUMMARY = {
    "llama70b_block_unit_n8": "rsa_n8_bf16_numel33m_67m_ncu.md",
    "gpt3_13b_block_unit_n8": "rsa_n8_bf16_numel33m_67m_ncu.md",
    "gpt2_large_block_unit_n2_fp16": "rsa_gpt2_large_block_unit_n2_fp16_ncu.md",
    "gpt2_small_block_unit_n8": "rsa_gpt2_small_block_unit_n8_ncu.md",
}


def read_summary(path: str) -> dict:
    """The `- key: value` lines of an ncu summary."""
    vals = {}
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line.startswith("- "):
                continue
            line = line[2:]
            if ":" in line:
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip().strip("`")
    return vals


def recorded_traffic(workload: str, padded_numel: int):
    """Per-launch DRAM traffic (read + write bytes) of the fused kernel on a
    unit of padded_numel elements, from a committed ncu summary; None when
    there is none for this workload or the kernel changed since.

    A summary gives either the traffic of the whole unit (`captured_numel`:
    one size, equal to padded_numel) or captures of two smaller cases of the
    same kernel build (`captured_numel: n1, n2`, `traffic_bytes: T1, T2`).
    Traffic is then per-element bytes plus a fixed part (the stores still
    dirty in L2 when the kernel ends, which the next kernel writes back), so
    the two points give both and the full launch is read off the same line:
    T2 + (T2 - T1) / (n2 - n1) * (padded_numel - n2)."""
    name = TRAFFIC_SUMMARY.get(workload.split("_numel")[0])
    if name is None:
        return None
    path = os.path.join(ROOT, "profiles", name)
    if not os.path.exists(path):
        return None
    vals = read_summary(path)
    if vals.get("kernel_source_sha256") != kernel_source_hash():
        return None
    try:
        ns = [int(x) for x in vals["captured_numel"].split(",")]
        ts = [float(x) for x in vals["traffic_bytes"].split(",")]
    except (KeyError, ValueError):
        return None
    if len(ns) == 1 and len(ts) == 1:
        return ts[0] if ns[0] == padded_numel else None
    if len(ns) != 2 or len(ts) != 2 or ns[1] <= ns[0]:
        return None
    slope = (ts[1] - ts[0]) / (ns[1] - ns[0])
    return round(ts[1] + slope * (padded_numel - ns[1]))


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.gpu)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.reader.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


class L2Flush:
    """Between timed iterations of units whose working set is not far larger
    than L2: write a buffer of twice L2, then read another of twice L2, so
    that L2 holds neither the unit's data nor dirty lines of the flush."""

    FAR_LARGER = 16  # units moving more than 16 x L2 per kernel need no flush

    def __init__(self, device, work_bytes: int):
        import torch

        props = torch.cuda.get_device_properties(device)
        self.l2 = int(getattr(props, "L2_cache_size", 0) or 129 * 2**20)
        self.active = work_bytes <= self.FAR_LARGER * self.l2
        if self.active:
            n = 2 * self.l2 // 4
            self.w = torch.empty(n, dtype=torch.int32, device=device)
            self.r = torch.ones(n, dtype=torch.int32, device=device)
            self.k = 0

    def __call__(self):
        if self.active:
            self.k += 1
            self.w.fill_(self.k)
            self.r.sum()

    def describe(self) -> str:
        if self.active:
            return (f"L2 flushed before every timed launch or step ({2 * self.l2 >> 20} MiB written, then "
                    f"{2 * self.l2 >> 20} MiB read); each timed between its own CUDA events")
        return "inputs larger than L2 (no flush needed)"


def timed_calls(fn, K: int, stream, flush: L2Flush) -> float:
    """Mean device time of fn() over K calls (ms): one pair of events around
    all K calls, or, with the flush active, a pair around each call."""
    import torch

    torch.cuda.synchronize()
    if not flush.active:
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for i in range(K):
            fn(i)
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / K
    evs = []
    for i in range(K):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn(i)
        b.record(stream)
        evs.append((a, b))
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in evs) / K


def timed_launches(fn, K: int, stream, flush: L2Flush):
    """Device time of each of K calls of fn(i) (ms): back to back with an
    event between consecutive calls, or, with the flush active, a pair of
    events around each call (the flush outside them)."""
    import torch

    torch.cuda.synchronize()
    if not flush.active:
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(K + 1)]
        ev[0].record(stream)
        for i in range(K):
            fn(i)
            ev[i + 1].record(stream)
        torch.cuda.synchronize()
        return [ev[i].elapsed_time(ev[i + 1]) for i in range(K)]
    pairs = []
    for i in range(K):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn(i)
        b.record(stream)
        pairs.append((a, b))
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in pairs]


GROUP_MAX_UNITS = 256          # the library's batched launches: units per launch
GROUP_MAX_NUMEL = 1 << 24      # and the largest unit they take


def model_launches(n_units: int, numel: int, gathers: int) -> int:
    """Kernel launches of one fsdp_step_units call (or captured step) over
    n_units equal units of numel elements whose buffers qualify for batched
    launches when small enough: one update and `gathers` gathers per unit, or
    per group of up to GROUP_MAX_UNITS units (a group of one is a unit)."""
    if numel > GROUP_MAX_NUMEL:
        return n_units * (1 + gathers)
    return -(-n_units // GROUP_MAX_UNITS) * (1 + gathers)


def measure_driver(F, fi, dev, stream, n_units: int = 12, steps: int = 20, numel: int = 0):
    """Host enqueue time and device time per model step of n_units GPT-2 small
    block units (or, with numel, n_units one-tensor units of numel elements
    with the same N, dtypes and hyperparameters; one gather each), stepped by
    a Python loop over the units, by the native step of a model validated
    once (UnitSequence.step: a StepPlan launch), by one fsdp_step_units call
    that validates every unit each time, and by one launch of the step
    captured as a CUDA graph; beside them the planned step with the gather
    fused into the update (`native_fused_gather`, its own byte model: no
    separate gather, the shard and every gathered buffer written by the
    update). Returns (result, timed launches)."""
    import torch

    cfg = fi.CONFIGS["gpt2_small"]
    gdt, odt = fi.torch_dtype(cfg.grad_dtype), fi.torch_dtype(cfg.out_dtype)
    params = [("flat", (numel,))] if numel else cfg.params
    units = []
    for k in range(n_units):
        u = F.FlatParamUnit(params, cfg.world, gdt, odt, device=dev)
        u.load_master([fi.gen_master(cfg, device=dev, seed_base=7000 + k, numel=u.numel)])
        for r in range(cfg.world):
            u.load_grad(r, [fi.gen_grad(cfg, r, 1, device=dev, seed_base=7000 + k, numel=u.numel)])
        units.append(u)
    seq = F.UnitSequence(units)
    t = [0]

    def hp():
        t[0] += 1
        return F.AdamWHParams(cfg.lr, cfg.beta1, cfg.beta2, cfg.eps, cfg.weight_decay, t[0], cfg.grad_scale)

    def python_loop():
        h = hp()
        for u in units:
            u.step(h, gathers=cfg.gathers)

    def native():
        seq.step(hp(), gathers=cfg.gathers)

    def native_unplanned():
        seq.step_unplanned(hp(), gathers=cfg.gathers)

    def native_fused_gather():
        seq.step(hp(), gathers=cfg.gathers, fuse_gather=True)

    graph = seq.capture(gathers=cfg.gathers)

    def captured():
        graph.launch(hp())

    out = {}
    for name, fn in (("python_loop", python_loop), ("native", native), ("native_unplanned", native_unplanned),
                     ("cuda_graph", captured), ("native_fused_gather", native_fused_gather)):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        t0 = time.perf_counter()
        for _ in range(steps):
            fn()
        t1 = time.perf_counter()
        b.record(stream)
        torch.cuda.synchronize()
        out[name] = {"host_enqueue_ms_per_step": round((t1 - t0) * 1e3 / steps, 4),
                     "device_ms_per_step": round(a.elapsed_time(b) / steps, 4)}
    rsa_b, ag_b = seq.step_bytes(cfg.gathers)
    out["bytes_per_step"] = rsa_b + ag_b
    for name in ("native", "native_unplanned", "cuda_graph"):
        out[name + "_GBs"] = round((rsa_b + ag_b) / (out[name]["device_ms_per_step"] * 1e-3) / 1e9, 1)
    out["native_over_cuda_graph"] = round(out["native"]["device_ms_per_step"]
                                          / out["cuda_graph"]["device_ms_per_step"], 3)
    fused_b = sum(u.padded_numel * (u.world * u.grads[0].element_size() + 3 * (4 + 4)
                                     + u.shard_out.element_size() * (1 + len(u.full))) for u in units)
    fused_b += sum(u.padded_numel * u.shard_out.element_size() * (1 + len(u.full)) for u in units) * (cfg.gathers - 1)
    out["native_fused_gather_bytes_per_step"] = fused_b
    out["native_fused_gather_GBs"] = round(fused_b / (out["native_fused_gather"]["device_ms_per_step"] * 1e-3)
                                           / 1e9, 1)
    per_unit = n_units * (1 + cfg.gathers)
    batched = model_launches(n_units, units[0].padded_numel, cfg.gathers)
    fused = seq.launches(gathers=cfg.gathers, fuse_gather=True)
    out["launches_per_step"] = {"python_loop": per_unit, "native": batched, "native_unplanned": batched,
                                "cuda_graph": batched, "native_fused_gather": fused}
    graph.close()
    del seq, units, graph
    torch.cuda.empty_cache()
    return out, steps * (per_unit + 3 * batched + fused)


def max_over_ranks(values, device):
    """Element-wise MAX of per-rank timings over the process group (every rank
    gets the result)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def all_ranks_agree(ok: bool, device) -> bool:
    """True on every rank when every rank says ok (a MIN over the process
    group), so that a leg runs on all ranks or on none."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([1 if ok else 0], device=device, dtype=torch.int32)
    dist.all_reduce(t, op=dist.ReduceOp.MIN)
    return bool(int(t.item()))


# ---------------------------------------------------------------- CPU oracle (baseline / reference arm)

def oracle_sample_run(cfg, n_elems: int, steps: int, warmup: int, time_budget_s: float | None):
    """The oracle as it stands, on an n_elems-element unit with the workload's
    N, dtypes, distributions and gathers. Returns (GB/s, elapsed, steps run, threads)."""
    import numpy as np
    import torch

    import fsdp_inputs as fi
    import oracle as orc

    threads = os.cpu_count() or 1
    orc.set_threads(threads)
    N = cfg.world
    P_pad = orc.padded_numel(n_elems, N)
    S = P_pad // N
    master = orc.flatten_pad([fi.gen_master(cfg, numel=n_elems).numpy()], N)
    m = np.zeros(P_pad, np.float32)
    v = np.zeros(P_pad, np.float32)

    def host_grad(r, t):
        g = fi.gen_grad(cfg, r, t, numel=n_elems)
        arr = g.numpy() if g.dtype == torch.float32 else g.view(torch.int16).numpy().view(np.uint16)
        return orc.flatten_pad([arr], N)

    grads = [host_grad(r, 1) for r in range(N)]
    gsize = 4 if cfg.grad_dtype == "f32" else 2
    osize = 4 if cfg.out_dtype == "f32" else 2
    rsa_b, ag_b = step_bytes(P_pad, N, gsize, osize, cfg.gathers, N)

    def one_step(t):
        hp = orc.hparams(cfg.lr, cfg.beta1, cfg.beta2, cfg.eps, cfg.weight_decay, t, cfg.grad_scale)
        shards, _ = orc.fsdp_step(grads, cfg.grad_dtype, N, master, m, v, cfg.out_dtype, hp)
        pieces = [shards[r * S:(r + 1) * S] for r in range(N)]
        for _ in range(cfg.gathers):
            for _dst in range(N):  # one gathered buffer per emulated rank
                orc.all_gather(pieces, N)

    for t in range(1, warmup + 1):
        one_step(t)
    t0 = time.perf_counter()
    done = 0
    while done < steps or (time_budget_s is not None and time.perf_counter() - t0 < time_budget_s):
        one_step(warmup + done + 1)
        done += 1
        if time_budget_s is None and done >= steps:
            break
    el = time.perf_counter() - t0
    return (rsa_b + ag_b) * done / el / 1e9, el, done, threads


# ---------------------------------------------------------------- our arm

def workload_config(args):
    """The unit to run: a named workload, or (--numel) a one-tensor unit of the
    same N, dtypes, distributions and gathers with fewer parameters."""
    import fsdp_inputs as fi
    cfg = fi.CONFIGS[args.config]
    name = WORKLOAD_NAMES[cfg.name]
    if args.numel:
        cfg = dataclasses.replace(cfg, params=(("flat", (int(args.numel),)),))
        name = f"{name}_numel{int(args.numel)}"
    return cfg, name


class _Run:
    """State shared by the legs of one bench run: the unit, its step counter
    (every launch takes the next step t), the stream, the L2 flush and the
    count of the library's launches inside timed regions."""

    def __init__(self, args, dev, rank, world_size):
        import torch

        import fsdp_inputs as fi
        import sharded_fsdp_reduce_gb300 as F

        self.args, self.dev, self.rank, self.world_size = args, dev, rank, world_size
        self.torch, self.F, self.fi = torch, F, fi
        self.cfg, self.workload = workload_config(args)
        cfg = self.cfg
        self.N = cfg.world
        self.gdt, self.odt = fi.torch_dtype(cfg.grad_dtype), fi.torch_dtype(cfg.out_dtype)
        self.unit = F.FlatParamUnit(cfg.params, self.N, self.gdt, self.odt, device=dev)
        self.P_pad = self.unit.padded_numel
        seed = 100_000 * rank  # each GPU owns a different unit
        self.unit.load_master([fi.gen_master(cfg, device=dev, seed_base=seed)])
        for r in range(self.N):
            self.unit.load_grad(r, [fi.gen_grad(cfg, r, 1, device=dev, seed_base=seed)])
        torch.cuda.synchronize()
        self.rsa_b, self.ag_b = self.unit.step_bytes(cfg.gathers)
        self.stream = torch.cuda.current_stream()
        self.K = args.steps
        self.flush = L2Flush(dev, self.rsa_b)
        self.t = 0
        self.launches = 0
        self.rsa_ms_median = None
        # the timed steps' gathers count their bounded waits that gave up here
        self.wait_timeouts = torch.zeros(1, dtype=torch.int32, device=dev)

    def hp(self, t):
        c = self.cfg
        return self.F.AdamWHParams(c.lr, c.beta1, c.beta2, c.eps, c.weight_decay, t, c.grad_scale)

    def next_hp(self):
        self.t += 1
        return self.hp(self.t)

    def barrier(self):
        if self.world_size > 1:
            import torch.distributed as dist
            dist.barrier()


def time_steps(run: _Run):
    """The timed region: K steps (fused kernel + gathers) after W warm-up
    steps; device time by CUDA events on the launching stream, clocks
    sampled meanwhile. Returns (step ms, fused-kernel ms, clock summary)."""
    torch, unit, cfg, K, flush, stream = run.torch, run.unit, run.cfg, run.K, run.flush, run.stream
    for _ in range(run.args.warmup):
        unit.step(run.next_hp(), gathers=cfg.gathers)
    torch.cuda.synchronize()
    ev = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in range(K)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    run.barrier()
    torch.cuda.synchronize()
    with ClockSampler(run.dev.index if "CUDA_VISIBLE_DEVICES" not in os.environ else 0) as clocks:
        time.sleep(0.25)  # let the sampler start before the timed launches
        start.record(stream)
        for i in range(K):
            hp = run.next_hp()
            flush()
            ev[i][0].record(stream)
            unit.reduce_scatter_adam_cast(hp)
            ev[i][1].record(stream)
            for _ in range(cfg.gathers):
                unit.all_gather(wait_timeouts=run.wait_timeouts)
            ev[i][2].record(stream)
        end.record(stream)
        torch.cuda.synchronize()
    run.barrier()
    if flush.active:  # the flushes between steps are not step time
        step_ms = sum(a.elapsed_time(c) for a, _, c in ev) / K
    else:
        step_ms = start.elapsed_time(end) / K
    rsa_each = [a.elapsed_time(b) for a, b, _ in ev]
    run.rsa_ms_median = statistics.median(rsa_each)
    rsa_ms = sum(rsa_each) / K
    run.launches += K * (1 + cfg.gathers)
    return step_ms, rsa_ms, clocks.summary()


def time_e2e(run: _Run):
    """End to end with the N gradient buffers in pinned host memory: every
    step brings its gradients from the host and reads the step's result
    back, its non-finite-gradient count (the metric a trainer checks every
    step; the gathered parameters stay on the GPU for the next forward), or
    with --e2e-read-params the compute-dtype parameters. Two forms, timed one
    after the other on the same host buffers:

    * copy_pipeline -- the binding's host-buffer step
      (FlatParamUnit.step_from_host): copies to device buffers on a copy
      stream, double-buffered so that a step's copies overlap the previous
      step's kernels;
    * zero_copy -- the C ABI call given the host buffers themselves (its
      gradients are "device or mapped host"): the fused kernel reads them
      over the host link, then the gathers run; no staging buffers.

    Every rank runs it or none does. Returns a dict: per form its ms per
    step, the steps timed, the bytes each way, and the ms of a bare copy of
    the gradients to the device (the host link's own bound); or
    {"unavailable": reason}."""
    torch, F, unit, cfg, args, dev = run.torch, run.F, run.unit, run.cfg, run.args, run.dev
    Ke = max(3, min(args.e2e_steps, run.K))
    unavailable = None
    try:  # N gradient buffers of pinned host memory (13.7 GB for the 70B unit)
        host_grads = [torch.empty(run.P_pad, dtype=run.gdt, pin_memory=True) for _ in range(run.N)]
    except RuntimeError as e:
        host_grads, unavailable = None, "pinned host buffers: " + str(e).splitlines()[0][:160]
    if run.world_size > 1 and not all_ranks_agree(host_grads is not None, dev) and host_grads is not None:
        host_grads, unavailable = None, "another rank could not pin its host buffers"
    if host_grads is None:
        return {"unavailable": unavailable}
    for r in range(run.N):
        host_grads[r].copy_(unit.grads[r])
    counter = torch.zeros(1, dtype=torch.int32, device=dev)
    if args.e2e_read_params:
        host_out, host_nf = torch.empty(run.P_pad, dtype=run.odt, pin_memory=True), None
        d2h = host_out.numel() * host_out.element_size()
    else:
        host_out, host_nf = None, torch.zeros(1, dtype=torch.int32, pin_memory=True)
        d2h = host_nf.numel() * host_nf.element_size()
    h2d = sum(g.numel() * g.element_size() for g in host_grads)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def pipeline_step():
        unit.step_from_host(host_grads, host_out, run.next_hp(), gathers=cfg.gathers, nonfinite_count=counter,
                            host_nonfinite=host_nf)

    def zero_copy_step():
        # the result is read back right after the update, so that it travels
        # while the gathers run
        hp = run.next_hp()
        if host_nf is not None:
            counter.zero_()
        F.fsdp_reduce_scatter_adam_cast(host_grads, unit.master, unit.exp_avg, unit.exp_avg_sq, unit.shard_out,
                                        hp, nonfinite_count=counter)
        if host_nf is not None:
            host_nf.copy_(counter, non_blocking=True)
        else:
            host_out.copy_(unit.shard_out, non_blocking=True)
        for _ in range(cfg.gathers):
            unit.all_gather()

    out = {"steps": Ke, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}
    for name, fn in (("copy_pipeline", pipeline_step), ("zero_copy", zero_copy_step)):
        fn()  # sets up the streams, warms the host mappings
        torch.cuda.synchronize()
        run.barrier()
        e0.record(run.stream)
        for _ in range(Ke):
            fn()
        e1.record(run.stream)
        torch.cuda.synchronize()
        out[name + "_ms"] = e0.elapsed_time(e1) / Ke
        if host_nf is not None and int(host_nf.item()) != 0:
            raise RuntimeError("e2e steps reported non-finite gradients")
        run.launches += Ke * (1 + cfg.gathers)
    # the host link's own bound, after the timed regions: the bare copy of the
    # same pinned gradients into the unit's gradient buffers (identical bytes)
    bare = []
    for _ in range(2):
        e0.record(run.stream)
        with torch.cuda.stream(run.stream):
            for r in range(run.N):
                unit.grads[r].copy_(host_grads[r], non_blocking=True)
        e1.record(run.stream)
        torch.cuda.synchronize()
        bare.append(e0.elapsed_time(e1))
    out["bare_h2d_ms"] = sum(bare) / len(bare)
    return out


def time_fused_gather_variants(run: _Run):
    """Two forms of the step with the gather fused into the update kernel,
    each on its own algorithmic bytes:

    * fused_gather -- the first gather written by the update kernel (the
      shard and every gathered buffer stored from registers, shard_out not
      read back), the second a separate gather: N*grad + 24 + (1 + n_full)*out
      bytes per element, plus (gathers - 1) * (1 + n_full) * out;
    * no_reshard_fused -- one fused gather kept for forward and backward,
      and no compute-dtype shard written (shard_out NULL: the gathered
      parameters are what is kept): N*grad + 24 + n_full*out."""
    F, unit, K, P, N = run.F, run.unit, run.K, run.P_pad, run.N
    gs, os_, nfull = unit.grads[0].element_size(), unit.shard_out.element_size(), len(unit.full)
    update = P * (N * gs + 3 * (4 + 4))
    g = run.cfg.gathers

    def fused(t):
        unit.step(run.hp(t), gathers=g, fuse_gather=True)

    def no_reshard(t):
        F.fsdp_reduce_scatter_adam_cast_gather(unit.grads, unit.master, unit.exp_avg, unit.exp_avg_sq, None,
                                               unit.full, run.hp(t))

    forms = (("fused_gather", fused, g, update + P * os_ * (1 + nfull) * g),
             ("no_reshard_fused", no_reshard, 1, update + P * os_ * nfull))
    variants = {}
    for vname, fn, launches, nbytes in forms:
        for _ in range(3):
            run.t += 1
            fn(run.t)
        t0 = run.t
        vms = timed_calls(lambda i, fn=fn: fn(t0 + 1 + i), K, run.stream, run.flush)
        run.t += K
        run.launches += K * launches
        variants[vname] = {"gathers_per_step": 1 if vname == "no_reshard_fused" else g,
                           "launches_per_step": launches, "ms_per_step": round(vms, 4), "bytes_per_step": nbytes}
    return variants


def time_variant_kernels(run: _Run):
    """The variant steps' kernels on the same unit, each on its own byte
    model: N*grad + (1 + states)*(read + write) + out, each optimizer from its
    own zero state."""
    torch, F, unit, cfg, dev, P, N = run.torch, run.F, run.unit, run.cfg, run.dev, run.P_pad, run.N
    gb = unit.grads[0].element_size()
    low = [unit.master.to(torch.bfloat16), torch.zeros(P, dtype=torch.bfloat16, device=dev),
           torch.zeros(P, dtype=torch.bfloat16, device=dev)]
    vsets = {
        "adamw_grad_dtype_reduce": ("adamw", True, unit.master, unit.exp_avg, unit.exp_avg_sq, unit.shard_out),
        "adamw_bf16_state": ("adamw", False, low[0], low[1], low[2], None),
        "sgd_momentum": ("sgd", False, unit.master, unit.exp_avg, None, unit.shard_out),
        "adamax": ("adamax", False, unit.master, unit.exp_avg, unit.exp_avg_sq, unit.shard_out),
        "adadelta": ("adadelta", False, unit.master, unit.exp_avg, unit.exp_avg_sq, unit.shard_out),
    }
    kernels = {}
    for vname, (opt, lowp, prm, s0, s1, out) in vsets.items():
        ss = prm.element_size()
        nstates = 1 + (s0 is not None) + (s1 is not None)
        nbytes = P * (N * gb + nstates * 2 * ss + (out.element_size() if out is not None else 0))
        lrv = 1.0 if opt == "adadelta" else cfg.lr
        for st in (s0, s1):
            if st is not None:
                st.zero_()

        def launch(tt, opt=opt, lowp=lowp, prm=prm, s0=s0, s1=s1, out=out, lrv=lrv):
            F.fsdp_reduce_scatter_step(unit.grads, prm, s0, s1, out,
                                       F.StepConfig(opt, lrv, cfg.beta1, cfg.beta2, cfg.eps, cfg.weight_decay,
                                                    tt, cfg.grad_scale, reduce_dtype=run.gdt if lowp else None))
        for i in range(3):
            launch(i + 1)
        kms = timed_calls(lambda i, launch=launch: launch(i + 4), run.K, run.stream, run.flush)
        run.launches += run.K
        kernels[vname] = {"ms": round(kms, 4), "bytes_per_launch": nbytes,
                          "achieved_GBs": round(nbytes / (kms * 1e-3) / 1e9, 1)}
    return kernels


def time_offload(run: _Run, rsa_ms: float):
    """The offload mode: master, m and v in pinned host memory, updated in
    place by the same fused kernel over the host link (12 B read and 12 B
    written per element there; gradients and the shard stay in HBM)."""
    torch, F, unit, P = run.torch, run.F, run.unit, run.P_pad
    try:
        hstate = [torch.zeros(P, dtype=torch.float32, pin_memory=True) for _ in range(3)]
    except RuntimeError as e:  # not enough page-locked host memory
        return {"unavailable": str(e).splitlines()[0][:200]}
    hstate[0].copy_(unit.master)
    torch.cuda.synchronize()

    def launch(i):
        F.fsdp_reduce_scatter_adam_cast(unit.grads, *hstate, unit.shard_out, run.hp(i + 1))

    for i in range(3):
        launch(i)
    Ko = max(3, min(run.K, 5))
    oms = timed_calls(lambda i: launch(i + 3), Ko, run.stream, run.flush)
    run.launches += Ko
    link_b = P * 3 * (4 + 4)
    hbm_b = P * (run.N * unit.grads[0].element_size() + unit.shard_out.element_size())
    return {"ms": round(oms, 3), "launches": Ko, "host_link_bytes_per_launch": link_b,
            "hbm_bytes_per_launch": hbm_b,
            "host_link_GBs": round(link_b / (oms * 1e-3) / 1e9, 1),
            "host_link_GBs_per_direction": round(link_b / 2 / (oms * 1e-3) / 1e9, 1),
            "slowdown_vs_device_state": round(oms / rsa_ms, 2)}


PER_CONFIG = ("gpt3_13b", "gpt2_large", "gpt2_small")
PER_CONFIG_MAX_LAUNCHES = 5000


def time_per_config(run: _Run, peak: float):
    """The fused kernel alone on each other block unit of the set (GPT-3
    13B, GPT-2 Large, GPT-2 small), built one at a time after the run's own
    unit is freed: CUDA events around every launch (L2 flushed before each
    launch of a unit that moves less than 16x L2), enough launches for about
    --per-config-seconds of device time (at least --steps), so that the
    clocks are sampled under load. Returns {workload: record}."""
    torch, F, fi, dev, stream = run.torch, run.F, run.fi, run.dev, run.stream
    out = {}
    for name in PER_CONFIG:
        if name == run.cfg.name:
            continue
        cfg = fi.CONFIGS[name]
        workload = WORKLOAD_NAMES[name]
        unit = F.FlatParamUnit(cfg.params, cfg.world, fi.torch_dtype(cfg.grad_dtype), fi.torch_dtype(cfg.out_dtype),
                               device=dev)
        unit.load_master([fi.gen_master(cfg, device=dev)])
        for r in range(cfg.world):
            unit.load_grad(r, [fi.gen_grad(cfg, r, 1, device=dev)])
        P = unit.padded_numel
        rsa_b, _ = unit.step_bytes(cfg.gathers)
        flush = L2Flush(dev, rsa_b)

        def launch(t, unit=unit, cfg=cfg):
            unit.reduce_scatter_adam_cast(F.AdamWHParams(cfg.lr, cfg.beta1, cfg.beta2, cfg.eps, cfg.weight_decay,
                                                         t, cfg.grad_scale))

        warm = timed_launches(lambda i: launch(i + 1), 3, stream, flush)
        want = int(run.args.per_config_seconds * 1e3 / max(min(warm), 1e-3)) + 1
        K = min(PER_CONFIG_MAX_LAUNCHES, max(run.K, want))
        torch.cuda.synchronize()
        with ClockSampler(dev.index if "CUDA_VISIBLE_DEVICES" not in os.environ else 0) as clocks:
            time.sleep(0.25)  # let the sampler start before the timed launches
            each = timed_launches(lambda i: launch(4 + i), K, stream, flush)
        run.launches += K  # the timed launches (the three warm-up launches are not counted)
        mean = sum(each) / K
        achieved = rsa_b / (mean * 1e-3) / 1e9
        out[workload] = {
            "padded_numel": P, "world": cfg.world, "grad_dtype": cfg.grad_dtype, "out_dtype": cfg.out_dtype,
            "launches": K, "ms": round(mean, 5), "ms_median": round(statistics.median(each), 5),
            "bytes_per_launch": rsa_b, "achieved_GBs": round(achieved, 1),
            "frac": round(achieved / peak, 4), "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
            "traffic": recorded_traffic(workload, P), "l2": flush.describe(), "clocks": clocks.summary(),
        }
        del unit, flush
        torch.cuda.empty_cache()
    return out


def e2e_record(e2e: dict, total_bytes: int, args) -> dict:
    """The bench line's e2e: the faster of the two host-buffer forms, the
    other beside it, each with its share of the bare host-to-device copy."""
    if "unavailable" in e2e:
        return {"unavailable": e2e["unavailable"]}
    forms = ("copy_pipeline", "zero_copy")
    best = min(forms, key=lambda k: e2e[k + "_ms"])
    other = forms[1 - forms.index(best)]
    bare = e2e["bare_h2d_ms"]

    def form(k):
        ms = e2e[k + "_ms"]
        return {"value": round(total_bytes / (ms * 1e-3) / 1e9, 2), "ms_per_step": round(ms, 3),
                "bare_h2d_over_e2e": round(bare / ms, 4)}

    rec = {"unit": "GB/s", **form(best), "path": best, "steps": e2e["steps"],
           "h2d_bytes_per_step": e2e["h2d_bytes_per_step"], "d2h_bytes_per_step": e2e["d2h_bytes_per_step"],
           "d2h": "compute-dtype parameters" if args.e2e_read_params else "non-finite gradient count",
           "bare_h2d_ms": round(bare, 3), "bare_h2d_GBs": round(e2e["h2d_bytes_per_step"] / (bare * 1e-3) / 1e9, 1)}
    rec[other] = form(other)
    return rec


def run_ours(args):
    import torch
    import torch.distributed as dist

    import sharded_fsdp_reduce_gb300 as F
    from sharded_fsdp_reduce_gb300 import build as _build

    rank, local_rank, world_size = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (GB300); there is no CPU path")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world_size > 1:
        dist.init_process_group("nccl", device_id=dev)
    if rank == 0:  # one build (a no-op when up to date); the other ranks wait for it
        _build.build()
    if world_size > 1:
        dist.barrier()
    F._lib.load()

    run = _Run(args, dev, rank, world_size)
    step_ms, rsa_ms, clocks = time_steps(run)
    e2e = time_e2e(run)
    variants = time_fused_gather_variants(run) if not args.no_variants else {}
    kernels = time_variant_kernels(run) if not args.no_variants else {}
    offload = None
    if not args.no_variants and not args.no_offload and world_size == 1:  # pins 12 B/param of host memory
        offload = time_offload(run, rsa_ms)
    driver = small_units = None
    if not args.no_variants and not args.no_driver and world_size == 1:
        driver, n_launch = measure_driver(F, run.fi, dev, run.stream)
        run.launches += n_launch
        small_units, n_launch = measure_driver(F, run.fi, dev, run.stream, n_units=200, numel=50000)
        run.launches += n_launch

    if int(run.wait_timeouts.item()) != 0:
        raise RuntimeError("a bounded wait of the timed steps' gathers gave up: their results are not trustworthy")
    if world_size > 1:
        step_ms, rsa_ms = max_over_ranks([step_ms, rsa_ms], dev)
        if "unavailable" not in e2e:
            e2e["copy_pipeline_ms"], e2e["zero_copy_ms"] = max_over_ranks(
                [e2e["copy_pipeline_ms"], e2e["zero_copy_ms"]], dev)
        for v in variants.values():
            v["ms_per_step"] = max_over_ranks([v["ms_per_step"]], dev)[0]

    if rank != 0:
        if world_size > 1:
            dist.barrier()
            dist.destroy_process_group()
        return

    unit, cfg, N, P_pad, rsa_b, ag_b = run.unit, run.cfg, run.N, run.P_pad, run.rsa_b, run.ag_b
    workload, flush = run.workload, run.flush
    peak, peak_kind = measured_peak()
    achieved = rsa_b / (rsa_ms * 1e-3) / 1e9
    traffic = recorded_traffic(workload, P_pad)
    total_bytes = (rsa_b + ag_b) * world_size
    unit_numel = unit.numel
    per_config = None
    if world_size == 1 and not args.no_per_config:
        run.unit = unit = None  # the other block units are built after this one is freed
        torch.cuda.empty_cache()
        per_config = time_per_config(run, peak)
    result = {
        "metric": METRIC,
        "value": round(total_bytes / (step_ms * 1e-3) / 1e9, 2),
        "unit": "GB/s",
        "n_gpus": world_size,
        "steps": run.K,
        "warmup": args.warmup,
        "ms_per_step": round(step_ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded; no dataset or weights)",
        "config": {
            "workload": workload, "params": unit_numel, "padded_numel": P_pad, "world": N,
            "grad_dtype": cfg.grad_dtype, "out_dtype": cfg.out_dtype, "gathers_per_step": cfg.gathers,
            "bytes_per_step": rsa_b + ag_b, "fused_bytes_per_launch": rsa_b,
            "l2": flush.describe(),
            "units_per_gpu": 1,
        },
        "params_per_s": round(P_pad * world_size / (step_ms * 1e-3), 1),
        "fused_params_per_s": round(P_pad / (rsa_ms * 1e-3), 1),
        "roofline": {
            "bound": "hbm", "kernel": "rsa_kernel (fused reduce-scatter + AdamW + cast)",
            "achieved": round(achieved, 1), "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "traffic": traffic,
            "fused_ms": round(rsa_ms, 4), "fused_ms_median": round(run.rsa_ms_median, 4),
            "nominal_peak": NOMINAL_HBM_GBS, "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
        },
        "e2e": e2e_record(e2e, total_bytes, args),
        "gpu_launches": run.launches,
        "wait_timeouts": int(run.wait_timeouts.item()),
        "variants": {k: dict(v, value=round(world_size * v["bytes_per_step"] / (v["ms_per_step"] * 1e-3) / 1e9, 2),
                             frac=round(v["bytes_per_step"] / (v["ms_per_step"] * 1e-3) / 1e9 / peak, 4))
                     for k, v in variants.items()},
        "variant_kernels": {k: dict(v, frac=round(v["achieved_GBs"] / peak, 4)) for k, v in kernels.items()},
        "offload_state_on_host": offload,
        "driver_gpt2_small_model_12_units": driver,
        "driver_model_200_units_of_50k": small_units,
        "per_config": per_config,
        "clocks": clocks,
    }
    if world_size == 1 and not args.no_cpu_baseline:
        n_s = min(unit_numel, args.cpu_sample)
        gbs, el, done, threads = oracle_sample_run(cfg, n_s, 1, 1, args.cpu_seconds)
        result["cpu_baseline"] = {
            "value": round(gbs, 3), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{done} steps of a {n_s}-element unit with the workload's N, dtypes, distributions and "
                      f"all-gathers ({el:.1f} s)", **host_info()}
    print(json.dumps(result), flush=True)
    if world_size > 1:
        dist.barrier()
        dist.destroy_process_group()


# ---------------------------------------------------------------- reference arm (the oracle)

def run_reference(args):
    import fsdp_inputs as fi

    rank, _, world_size = dist_env()
    if rank != 0:
        return  # the CPU oracle runs on rank 0 only
    cfg, workload = workload_config(args)
    n_s = min(fi.unit_numel(cfg), args.ref_sample)
    gbs, el, done, threads = oracle_sample_run(cfg, n_s, args.steps, args.warmup, None)
    sample = f"each step: a {n_s}-element unit with the workload's N, dtypes, distributions and all-gathers"
    print(json.dumps({
        "impl": "reference",
        "metric": METRIC, "value": round(gbs, 3), "unit": "GB/s", "n_gpus": world_size,
        "steps": done, "warmup": args.warmup, "ms_per_step": round(el / done * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded; no dataset or weights)",
        "config": {"workload": workload, "world": cfg.world, "grad_dtype": cfg.grad_dtype,
                   "out_dtype": cfg.out_dtype, "gathers_per_step": cfg.gathers, "sample_numel": n_s},
        "cpu_baseline": {"value": round(gbs, 3), "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": sample, **host_info()},
        "e2e": {"value": round(gbs, 3), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="llama70b", choices=sorted(WORKLOAD_NAMES))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--numel", type=int, default=0,
                    help="replace the unit by one flat tensor of this many parameters (small profiling cases)")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-read-params", action="store_true",
                    help="e2e reads the compute-dtype parameters back each step instead of the step's metric")
    ap.add_argument("--no-variants", action="store_true", help="skip the fused-gather variant timings")
    ap.add_argument("--no-driver", action="store_true",
                    help="skip the per-unit driver timing on a 12-unit GPT-2 small model")
    ap.add_argument("--no-offload", action="store_true",
                    help="skip the offload-mode timing (state in pinned host memory)")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the fused kernel's timing on the other block units (13B, GPT-2 Large, GPT-2 small)")
    ap.add_argument("--per-config-seconds", type=float, default=0.6,
                    help="device time of each of those units' timed launches (clocks are sampled meanwhile)")
    ap.add_argument("--cpu-sample", type=int, default=1 << 24, help="elements in the CPU-baseline sample")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="CPU-baseline time budget")
    ap.add_argument("--ref-sample", type=int, default=1 << 22, help="elements per reference-arm step")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        raise SystemExit("--warmup must be at least 3")
    _, _, world_size = dist_env()
    if args.gpus != world_size:
        raise SystemExit(f"--gpus {args.gpus} but WORLD_SIZE={world_size}: launch N>1 with torchrun")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
