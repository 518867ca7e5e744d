#!/usr/bin/env python
"""Benchmark of the RMSNorm hot path on GB300: achieved HBM GB/s (and the
fraction of the measured HBM copy bandwidth) of the fused add-RMSNorm forward
and the RMSNorm VJP.

One step = the prefill workload, bf16, rows 16384:
    fwd(D=4096, with residual); fwd(D=8192, with residual);
    vjp(D=4096, x = new_residual); vjp(D=8192, x = new_residual)
(each VJP is its main kernel plus the gw stage-2 kernel).  The order puts at
least one other launch of >= 400 MB between a tensor's write and its re-read,
and every operand (134 or 268 MB) is larger than the 129 MB L2, so each step
streams from HBM.  Algorithmic bytes: forward 4*R*D*2 + D*2, VJP
3*R*D*2 + D*2 + 4*D (the gw partials are scratch and not counted).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  N > 1 runs N independent replicas of the step
(torchrun, one process per GPU): the path has no exchange step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import torch
import torch.distributed as dist

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "achieved HBM GB/s and % of GB300 peak for add-RMSNorm fwd and RMSNorm VJP"
UNIT = "GB/s"
ROWS = 16384
DS = (4096, 8192)
ITEM = 2  # bf16
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0  # the ~8 TB/s HBM3e figure the target is quoted against


def fwd_bytes(rows, D, residual=True, s=ITEM):
    return (4 if residual else 2) * rows * D * s + D * s


def vjp_bytes(rows, D, s=ITEM):
    return 3 * rows * D * s + D * s + 4 * D


def gate_bytes(rows, d, s=ITEM):
    """Gated activation: 2d values read, d written per row."""
    return 3 * rows * d * s


def rope_bytes(T, Hq, Hkv, Dh, s=ITEM):
    """Rope + append: q read and written, k and v read and written once."""
    return (2 * Hq + 4 * Hkv) * T * Dh * s + 16 * T


def fused_vjp_bytes(rows, D, s=ITEM):
    """The two-output op's VJP: h, g_out and g_residual read, g_h written."""
    return 4 * rows * D * s + D * s + 4 * D


STEP_BYTES = sum(fwd_bytes(ROWS, D) + vjp_bytes(ROWS, D) for D in DS)
OPS = [("fwd_d%d" % D, D) for D in DS] + [("vjp_d%d" % D, D) for D in DS]
OP_BYTES = {"fwd_d%d" % D: fwd_bytes(ROWS, D) for D in DS}
OP_BYTES.update({"vjp_d%d" % D: vjp_bytes(ROWS, D) for D in DS})
KERNELS_PER_STEP = 6  # two forward kernels, two VJP main kernels, two gw reductions

# The POC workload (fp16, rows 8192, D 4096, x, w, g ~ U(0,1), eps 1e-5): its
# VJP and the forward without a residual, timed per op beside the step.
C3_ROWS, C3_D, C3_ITEM = 8192, 4096, 2
C3_OPS = {"c3_vjp_f16": vjp_bytes(C3_ROWS, C3_D, C3_ITEM),
          "c3_fwd_nores_f16": fwd_bytes(C3_ROWS, C3_D, residual=False, s=C3_ITEM)}

CONFIG = {
    "workload": "prefill fused add-RMSNorm fwd (with residual) + RMSNorm VJP on new_residual, "
                "rows 16384, D 4096 and 8192, bf16, eps 1e-6, weight_bias 0",
    "rows": ROWS,
    "D": list(DS),
    "l2": "inputs larger than L2: every operand is 134-268 MB vs 129 MB L2; no operand is "
          "re-read from L2 between steps",
    "parallelism": "replicas",
}


# ---------------------------------------------------------------------------
# ranks
# ---------------------------------------------------------------------------

def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and not dist.is_initialized():
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return rank, world, local


def barrier():
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def max_over_ranks(value: float, device) -> float:
    """Largest value over all ranks (the value itself without a process group)."""
    if not (dist.is_available() and dist.is_initialized()):
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

CLOCK_FIELDS = ("pci.bus_id,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
REASON_NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")


class ClockSampler:
    def __init__(self, device_index: int):
        self.samples = []
        self.proc = None
        self.bus = None
        try:
            props = torch.cuda.get_device_properties(device_index)
            self.bus = "%08X:%02X:%02X" % (props.pci_domain_id, props.pci_bus_id, props.pci_device_id)
        except Exception:
            self.bus = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + CLOCK_FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        threading.Thread(target=self._read, daemon=True).start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [f.strip() for f in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        rows = [(t, f) for (t, f) in self.samples if len(f) >= 9]
        buses = {f[0] for _, f in rows}
        if len(buses) > 1 and self.bus:
            rows = [(t, f) for (t, f) in rows if f[0].upper().startswith(self.bus.upper())] or rows
        window = [f for (t, f) in rows if t0 - 0.1 <= t <= t1 + 0.1]
        use = window or [f for _, f in rows]
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [num(f[1]) for f in use if num(f[1]) is not None]
        mx = [num(f[2]) for f in use if num(f[2]) is not None]
        reasons = set()
        for f in use:
            for name, flag in zip(REASON_NAMES, f[5:9]):
                if flag.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(use),
                "in_timed_window": bool(window)}


# ---------------------------------------------------------------------------
# the measured path
# ---------------------------------------------------------------------------

def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, copy)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# Files that define the staged kernels and their launch plans: a change to any
# of them invalidates recorded DRAM traffic.
STAGED_SOURCES = ("common.cuh", "plan.h", "planner.h", "launch_util.h", "launch_staged.cuh",
                  "staged.cuh", "staged_bf16.cu", "staged_f16.cu")


def source_hash(files=STAGED_SOURCES):
    h = hashlib.sha256()
    pkg = os.path.join(ROOT, "rmsnorm_fwd_bwd_add_gb300", "csrc")
    for name in files:
        with open(os.path.join(pkg, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic_prefill_r16384_bf16.md")


def recorded_traffic(op):
    """DRAM bytes (read + write) per launch of `op`'s main kernel from the
    committed ncu summary, if it was taken on the current staged-kernel
    sources; otherwise None.  The summary's lines `staged sources: <hash>` and
    `<op>: <bytes>` are read."""
    try:
        with open(TRAFFIC_FILE) as f:
            text = f.read()
    except OSError:
        return None
    rec = {}
    for line in text.splitlines():
        line = line.strip().strip("`")
        if ":" in line:
            k, v = line.split(":", 1)
            rec[k.strip()] = v.strip()
    if rec.get("staged sources") != source_hash():
        return None
    try:
        return int(rec[op])
    except (KeyError, ValueError):
        return None


def device_inputs(device):
    """The workload drawn on the GPU (seeded CUDA generator, same
    distributions as the tests' CPU draws): fast at any number of ranks."""
    from rmsnorm_fwd_bwd_add_gb300 import workloads as W
    return {D: W.config4_on_device(D, device, ROWS) for D in DS}


def to_host(cases, rows=None):
    """Host copies of the cases (all rows, or the first `rows`)."""
    import copy
    out = {}
    for D, c in cases.items():
        h = copy.copy(c)
        sl = slice(None) if rows is None else slice(0, rows)
        h.x, h.residual, h.g = (t[sl].cpu() for t in (c.x, c.residual, c.g))
        h.w = c.w.cpu()
        h.rows = h.x.shape[0]
        out[D] = h
    return out


class Step:
    """Device buffers for one step and the calls that make it."""

    def __init__(self, cases, device):
        import rmsnorm_fwd_bwd_add_gb300 as rn
        self.rn = rn
        self.dev = device
        self.t = {}
        for D, c in cases.items():
            self.t[D] = dict(
                x=c.x, res=c.residual, w=c.w, g=c.g,
                out=torch.empty_like(c.x, device=device), nr=torch.empty_like(c.x, device=device),
                gx=torch.empty_like(c.x, device=device),
                gw=torch.empty(D, dtype=torch.float32, device=device))
        self.eps = {D: c.eps for D, c in cases.items()}

    def op(self, name, D):
        t = self.t[D]
        if name.startswith("fwd"):
            self.rn.rmsnorm_fwd(t["x"], t["w"], self.eps[D], 0.0, t["res"], out=t["out"],
                                new_residual=t["nr"])
        else:
            self.rn.rmsnorm_vjp(t["nr"], t["w"], t["g"], self.eps[D], 0.0, gx=t["gx"], gw=t["gw"])

    def run(self):
        for name, D in OPS:
            self.op(name, D)


PROBE_EVERY = 8  # steps between per-op event probes


def time_device(step: Step, steps: int, warmup: int, sampler: ClockSampler):
    """Times `steps` steps on the launching stream.  Every PROBE_EVERY-th step
    brackets each op with CUDA events (for the per-op durations behind the
    roofline); the other steps run back to back exactly as a user's loop
    would, so the library's launches overlap their predecessors' tails."""
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        step.run()
    torch.cuda.synchronize()
    probes = [k for k in range(steps) if k % PROBE_EVERY == 0]
    ev = {name: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                 for _ in probes] for name, _ in OPS}
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    start.record(stream)
    pi = 0
    for k in range(steps):
        if k % PROBE_EVERY == 0:
            for name, D in OPS:
                a, b = ev[name][pi]
                a.record(stream)
                step.op(name, D)
                b.record(stream)
            pi += 1
        else:
            step.run()
    end.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    barrier()
    total_ms = start.elapsed_time(end)
    per_op_us = {name: 1e3 * statistics.mean(a.elapsed_time(b) for a, b in ev[name])
                 for name, _ in OPS}
    return total_ms, per_op_us, sampler.summary(t0, t1)


def time_sustained(call, sets, reps=20, min_ms=1.0, warmup=10):
    """µs per call under the sustained protocol: calls back to back over the
    rotating `sets` (together at least twice the L2, so no call finds its
    operands in L2), N calls per repetition (a multiple of len(sets), at least
    `min_ms` of work), CUDA events on the launching stream, median of `reps`
    repetitions.  Consecutive calls overlap their launch and prologue with the
    previous call's tail, as they do in a user's loop."""
    K = len(sets)
    for i in range(max(warmup, K)):
        call(sets[i % K])
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for i in range(K):
        call(sets[i])
    b.record()
    torch.cuda.synchronize()
    est_us = max(1.0, 1e3 * a.elapsed_time(b) / K)
    calls = K * max(1, -(-int(1e3 * min_ms / est_us) // K))
    times = []
    for _ in range(reps):
        a.record()
        for i in range(calls):
            call(sets[i % K])
        b.record()
        torch.cuda.synchronize()
        times.append(1e3 * a.elapsed_time(b) / calls)
    return statistics.median(times)


def sets_for_l2(set_bytes: int, device) -> int:
    """Rotating sets needed for at least twice the device's L2 in total."""
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    return max(1, -(-2 * l2 // set_bytes))


def sustained_ops(step: "Step", device):
    """Per-op µs per call under the sustained protocol for the step's four ops
    (their own buffers: each op's operands are 0.4-1.1 GB, one set is already
    more than twice the L2) and for the POC workload's VJP and forward without
    a residual (fp16 8192 x 4096, two rotating sets)."""
    import rmsnorm_fwd_bwd_add_gb300 as rn
    from rmsnorm_fwd_bwd_add_gb300 import workloads as W
    us = {}
    for name, D in OPS:
        t = step.t[D]
        n_sets = sets_for_l2(OP_BYTES[name], device)
        sets = [t] + [{k: torch.empty_like(v) if v.dim() == 2 else v for k, v in t.items()}
                      for _ in range(n_sets - 1)]
        for s_ in sets[1:]:
            for k in ("x", "res", "g", "nr"):
                s_[k].copy_(t[k])
        if name.startswith("fwd"):
            def call(s_, D=D):
                rn.rmsnorm_fwd(s_["x"], s_["w"], step.eps[D], 0.0, s_["res"], out=s_["out"],
                               new_residual=s_["nr"])
        else:
            def call(s_, D=D):
                rn.rmsnorm_vjp(s_["nr"], s_["w"], s_["g"], step.eps[D], 0.0, gx=s_["gx"],
                               gw=s_["gw"])
        us[name] = time_sustained(call, sets)
        del sets
    c = W.config3(C3_ROWS, C3_D)
    x, w, g = c.x.to(device), c.w.to(device), c.g.to(device)
    for name, nbytes in C3_OPS.items():
        n_sets = sets_for_l2(nbytes, device)
        sets = [dict(x=x.clone(), g=g.clone(), out=torch.empty_like(x),
                     gw=torch.empty(C3_D, dtype=torch.float32, device=device))
                for _ in range(n_sets)]
        if name.startswith("c3_vjp"):
            def call(s_):
                rn.rmsnorm_vjp(s_["x"], w, s_["g"], c.eps, 0.0, gx=s_["out"], gw=s_["gw"])
        else:
            def call(s_):
                rn.rmsnorm_fwd(s_["x"], w, c.eps, 0.0, out=s_["out"])
        us[name] = time_sustained(call, sets)
        del sets
    return us


def bind_to_gpu_numa_node(device_index: int) -> None:
    """Run this process on the CPUs next to the GPU (sysfs local_cpulist of
    its PCI function) so that pinned host buffers are allocated in the GPU's
    NUMA node; a no-op where the information is missing."""
    try:
        props = torch.cuda.get_device_properties(device_index)
        bus = "%04x:%02x:%02x.0" % (props.pci_domain_id, props.pci_bus_id, props.pci_device_id)
        with open("/sys/bus/pci/devices/%s/local_cpulist" % bus) as f:
            text = f.read().strip()
        cpus = set()
        for part in text.split(","):
            lo, _, hi = part.partition("-")
            cpus.update(range(int(lo), int(hi or lo) + 1))
        cpus &= os.sched_getaffinity(0)
        if cpus:
            os.sched_setaffinity(0, cpus)
    except Exception:
        pass


def time_e2e(cases, device, steps: int, warmup: int):
    """The step through the public Python API with pinned host buffers: every
    step copies its inputs (x, residual, g, w of both D) host->device and its
    results (out, new_residual, gx, gw) device->host.  Copies run on their own
    streams with two device buffer sets, so step k's upload, step k-1's
    compute and step k-2's download overlap, as a user streaming batches
    would arrange it; the timed region ends when the last download is done."""
    import rmsnorm_fwd_bwd_add_gb300 as rn
    bind_to_gpu_numa_node(device.index if device.index is not None else 0)
    ins = ("x", "res", "g", "w")
    outs = ("out", "nr", "gx", "gw")
    host = {}
    for D, c in cases.items():
        host[D] = dict(x=c.x.pin_memory(), res=c.residual.pin_memory(), g=c.g.pin_memory(),
                       w=c.w.pin_memory(),
                       out=torch.empty_like(c.x).pin_memory(), nr=torch.empty_like(c.x).pin_memory(),
                       gx=torch.empty_like(c.x).pin_memory(),
                       gw=torch.empty(D, dtype=torch.float32).pin_memory())
    sets = [{D: {k: torch.empty_like(v, device=device) for k, v in host[D].items()} for D in DS}
            for _ in range(2)]
    h2d = sum(host[D][k].numel() * host[D][k].element_size() for D in DS for k in ins)
    d2h = sum(host[D][k].numel() * host[D][k].element_size() for D in DS for k in outs)
    compute = torch.cuda.current_stream(device)
    up = torch.cuda.Stream(device)
    down = torch.cuda.Stream(device)
    ev = [dict(inputs=torch.cuda.Event(), computed=torch.cuda.Event(), fetched=torch.cuda.Event())
          for _ in range(2)]

    def one(k):
        s, e = sets[k % 2], ev[k % 2]
        with torch.cuda.stream(up):
            up.wait_event(e["computed"])  # step k-2 is done reading this set's inputs
            for D in DS:
                for name in ins:
                    s[D][name].copy_(host[D][name], non_blocking=True)
            e["inputs"].record(up)
        compute.wait_event(e["inputs"])
        compute.wait_event(e["fetched"])  # step k-2's results have left this set
        for D in DS:
            d = s[D]
            rn.rmsnorm_fwd(d["x"], d["w"], cases[D].eps, 0.0, d["res"], out=d["out"],
                           new_residual=d["nr"])
        for D in DS:
            d = s[D]
            rn.rmsnorm_vjp(d["nr"], d["w"], d["g"], cases[D].eps, 0.0, gx=d["gx"], gw=d["gw"])
        e["computed"].record(compute)
        with torch.cuda.stream(down):
            down.wait_event(e["computed"])
            for D in DS:
                for name in outs:
                    host[D][name].copy_(s[D][name], non_blocking=True)
            e["fetched"].record(down)

    for k in range(warmup):
        one(k)
    torch.cuda.synchronize()
    barrier()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(compute)
    for k in range(steps):
        one(warmup + k)
    compute.wait_stream(down)
    b.record(compute)
    torch.cuda.synchronize()
    ms = max_over_ranks(a.elapsed_time(b), device)
    return ms / steps, h2d, d2h


# ---------------------------------------------------------------------------
# the oracle on the host cores (reported baseline and the reference arm)
# ---------------------------------------------------------------------------

def oracle_sample(cases, rows):
    """float64 copies of the first `rows` rows of each D of the workload."""
    import numpy as np
    out = {}
    for D, c in cases.items():
        def f(t):
            return np.ascontiguousarray(t[:rows].to(torch.float64).numpy())
        out[D] = dict(x=f(c.x), res=f(c.residual), g=f(c.g),
                      w=c.w.to(torch.float64).numpy(), eps=c.eps)
    return out


def host_cores() -> int:
    """CPU cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _oracle_block(s, lo, hi):
    import oracle
    _, h = oracle.fwd(s["x"][lo:hi], s["w"], s["eps"], 0.0, s["res"][lo:hi])
    return oracle.vjp(h, s["w"], s["g"][lo:hi], s["eps"], 0.0)[1]


def oracle_pass(sample, threads=1, pool=None):
    """One forward (with residual) + VJP on new_residual per D.  With
    threads > 1 the rows are split into that many contiguous blocks, each run
    by the unchanged oracle functions on a thread of `pool` (the C oracle
    releases the GIL while it runs), and the blocks' gw are added in block
    order.  Returns the algorithmic bytes it stands for and each D's gw."""
    nbytes = 0
    gws = {}
    for D, s in sample.items():
        rows = s["x"].shape[0]
        if threads <= 1 or pool is None:
            gws[D] = _oracle_block(s, 0, rows)
        else:
            bounds = [rows * i // threads for i in range(threads + 1)]
            parts = [pool.submit(_oracle_block, s, lo, hi)
                     for lo, hi in zip(bounds, bounds[1:]) if hi > lo]
            gw = None
            for f in parts:  # block order
                gw = f.result() if gw is None else gw + f.result()
            gws[D] = gw
        nbytes += fwd_bytes(rows, D) + vjp_bytes(rows, D)
    return nbytes, gws


def _timed_passes(sample, seconds, threads, pool):
    oracle_pass(sample, threads, pool)  # load and warm
    t0 = time.perf_counter()
    nbytes = passes = 0
    while True:
        nbytes += oracle_pass(sample, threads, pool)[0]
        passes += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            return nbytes / el / 1e9, passes, el


def cpu_baseline(cases, seconds_one=5.0, seconds_all=10.0, rows=None):
    """The fp64 C oracle on the host: one thread, then one thread per host
    core over contiguous row blocks.  `value` is the all-core figure."""
    import concurrent.futures as cf
    import oracle
    oracle.build()
    cores = host_cores()
    rows = rows or max(256, 32 * cores)
    sample = oracle_sample(cases, rows)
    one, passes1, el1 = _timed_passes(sample, seconds_one, 1, None)
    with cf.ThreadPoolExecutor(max_workers=cores) as pool:
        allc, passes, el = _timed_passes(sample, seconds_all, cores, pool)
    return {"value": allc, "unit": UNIT, "cores": cores, "kind": "oracle",
            "host_cores": cores, "single_thread_value": one,
            "sample": "first %d rows of each D (4096, 8192) of the prefill workload: fp64 C oracle "
                      "forward with residual + VJP; %d threads over contiguous row blocks, %d "
                      "passes in %.1f s (one thread: %d passes in %.1f s)"
                      % (rows, cores, passes, el, passes1, el1)}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import concurrent.futures as cf
    import oracle
    oracle.build()
    from rmsnorm_fwd_bwd_add_gb300 import workloads as W
    cores = host_cores()
    cases = {D: W.config4(D, 1024) for D in DS}  # rows of the same recipe; a sample is taken below
    with cf.ThreadPoolExecutor(max_workers=cores) as pool:
        # size each step's sample so the whole run takes about a minute
        cal = oracle_sample(cases, 4 * cores)
        oracle_pass(cal, cores, pool)
        t0 = time.perf_counter()
        cal_bytes = oracle_pass(cal, cores, pool)[0]
        rate = cal_bytes / max(time.perf_counter() - t0, 1e-6)
        per_row = sum(fwd_bytes(1, D) + vjp_bytes(1, D) for D in DS)
        rows = int(60.0 * rate / max(1, args.steps + args.warmup) / per_row)
        rows = max(cores, min(1024, rows))
        sample = oracle_sample(cases, rows)
        for _ in range(args.warmup):
            oracle_pass(sample, cores, pool)
        t0 = time.perf_counter()
        nbytes = 0
        for _ in range(args.steps):
            nbytes += oracle_pass(sample, cores, pool)[0]
        el = time.perf_counter() - t0
    value = nbytes / el / 1e9
    desc = ("first %d rows of each D (4096, 8192) of the prefill workload per step: fp64 C oracle "
            "forward with residual + VJP, %d threads over contiguous row blocks" % (rows, cores))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * el / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": CONFIG,
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "host_cores": cores, "sample": desc},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_rope(args, rn, dev):
    """rope + KV append with Llama-3-8B heads (32 q, 8 kv, head 128): --rows
    tokens at positions 50000.., slots = positions mod 2 * rows."""
    T, Hq, Hkv, Dh = args.rows, 32, 8, 128
    gen = torch.Generator(device=dev).manual_seed(7)
    q = torch.randn(T, Hq, Dh, device=dev, generator=gen).to(torch.bfloat16)
    k = torch.randn(T, Hkv, Dh, device=dev, generator=gen).to(torch.bfloat16)
    v = torch.randn(T, Hkv, Dh, device=dev, generator=gen).to(torch.bfloat16)
    pos = torch.arange(50000, 50000 + T, device=dev)
    slots = pos % (2 * T)
    kc = torch.zeros(2 * T, Hkv, Dh, device=dev, dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    q_out = torch.empty_like(q)

    def once():
        rn.rmsnorm_rope_kv_append(q, k, v, pos, slots, kc, vc, rope_base=500000.0, q_out=q_out)
    for _ in range(max(1, args.warmup)):
        once()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(args.reps):
        once()
    b.record()
    torch.cuda.synchronize()
    us = 1e3 * a.elapsed_time(b) / args.reps
    print("op=rope tokens=%d heads=%d/%d Dh=%d us=%.2f GB/s=%.1f" % (
        T, Hq, Hkv, Dh, us, rope_bytes(T, Hq, Hkv, Dh) / us / 1e3), flush=True)
    return 0


def run_single_op(args):
    """One op on a case of the prefill recipe (for ncu captures of one kernel)."""
    from rmsnorm_fwd_bwd_add_gb300 import build, workloads as W
    import rmsnorm_fwd_bwd_add_gb300 as rn
    build.build()
    dev = torch.device("cuda", 0)
    if args.op == "rope":
        return run_rope(args, rn, dev)
    c = W.config4_on_device(args.D, dev, args.rows)
    dtype = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}[args.dtype]
    es = torch.empty(0, dtype=dtype).element_size()
    x, res, w, g = (t.to(dtype) for t in (c.x, c.residual, c.w, c.g))
    if args.layout == "strided":
        # x and residual (and g and g_residual, out and new_residual) as the
        # two halves of [rows, 2D] buffers: row stride 2D
        xr = torch.cat([x, res], dim=1)
        x, res = xr[:, :args.D], xr[:, args.D:]
        gr = torch.cat([g, res], dim=1)
        g, g_res = gr[:, :args.D], gr[:, args.D:]
        ob = torch.empty_like(xr)
        out, nr = ob[:, :args.D], ob[:, args.D:]
        gx = torch.empty_like(xr)[:, :args.D]
    elif args.layout == "offset":
        # every tensor one element past a 16-byte boundary (a slice of a
        # bigger buffer): rows at one shared offset
        def offset(t):
            buf = torch.empty(t.numel() + 16, dtype=dtype, device=dev)
            v = buf[1:1 + t.numel()].view(t.shape)
            v.copy_(t)
            return v
        x, res, g = offset(x), offset(res), offset(g)
        g_res = res
        out, nr, gx = offset(x), offset(x), offset(x)
    elif args.layout == "padded":
        # every tensor in its own buffer with rows of D + 64 elements
        def padded(t):
            buf = torch.empty(args.rows, args.D + 64, dtype=dtype, device=dev)
            buf[:, :args.D] = t
            return buf[:, :args.D]
        x, res, g = padded(x), padded(res), padded(g)
        g_res = res
        out, nr, gx = padded(x), padded(x), padded(x)
    else:
        g_res = res
        out, nr, gx = torch.empty_like(x), torch.empty_like(x), torch.empty_like(x)
    gw = torch.empty(args.D, dtype=torch.float32, device=dev)
    rstd = torch.empty(args.rows, dtype=torch.float32, device=dev) if args.rstd else None
    if args.rstd and args.op == "vjp":
        rn.rmsnorm_fwd_ex(x, w, c.eps, 0.0, rstd=rstd)  # a valid saved scale to read
    general = args.rstd or args.layout in ("strided", "padded") or args.dtype == "f32"

    if args.op == "gate":  # x = [a | b] of width 2D from the same draws
        xg = torch.cat([x, res], dim=1)
        og = torch.empty_like(x)

    def once():
        if args.op == "gate":
            rn.rmsnorm_gated_silu(xg, out=og)
        elif args.op == "fwd" and general:
            rn.rmsnorm_fwd_ex(x, w, c.eps, 0.0, res, out=out, new_residual=nr, rstd=rstd)
        elif args.op == "fwd":
            rn.rmsnorm_fwd(x, w, c.eps, 0.0, res, out=out, new_residual=nr)
        elif args.op == "vjp" and general:
            rn.rmsnorm_vjp_ex(x, w, g, c.eps, 0.0, rstd=rstd, gx=gx, gw=gw)
        elif args.op == "vjp":
            rn.rmsnorm_vjp(x, w, g, c.eps, 0.0, gx=gx, gw=gw)
        elif general:
            rn.rmsnorm_vjp_ex(x, w, g, c.eps, 0.0, g_res, rstd=rstd, gx=gx, gw=gw)
        else:
            rn.rmsnorm_fused_vjp(x, w, g, c.eps, 0.0, g_res, g_h=gx, gw=gw)
    for _ in range(args.warmup):
        once()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(args.reps):
        once()
    b.record()
    torch.cuda.synchronize()
    us = 1e3 * a.elapsed_time(b) / args.reps
    nbytes = {"fwd": fwd_bytes, "vjp": vjp_bytes, "fvjp": fused_vjp_bytes,
              "gate": gate_bytes}[args.op](args.rows, args.D, s=es)
    if args.rstd and args.op != "gate":
        nbytes += 4 * args.rows  # written by the forward, read by the VJP
    plan = ("gate" if args.op == "gate" else
            rn.rmsnorm_describe_dispatch("fwd" if args.op == "fwd" else "vjp", args.rows, args.D,
                                         dtype, args.op != "vjp",
                                         2 if args.layout == "offset" else
                                         1 if args.layout == "dense" else 0))
    print("op=%s dtype=%s layout=%s rstd=%d rows=%d D=%d plan=%s us=%.2f GB/s=%.1f" % (
        args.op, args.dtype, args.layout, int(args.rstd), args.rows, args.D, plan, us,
        nbytes / us / 1e3), flush=True)
    return 0


def run_all_configs(args):
    """Every workload configuration, fwd and VJP: µs per call with L2 flushed
    before each call (cold), back to back (warm: small problems then live in
    L2), replayed from a CUDA graph of back-to-back calls (launch cost
    amortised), and back to back over K copies of the problem's tensors whose
    total is at least twice the L2 (rotating: sustained HBM bandwidth, no
    reuse between calls; median of 20 repetitions of at least 1 ms); GB/s of
    algorithmic bytes, cold and rotating.  Prints one table row per case."""
    from rmsnorm_fwd_bwd_add_gb300 import build, workloads as W
    import rmsnorm_fwd_bwd_add_gb300 as rn
    build.build()
    dev = torch.device("cuda", 0)
    # Evicts L2 by reading 512 MB (a read leaves clean lines: the timed call does
    # not pay for write-backs of the flush itself).
    flush = torch.ones(128 << 20, dtype=torch.float32, device=dev)
    cases = [W.config1()]
    cases += [W.config2(r, D, gm) for r in W.DECODE_ROWS for D in W.DECODE_D for gm in (False, True)]
    cases += [W.config3()]
    cases += [W.config4(D) for D in W.PREFILL_D]
    cases += [W.config5(D, dt) for D in W.SWEEP_D for dt in (torch.float16, torch.bfloat16)]
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    print("%-22s %-4s %-62s %9s %9s %9s %9s %9s %9s" % (
        "case", "op", "plan", "cold_us", "warm_us", "graph_us", "rot_us", "cold_GB/s", "rot_GB/s"),
        flush=True)
    for c in cases:
        x, w = c.x.to(dev), c.w.to(dev)
        res = c.residual.to(dev) if c.residual is not None else None
        g = c.g.to(dev)
        out, nr, gx = torch.empty_like(x), torch.empty_like(x) if res is not None else None, torch.empty_like(x)
        gw = torch.empty(c.D, dtype=torch.float32, device=dev)
        ws = torch.empty(max(256, rn.rmsnorm_vjp_workspace_size(c.rows, c.D, c.dtype)),
                         dtype=torch.uint8, device=dev)
        ops = [("fwd", lambda: rn.rmsnorm_fwd(x, w, c.eps, c.weight_bias, res, out=out, new_residual=nr),
                fwd_bytes(c.rows, c.D, res is not None, 2))]
        ops.append(("vjp", lambda: rn.rmsnorm_vjp_ws(x, w, g, c.eps, c.weight_bias, workspace=ws,
                                                     gx=gx, gw=gw), vjp_bytes(c.rows, c.D, 2)))
        if res is not None and c.config == 4:
            # the two-output op's VJP, with the residual standing in for g_residual
            ops.append(("fvjp", lambda: rn.rmsnorm_fused_vjp(x, w, g, c.eps, c.weight_bias, res,
                                                             g_h=gx, gw=gw),
                        fused_vjp_bytes(c.rows, c.D, 2)))
        # K copies of every [rows, D] tensor for the rotating measurement (at
        # most 256: the decode shapes stay launch-bound whatever K is)
        per_set = (5 if res is not None else 4) * x.numel() * x.element_size()
        K = int(min(256, max(2, -(-2 * l2 // per_set))))

        def stack(t):
            return None if t is None else t.unsqueeze(0).repeat(K, *([1] * t.dim()))
        xs, gs, rs = stack(x), stack(g), stack(res)
        outs, gxs = torch.empty_like(xs), torch.empty_like(xs)
        nrs = None if res is None else torch.empty_like(xs)
        sets = [dict(x=xs[i], g=gs[i], out=outs[i], gx=gxs[i],
                     res=None if rs is None else rs[i], nr=None if nrs is None else nrs[i])
                for i in range(K)]
        rot_ops = {
            "fwd": lambda t: rn.rmsnorm_fwd(t["x"], w, c.eps, c.weight_bias, t["res"], out=t["out"],
                                            new_residual=t["nr"]),
            "vjp": lambda t: rn.rmsnorm_vjp_ws(t["x"], w, t["g"], c.eps, c.weight_bias, workspace=ws,
                                               gx=t["gx"], gw=gw),
            "fvjp": lambda t: rn.rmsnorm_fused_vjp(t["x"], w, t["g"], c.eps, c.weight_bias, t["res"],
                                                   g_h=t["gx"], gw=gw),
        }
        for name, f, nbytes in ops:
            for _ in range(5):
                f()
            torch.cuda.synchronize()
            cold = []
            for _ in range(20):
                flush.sum()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                f()
                b.record()
                torch.cuda.synchronize()
                cold.append(1e3 * a.elapsed_time(b))
            n = 50
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(n):
                f()
            b.record()
            torch.cuda.synchronize()
            warm = 1e3 * a.elapsed_time(b) / n
            s_ = torch.cuda.Stream()
            s_.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s_):
                f()
            torch.cuda.current_stream().wait_stream(s_)
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                for _ in range(n):
                    f()
            graph.replay()
            torch.cuda.synchronize()
            a.record()
            graph.replay()
            b.record()
            torch.cuda.synchronize()
            graph_us = 1e3 * a.elapsed_time(b) / n
            cold_us = statistics.median(cold)
            rf = rot_ops[name]
            calls = K * max(1, -(-int(1000.0 / max(cold_us, 1.0)) // K))  # >= ~1 ms per repetition
            for i in range(K):
                rf(sets[i])
            torch.cuda.synchronize()
            rot = []
            for _ in range(20):
                a.record()
                for i in range(calls):
                    rf(sets[i % K])
                b.record()
                torch.cuda.synchronize()
                rot.append(1e3 * a.elapsed_time(b) / calls)
            rot_us = statistics.median(rot)
            plan = rn.rmsnorm_describe_dispatch("fwd" if name == "fwd" else "vjp", c.rows, c.D,
                                                c.dtype, name != "vjp" and res is not None)
            print("%-22s %-4s %-62s %9.2f %9.2f %9.2f %9.2f %9.1f %9.1f" % (
                c.name, name, plan, cold_us, warm, graph_us, rot_us, nbytes / cold_us / 1e3,
                nbytes / rot_us / 1e3), flush=True)
        del sets, xs, gs, rs, outs, gxs, nrs
    return 0


# ---------------------------------------------------------------------------

def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)  # ~0.5 s of timed GPU work
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--op", choices=("fwd", "vjp", "fvjp", "gate", "rope"),
                    help="profiling mode: run one op of the prefill recipe at --rows x --D "
                         "(--reps launches after --warmup) and print its mean time; no JSON line")
    ap.add_argument("--rows", type=int, default=8192)
    ap.add_argument("--D", type=int, default=8192)
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--dtype", choices=("bf16", "f16", "f32"), default="bf16",
                    help="profiling mode: element type")
    ap.add_argument("--layout", choices=("dense", "strided", "padded", "offset"), default="dense",
                    help="profiling mode: strided = the tensors are halves of [rows, 2D] "
                         "buffers; padded = rows of D + 64 elements; offset = every tensor one "
                         "element past a 16-byte boundary")
    ap.add_argument("--rstd", action="store_true",
                    help="profiling mode: the forward writes rstd / the VJP reads it")
    ap.add_argument("--all-configs", action="store_true",
                    help="table of µs/call and GB/s for every workload configuration; no JSON line")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.op is None:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        return run_reference(args)
    if args.op is not None:
        return run_single_op(args)
    if args.all_configs:
        return run_all_configs(args)

    from rmsnorm_fwd_bwd_add_gb300 import build
    rank, world, local = dist_setup(args.gpus)
    if rank == 0:
        build.build()
    barrier()
    if world > 1:
        build.build()  # no-op once rank 0 has built it
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)

    if world > 1:
        torch.set_num_threads(max(1, (os.cpu_count() or 1) // world))
    cases = device_inputs(device)
    step = Step(cases, device)
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    total_ms, per_op_us, clocks = time_device(step, args.steps, args.warmup, sampler)
    sampler.stop()
    total_ms = max_over_ranks(total_ms, device)
    ms_per_step = total_ms / args.steps
    value = world * STEP_BYTES * args.steps / (total_ms * 1e-3) / 1e9

    peak, peak_src = measured_peak()
    sustained = sustained_ops(step, device)
    all_bytes = dict(OP_BYTES, **C3_OPS)
    ops = {}
    for name, us in sustained.items():
        gbs = all_bytes[name] / (us * 1e-6) / 1e9
        ops[name] = {"us": round(us, 2), "gbs": round(gbs, 1), "frac": round(gbs / peak, 4),
                     "frac_nominal": round(gbs / NOMINAL_HBM_GBS, 4), "bytes": all_bytes[name]}
    for name, _ in OPS:
        gbs = OP_BYTES[name] / (per_op_us[name] * 1e-6) / 1e9
        ops[name].update({"us_step": round(per_op_us[name], 2), "gbs_step": round(gbs, 1),
                          "frac_step": round(gbs / peak, 4)})
    dom = max(per_op_us, key=per_op_us.get)
    dom_gbs = OP_BYTES[dom] / (per_op_us[dom] * 1e-6) / 1e9
    roofline = {"bound": "hbm", "achieved": round(dom_gbs, 1), "peak": peak, "unit": UNIT,
                "frac": dom_gbs / peak, "frac_nominal": dom_gbs / NOMINAL_HBM_GBS,
                "traffic": recorded_traffic(dom), "kernel": dom, "peak_source": peak_src,
                "achieved_sustained": ops[dom]["gbs"],
                "note": "achieved = algorithmic bytes per launch / mean CUDA-event duration of "
                        "the op inside the timed steps (events around each op on every %dth "
                        "step); achieved_sustained = the same op timed back to back over "
                        "rotating buffers (ops[...].us)" % PROBE_EVERY}

    e2e = None
    if not args.no_e2e:
        del step
        host_cases = to_host(cases)
        torch.cuda.empty_cache()
        e2e_steps = max(3, min(args.steps, 30))
        ms_e2e, h2d, d2h = time_e2e(host_cases, device, e2e_steps, 3)
        e2e = {"value": world * STEP_BYTES / (ms_e2e * 1e-3) / 1e9, "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
               "ms_per_step": ms_e2e,
               "note": "public Python API, pinned host buffers; uploads, compute and "
                       "downloads of consecutive steps overlap on three streams"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(to_host(cases, rows=256))

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16", "data": "synthetic", "config": CONFIG,
                "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": KERNELS_PER_STEP * args.steps, "clocks": clocks, "ops": ops}
        print(json.dumps(line), flush=True)
    if dist.is_available() and dist.is_initialized():
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
