#!/usr/bin/env python3
"""Benchmark of the fused ZeRO shard-step (params/s and HBM GB/s) on GB300.

One "step" is one optimizer step of the whole workload: for every FSDP unit,
reduce-scatter by averaging of the N_d bf16 gradient buffers, AdamW on every
rank's fp32 shard, bf16 cast and all-gather -- one zero_step_units call,
which packs the units into as few fused launches as it can.  Inputs
(gradients, optimizer state) are synthetic and resident in HBM before the
timed region; they are larger than L2, so no flush is needed.  The JSON line
also carries the same step end to end through the host-buffer entry point
(gradients copied in, parameters copied out every step), the roofline of the
fused kernel, the CPU oracle's throughput, the clocks seen during the timed
region and, unless --no-extra, the secondary workloads.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload gpt2-small] [--variant plain|clip|per-param|zero1]
                  [--no-extra] [--no-e2e] [--no-cpu] [--sweep [--sweep-sizes ...]]
                  [--seed S]

With N > 1 (launched under torch.distributed.run) every rank runs an
independent replica of the workload on its own GPU (replicas only: no
collective on the data path); value = all ranks' parameters / max-over-ranks
step time.  `--impl reference` times the CPU oracle on a bounded sample, one
contiguous chunk per host core.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused ZeRO shard-step params/s and achieved HBM GB/s vs GB300 peak (1 GPU)"
UNIT = "params/s"
FALLBACK_HBM_GBS = 6800.0
WORKLOAD_NAMES = {
    "gpt2-small": "gpt2-small-124M-13units-Nd8",
    "llama3-8b-layer": "llama3-8b-decoder-layer-218M-Nd64",
    "7.5b": "7.5B-32units-Nd64",
    "7.5b-accum": "7.5B-32units-Nd64-fp32-accum-4-micro",
    "tiny": "tiny-4.2M-Nd4",
}


def workload_label(name: str) -> str:
    if name.startswith("sweep:"):
        _, p, n = name.split(":")
        return f"flat-{p}-Nd{n}"
    return WORKLOAD_NAMES[name]


# ------------------------------------------------------------------ env ----

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(ws, backend):
    """Process group of the N > 1 replicas.  Its collectives (the barriers
    around the timed region, the max over ranks) give up after
    BENCH_DIST_TIMEOUT_S seconds (default 600), so a rank that died is
    reported as an error on the others instead of a hang."""
    import datetime
    import torch.distributed as dist
    if ws > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        timeout = float(os.environ.get("BENCH_DIST_TIMEOUT_S", "600"))
        dist.init_process_group(backend=backend, timeout=datetime.timedelta(seconds=timeout))
    return dist


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, ws: int, device) -> float:
    if ws <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


KERNEL_SOURCES = ("zero_step_tma.cu", "zero_common.cuh", "zero_kernels.cuh")


def kernel_source_hash() -> str:
    """Hash of the sources of the timed kernel (staged fused step)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "fsdp_sharded_mixed_flatten_gb300", "csrc")
    for name in KERNEL_SOURCES:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def traffic_class(n_ranks: int, aligned: bool) -> str:
    """Kernel form a launch runs, as far as its DRAM traffic per element goes:
    the rank count and whether every shard starts on the 16-byte grid."""
    return f"nd{n_ranks}-{'aligned' if aligned else 'misaligned'}"


def recorded_traffic(tclass: str, padded_elements: int):
    """DRAM bytes the fused kernel moves for `padded_elements` flat elements,
    scaled from a committed ncu capture of a small case of the same kernel form
    (DRAM read + write bytes per padded element; the kernel streams every
    element once, so traffic grows in proportion to the elements).  None when
    no capture of that form exists or the kernel sources changed since."""
    path = os.path.join(ROOT, "profiles", "fused_step_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except Exception:
        return None
    if d.get("kernel_source_hash") != kernel_source_hash():
        return None
    entry = d.get("captures", {}).get(tclass)
    if entry is None:
        return None
    return float(entry["dram_bytes_per_padded_element"]) * padded_elements


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms; each sample
    is stamped with the host time it arrived, so that a summary can be taken
    over chosen time windows (the timed regions) only."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self, windows=None):
        """Stop sampling; summarise the samples inside `windows` (a list of
        (t0, t1) host times), or all of them."""
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=2)
        return self.summary(windows)

    def summary(self, windows=None):
        sm, power, smax, reasons = [], [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, ln in self.lines:
            if windows is not None and not any(a <= ts <= b for a, b in windows):
                continue
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax = float(parts[1])
                power.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm), "sm_mhz_min": min(sm), "power_w_max": max(power)}


# ------------------------------------------------------------- workloads ----

# Launch packing of zero_step_units (ZERO_UNITS_PER_LAUNCH, ZERO_POINTERS_PER_LAUNCH in
# include/zero_flat.h): used only to report how many kernels a step launches.
UNITS_PER_LAUNCH = 64
POINTERS_PER_LAUNCH = 3392


def staged_launches(n_ranks_per_unit, n_out=1, pointers=None):
    """Launches zero_step_units issues for these units; `pointers(n)` is the
    pointer count one unit of n ranks needs (default: a plain fused step)."""
    if os.environ.get("ZERO_STEP_KERNEL") == "direct":
        return len(n_ranks_per_unit)        # the direct-load kernels: one launch per unit
    if pointers is None:
        pointers = lambda n: 4 * n + n_out
    launches, units, ptrs = 0, 0, 0
    for n in n_ranks_per_unit:
        need = pointers(n)
        if units == UNITS_PER_LAUNCH or ptrs + need > POINTERS_PER_LAUNCH or units == 0:
            launches += 1
            units, ptrs = 0, 0
        units += 1
        ptrs += need
    return launches


def unit_bytes(P_pad, n_ranks, n_out=1, n_micro=1):
    """Algorithmic HBM bytes of one optimizer step of one unit: each gradient,
    state and parameter byte crosses HBM exactly once.  With K > 1 micro-steps:
    the first reduce-scatter writes the fp32 accumulator (2N + 4 per element),
    the middle ones read and write it (2N + 8), the fused last one reads it
    with the state (2N + 4 + 24 + 2 n_out)."""
    if n_micro <= 1:
        return P_pad * (2 * n_ranks + 24 + 2 * n_out)
    per = (2 * n_ranks + 4) + (n_micro - 2) * (2 * n_ranks + 8) + (2 * n_ranks + 28 + 2 * n_out)
    return P_pad * per


class Resident:
    """All units of a workload resident in HBM (per-unit gradient buffers),
    or, with shared_grads, one gradient buffer reused by every unit (the
    7.5B model streams its gradients unit by unit)."""

    def __init__(self, w, shared_grads=False, n_units=None):
        import torch
        from fsdp_sharded_mixed_flatten_gb300 import synthetic
        from fsdp_sharded_mixed_flatten_gb300.buffers import FlatUnit
        self.w = w
        units = w.units if n_units is None else w.units[:n_units]
        self.units = []
        shared = None
        self.n_micro = w.n_micro
        for ui, u in enumerate(units):
            fu = FlatUnit(u.numels, w.n_ranks, accum=w.n_micro > 1,
                          with_grads=not (shared_grads and shared is not None))
            if shared_grads:
                if shared is None:
                    shared = fu.grads
                else:
                    fu.grads = shared
            master = synthetic.make_master_flat(u.numel, w.n_ranks, w.master_std,
                                                (w.name, u.name), device="cuda")
            fu.set_master_flat(master)
            del master
            if not (shared_grads and ui > 0):
                for r in range(w.n_ranks):
                    synthetic.fill_grad_(fu.grads[r], fu.P, w.grad_std,
                                         synthetic.seed_for(w.name, u.name, "grad", r),
                                         w.outlier_frac, w.outlier_scale)
            self.units.append(fu)
        torch.cuda.synchronize()
        self.numel = sum(fu.P for fu in self.units)
        self.bytes = sum(unit_bytes(fu.P_pad, w.n_ranks, n_micro=w.n_micro) for fu in self.units)
        self.ptrs = [(fu.grad_rows(), *fu.state_rows(), fu.accum_rows(), fu.param_rows(),
                      fu.layout) for fu in self.units]
        from fsdp_sharded_mixed_flatten_gb300.zero import prepare_units
        self.prepared = prepare_units(self.ptrs)      # pointer tables marshalled once
        nr = [fu.n_ranks for fu in self.units]
        if w.n_micro > 1:
            self.launches_per_step = (
                (w.n_micro - 1) * staged_launches(nr, pointers=lambda n: 2 * n)
                + staged_launches(nr, pointers=lambda n: 5 * n + 1))
        else:
            self.launches_per_step = staged_launches(nr, n_out=1)

    def launch(self, step, hp_base, events=None):
        """One optimizer step over every unit: one zero_step_units call per
        micro-step (the library packs the units into as few launches as it can)."""
        from fsdp_sharded_mixed_flatten_gb300 import zero_step_units
        hp = dict(hp_base, step=step)
        if events is not None:
            events[0][0].record()
        for k in range(1, self.n_micro + 1):
            zero_step_units(self.prepared, k, self.n_micro, hp)
        if events is not None:
            events[0][1].record()
        return self.launches_per_step


class PerParamResident:
    """The workload as FSDP2 per-parameter units: every tensor its own unit,
    split along dim 0 into N_d chunks with no padding (Shard(0)), all stepped
    by one zero_step_units call (the library packs them into launches)."""

    def __init__(self, w):
        import torch
        from fsdp_sharded_mixed_flatten_gb300 import synthetic
        from fsdp_sharded_mixed_flatten_gb300.buffers import ParamUnit
        from fsdp_sharded_mixed_flatten_gb300.zero import prepare_units
        self.w = w
        self.n_micro = 1
        self.units = []
        for u in w.units:
            for i, (d0, row) in enumerate(u.rows()):
                pu = ParamUnit(d0, row, w.n_ranks)
                pu.set_master_flat(synthetic.make_master_flat(
                    pu.numel, 1, w.master_std, (w.name, u.name, "param", i), device="cuda"))
                for r in range(w.n_ranks):
                    synthetic.fill_grad_(pu.grads[r], pu.numel, w.grad_std,
                                         synthetic.seed_for(w.name, u.name, "param", i, "grad", r),
                                         w.outlier_frac, w.outlier_scale)
                self.units.append(pu)
        torch.cuda.synchronize()
        self.numel = sum(pu.numel for pu in self.units)
        # every element once: N_d bf16 gradients, fp32 state read + written, bf16 output
        self.bytes = sum(pu.numel * (2 * w.n_ranks + 26) for pu in self.units)
        self.prepared = prepare_units([pu.unit_tuple() for pu in self.units])
        self.launches_per_step = staged_launches([w.n_ranks] * len(self.units))

    def launch(self, step, hp_base, events=None):
        from fsdp_sharded_mixed_flatten_gb300 import zero_step_units
        if events is not None:
            events[0][0].record()
        zero_step_units(self.prepared, 1, 1, dict(hp_base, step=step))
        if events is not None:
            events[0][1].record()
        return self.launches_per_step


class ClipResident(Resident):
    """Resident units stepped with global gradient-norm clipping: a norm pass
    (the averaged gradient written to each unit's accumulator with per-CTA
    partial sums of squares) and an update pass (AdamW from the accumulator
    times the clip coefficient)."""

    def __init__(self, w, max_norm):
        import torch
        from fsdp_sharded_mixed_flatten_gb300 import zero_clip_workspace_bytes
        from fsdp_sharded_mixed_flatten_gb300.buffers import aligned_rows
        from fsdp_sharded_mixed_flatten_gb300.zero import prepare_units
        super().__init__(w)
        for fu in self.units:
            fu.accum = aligned_rows(fu.n_ranks, fu.S, torch.float32, "cuda", 0)
        self.prepared = prepare_units([(fu.grad_rows(), *fu.state_rows(), fu.accum_rows(),
                                        fu.param_rows(), fu.layout) for fu in self.units])
        self.ws_bytes = zero_clip_workspace_bytes(self.prepared, 1)
        self.workspace = torch.empty(max(self.ws_bytes // 8, 1), dtype=torch.float64,
                                     device="cuda")
        self.norm = torch.zeros(1, dtype=torch.float32, device="cuda")
        self.max_norm = max_norm
        # pass 1: gradients in, averaged gradient out; pass 2: it and the state in, state
        # and parameters out
        self.bytes = sum(fu.P_pad * ((2 * fu.n_ranks + 4) + (4 + 24 + 2)) for fu in self.units)
        nr = [fu.n_ranks for fu in self.units]
        self.launches_per_step = (staged_launches(nr, pointers=lambda n: 2 * n)
                                  + staged_launches(nr, pointers=lambda n: 4 * n + 1))

    def launch(self, step, hp_base, events=None):
        from fsdp_sharded_mixed_flatten_gb300 import zero_step_units_clip
        if events is not None:
            events[0][0].record()
        zero_step_units_clip(self.prepared, 1, 1, dict(hp_base, step=step), self.max_norm,
                             self.workspace, self.ws_bytes, self.norm)
        if events is not None:
            events[0][1].record()
        return self.launches_per_step


class Zero1Resident:
    """The ZeRO-1 form of a step of K micro-batches on one unit: each rank
    accumulates its full fp32 gradient locally (zero1_accumulate), then one
    reduce-scatter of the accumulators with the update (zero1_step)."""

    def __init__(self, w, n_micro=4):
        import torch
        from fsdp_sharded_mixed_flatten_gb300 import synthetic
        from fsdp_sharded_mixed_flatten_gb300.buffers import FlatUnit, aligned_rows, rows
        self.w = w
        self.n_micro = n_micro
        u = w.units[0]
        self.fu = FlatUnit(u.numels, w.n_ranks)
        self.fu.set_master_flat(synthetic.make_master_flat(u.numel, w.n_ranks, w.master_std,
                                                           (w.name, u.name), device="cuda"))
        for r in range(w.n_ranks):
            synthetic.fill_grad_(self.fu.grads[r], self.fu.P, w.grad_std,
                                 synthetic.seed_for(w.name, u.name, "grad", r),
                                 w.outlier_frac, w.outlier_scale)
        self.full_acc = aligned_rows(w.n_ranks, self.fu.P_pad, torch.float32, "cuda", 0)
        self.acc_rows = rows(self.full_acc)
        torch.cuda.synchronize()
        self.units = [self.fu]
        self.numel = self.fu.P
        N, P_pad = w.n_ranks, self.fu.P_pad
        self.bytes = P_pad * N * (6 + 10 * (n_micro - 1)) + P_pad * (4 * N + 26)
        self.launches_per_step = n_micro + 1

    def launch(self, step, hp_base, events=None):
        import fsdp_sharded_mixed_flatten_gb300 as zf
        fu = self.fu
        if events is not None:
            events[0][0].record()
        for k in range(1, self.n_micro + 1):
            zf.zero1_accumulate(fu.grad_rows(), self.acc_rows, k == 1, fu.layout)
        zf.zero1_step(self.acc_rows, self.n_micro, *fu.state_rows(), fu.param_rows(), fu.layout,
                      dict(hp_base, step=step))
        if events is not None:
            events[0][1].record()
        return self.launches_per_step


def timed_extra(res, steps, warmup, ws, device, hbm_peak):
    import gc
    import torch
    el, kern, launches, _ = time_resident(res, steps, warmup, ws, device)
    gbs = res.bytes * steps / kern / 1e9
    out = {"params_per_s": ws * res.numel * steps / el, "ms_per_step": el / steps * 1e3,
           "kernel_gbs": gbs, "frac_of_measured_hbm": gbs / hbm_peak,
           "bytes_per_step": res.bytes, "units": len(res.units), "n_ranks": res.w.n_ranks,
           "params": res.numel, "launches_per_step": res.launches_per_step, "steps": steps}
    del res
    gc.collect()
    torch.cuda.empty_cache()
    return out


def time_resident(res, steps, warmup, ws, device, per_kernel=True, clocks=None):
    import torch
    from fsdp_sharded_mixed_flatten_gb300 import synthetic
    hp = dict(synthetic.ADAMW_DEFAULTS)
    t = 0
    for _ in range(warmup):
        t += 1
        res.launch(t, hp)
    torch.cuda.synchronize()
    ev = [[[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)]]
          for _ in range(steps)] if per_kernel else None
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(ws)
    torch.cuda.synchronize()
    if clocks is not None:
        clocks.start()
    launches = 0
    torch.cuda.nvtx.range_push("timed")      # lets a profiler list the timed launches only
    start.record()
    for s in range(steps):
        t += 1
        launches += res.launch(t, hp, ev[s] if ev else None)
    stop.record()
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    clock_info = clocks.stop() if clocks is not None else None
    barrier(ws)
    elapsed = start.elapsed_time(stop) / 1e3
    elapsed_max = max_over_ranks(elapsed, ws, device)
    kern = None
    if ev:
        kern = sum(a.elapsed_time(b) for row in ev for a, b in row) / 1e3
    return elapsed_max, kern, launches, clock_info


def time_graph(step_fn, n_steps, reps=5, windows=None):
    """Seconds per step of step_fn(t) replayed from a CUDA graph of n_steps
    consecutive steps: the kernels run back to back, without the host's
    per-call launch cost (tens of microseconds through Python and ctypes),
    which would otherwise hide short kernels.  The graph fixes the step
    number t of every captured call; the bytes and the work do not depend on
    it.  The step is warmed up eagerly first (kernel attributes, caches).
    The host times of the timed replays are appended to `windows`."""
    import torch
    step_fn(1)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for t in range(n_steps):
            step_fn(2 + t)
    g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    a.record()
    for _ in range(reps):
        g.replay()
    b.record()
    torch.cuda.synchronize()
    if windows is not None:
        windows.append((t0, time.time()))
    del g
    return a.elapsed_time(b) / 1e3 / (reps * n_steps)


def time_e2e(res, steps, warmup, ws, device):
    """The same step through the host-buffer entry point
    (zero_step_units_host): every step copies every unit's gradients from
    pinned host memory and the gathered bf16 parameters back, through the SMs
    (ZERO_HOST_SM_COPY: the copy engines stall periodically on this host
    link).  Two device gradient sets alternate, so a step's copies overlap the
    previous step's update; the copies of a set wait for the step that last
    read it."""
    import torch
    from fsdp_sharded_mixed_flatten_gb300 import (ZERO_HOST_GRADS_FREE, ZERO_HOST_SM_COPY,
                                                  HostTables, synthetic, zero_step_units_host)
    from fsdp_sharded_mixed_flatten_gb300.buffers import aligned_rows
    from fsdp_sharded_mixed_flatten_gb300.zero import prepare_units
    hp = dict(synthetic.ADAMW_DEFAULTS)
    host_g = [fu.grads.cpu().pin_memory() for fu in res.units]          # (N_d, P_pad) each
    host_p = [torch.empty(fu.P_pad, dtype=torch.bfloat16).pin_memory() for fu in res.units]
    h2d = sum(x.numel() * 2 for x in host_g) * res.n_micro
    d2h = sum(x.numel() * 2 for x in host_p)
    tables = HostTables([[hg[k] for k in range(hg.shape[0])] for hg in host_g], host_p)
    spare = [aligned_rows(fu.n_ranks, fu.P_pad, torch.bfloat16, device, 0) for fu in res.units]
    sets = [prepare_units([([g[k] for k in range(fu.n_ranks)], *fu.state_rows(),
                            fu.accum_rows(), fu.param_rows(), fu.layout)
                           for fu, g in zip(res.units, grads)])
            for grads in ([fu.grads for fu in res.units], spare)]
    comp = torch.cuda.current_stream()
    s_h2d, s_d2h = torch.cuda.Stream(), torch.cuda.Stream()
    done = {}

    def one(i, step):
        if i - 2 in done:
            s_h2d.wait_event(done.pop(i - 2))    # the last step that read this set is done
        for k in range(1, res.n_micro + 1):
            zero_step_units_host(sets[i % 2], tables, k, res.n_micro, dict(hp, step=step),
                                 ZERO_HOST_GRADS_FREE | ZERO_HOST_SM_COPY, s_h2d, comp, s_d2h)
        done[i] = comp.record_event()

    t = 1000
    for i in range(warmup):
        t += 1
        one(i, t)
    torch.cuda.synchronize()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(ws)
    torch.cuda.nvtx.range_push("timed_e2e")
    start.record(comp)
    s_h2d.wait_stream(comp)
    for i in range(warmup, warmup + steps):
        t += 1
        one(i, t)
    comp.wait_stream(s_h2d)
    comp.wait_stream(s_d2h)
    stop.record(comp)
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    barrier(ws)
    el = max_over_ranks(start.elapsed_time(stop) / 1e3, ws, device)
    del host_g, host_p, spare, sets
    return el, h2d, d2h


def time_e2e_streamed(res, steps, warmup, ws, device):
    """The 7.5B step end to end with gradients streamed unit by unit from host
    memory, as the model's units would arrive: every step, each of the 32
    units' N_d gradient rows (N_d x P_pad bf16, 30 GB) crosses the host link
    into one of two device gradient buffers, the unit is stepped from it
    (zero_step_units_host, one unit per call), and its gathered bf16 parameters
    cross back into the unit's pinned host buffer.  Unit i's copy overlaps the
    step of unit i - 1; a buffer is refilled only after the step that read it.
    The host holds one set of gradient rows that every unit reads in turn (the
    resident step also shares one gradient buffer between its units); every
    byte still crosses the link each time.  Transfers go through the SMs
    (ZERO_HOST_SM_COPY)."""
    import torch
    from fsdp_sharded_mixed_flatten_gb300 import (ZERO_HOST_GRADS_FREE, ZERO_HOST_SM_COPY,
                                                  HostTables, synthetic, zero_step_units_host)
    from fsdp_sharded_mixed_flatten_gb300.buffers import aligned_rows, rows
    from fsdp_sharded_mixed_flatten_gb300.zero import prepare_units
    hp = dict(synthetic.ADAMW_DEFAULTS)
    fu0 = res.units[0]
    N, P_pad = fu0.n_ranks, fu0.P_pad
    # Distinct host gradient rows: all N_d when a quarter of the host's free
    # memory, shared by the replicas on this host, holds them; else fewer,
    # each standing in for several ranks.  Every rank's row still crosses the
    # link every step, so the bytes moved do not change.
    row_bytes = P_pad * 2
    params_bytes = sum(fu.P_pad * 2 for fu in res.units)
    budget = host_available_bytes() // 4 // max(ws, 1) - params_bytes
    n_rows = int(max(1, min(N, budget // row_bytes)))
    host_g = torch.empty((n_rows, P_pad), dtype=torch.bfloat16, pin_memory=True)
    for k in range(n_rows):
        host_g[k].copy_(fu0.grads[k])
    host_p = [torch.empty(fu.P_pad, dtype=torch.bfloat16, pin_memory=True) for fu in res.units]
    spare = aligned_rows(N, P_pad, torch.bfloat16, device, 0)
    dev_sets = (fu0.grad_rows(), rows(spare))
    prepared = [[prepare_units([(g, *fu.state_rows(), None, fu.param_rows(), fu.layout)])
                 for g in dev_sets] for fu in res.units]
    host_rows = [host_g[k % n_rows] for k in range(N)]
    tables = [HostTables([host_rows], [hp_buf]) for hp_buf in host_p]
    h2d = len(res.units) * N * P_pad * 2
    d2h = sum(fu.P_pad * 2 for fu in res.units)
    comp = torch.cuda.current_stream()
    s_h2d, s_d2h = torch.cuda.Stream(), torch.cuda.Stream()
    done = {}
    counter = [0]

    def one_step(t):
        for ui in range(len(res.units)):
            i = counter[0]
            counter[0] += 1
            if i - 2 in done:
                s_h2d.wait_event(done.pop(i - 2))    # the step that last read this buffer
            zero_step_units_host(prepared[ui][i % 2], tables[ui], 1, 1, dict(hp, step=t),
                                 ZERO_HOST_GRADS_FREE | ZERO_HOST_SM_COPY, s_h2d, comp, s_d2h)
            done[i] = comp.record_event()

    t = 1000
    for _ in range(warmup):
        t += 1
        one_step(t)
    torch.cuda.synchronize()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(ws)
    torch.cuda.nvtx.range_push("timed_e2e")
    start.record(comp)
    s_h2d.wait_stream(comp)
    for _ in range(steps):
        t += 1
        one_step(t)
    comp.wait_stream(s_h2d)
    comp.wait_stream(s_d2h)
    stop.record(comp)
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    barrier(ws)
    el = max_over_ranks(start.elapsed_time(stop) / 1e3, ws, device)
    del host_g, host_p, spare, prepared, tables, dev_sets
    return el, h2d, d2h, n_rows


def host_available_bytes() -> int:
    """Host memory available to this process now (MemAvailable), else the
    physical memory, else a conservative 64 GB."""
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        pass
    try:
        return os.sysconf("SC_PAGE_SIZE") * os.sysconf("SC_PHYS_PAGES")
    except (ValueError, OSError, AttributeError):
        return 64 << 30


def _oracle_sample(E, workload="gpt2-small"):
    """Seeded inputs of one contiguous sample of E flat elements x N_d ranks
    of a workload, for the CPU oracle."""
    import numpy as np
    from fsdp_sharded_mixed_flatten_gb300 import synthetic
    w = synthetic.workload(workload)
    g = synthetic.make_grads(E, w.n_ranks, w.grad_std, ("cpu-sample",))
    master = synthetic.make_master_flat(E, w.n_ranks, w.master_std, ("cpu-sample",)).numpy()
    return w, synthetic.bf16_bits(g), master, np.zeros_like(master), np.zeros_like(master)


def host_threads():
    """Host cores this process may run on."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine)."""
    import platform
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.machine()


class OracleRun:
    """The oracle over one contiguous sample of E elements, cut into one
    contiguous chunk per host thread.  The step is element-wise, so the chunks
    are independent, and the oracle's C calls release the interpreter lock, so
    the threads run in parallel."""

    def __init__(self, E, threads, workload="gpt2-small"):
        from concurrent.futures import ThreadPoolExecutor
        import numpy as np
        from fsdp_sharded_mixed_flatten_gb300 import synthetic
        from oracle import Oracle
        self.o, self.hp = Oracle(), synthetic.ADAMW_DEFAULTS
        self.w, gb, master, m, v = _oracle_sample(E, workload)
        self.E = E
        edges = [(E * i // threads) & ~7 for i in range(threads)] + [E]
        self.chunks = [(np.ascontiguousarray(gb[:, a:b]), master[a:b], m[a:b], v[a:b])
                       for a, b in zip(edges, edges[1:]) if b > a]
        self.pool = ThreadPoolExecutor(len(self.chunks))

    def step(self, step):
        for f in [self.pool.submit(self.o.sampled_step, *c, step=step, **self.hp)
                  for c in self.chunks]:
            f.result()

    def close(self):
        self.pool.shutdown()


def _timed_oracle_steps(run, seconds):
    """Step an OracleRun until `seconds` have passed; (steps, elapsed s)."""
    reps = 0
    t0 = time.perf_counter()
    while True:
        reps += 1
        run.step(reps)
        el = time.perf_counter() - t0
        if el >= seconds:
            return reps, el


def cpu_baseline(workload="7.5b", seconds=8.0):
    """The CPU oracle as it stands, on a bounded contiguous sample of the
    workload (all N_d ranks): one chunk per host core of 2^23 / N_d flat
    elements (so that a chunk holds 2^23 gradient values whatever N_d is), the
    chunks stepped in parallel for about `seconds`; then one such chunk on a
    single thread for a quarter of that (the single-core rate)."""
    from fsdp_sharded_mixed_flatten_gb300 import synthetic
    threads = host_threads()
    n_ranks = synthetic.workload(workload).n_ranks
    per = max(1 << 12, (1 << 23) // n_ranks) & ~7
    run = OracleRun(threads * per, threads, workload)
    reps, el = _timed_oracle_steps(run, seconds)
    run.close()
    rate = reps * run.E / el
    one = OracleRun(per, 1, workload)
    reps1, el1 = _timed_oracle_steps(one, seconds / 4)
    one.close()
    rate1 = reps1 * one.E / el1
    return {"value": rate, "unit": UNIT, "cores": threads, "kind": "oracle",
            "cpu": cpu_model(),
            "extrapolated_full_step_s": sum(u.numel for u in run.w.units) / rate,
            "single_thread_value": rate1,
            "sample": f"{run.E} contiguous flat elements x {run.w.n_ranks} ranks of the {workload} "
                      f"workload in {len(run.chunks)} chunks, one per thread; {reps} oracle steps "
                      f"in {el:.1f} s (double arithmetic); single thread: {one.E} elements, "
                      f"{reps1} steps in {el1:.1f} s"}


# ----------------------------------------------------------------- arms ----

def run_reference(args, ws, rank, budget_s=90.0):
    """The oracle as the reference arm: W untimed and K timed steps, each over
    a contiguous sample of the workload sized from a short calibration so that
    the whole run takes at most about budget_s seconds.  The sample is also
    capped at 2^21 flat elements and 2^25 gradient values per thread, which
    bound its host memory (at N_d = 64 the second cap binds: 2^19 elements
    per thread)."""
    if rank != 0:
        return 0
    from fsdp_sharded_mixed_flatten_gb300 import synthetic
    threads = host_threads()
    cal = OracleRun(threads << 14, threads, args.workload)
    t0 = time.perf_counter()
    cal.step(1)
    cal.step(2)
    rate = 2 * cal.E / (time.perf_counter() - t0)          # elements per second
    cal.close()
    E = int(budget_s * rate / (args.steps + args.warmup))
    n_ranks = cal.w.n_ranks
    E = max(threads << 10, min(threads << 21, (threads << 25) // n_ranks, E)) & ~7
    run = OracleRun(E, threads, args.workload)
    step = 0
    for _ in range(args.warmup):
        step += 1
        run.step(step)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step += 1
        run.step(step)
    el = time.perf_counter() - t0
    run.close()
    value = E * args.steps / el
    sample = (f"{E} contiguous flat elements x {run.w.n_ranks} ranks of the {args.workload} "
              f"workload per step in {len(run.chunks)} chunks, one per thread; {args.steps} "
              f"timed oracle steps in {el:.1f} s (double arithmetic)")
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": workload_label(args.workload), "variant": args.variant,
                       "seed": args.seed, "n_ranks_logical": run.w.n_ranks,
                       "units": len(run.w.units), "params": sum(u.numel for u in run.w.units),
                       "padded_elements": sum(synthetic.padded(u.numel, run.w.n_ranks)
                                              for u in run.w.units),
                       "storage": "bf16 grads/params, fp32 master/m/v", "n_out": 1,
                       "sample": sample},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "cpu": cpu_model(), "sample": sample,
                             "extrapolated_full_step_s":
                                 sum(u.numel for u in run.w.units) / value},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def secondary(name, steps, warmup, ws, device, hbm_peak, shared=False, n_units=None):
    import gc
    import torch
    from fsdp_sharded_mixed_flatten_gb300 import synthetic
    w = synthetic.workload(name)
    res = Resident(w, shared_grads=shared, n_units=n_units)
    el, kern, launches, _ = time_resident(res, steps, warmup, ws, device)
    gbs = res.bytes * steps / kern / 1e9
    out = {"params_per_s": ws * res.numel * steps / el, "ms_per_step": el / steps * 1e3,
           "kernel_gbs": gbs, "frac_of_measured_hbm": gbs / hbm_peak,
           "bytes_per_step": res.bytes, "units": len(res.units), "n_ranks": w.n_ranks,
           "params": res.numel, "steps": steps}
    del res
    gc.collect()
    torch.cuda.empty_cache()
    return out


def run_sweep(args, device, hbm_peak):
    """Flat sizes 4^k and 4^k + 13 (k = 10..15) x N_d in {2, 8, 64}: the fused
    step (zero_step) against the unfused reduce-scatter + AdamW + all-gather
    sequence, one JSON line per point.  Points whose step moves less than
    4 x L2 (129 MB) stay partly cache-resident between steps and are marked."""
    import gc
    import torch
    import fsdp_sharded_mixed_flatten_gb300 as zf
    from fsdp_sharded_mixed_flatten_gb300 import synthetic
    from fsdp_sharded_mixed_flatten_gb300.buffers import aligned_rows, rows
    hp0 = dict(synthetic.ADAMW_DEFAULTS)
    sizes = synthetic.sweep_sizes() if not args.sweep_sizes else \
        [int(x) for x in args.sweep_sizes.split(",")]
    for P in sizes:
        for n in synthetic.SWEEP_RANKS:
            w = synthetic.workload(f"sweep:{P}:{n}")
            res = Resident(w)
            fu = res.units[0]
            steps = int(max(10, min(200, 2e10 // res.bytes)))
            el, kern, _, _ = time_resident(res, steps, 5, 1, device)
            fused_gbs = res.bytes * steps / kern / 1e9
            gsh = aligned_rows(n, fu.S, torch.float32, device, 0)
            psh = aligned_rows(n, fu.S, torch.bfloat16, device, 0)
            master, m, v = fu.state_rows()

            def unfused(t):
                hp = dict(hp0, step=t)
                zf.zero_reduce_scatter(fu.grad_rows(), rows(gsh), fu.layout, 0)
                zf.zero_adamw_shard_step(master, m, v, rows(gsh), 1.0, rows(psh), fu.layout, hp)
                zf.zero_all_gather(rows(psh), fu.param_rows(), fu.layout)

            for t in range(1, 4):
                unfused(1000 + t)
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for t in range(steps):
                unfused(2000 + t)
            b.record()
            torch.cuda.synchronize()
            un_el = a.elapsed_time(b) / 1e3
            un_bytes = fu.P_pad * (2 * n + 38)
            # the same two steps replayed from CUDA graphs (no host launch cost)
            n_graph = int(max(4, min(50, 5e9 // res.bytes)))
            fused_g = time_graph(lambda t: res.launch(t, hp0), n_graph)
            unfused_g = time_graph(unfused, n_graph)
            line = {"sweep": True, "P": P, "n_ranks": n, "P_pad": fu.P_pad, "S": fu.S,
                    "S_mod_8": fu.S % 8, "steps": steps,
                    "fused_bytes_per_step": res.bytes, "fused_ms": kern / steps * 1e3,
                    "fused_gbs": fused_gbs, "fused_frac_of_measured_hbm": fused_gbs / hbm_peak,
                    "unfused_bytes_per_step": un_bytes, "unfused_ms": un_el / steps * 1e3,
                    "unfused_gbs": un_bytes * steps / un_el / 1e9,
                    "unfused_frac_of_measured_hbm": un_bytes * steps / un_el / 1e9 / hbm_peak,
                    "fused_speedup": un_el / kern,
                    "graph_steps": n_graph,
                    "fused_graph_ms": fused_g * 1e3,
                    "fused_graph_frac_of_measured_hbm": res.bytes / fused_g / 1e9 / hbm_peak,
                    "unfused_graph_ms": unfused_g * 1e3,
                    "unfused_graph_frac_of_measured_hbm": un_bytes / unfused_g / 1e9 / hbm_peak,
                    "l2_resident": res.bytes < 4 * 129e6}
            print(json.dumps(line), flush=True)
            del res, fu, gsh, psh, master, m, v
            gc.collect()
            torch.cuda.empty_cache()
    return 0


L2_BYTES = 129e6


def sweep_points(gated_only=False):
    """(P, N_d, fused bytes per step, gated) of the flat-size x N_d sweep; a
    point is gated when its step moves at least 4 x L2 (smaller ones stay
    partly cache-resident between steps)."""
    from fsdp_sharded_mixed_flatten_gb300 import synthetic
    out = []
    for P in synthetic.sweep_sizes():
        for n in synthetic.SWEEP_RANKS:
            nbytes = unit_bytes(synthetic.padded(P, n), n)
            gated = nbytes >= 4 * L2_BYTES
            if gated or not gated_only:
                out.append((P, n, nbytes, gated))
    return out


def sweep_gated(device, hbm_peak, local, min_seconds=0.25):
    """The sweep's gated points, timed in the default run: for each (P, N_d)
    the fused step (one zero_step launch of the staged kernel) replayed from a
    CUDA graph (the kernels back to back; at least 10 steps and min_seconds of
    timed replays) and, beside it, timed eagerly with per-launch CUDA events
    (one Python call per step, at least 10 steps).  Clocks are sampled over
    the whole sweep and summarised over the timed windows only."""
    import gc
    import torch
    from fsdp_sharded_mixed_flatten_gb300 import synthetic
    hp0 = dict(synthetic.ADAMW_DEFAULTS)
    sampler = ClockSampler(local).start()
    windows, points = [], []
    for P, n, nbytes, _ in sweep_points(gated_only=True):
        res = Resident(synthetic.workload(f"sweep:{P}:{n}"))
        fu = res.units[0]
        # a rough step time from a few eager steps sizes both timings
        el, kern, _, _ = time_resident(res, 3, 3, 1, device)
        est = max(kern / 3, 1e-6)
        eager_steps = int(max(10, min(2000, min_seconds / est)))
        t0 = time.time()
        el, kern, _, _ = time_resident(res, eager_steps, 2, 1, device)
        windows.append((t0, time.time()))
        n_graph = int(max(4, min(50, 5e9 // nbytes)))
        reps = int(max(3, -(-10 // n_graph), min_seconds / (est * n_graph)))
        g = time_graph(lambda t: res.launch(t, hp0), n_graph, reps, windows)
        points.append({"P": P, "n_ranks": n, "S_mod_8": fu.S % 8, "bytes_per_step": nbytes,
                       "graph_steps": n_graph * reps, "graph_ms": g * 1e3,
                       "graph_frac_of_measured_hbm": nbytes / g / 1e9 / hbm_peak,
                       "eager_steps": eager_steps, "eager_kernel_ms": kern / eager_steps * 1e3,
                       "eager_frac_of_measured_hbm": nbytes * eager_steps / kern / 1e9 / hbm_peak})
        del res, fu
        gc.collect()
    clock_info = sampler.stop(windows)
    torch.cuda.empty_cache()
    worst = min(points, key=lambda p: p["graph_frac_of_measured_hbm"])
    return {"gate": "fused step >= 0.80 of the measured HBM copy peak on every point moving "
                    ">= 4 x L2 per step",
            "timing": "graph: CUDA-graph replays of the fused launch, kernels back to back "
                      "(the gated figure); eager: per-launch CUDA events, one Python call per step",
            "n_points": len(points),
            "min_graph_frac_of_measured_hbm": worst["graph_frac_of_measured_hbm"],
            "min_point": f"P={worst['P']} N_d={worst['n_ranks']}",
            "min_eager_frac_of_measured_hbm": min(p["eager_frac_of_measured_hbm"]
                                                  for p in points),
            "points_at_or_above_0.80": sum(p["graph_frac_of_measured_hbm"] >= 0.80
                                           for p in points),
            "clocks": clock_info, "points": points}


def zero1_vs_zero2(device, hbm_peak, n_micro=4, steps=2):
    """One optimizer step of K = 4 micro-batches on the Llama-3-8B layer
    (N_d = 64) in the ZeRO-2 form (reduce-scatter into the sharded fp32
    accumulator every micro-step, fused last step) and in the ZeRO-1 form
    (each rank accumulates its full fp32 gradient locally, one reduce-scatter
    at the end).  Both are timed with CUDA events; bytes are algorithmic."""
    import gc
    import torch
    import fsdp_sharded_mixed_flatten_gb300 as zf
    from fsdp_sharded_mixed_flatten_gb300 import synthetic
    from fsdp_sharded_mixed_flatten_gb300.buffers import FlatUnit, aligned_rows, rows
    w = synthetic.workload("llama3-8b-layer")
    u = FlatUnit(w.units[0].numels, w.n_ranks, accum=True)
    for r in range(w.n_ranks):
        synthetic.fill_grad_(u.grads[r], u.P, w.grad_std, synthetic.seed_for("z1z2", r))
    full_acc = aligned_rows(w.n_ranks, u.P_pad, torch.float32, device, 0)
    hp = dict(synthetic.ADAMW_DEFAULTS)
    N, P_pad = w.n_ranks, u.P_pad

    def zero2(t):
        for k in range(1, n_micro + 1):
            zf.zero_step(u.grad_rows(), *u.state_rows(), u.accum_rows(), k, n_micro,
                         u.param_rows(), u.layout, dict(hp, step=t))

    def zero1(t):
        for k in range(1, n_micro + 1):
            zf.zero1_accumulate(u.grad_rows(), rows(full_acc), k == 1, u.layout)
        zf.zero1_step(rows(full_acc), n_micro, *u.state_rows(), u.param_rows(), u.layout,
                      dict(hp, step=t))

    out = {}
    b2 = unit_bytes(P_pad, N, n_micro=n_micro)
    b1 = P_pad * N * (6 + 10 * (n_micro - 1)) + P_pad * (4 * N + 26)
    for name, fn, nbytes in (("zero2", zero2, b2), ("zero1", zero1, b1)):
        for t in range(1, 3):
            fn(t)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for t in range(steps):
            fn(100 + t)
        b.record()
        torch.cuda.synchronize()
        el = a.elapsed_time(b) / 1e3 / steps
        out[name] = {"ms_per_step": el * 1e3, "bytes_per_step": nbytes,
                     "gbs": nbytes / el / 1e9, "frac_of_measured_hbm": nbytes / el / 1e9 / hbm_peak}
    out["zero1_over_zero2_time"] = out["zero1"]["ms_per_step"] / out["zero2"]["ms_per_step"]
    del u, full_acc
    gc.collect()
    torch.cuda.empty_cache()
    return out


def run_ours(args, ws, rank, local):
    import gc
    import torch
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device for --impl ours")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    init_dist(ws, "nccl")
    import fsdp_sharded_mixed_flatten_gb300 as zf
    from fsdp_sharded_mixed_flatten_gb300 import synthetic
    zf.load()   # fails loudly if the CUDA library was not built
    hbm_peak, peak_kind = peaks()
    if args.sweep:
        return run_sweep(args, device, hbm_peak)

    w = synthetic.workload(args.workload)
    streamed = args.workload.startswith("7.5b")      # one gradient buffer for every unit
    if args.variant == "clip":
        res = ClipResident(w, max_norm=1.0)
    elif args.variant == "per-param":
        res = PerParamResident(w)
    elif args.variant == "zero1":
        res = Zero1Resident(w)
    else:
        res = Resident(w, shared_grads=streamed)
    clocks = ClockSampler(local)
    el, kern, launches, clock_info = time_resident(res, args.steps, args.warmup, ws, device,
                                                   clocks=clocks)
    value = ws * res.numel * args.steps / el
    n_launch = res.launches_per_step
    achieved = res.bytes * args.steps / kern / 1e9
    traffic = None
    if args.variant == "plain" and w.n_micro == 1:
        aligned = all(fu.S % 8 == 0 for fu in res.units)
        traffic = recorded_traffic(traffic_class(w.n_ranks, aligned),
                                   sum(fu.P_pad for fu in res.units))
    e2e = None
    if not args.no_e2e and args.variant == "plain" and w.n_micro == 1:
        if streamed:
            e2e_steps, e2e_warm = min(args.steps, 3), 1
            e2e_el, h2d, d2h, n_rows = time_e2e_streamed(res, e2e_steps, e2e_warm, ws, device)
            how = ("every unit's gradient rows copied in and its parameters copied out each step, "
                   "unit by unit through two device gradient buffers; SM loads/stores through "
                   "the pinned buffers' device mapping (ZERO_HOST_SM_COPY); "
                   f"{n_rows} distinct host gradient rows for the {w.n_ranks} ranks")
        else:
            e2e_steps, e2e_warm = args.steps, args.warmup
            e2e_el, h2d, d2h = time_e2e(res, e2e_steps, e2e_warm, ws, device)
            how = ("SM loads/stores through the pinned buffers' device mapping "
                   "(ZERO_HOST_SM_COPY)")
        e2e = {"value": ws * res.numel * e2e_steps / e2e_el, "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "steps": e2e_steps, "warmup": e2e_warm, "ms_per_step": e2e_el / e2e_steps * 1e3,
               "transport": how}
    step_bytes = res.bytes
    units_desc = {"units": len(res.units), "params": res.numel,
                  "padded_elements": sum(getattr(fu, "P_pad", getattr(fu, "numel", 0))
                                         for fu in res.units)}
    grad_bytes = w.n_ranks * sum(synthetic.padded(u.numel, w.n_ranks) for u in
                                 (w.units[:1] if streamed else w.units)) * 2
    del res
    gc.collect()
    torch.cuda.empty_cache()

    extra = {}
    if not args.no_extra:
        if args.workload != "7.5b":
            extra["7.5B-32units-Nd64-streamed-grads"] = secondary("7.5b", 5, 3, ws, device,
                                                                  hbm_peak, shared=True)
        if args.workload != "gpt2-small":
            extra["gpt2-small-124M-13units-Nd8"] = secondary("gpt2-small", 20, 3, ws, device,
                                                             hbm_peak)
        extra["llama3-8b-decoder-layer-Nd64"] = secondary("llama3-8b-layer", 10, 3, ws, device,
                                                          hbm_peak)
        extra["7.5B-32units-Nd64-fp32-accum-4-micro"] = secondary("7.5b-accum", 2, 1, ws, device,
                                                                  hbm_peak, shared=True)
        extra["llama3-8b-layer-K4-zero2-vs-zero1"] = zero1_vs_zero2(device, hbm_peak)
        extra["gpt2-small-global-norm-clip"] = timed_extra(
            ClipResident(synthetic.workload("gpt2-small"), max_norm=1.0), 20, 3, ws, device,
            hbm_peak)
        extra["gpt2-small-fsdp2-per-parameter-148-units"] = timed_extra(
            PerParamResident(synthetic.workload("gpt2-small")), 20, 3, ws, device, hbm_peak)
        extra["llama3-8b-layer-fsdp2-per-parameter-9-units"] = timed_extra(
            PerParamResident(synthetic.workload("llama3-8b-layer")), 5, 3, ws, device, hbm_peak)
        if not args.no_sweep:
            extra["sweep_gated"] = sweep_gated(device, hbm_peak, local)

    base = cpu_baseline(args.workload) if (rank == 0 and ws == 1 and not args.no_cpu) else None
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": workload_label(args.workload), "variant": args.variant,
                   "seed": args.seed,
                   "n_ranks_logical": w.n_ranks, **units_desc,
                   "storage": "bf16 grads/params, fp32 master/m/v", "n_out": 1,
                   "bytes_per_step": step_bytes,
                   "hbm_gbs_per_step": step_bytes / (el / args.steps) / 1e9,
                   "l2": "inputs larger than L2 (%.2f GB of gradients read per unit pass)" % (
                       grad_bytes / 1e9),
                   "gradients": ("one N_d x P_pad buffer read by every unit in turn (streamed "
                                 "unit by unit)" if streamed else "resident per unit"),
                   "parallelism": f"replicas x{ws}" if ws > 1 else "1 GPU, N_d logical ranks"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "peak_kind": peak_kind,
                     "kernel": ("fused_step_kernel" if os.environ.get("ZERO_STEP_KERNEL") == "direct"
                                else "staged_step_kernel"),
                     "launches_per_step": n_launch,
                     "algorithmic_bytes_per_launch": step_bytes / n_launch,
                     "traffic": traffic / n_launch if traffic is not None else None,
                     "traffic_source": ("DRAM read+write bytes per padded element from a small "
                                        "ncu capture of the same kernel form, scaled to this "
                                        "launch's elements (profiles/fused_step_traffic.json)")
                     if traffic is not None else None},
        "cpu_baseline": base,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clock_info,
        "workloads": extra,
    }
    if rank == 0:
        print(json.dumps(line))
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="7.5b",
                    help="7.5b (default) | 7.5b-accum | gpt2-small | llama3-8b-layer | tiny | "
                         "sweep:<P>:<N_d>")
    ap.add_argument("--variant", default="plain", choices=["plain", "clip", "per-param", "zero1"],
                    help="the timed step: plain (default), with global-norm clipping, as FSDP2 "
                         "per-parameter units, or the ZeRO-1 form of 4 micro-steps (first unit)")
    ap.add_argument("--no-extra", action="store_true", help="skip the secondary workloads")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer leg")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline")
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the gated sweep points of the default run")
    ap.add_argument("--sweep", action="store_true",
                    help="fused vs unfused over the flat-size x N_d sweep (JSON line per point)")
    ap.add_argument("--sweep-sizes", default="", help="comma-separated flat sizes for --sweep")
    ap.add_argument("--seed", type=int, default=None,
                    help="base seed of the synthetic draws (default: the library's fixed base)")
    args = ap.parse_args()
    from fsdp_sharded_mixed_flatten_gb300 import synthetic
    if args.seed is not None:
        synthetic.BASE_SEED = args.seed
    args.seed = synthetic.BASE_SEED
    if args.workload not in WORKLOAD_NAMES and not args.workload.startswith("sweep:"):
        ap.error(f"unknown workload {args.workload}")
    if args.warmup < 3:
        args.warmup = 3
    ws, rank, local = dist_env()
    if args.impl == "reference":
        return run_reference(args, ws, rank)
    return run_ours(args, ws, rank, local)


if __name__ == "__main__":
    sys.exit(main())
