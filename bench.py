"""Benchmark: exact attention forward + backward on one GB300 (or N replicas).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

A step is one forward and one backward pass of the whole workload through the
C ABI on inputs already resident in HBM; L2 is flushed (a 256 MiB write)
before every timed step and the flush is outside the timed events (the decode
workload, whose K/V cache alone exceeds L2, rotates over copies of its inputs
instead, so no flush's dirty lines are written back inside its step). The JSON
line reports nominal fwd+bwd TFLOP/s (12 c N^2 d per head, recompute FLOPs
excluded and reported separately), the roofline of the dominant kernel, the
end-to-end number through host buffers (every step uploads its inputs and
downloads its outputs; the copies overlap the neighbouring steps' compute, and
the serial schedule is reported beside it), the oracle on host cores, peak
activation memory and the SM clocks seen while timing.

--impl reference times the fp64 CPU oracle instead (the only reference this
method has): each step is a bounded sample of heads of the same workload.
Under torchrun each rank runs the workload on its own GPU (heads are
independent: weak scaling, no collective on the data path).
"""

from __future__ import annotations

import argparse
import copy
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "attention fwd+bwd TFLOP/s (bf16, 1×GB300) and % of tensor-core peak; peak mem"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while it runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.t_start = self.t_stop = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=timestamp," + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            rows.append((ts, parts))
        inside = [r for ts, r in rows if self.t_start and self.t_stop and self.t_start <= ts <= self.t_stop + 0.1]
        use = inside or rows
        sm = [float(r[1]) for r in use if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in use if r[2].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in use:
            for name, val in zip(names, r[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(inside), "samples_total": len(rows)}


# ------------------------------------------------------------------ multi-rank aggregation
def job_throughput(ms_local: float, units_local: float, device=None):
    """Whole-job rate over all ranks: every rank processes its own copy of the
    workload (heads are independent, no collective on the data path), so the
    job takes the slowest rank's time and does world_size times the units.
    Returns (ms_max, total_units_per_s). Single process: the local values."""
    import torch
    ws = 1
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        ws = torch.distributed.get_world_size()
    ms = float(ms_local)
    units = float(units_local)
    if ws > 1:
        t = torch.tensor([ms, units], dtype=torch.float64, device=device)
        tmax = t.clone()
        torch.distributed.all_reduce(tmax, op=torch.distributed.ReduceOp.MAX)
        tsum = t.clone()
        torch.distributed.all_reduce(tsum, op=torch.distributed.ReduceOp.SUM)
        ms, units = float(tmax[0]), float(tsum[1])
    return ms, units / (ms * 1e-3)


# ------------------------------------------------------------------ oracle on host cores
ORACLE_ROWS = 2048  # query rows per oracle unit on long rows


def oracle_units(w):
    """Units of oracle work over a workload, in order: whole heads up to 4096 rows; beyond
    that the last ORACLE_ROWS query rows of each head (with all keys), the heaviest rows of a
    causal head, computed by the oracle as a problem of ORACLE_ROWS queries over N_k keys
    aligned with the last keys (exactly those rows' share of the head's work)."""
    r = w.N if w.N <= 4096 else ORACLE_ROWS
    return [(b, h, w.N - r) for b in range(w.B) for h in range(w.H)]


def oracle_sample(w, x, budget_s: float, max_heads=None):
    """Time the fp64 oracle on as many units of the workload as fit in budget_s."""
    from oracle import ref

    f64 = lambda t: t.to(dtype=__import__("torch").float64).numpy()  # noqa: E731
    kv = None if x["kv_len"] is None else x["kv_len"].numpy()
    units = oracle_units(w)
    done, flops = 0, 0.0
    t0 = time.perf_counter()
    for b, h, r0 in units:
        q, do = (f64(x[n][b, h, r0:]) for n in ("q", "do"))
        k, v = (f64(x[n][b, h]) for n in ("k", "v"))
        kl = None if kv is None else int(kv[b])
        nq = w.N - r0
        if w.infer:  # forward only
            ref.head_forward(q, k, v, w.scale, w.causal, kl)
            flops += 4 * w.d * workloads.visible_pairs(nq, w.nk, w.causal, kl)
        else:
            ref.head_backward(q, k, v, do, w.scale, w.causal, kl)
            flops += 12 * w.d * workloads.visible_pairs(nq, w.nk, w.causal, kl)
        done += 1
        if time.perf_counter() - t0 > budget_s or (max_heads and done >= max_heads):
            break
    dt = time.perf_counter() - t0
    cores = len(os.sched_getaffinity(0))
    what = "heads" if units and units[0][2] == 0 else f"(head, last {w.N - units[0][2]} query rows) units"
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{done} of {len(units)} {what} of {w.name} (fp64 numpy, {'fwd' if w.infer else 'fwd+bwd'}, "
                      f"S and P materialised), "
                      f"{dt:.1f} s", "seconds": dt, "heads": done}


# ------------------------------------------------------------------ traffic record
def traffic_record(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if its source hash still matches."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}_traffic.txt")
    try:
        with open(path) as f:
            kv = dict(line.split(":", 1) for line in f if ":" in line and not line.startswith("#"))
    except OSError:
        return None
    src = kv.get("source_sha256", "").strip()
    files = [s.strip() for s in kv.get("source_files", "").split(",") if s.strip()]
    h = hashlib.sha256()
    for fn in files:
        with open(os.path.join(ROOT, fn), "rb") as f:
            h.update(f.read())
    if not files or h.hexdigest() != src:
        return None
    try:
        return float(kv["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def io_accounting(w, kv_len=None, measured=None):
    """HBM bytes of one fwd+bwd step under the pages' access model, per workload.

    compulsory: what any exact method must move (bf16 tensors, fp32 LSE): the forward
    reads Q, K, V and writes O, LSE; the backward reads Q, K, V, O, dO, LSE, writes dQ,
    dK, dV, and here also writes and reads -D, -LSE2 (fp32) and the fp32 dQ accumulator.
    standard: the same plus the N x N matrices of standard attention in bf16, written
    and read back (S written, S read, P written, P read in the forward; P read in the
    backward: five passes of 2 bytes per entry, the IO analysis' N^2 term).
    tiled_term: N^2 d^2 / M elements (bf16) per head for M = 116736 on-chip elements
    (228 KB of shared memory in bf16): the order of the tiled method's HBM accesses.
    measured: DRAM bytes of the two main kernels from the committed ncu records, if any;
    step_bytes adds the modelled bytes of the two streaming backward kernels to them.
    """
    heads = w.B * w.H
    N, Nk, d = w.N, w.nk, w.d
    npad = (N + 127) // 128 * 128
    fwd = heads * (2 * N * d + 2 * 2 * Nk * d + 2 * N * d + 4 * N)
    bwd = heads * (2 * N * d + 2 * 2 * Nk * d + 2 * 2 * N * d + 4 * N + 2 * N * d + 2 * 2 * Nk * d
                   + 2 * 8 * npad + 2 * 4 * npad * d)
    if kv_len is not None:  # key padding: only valid keys' columns exist in the N x N matrix
        cols = float(sum(int(x) for x in kv_len)) * w.H * N
    else:
        cols = float(heads) * N * Nk
    standard = fwd + bwd + 5 * 2 * cols
    tiled_term = heads * 2.0 * N * N * d * d / 116736
    # the two streaming kernels of the backward move what they must: pre reads O, dO, LSE and
    # writes -D, -LSE2 and the zeroed accumulator; the rounding reads the accumulator, writes dQ
    small = heads * (2 * 2 * N * d + 4 * N + 8 * npad + 4 * npad * d) + heads * (4 * npad * d + 2 * N * d)
    out = {"compulsory_bytes": fwd + bwd, "standard_attention_bytes": standard,
           "tiled_order_term_bytes": tiled_term,
           "model": "bf16 tensors, fp32 LSE / D / dQ accumulator; standard adds 5 passes over N x N bf16"}
    if measured:
        out["measured_main_kernels_bytes"] = measured
        out["pre_and_rounding_bytes_model"] = small
        out["step_bytes"] = measured + small
        out["standard_over_step"] = standard / (measured + small)
    return out


def source_hash(files):
    h = hashlib.sha256()
    for fn in files:
        with open(os.path.join(ROOT, fn), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


E2E_PIPELINED = ("pipelined: each step uploads its inputs (pinned host -> device, copy stream), runs fwd+bwd and "
                 "downloads O, LSE, dQ, dK, dV (device -> pinned host, a second copy stream); uploads and downloads "
                 "overlap the neighbouring steps' compute, two device buffer sets, L2 flushed before every step "
                 "inside the timed region")
E2E_SERIAL = ("upload, compute, download, synchronise, step after step; L2 flushed before each step, outside the "
              "timed region")


def pipelined_e2e(dev, sets, host_in, host_out, flush, steps):
    """Milliseconds per step of `steps` end-to-end steps whose host copies overlap compute.

    Each step uploads its inputs from pinned host memory, runs the whole path and downloads
    its outputs, as in a training or serving loop that prefetches. Step i's upload (one
    copy stream) runs while step i - 1 computes. Its download (another copy stream) runs
    while step i + 1 computes. `sets` are two device buffer sets used in turn, each an
    (inputs, outputs, step) triple. A set is reused only after the step two back has
    finished with it: its compute for the inputs, its download for the outputs. L2 is
    flushed on the compute stream before every step's kernels, inside the timed region.
    The timed region runs from the first upload to the last download, between device
    synchronisations."""
    import torch
    comp = torch.cuda.current_stream(dev)
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def run(k):
        ready = [torch.cuda.Event() for _ in range(k)]
        done = [torch.cuda.Event() for _ in range(k)]
        read = [torch.cuda.Event() for _ in range(k)]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        t0.record(comp)
        up.wait_event(t0)
        for i in range(k):
            ins, outs, step = sets[i % 2]
            with torch.cuda.stream(up):
                if i >= 2:
                    up.wait_event(done[i - 2])  # the set's inputs are no longer read
                for dst, src in zip(ins, host_in):
                    dst.copy_(src, non_blocking=True)
                ready[i].record(up)
            comp.wait_event(ready[i])
            if i >= 2:
                comp.wait_event(read[i - 2])  # the set's outputs have been downloaded
            flush.zero_()
            step()
            done[i].record(comp)
            with torch.cuda.stream(down):
                down.wait_event(done[i])
                for dst, src in zip(host_out, outs):
                    dst.copy_(src, non_blocking=True)
                read[i].record(down)
        comp.wait_event(read[k - 1])
        t1.record(comp)
        t1.synchronize()
        return t0.elapsed_time(t1)

    run(2)  # the streams, events and second buffer set warmed up
    return run(steps) / steps


# ------------------------------------------------------------------ main arms
def run_reference(args, w):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    x = workloads.make_inputs(w)
    budget = min(20.0, 150.0 / max(1, args.steps + args.warmup))  # whole run within a few minutes
    sample = oracle_sample_packed if w.packed else oracle_sample
    for _ in range(args.warmup):
        sample(w, x, budget, 1)
    vals, secs, heads = [], 0.0, 0
    for _ in range(args.steps):
        r = sample(w, x, budget)
        vals.append(r["value"])
        secs += r["seconds"]
        heads += r["heads"]
    value = statistics.median(vals)
    cores = len(os.sched_getaffinity(0))
    unit = "heads" if w.packed or oracle_units(w)[0][2] == 0 else f"(head, last {ORACLE_ROWS} query rows) units"
    sample = (f"each step: the fp64 oracle on as many {unit} of {w.name} as fit in {budget:.1f} s "
              f"({heads} over {args.steps} steps)")
    line = {
        "impl": "reference", "metric": INFER_METRIC if w.infer else METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / max(1, args.steps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1), bf16-rounded, upcast to fp64)",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "N_k": w.nk, "d": w.d, "causal": w.causal},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


class TrainingSetup:
    """One workload's tensors on the device and its fwd+bwd step through the C ABI."""

    KERNELS = ["fwd_kernel", "bwd_pre_kernel", "bwd_kernel", "dq_convert_kernel"]

    def __init__(self, w, dev, lib, flush):
        import ctypes

        import torch

        from io_aware_exact_04_gb300 import _lib
        self.w, self.dev, self.lib, self.flush = w, dev, lib, flush
        self.x = x = workloads.make_inputs(w, seed=0)
        B, H, N, Nk, d = w.B, w.H, w.N, w.nk, w.d
        self.q, self.k, self.v, self.do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
        self.kv = None if x["kv_len"] is None else x["kv_len"].to(dev)
        self.o = torch.empty_like(self.q)
        self.lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
        self.dq, self.dk, self.dv = torch.empty_like(self.q), torch.empty_like(self.k), torch.empty_like(self.k)
        self.wsb = int(lib.fa_backward_workspace_size(B, H, N, d))
        self.work = torch.empty(self.wsb, dtype=torch.uint8, device=dev)
        self.stream = torch.cuda.current_stream(dev)
        self.sp = ctypes.c_void_p(self.stream.cuda_stream)
        self._check = _lib.check
        self.fl = workloads.flop_counts(w, x["kv_len"])

    @staticmethod
    def _p(t):
        import ctypes
        return ctypes.c_void_p(t.data_ptr()) if t is not None else None

    def fwd(self):
        w, P = self.w, self._p
        self._check(self.lib.fa_forward_qk(P(self.q), P(self.k), P(self.v), P(self.o), P(self.lse), w.B, w.H, w.N,
                                           w.nk, w.d, w.scale, int(w.causal), P(self.kv), self.sp), "fwd")

    def bwd_stage(self, s):
        w, P = self.w, self._p
        self._check(self.lib.fa_backward_stage_qk(s, P(self.q), P(self.k), P(self.v), P(self.o), P(self.do),
                                                  P(self.lse), P(self.dq), P(self.dk), P(self.dv), w.B, w.H, w.N,
                                                  w.nk, w.d, w.scale, int(w.causal), P(self.kv), P(self.work),
                                                  self.wsb, self.sp), "bwd")

    def step(self, ev=None):
        if ev is None:
            self.fwd()
            for s in range(3):
                self.bwd_stage(s)
            return
        ev[0].record(self.stream)
        self.fwd()
        ev[1].record(self.stream)
        for s in range(3):
            self.bwd_stage(s)
            ev[2 + s].record(self.stream)

    def status(self, when):
        import ctypes
        detail = (ctypes.c_int * 4)()
        if self.lib.fa_get_last_device_status_detail(self.sp, detail) != 0:
            raise RuntimeError(f"device status {when}: {list(detail)}")

    def warmup(self, n):
        import torch
        for _ in range(max(3, n)):
            self.flush.zero_()
            self.step()
        torch.cuda.synchronize(self.dev)
        self.status("after warm-up")

    def time_steps(self, steps):
        """(step ms total, per-kernel ms totals, step ms with an event after every kernel).

        Step time: events at step boundaries only. The four kernels of a step are launched with
        programmatic dependent launch, and an event recorded between two of them would serialise
        that overlap, so the per-kernel breakdown comes from a second timed pass of the same
        steps with an event after every kernel."""
        import torch
        step_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
        events = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(steps)]
        for i in range(steps):
            self.flush.zero_()
            step_ev[i][0].record(self.stream)
            self.step()
            step_ev[i][1].record(self.stream)
        torch.cuda.synchronize(self.dev)
        for i in range(steps):
            self.flush.zero_()
            self.step(events[i])
        torch.cuda.synchronize(self.dev)
        per_kernel = {k: 0.0 for k in self.KERNELS}
        total_ms = sum(ev[0].elapsed_time(ev[1]) for ev in step_ev)
        for ev in events:
            t = [ev[0].elapsed_time(ev[j]) for j in range(1, 5)]
            per_kernel["fwd_kernel"] += t[0]
            per_kernel["bwd_pre_kernel"] += t[1] - t[0]
            per_kernel["bwd_kernel"] += t[2] - t[1]
            per_kernel["dq_convert_kernel"] += t[3] - t[2]
        with_events = sum(ev[0].elapsed_time(ev[4]) for ev in events)
        return total_ms, per_kernel, with_events

    def activation_memory(self):
        """Peak device memory that one fwd+bwd through the public API holds beyond its inputs
        (Q, K, V, dO) and its gradient outputs (dQ, dK, dV), as torch's allocator measures it:
        O and LSE from the forward call, the backward call's workspace."""
        import torch

        from io_aware_exact_04_gb300 import api
        w = self.w
        torch.cuda.synchronize(self.dev)
        base = torch.cuda.memory_allocated(self.dev)
        torch.cuda.reset_peak_memory_stats(self.dev)
        o, lse = api.forward(self.q, self.k, self.v, causal=w.causal, kv_len=self.kv)
        api.backward(self.q, self.k, self.v, o, self.do, lse, causal=w.causal, kv_len=self.kv,
                     dq=self.dq, dk=self.dk, dv=self.dv)
        torch.cuda.synchronize(self.dev)
        peak = torch.cuda.max_memory_allocated(self.dev) - base
        del o, lse
        self.status("after the memory measurement")
        return int(peak)


# the long-context sweep of the GPT-2 memory-table configuration (12 heads, d 64, causal)
LONG_SWEEP = ["long2048", "long8192", "long16384", "long32768"]


def sweep_entry(w, setup, peaks, steps):
    """TFLOP/s and measured activation memory of one workload of the sweep."""
    setup.warmup(3)
    total, per_kernel, _ = setup.time_steps(steps)
    ms = total / steps
    fl = setup.fl
    nominal = fl["fwd_bwd_nominal"] / (ms * 1e-3) / 1e12
    executed = fl["fwd_bwd_executed"] / (ms * 1e-3) / 1e12
    mem = setup.activation_memory()
    peak = float(peaks["bf16_tflops"])
    bwd_ms = (per_kernel["bwd_pre_kernel"] + per_kernel["bwd_kernel"] + per_kernel["dq_convert_kernel"]) / steps
    return {"N": w.N, "ms_per_step": ms, "tflops_nominal": nominal, "tflops_executed": executed,
            "pct_of_peak": 100 * nominal / peak, "pct_of_peak_executed": 100 * executed / peak,
            "fwd_tflops": fl["fwd"] / (per_kernel["fwd_kernel"] / steps * 1e-3) / 1e12,
            "bwd_tflops_nominal": fl["bwd_nominal"] / (bwd_ms * 1e-3) / 1e12,
            "bwd_kernel_frac": (fl["bwd_nominal"] + fl["bwd_recompute"])
            / (per_kernel["bwd_kernel"] / steps * 1e-3) / 1e12 / peak,
            "peak_act_mem_bytes": mem, "act_bytes_per_head_row": mem / (w.B * w.H * w.N),
            "std_attention_matrix_bytes_bf16": w.B * w.H * w.N * w.nk * 2}


def standard_records():
    """Measured DRAM bytes and times of standard (materialising) attention and of this
    library's step on the same workloads, from the committed ncu records."""
    out = {}
    for wl in ("gpt2", "long8192"):
        rec = {}
        for kind in ("standard_attention", "flash_step"):
            path = os.path.join(ROOT, "profiles", f"{kind}_{wl}_dram.txt")
            try:
                with open(path) as f:
                    kv = dict(line.split(":", 1) for line in f if ":" in line and not line.startswith("#"))
                files = [x.strip() for x in kv.get("source_files", "").split(",") if x.strip()]
                if files and source_hash(files) != kv.get("source_sha256", "").strip():
                    continue  # this library's kernels changed since the record was taken
                rec[kind + "_dram_bytes"] = float(kv["dram_bytes_per_step"])
            except (OSError, KeyError, ValueError):
                pass
        if len(rec) == 2:
            rec["standard_over_flash"] = rec["standard_attention_dram_bytes"] / rec["flash_step_dram_bytes"]
            out[wl] = rec
    return out


def run_gpu(args, w):
    import torch

    from io_aware_exact_04_gb300 import _lib, memmodel

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    lib = _lib.load("libfa.so")
    peaks, peak_src = load_peaks()

    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    S = TrainingSetup(w, dev, lib, flush)
    x = S.x
    B, H, N, Nk, d = w.B, w.H, w.N, w.nk, w.d
    S.warmup(args.warmup)
    # peak activation memory, measured: what one fwd+bwd holds besides inputs and gradients
    act_bytes = S.activation_memory()
    S.warmup(3)

    sampler = ClockSampler(local if "CUDA_VISIBLE_DEVICES" not in os.environ else 0)
    if rank == 0:
        sampler.start()
        time.sleep(0.3)
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    sampler.mark("t_start")
    total_ms, per_kernel, with_events = S.time_steps(args.steps)
    sampler.mark("t_stop")
    if ws > 1:
        torch.distributed.barrier()
    S.status("after timing")
    fl = S.fl
    ms_step, nominal_rate = job_throughput(total_ms / args.steps, fl["fwd_bwd_nominal"], device=dev)
    value = nominal_rate / 1e12
    executed = value * fl["fwd_bwd_executed"] / fl["fwd_bwd_nominal"]

    # dominant kernel and its roofline (tensor-bound: algorithmic flops per launch / event time)
    avg = {kname: t / args.steps for kname, t in per_kernel.items()}
    dom = max(avg, key=avg.get)
    alg_flops = {"fwd_kernel": fl["fwd"], "bwd_kernel": fl["bwd_nominal"] + fl["bwd_recompute"]}
    if dom in alg_flops:
        achieved = alg_flops[dom] / (avg[dom] * 1e-3) / 1e12
        peak = float(peaks["bf16_tflops"])
        traffic = traffic_record(dom, w.name)
        roof = {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": traffic,
                "peak_source": f"{peak_src} bf16 dense (burst)", "avg_launch_ms": avg[dom],
                "flops_per_launch": alg_flops[dom]}
    else:  # a memory-bound helper dominating would be reported against HBM
        nbytes = {"bwd_pre_kernel": B * H * N * d * 2 * 2 + B * H * (N + 127) // 128 * 128 * (8 + 4 * d),
                  "dq_convert_kernel": B * H * N * d * (4 + 2)}[dom]
        achieved = nbytes / (avg[dom] * 1e-3) / 1e9
        peak = float(peaks["hbm_gbs"])
        roof = {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": traffic_record(dom, w.name), "peak_source": peak_src,
                "avg_launch_ms": avg[dom]}

    # end to end through host buffers: H2D inputs, fwd+bwd, D2H outputs, every step
    hq, hk, hv, hdo = (x[n].pin_memory() for n in ("q", "k", "v", "do"))
    ho, hdq = (torch.empty_like(hq).pin_memory() for _ in range(2))
    hdk, hdv = (torch.empty_like(hk).pin_memory() for _ in range(2))
    hlse = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hdo))
    d2h = sum(t.numel() * t.element_size() for t in (ho, hlse, hdq, hdk, hdv))
    e2e_steps = max(3, min(args.steps, 50))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_ms = 0.0
    stream = S.stream
    for i in range(e2e_steps + 2):
        flush.zero_()
        torch.cuda.synchronize(dev)
        e0.record(stream)
        S.q.copy_(hq, non_blocking=True)
        S.k.copy_(hk, non_blocking=True)
        S.v.copy_(hv, non_blocking=True)
        S.do.copy_(hdo, non_blocking=True)
        S.step()
        ho.copy_(S.o, non_blocking=True)
        hlse.copy_(S.lse, non_blocking=True)
        hdq.copy_(S.dq, non_blocking=True)
        hdk.copy_(S.dk, non_blocking=True)
        hdv.copy_(S.dv, non_blocking=True)
        e1.record(stream)
        e1.synchronize()
        if i >= 2:
            e2e_ms += e0.elapsed_time(e1)
    e2e_ms /= e2e_steps
    serial_ms, serial_rate = job_throughput(e2e_ms, fl["fwd_bwd_nominal"], device=dev)
    # ... and pipelined: the same steps with their copies overlapping the neighbouring steps'
    # compute (two device buffer sets; the workspace and the compute stream are shared)
    T = copy.copy(S)
    T.q, T.k, T.v, T.do = (torch.empty_like(t) for t in (S.q, S.k, S.v, S.do))
    T.o, T.lse, T.dq, T.dk, T.dv = (torch.empty_like(t) for t in (S.o, S.lse, S.dq, S.dk, S.dv))
    sets = [((b.q, b.k, b.v, b.do), (b.o, b.lse, b.dq, b.dk, b.dv), b.step) for b in (S, T)]
    e2e_ms = pipelined_e2e(dev, sets, (hq, hk, hv, hdo), (ho, hlse, hdq, hdk, hdv), flush, e2e_steps)
    S.status("after the end-to-end steps")
    e2e_ms, e2e_rate = job_throughput(e2e_ms, fl["fwd_bwd_nominal"], device=dev)
    e2e_val = e2e_rate / 1e12
    del T, sets

    clocks = sampler.stop() if rank == 0 else None

    # the rest of the long-context sweep (same configuration, other N): TFLOP/s and measured
    # activation memory at each N, so that linearity in N is observed, not assumed
    sweep = None
    if w.name in LONG_SWEEP and not args.no_sweep:
        del S
        torch.cuda.empty_cache()
        sweep = []
        for name in LONG_SWEEP:
            ww = workloads.WORKLOADS[name]
            if name == w.name:
                sweep.append({"N": w.N, "ms_per_step": ms_step, "tflops_nominal": value, "tflops_executed": executed,
                              "pct_of_peak": 100 * value / float(peaks["bf16_tflops"]),
                              "pct_of_peak_executed": 100 * executed / float(peaks["bf16_tflops"]),
                              "peak_act_mem_bytes": act_bytes, "act_bytes_per_head_row": act_bytes / (B * H * N),
                              "std_attention_matrix_bytes_bf16": B * H * N * Nk * 2, "source": "main timing above"})
                continue
            st = TrainingSetup(ww, dev, lib, flush)
            sweep.append(sweep_entry(ww, st, peaks, max(10, min(args.steps, 100))))
            del st
            torch.cuda.empty_cache()
        per_row = [e["act_bytes_per_head_row"] for e in sweep]
        sweep = {"workloads": LONG_SWEEP, "entries": sweep,
                 "act_bytes_per_head_row_spread": (max(per_row) - min(per_row)) / min(per_row),
                 "note": "each N: L2 flushed before every step; peak memory = torch max_memory_allocated over "
                         "one fwd+bwd through the public API minus the resident inputs and gradient outputs"}

    if ws > 1:
        torch.distributed.barrier()
    if rank != 0:
        return
    cpu = oracle_sample(w, x, budget_s=args.cpu_budget) if not args.no_cpu_baseline else None
    std = memmodel.training_memory(N, d_model=H * d, heads=H, layers=1)
    io = io_accounting(w, x["kv_len"], measured=(
        (traffic_record("fwd_kernel", w.name) or 0) + (traffic_record("bwd_kernel", w.name) or 0)
        if traffic_record("fwd_kernel", w.name) and traffic_record("bwd_kernel", w.name) else None))
    io["standard_measured"] = standard_records()
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) inputs, bf16)",
        "config": {"workload": w.name, "B": B, "H": H, "N": N, "N_k": Nk, "d": d, "causal": w.causal,
                   "key_padding": w.padded, "l2": "flushed before every step (256 MiB write, untimed)",
                   "flops": "nominal fwd+bwd 12*c*N*Nk*d per head (c = 1/2 causal), recompute excluded",
                   "parallelism": f"replicas x{ws} (heads independent)"},
        "tflops_executed": executed,
        "pct_of_peak": 100.0 * value / float(peaks["bf16_tflops"]),
        "pct_of_peak_executed": 100.0 * executed / float(peaks["bf16_tflops"]),
        "peak_source": f"{peak_src} MEASURED_PEAKS bf16_tflops" if peak_src == "measured" else "fallback 1900 TFLOP/s",
        "fwd_ms": avg["fwd_kernel"], "bwd_ms": avg["bwd_pre_kernel"] + avg["bwd_kernel"] + avg["dq_convert_kernel"],
        "fwd_tflops": fl["fwd"] / (avg["fwd_kernel"] * 1e-3) / 1e12,
        "bwd_tflops_nominal": fl["bwd_nominal"] / ((avg["bwd_pre_kernel"] + avg["bwd_kernel"] + avg["dq_convert_kernel"]) * 1e-3) / 1e12,
        "kernel_ms": avg,
        "kernel_ms_source": "second timed pass of the same steps, an event after every kernel",
        "step_ms_with_kernel_events": with_events / args.steps,
        "peak_act_mem_bytes": act_bytes,
        "peak_act_mem_source": "measured: torch max_memory_allocated over one fwd+bwd through the public API, "
                               "minus the resident inputs and gradient outputs (O, LSE and the backward workspace)",
        "act_bytes_per_head_row": act_bytes / (B * H * N),
        "std_attention_matrix_bytes_bf16": B * H * N * Nk * 2,
        "io": io,
        "std_attention_memmodel_gb_per_layer_B1": std["standard_gb"],
        "long_sweep": sweep,
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_val, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms, "steps": e2e_steps,
                "schedule": E2E_PIPELINED,
                "serial": {"value": serial_rate / 1e12, "ms_per_step": serial_ms, "schedule": E2E_SERIAL}},
        "gpu_launches": 4 * args.steps,
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ standard attention (comparison)
def run_standard(args, w):
    """Standard attention, forward and backward, with every N x N matrix in HBM: the
    comparison the pages' IO analysis makes (the tiled method against the one that writes S
    and P out and reads them back). PyTorch bf16 matmuls and softmax; not this library."""
    import torch

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peaks, peak_src = load_peaks()
    x = workloads.make_inputs(w, seed=0)
    B, H, N, Nk, d = w.B, w.H, w.N, w.nk, w.d
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    scale = w.scale
    keep = None
    if w.causal:
        i = torch.arange(N, device=dev)[:, None]
        j = torch.arange(Nk, device=dev)[None, :]
        keep = j <= i + (Nk - N)
    if x["kv_len"] is not None:
        kvm = torch.arange(Nk, device=dev)[None, :] < x["kv_len"].to(dev)[:, None]   # [B, Nk]
        kvm = kvm[:, None, None, :]
        keep = kvm if keep is None else (keep & kvm)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    drop = None if keep is None else ~keep
    qs = (q * scale).to(torch.bfloat16)  # the scale folded into Q once (not an N x N pass)

    # Every N x N matrix is a bf16 tensor in HBM; the elementwise steps run in place, so the
    # N x N passes are: S written; S read and written (mask); S read, P written (softmax); P read
    # twice (O, dV); dP written; dP read and written twice (- D, * P), giving dS; dS read twice.
    def step():
        s_ = torch.matmul(qs, k.transpose(-1, -2))                      # S = s Q K^T
        if drop is not None:
            s_.masked_fill_(drop, float("-inf"))
        p_ = torch.softmax(s_, dim=-1)                                   # P
        del s_
        o_ = torch.matmul(p_, v)                                         # O = P V
        dv_ = torch.matmul(p_.transpose(-1, -2), do)                     # dV = P^T dO
        ds_ = torch.matmul(do, v.transpose(-1, -2))                      # dP = dO V^T
        dd = (do.float() * o_.float()).sum(-1, keepdim=True).to(torch.bfloat16)  # D (per row)
        ds_.sub_(dd).mul_(p_)                                            # dS = P (dP - D)
        del p_
        dq_ = torch.matmul(ds_, k).mul_(scale)                           # dQ = s dS K
        dk_ = torch.matmul(ds_.transpose(-1, -2), q).mul_(scale)        # dK = s dS^T Q
        return o_, dq_, dk_, dv_

    for _ in range(max(3, args.warmup)):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    torch.cuda.reset_peak_memory_stats(dev)
    base = torch.cuda.memory_allocated(dev)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    for i in range(args.steps):
        flush.zero_()
        evs[i][0].record(stream)
        out = step()
        evs[i][1].record(stream)
        del out
    torch.cuda.synchronize(dev)
    peak_mem = torch.cuda.max_memory_allocated(dev) - base
    ms = sum(e[0].elapsed_time(e[1]) for e in evs) / args.steps
    fl = workloads.flop_counts(w, x["kv_len"])
    value = fl["fwd_bwd_nominal"] / (ms * 1e-3) / 1e12
    rec = standard_records().get(w.name)
    line = {"impl": "standard", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "dtype": "bf16", "data": "synthetic (seeded N(0,1) inputs, bf16)",
            "config": {"workload": w.name, "B": B, "H": H, "N": N, "N_k": Nk, "d": d, "causal": w.causal,
                       "method": "standard attention: S, P, dP, dS materialised in HBM (torch bf16 matmul, "
                                 "softmax; comparison only, not this library)",
                       "l2": "flushed before every step (256 MiB write, untimed)"},
            "pct_of_peak": 100.0 * value / float(peaks["bf16_tflops"]),
            "peak_mem_bytes_beyond_inputs": int(peak_mem),
            "dram": rec, "peak_source": peak_src}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ inference workloads
INFER_METRIC = "attention forward-only TFLOP/s (inference, split keys; bf16, 1×GB300); roofline in GB/s"


INFER_ROTATE_BYTES = 800 << 20  # inference inputs rotated over copies of at least this much in all


def infer_bytes(w):
    """Algorithmic bytes of one inference forward step: Q, K and V read once (bf16), O written
    (bf16). The partial results that a split head's CTAs exchange are not counted."""
    rows_q = w.B * w.H * w.N
    return 2 * rows_q * w.d + 2 * 2 * w.B * w.H * w.nk * w.d + 2 * rows_q * w.d


def infer_launches(w, n_split, sms, has_kv_len):
    """Kernels one fa_forward_split call launches. Decode (N_q <= 8) with n_split = 1: whole
    heads a CTA, one kernel. With n_split > 1: the stream-K kernel over G = min(SMs, 256,
    n_split B H, T) CTAs, plus the join of split heads when key padding is given or some CTA's
    run of key tiles starts inside a head. Otherwise: the split kernel and its combine
    (n_split = 1 with an LSE is the plain forward, which the bench does not use)."""
    if w.N > 8:
        return 2
    if n_split == 1:
        return 1
    bh, t_head = w.B * w.H, -(-w.nk // 128)
    t_max = max(1, bh * t_head)
    G = max(1, min(sms, 256, n_split * bh, t_max))
    split = has_kv_len or any((c * t_max // G) % t_head for c in range(1, G))
    return 2 if split else 1


def run_gpu_infer(args, w):
    """Forward only through fa_forward_split: a step is one split-key forward and its combine."""
    import ctypes

    import torch

    from io_aware_exact_04_gb300 import _lib

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    lib = _lib.load("libfa.so")
    peaks, peak_src = load_peaks()
    x = workloads.make_inputs(w, seed=0)
    B, H, N, Nk, d = w.B, w.H, w.N, w.nk, w.d
    # The K/V cache is larger than L2, so instead of a flush (whose dirty lines would be
    # written back during the next step's reads) the steps rotate over R copies of the inputs:
    # a step's inputs were last read R - 1 steps (at least 600 MB of other reads) earlier.
    in_bytes = sum(x[n].numel() * x[n].element_size() for n in ("q", "k", "v"))
    R = max(1, -(-INFER_ROTATE_BYTES // in_bytes))
    copies = [tuple(x[n].to(dev) for n in ("q", "k", "v")) for _ in range(R)]
    q, k, v = copies[0]
    kv = None if x["kv_len"] is None else x["kv_len"].to(dev)
    o = torch.empty_like(q)
    n_split = int(lib.fa_forward_split_count(B, H, N, Nk, d))
    wsb = int(lib.fa_forward_split_workspace_size(B, H, N, d, n_split))
    work = torch.empty(max(wsb, 1), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    sp = ctypes.c_void_p(stream.cuda_stream)
    P = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None  # noqa: E731

    def step(i=0):
        qi, ki, vi = copies[i % R]
        _lib.check(lib.fa_forward_split(P(qi), P(ki), P(vi), P(o), None, B, H, N, Nk, d, w.scale, int(w.causal),
                                        P(kv), n_split, P(work), wsb, sp), "fwd_split")

    for i in range(max(3, args.warmup)):
        step(i)
    torch.cuda.synchronize(dev)
    detail = (ctypes.c_int * 4)()
    if lib.fa_get_last_device_status_detail(sp, detail) != 0:
        raise RuntimeError(f"device status after warm-up: {list(detail)}")
    # The K steps run back to back between one pair of events, as a decode loop runs them (each
    # launch may start while the previous one drains); a second pass times every step between
    # events of its own (which serialises the launches) for comparison.
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    step_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    sampler = ClockSampler(local if "CUDA_VISIBLE_DEVICES" not in os.environ else 0)
    if rank == 0:
        sampler.start()
        time.sleep(0.3)
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    sampler.mark("t_start")
    ev0.record(stream)
    for i in range(args.steps):
        step(i)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    sampler.mark("t_stop")
    if ws > 1:
        torch.distributed.barrier()
    total_ms = ev0.elapsed_time(ev1)
    for i in range(args.steps):
        step_ev[i][0].record(stream)
        step(i)
        step_ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    isolated_ms = sum(e[0].elapsed_time(e[1]) for e in step_ev) / args.steps
    fwd_flops = 4.0 * d * workloads.visible_pairs(N, Nk, w.causal) * B * H
    ms_step, rate = job_throughput(total_ms / args.steps, fwd_flops, device=dev)
    value = rate / 1e12
    # roofline of the step's two launches together (the combine reads back only the shares'
    # small fp32 rows): algorithmic bytes over the event-timed step
    bytes_alg = infer_bytes(w)
    achieved = bytes_alg / (ms_step * 1e-3) / 1e9
    peak = float(peaks["hbm_gbs"])
    roof = {"bound": "hbm", "kernel": "decode_kernel (+ join of split heads): whole step", "achieved": achieved, "peak": peak,
            "unit": "GB/s", "frac": achieved / peak, "traffic": traffic_record("decode_kernel", w.name),
            "peak_source": f"{peak_src} hbm_gbs (copy)", "avg_launch_ms": ms_step,
            "bytes_per_launch": bytes_alg,
            "isolated_step_ms": isolated_ms, "isolated_frac": bytes_alg / (isolated_ms * 1e-3) / 1e9 / peak}
    # end to end through host buffers
    hq, hk, hv = (x[n].pin_memory() for n in ("q", "k", "v"))
    ho = torch.empty_like(hq).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
    d2h = ho.numel() * ho.element_size()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_steps, e2e_ms = max(3, min(args.steps, 50)), 0.0
    for i in range(e2e_steps + 2):
        torch.cuda.synchronize(dev)
        e0.record(stream)
        q.copy_(hq, non_blocking=True)
        k.copy_(hk, non_blocking=True)
        v.copy_(hv, non_blocking=True)
        step()
        ho.copy_(o, non_blocking=True)
        e1.record(stream)
        e1.synchronize()
        if i >= 2:
            e2e_ms += e0.elapsed_time(e1)
    e2e_ms, e2e_rate = job_throughput(e2e_ms / e2e_steps, fwd_flops, device=dev)
    clocks = sampler.stop() if rank == 0 else None
    if ws > 1:
        torch.distributed.barrier()
    if rank != 0:
        return
    cpu = oracle_sample(w, x, budget_s=args.cpu_budget) if not args.no_cpu_baseline else None
    line = {
        "metric": INFER_METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) inputs, bf16)",
        "config": {"workload": w.name, "B": B, "H": H, "N": N, "N_k": Nk, "d": d, "causal": w.causal,
                   "n_split": n_split, "lse": False,
                   "l2": f"no flush: inputs larger than L2, rotated over {R} copies ({R * in_bytes / 1e6:.0f} MB), "
                         "so a step's inputs were last read R - 1 steps earlier",
                   "timing": "K steps back to back between one event pair (isolated_step_ms: an event pair "
                             "around every step)",
                   "flops": "nominal forward 4*P*d per head, P = visible query-key pairs",
                   "parallelism": f"replicas x{ws} (heads independent)"},
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_rate / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms, "steps": e2e_steps},
        "gpu_launches": infer_launches(w, n_split, torch.cuda.get_device_properties(dev).multi_processor_count,
                                       kv is not None) * args.steps,
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ packed sequences
def oracle_sample_packed(w, x, budget_s: float, max_problems=None):
    """Time the fp64 oracle on as many (sequence, head) problems of a packed workload as fit."""
    import torch

    from oracle import ref
    pk = workloads.pack(x)
    lens = x["kv_len"].tolist()
    f64 = lambda t: t.to(torch.float64).numpy()  # noqa: E731
    cuh = pk["cu_seqlens"].tolist()
    t0, done, flops = time.perf_counter(), 0, 0.0
    for b in range(w.B):
        for h in range(w.H):
            sl = slice(cuh[b], cuh[b + 1])
            ref.head_backward(f64(pk["q"][h, sl]), f64(pk["k"][h, sl]), f64(pk["v"][h, sl]), f64(pk["do"][h, sl]),
                              w.scale, w.causal)
            flops += 12.0 * w.d * workloads.visible_pairs(lens[b], lens[b], w.causal)
            done += 1
            if time.perf_counter() - t0 > budget_s or (max_problems and done >= max_problems):
                break
        if time.perf_counter() - t0 > budget_s or (max_problems and done >= max_problems):
            break
    dt = time.perf_counter() - t0
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
            "sample": f"{done} of {w.B * w.H} (sequence, head) problems of {w.name} (fp64 numpy, fwd+bwd), {dt:.1f} s",
            "seconds": dt, "heads": done}


def run_gpu_packed(args, w):
    """fwd+bwd over packed sequences through fa_forward_varlen / fa_backward_varlen."""
    import ctypes

    import torch

    from io_aware_exact_04_gb300 import _lib

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    lib = _lib.load("libfa.so")
    peaks, peak_src = load_peaks()
    x = workloads.make_inputs(w, seed=0)
    pk = workloads.pack(x)
    lens = x["kv_len"].tolist()
    H, d, B = w.H, w.d, w.B
    T, maxlen = int(pk["cu_seqlens"][-1]), max(lens)
    q, k, v, do = (pk[n].to(dev) for n in ("q", "k", "v", "do"))
    cu = pk["cu_seqlens"].to(dev)
    o = torch.empty_like(q)
    lse = torch.empty((H, T), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    wsb = int(lib.fa_backward_varlen_workspace_size(B, H, T, d))
    work = torch.empty(wsb, dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    sp = ctypes.c_void_p(stream.cuda_stream)
    P = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None  # noqa: E731
    causal = int(w.causal)

    def make_step(q, k, v, do, o, lse, dq, dk, dv):
        def step():
            _lib.check(lib.fa_forward_varlen(P(q), P(k), P(v), P(o), P(lse), P(cu), B, H, T, maxlen, d, w.scale,
                                             causal, sp), "fwd_varlen")
            _lib.check(lib.fa_backward_varlen(P(q), P(k), P(v), P(o), P(do), P(lse), P(dq), P(dk), P(dv), P(cu), B, H,
                                              T, maxlen, d, w.scale, causal, P(work), wsb, sp), "bwd_varlen")
        return step

    step = make_step(q, k, v, do, o, lse, dq, dk, dv)

    for _ in range(max(3, args.warmup)):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    detail = (ctypes.c_int * 4)()
    if lib.fa_get_last_device_status_detail(sp, detail) != 0:
        raise RuntimeError(f"device status after warm-up: {list(detail)}")
    step_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    sampler = ClockSampler(local if "CUDA_VISIBLE_DEVICES" not in os.environ else 0)
    if rank == 0:
        sampler.start()
        time.sleep(0.3)
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    sampler.mark("t_start")
    for i in range(args.steps):
        flush.zero_()
        step_ev[i][0].record(stream)
        step()
        step_ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    sampler.mark("t_stop")
    if ws > 1:
        torch.distributed.barrier()
    pairs = sum(workloads.visible_pairs(n, n, w.causal) for n in lens) * H
    fl = 12.0 * d * pairs
    ms_step, rate = job_throughput(sum(e[0].elapsed_time(e[1]) for e in step_ev) / args.steps, fl, device=dev)
    value = rate / 1e12
    peak = float(peaks["bf16_tflops"])
    # whole-step roofline (the packed calls launch their three backward stages inside one call)
    roof = {"bound": "tensor", "kernel": "fwd+bwd step (packed calls)", "achieved": value * 14.0 / 12.0,
            "peak": peak, "unit": "TFLOP/s", "frac": value * 14.0 / 12.0 / peak, "traffic": None,
            "peak_source": f"{peak_src} MEASURED_PEAKS bf16_tflops", "avg_launch_ms": ms_step,
            "flops": "executed 14*P*d per head (recompute included) over the event-timed step"}
    hb = {n: pk[n].pin_memory() for n in ("q", "k", "v", "do")}
    ho = [torch.empty_like(hb["q"]).pin_memory() for _ in range(4)]
    hlse = torch.empty((H, T), dtype=torch.float32).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in hb.values())
    d2h = sum(t.numel() * t.element_size() for t in ho) + hlse.numel() * 4
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_steps, e2e_ms = max(3, min(args.steps, 50)), 0.0
    for i in range(e2e_steps + 2):
        flush.zero_()
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for n, t in (("q", q), ("k", k), ("v", v), ("do", do)):
            t.copy_(hb[n], non_blocking=True)
        step()
        for h_, t in zip(ho, (o, dq, dk, dv)):
            h_.copy_(t, non_blocking=True)
        hlse.copy_(lse, non_blocking=True)
        e1.record(stream)
        e1.synchronize()
        if i >= 2:
            e2e_ms += e0.elapsed_time(e1)
    serial_ms, serial_rate = job_throughput(e2e_ms / e2e_steps, fl, device=dev)
    # ... and pipelined (two device buffer sets; the workspace and the compute stream are shared)
    second = [torch.empty_like(t) for t in (q, k, v, do, o, lse, dq, dk, dv)]
    sets = [((q, k, v, do), (o, dq, dk, dv, lse), step),
            (tuple(second[:4]), (second[4], second[6], second[7], second[8], second[5]), make_step(*second))]
    e2e_ms = pipelined_e2e(dev, sets, tuple(hb[n] for n in ("q", "k", "v", "do")), (*ho, hlse), flush, e2e_steps)
    if lib.fa_get_last_device_status_detail(sp, detail) != 0:
        raise RuntimeError(f"device status after the end-to-end steps: {list(detail)}")
    e2e_ms, e2e_rate = job_throughput(e2e_ms, fl, device=dev)
    del second, sets
    clocks = sampler.stop() if rank == 0 else None
    if ws > 1:
        torch.distributed.barrier()
    if rank != 0:
        return
    cpu = oracle_sample_packed(w, x, args.cpu_budget) if not args.no_cpu_baseline else None
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) inputs, bf16), valid rows packed",
        "config": {"workload": w.name, "B": B, "H": H, "T": T, "max_seqlen": maxlen, "d": d, "causal": w.causal,
                   "lengths": f"U[{w.len_lo},{w.len_hi}] (the bert draw)",
                   "l2": "flushed before every step (256 MiB write, untimed)",
                   "flops": "nominal fwd+bwd 12*P*d per head, P = len^2 per sequence (non-causal)",
                   "parallelism": f"replicas x{ws} (heads independent)"},
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_rate / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms, "steps": e2e_steps, "schedule": E2E_PIPELINED,
                "serial": {"value": serial_rate / 1e12, "ms_per_step": serial_ms, "schedule": E2E_SERIAL}},
        "gpu_launches": 4 * args.steps,
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="long32768", choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--impl", default="native", choices=["native", "reference", "standard"])
    ap.add_argument("--no-sweep", action="store_true", help="skip the long-context sweep's other N")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    w = workloads.WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, w)
    elif args.impl == "standard":
        run_standard(args, w)
    elif w.infer:
        run_gpu_infer(args, w)
    elif w.packed:
        run_gpu_packed(args, w)
    else:
        run_gpu(args, w)


if __name__ == "__main__":
    main()
