"""Benchmark of the Cut Cross-Entropy hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]
                    [--config long] [--filter on|off] [--vocab-sort] [--mode two-call|single]
                    [--g-budget-mib M] [--quick]

One step = cce_forward + cce_backward (every stage of the path: LSE GEMM with
target capture, combine + reduction, target count, recompute + G + filter,
dC GEMM, dE GEMM, dE finalise) over one batch of the seeded synthetic
workload, inputs resident in HBM.  The forward first compacts away the rows
whose target is ignore_index (CCE_FWD_SKIP_IGNORED, "Cut Your Losses ...",
Table A1): the loss and the gradients are unchanged and only those rows' LSE
reads 0; --all-rows-forward computes every row's LSE.  --mode single times the single call
instead (cce_loss_and_grad: staged logits, no recompute).  Prints one JSON
line (rank 0): the headline workload (default: the long-context batch,
65,536 x 2,048 x 128,256, the largest that the workloads define) with its
end-to-end run through the public API and the CPU baseline, and under
"per_config" every other workload and filter mode, measured in the same run.

Timing: W untimed warm-up steps, then exactly K steps bracketed by a barrier
and torch.cuda.synchronize() on both sides, CUDA events on the launching
stream, max over ranks.  Multi-GPU runs (torchrun) are independent replicas
(the path does not shard): value = tokens of all ranks / max time.
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
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import cce_workloads as W  # noqa: E402

METRIC = "CCE fwd+bwd tokens/s and % of bf16 tensor peak; peak extra HBM bytes"
UNIT = "tokens/s"
DEFAULT_CONFIG = "long"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
GEMM_PHASES = ("fwd_lse_gemm", "bwd_recompute_g", "bwd_grad_gemm")
SOURCE_FILES = ("linear_cross_entropy_gb300/csrc/gemm.cuh", "linear_cross_entropy_gb300/csrc/ptx.cuh",
                "linear_cross_entropy_gb300/csrc/gemm_args.h")
WORKLOAD_NAMES = {
    "tiny": "tiny CCE head", "qwen": "Qwen2.5-0.5B-shaped head", "gemma": "Gemma-2-2B-shaped head",
    "llama": "Llama-3-8B-shaped head", "long": "long-context filter stress",
    "freq": "Qwen2.5-0.5B-shaped head, frequent tokens scattered",
    "freq16k": "Qwen2.5-0.5B-shaped head, frequent tokens scattered, 16384 tokens",
    "freq64k": "Qwen2.5-0.5B-shaped head, frequent tokens scattered, 65536 tokens",
}


# --------------------------------------------------------------- helpers
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            p = json.load(fh)
        return {k: float(p[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def source_digest() -> str:
    h = hashlib.sha256()
    for rel in SOURCE_FILES:
        with open(os.path.join(ROOT, rel), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel_phase: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    cur = source_digest()
    with open(path) as fh:
        for line in fh:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            f = dict(kv.split("=", 1) for kv in line.split())
            if f.get("phase") == kernel_phase and f.get("workload") == workload and f.get("source") == cur:
                return float(f["dram_bytes_per_launch"])
    return None


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu = gpu_id
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        return False

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


def reduce_max(value: float, dist, device) -> float:
    """Max of a per-rank float over all ranks (identity without a process group)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(elapsed_ms_by_rank, tokens_per_step, steps):
    """Whole-job throughput: tokens of all ranks / max time over ranks."""
    t = max(elapsed_ms_by_rank)
    world = len(elapsed_ms_by_rank)
    return {"value": tokens_per_step * steps * world / (t / 1e3), "ms_per_step": t / steps}


# ---------------------------------------------------------- CPU oracle
def oracle_sample_rate(w: W.Workload, E_bits, C_bits, x, target_s: float = 12.0):
    """Times the fp64 oracle (as it stands) on a bounded sample: forward +
    backward of the first k token rows as a standalone batch, k grown until a
    run takes a few seconds.  Returns (tokens/s, sample description, cores)."""
    import oracle
    C = oracle.widen_bf16(C_bits)
    E = oracle.widen_bf16(E_bits[: min(w.N, 4096)])
    k, spent, rate = 8, 0.0, None
    while True:
        rows = np.arange(k)
        t0 = time.perf_counter()
        oracle.fwd_bwd_rows(E, C, x, rows, reduction=w.reduction)
        dt = time.perf_counter() - t0
        spent += dt
        rate = k / dt
        if dt > target_s / 3 or spent > target_s or 2 * k > E.shape[0]:
            break
        k = min(E.shape[0], max(2 * k, int(k * (target_s / 3) / max(dt, 1e-3))))
    sample = (f"fp64 oracle forward+backward of the first {k} tokens of the workload as a standalone batch "
              f"(V={w.V}, D={w.D}); {dt:.1f} s")
    return rate, sample, os.cpu_count() or 1


# ----------------------------------------------------------- GPU arm
L2_BYTES = 129 * 1000 * 1000  # GB300 L2 (bytes); inputs below twice this get an L2 flush between steps

# The pages' own throughput for this metric on this exact workload shape: the
# "cut-cross-entropy" kernel card, section "Measured", runs forward and
# backward of 65,536 tokens against V = 128,256 at D = 2048 in 2.0 s on a
# 48 GB card (model not named) -- another machine's number, context only.
PAGE_TOKENS_PER_S = {"long": (65536 / 2.0, "cut-cross-entropy kernel card, 'Measured': 65,536 tokens, "
                                           "V=128,256, D=2048, fwd+bwd in 2.0 s on a 48 GB card")}


def work_flops(n_fwd, n_part, D, V, kept, single):
    """Algorithmic flops of one step over the work actually done: the logit
    GEMM of the forward over the rows it covers, the recompute over the rows
    that take part (none in the single call), and dE + dC over the kept
    filter tiles."""
    fwd = 2.0 * (n_part if single else n_fwd) * D * V
    rec = 0.0 if single else 2.0 * n_part * D * V
    return fwd + rec + 4.0 * n_part * D * V * kept


class Case:
    """Device inputs and buffers of one workload, and its step function."""

    def __init__(self, cce, torch, dev, name, filter_mode, sort, skip, single, budget, inputs=None):
        self.w = w = W.ALL_CONFIGS[name]
        self.name = name
        self.eps = W_FILTER_EPS if filter_mode == "on" else 0.0
        self.filter_mode = filter_mode
        self.sort, self.skip, self.single, self.budget = sort, skip, single, budget
        self.E_bits, self.C_bits, self.x = inputs if inputs is not None else W.make_inputs(w)
        N, D, V = w.N, w.D, w.V
        self.E = torch.from_numpy(self.E_bits.view(np.int16)).to(dev).view(torch.bfloat16)
        self.C = torch.from_numpy(self.C_bits.view(np.int16)).to(dev).view(torch.bfloat16)
        self.xt = torch.from_numpy(self.x).to(dev)
        red = w.reduction
        self.g = torch.ones(N if red == "none" else 1, dtype=torch.float32, device=dev)
        self.ws_f = torch.empty(max(16, cce.forward_workspace_bytes(N, D, V, skip_ignored=skip)), dtype=torch.uint8,
                                device=dev)
        if single:
            self.ws_b = torch.empty(cce.loss_and_grad_workspace_bytes(N, D, V), dtype=torch.uint8, device=dev)
        else:
            self.ws_b = torch.empty(cce.backward_workspace_bytes(N, D, V, vocab_sort=sort, max_staging_bytes=budget),
                                    dtype=torch.uint8, device=dev)
        self.dE = torch.empty_like(self.E)
        self.dC = torch.empty_like(self.C)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.cce, self.torch, self.dev = cce, torch, dev
        self.n_part = int((self.x != W.IGNORE_INDEX).sum())

    def step(self):
        cce, w = self.cce, self.w
        if self.single:
            loss, _, _, _ = cce.cce_loss_and_grad(self.E, self.C, self.xt, -100, w.reduction, self.eps,
                                                  workspace=self.ws_b, dev_err=self.err, check_errors=False,
                                                  lse=False, dE=self.dE, dC=self.dC)
            return loss
        loss, lse = cce.cce_forward(self.E, self.C, self.xt, -100, w.reduction, workspace=self.ws_f,
                                    dev_err=self.err, check_errors=False, skip_ignored=self.skip)
        cce.cce_backward(self.E, self.C, self.xt, lse, self.g, -100, w.reduction, self.eps, workspace=self.ws_b,
                         dev_err=self.err, check_errors=False, dE=self.dE, dC=self.dC, vocab_sort=self.sort,
                         max_staging_bytes=self.budget)
        return loss

    def stats_step(self):
        """One untimed step with fresh workspaces: filter statistics and the
        peak device memory beyond inputs and outputs."""
        cce, torch, w, dev = self.cce, self.torch, self.w, self.dev
        torch.cuda.synchronize()
        torch.cuda.reset_peak_memory_stats(dev)
        base = torch.cuda.memory_allocated(dev)
        red = w.reduction
        if self.single:
            loss, lse, _, _, st = cce.cce_loss_and_grad(self.E, self.C, self.xt, -100, red, self.eps,
                                                        dev_err=self.err, check_errors=False, stats=True)
            outs = [loss, lse]
        else:
            loss, lse = cce.cce_forward(self.E, self.C, self.xt, -100, red, dev_err=self.err, check_errors=False,
                                        skip_ignored=self.skip)
            dE, dC, st = cce.cce_backward(self.E, self.C, self.xt, lse, self.g, -100, red, self.eps,
                                          dev_err=self.err, check_errors=False, stats=True, vocab_sort=self.sort,
                                          max_staging_bytes=self.budget)
            outs = [loss, lse, dE, dC]
        torch.cuda.synchronize()
        N, D, V = w.N, w.D, w.V
        outputs = N * D * 2 + V * D * 2 + N * 4 + (N * 4 if red == "none" else 4) + 16
        peak_extra = torch.cuda.max_memory_allocated(dev) - base - outputs
        del outs
        return st, int(peak_extra)

    def inputs_bytes(self):
        return self.E.numel() * 2 + self.C.numel() * 2 + self.xt.numel() * 8


def time_steps(case, steps, stream, flush):
    """Device time of `steps` steps (CUDA events on the launching stream).
    flush: the inputs fit in L2, so a buffer larger than L2 is written
    between steps, outside the timed events."""
    torch = case.torch
    torch.cuda.synchronize()
    if not flush:
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for _ in range(steps):
            case.step()
        ev1.record(stream)
        torch.cuda.synchronize()
        return ev0.elapsed_time(ev1)
    scrub = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=case.dev)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in evs:
        scrub.fill_(1.0)
        a.record(stream)
        case.step()
        b.record(stream)
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in evs)


def phase_report(phases, steps, flops):
    rep = {}
    for name, ms in phases.ms.items():
        n_l = phases.launches[name]
        if n_l == 0:
            continue
        r = {"ms_per_step": ms / steps, "launches_per_step": n_l / steps}
        if name in flops:
            r["tflops"] = flops[name] * steps / (ms / 1e3) / 1e12
        rep[name] = r
    return rep


def gemm_phase_flops(case, kept):
    w = case.w
    n_fwd = case.n_part if (case.skip or case.single) else w.N
    return {"fwd_lse_gemm": 2.0 * n_fwd * w.D * w.V,
            "bwd_recompute_g": 2.0 * case.n_part * w.D * w.V,
            "bwd_grad_gemm": 4.0 * case.n_part * w.D * w.V * kept}


def measure_case(case, steps, warmup, stream, peaks, gpu_id):
    """Timed steps of one workload: the summary the per-config table carries."""
    cce = case.cce
    st, peak_extra = case.stats_step()
    kept = 1.0 - st["skipped"] / max(st["tiles"], 1)
    flush = case.inputs_bytes() < 2 * L2_BYTES
    for _ in range(warmup):
        case.step()
    with ClockSampler(gpu_id) as clocks, cce.Profiler():
        elapsed = time_steps(case, steps, stream, flush)
    phases = cce.Profiler.read()
    if int(case.err.item()) != 0:
        raise RuntimeError(f"device error word {int(case.err.item())} set during the timed steps")
    w = case.w
    ms = elapsed / steps
    n_fwd = case.n_part if (case.skip or case.single) else w.N
    work = work_flops(n_fwd, case.n_part, w.D, w.V, kept, case.single)
    flops8 = 8.0 * w.N * w.D * w.V
    return {
        "workload": f"{WORKLOAD_NAMES[case.name]} N={w.N} D={w.D} V={w.V}", "config": case.name,
        "filter": case.filter_mode, "reduction": w.reduction, "steps": steps, "warmup": warmup,
        "ms_per_step": round(ms, 4), "tokens_per_s": round(w.N / (ms / 1e3), 1),
        "tflops_8NDV": round(flops8 / (ms / 1e3) / 1e12, 1),
        "achieved_tflops": round(work / (ms / 1e3) / 1e12, 1),
        "frac_of_burst_peak": round(work / (ms / 1e3) / 1e12 / peaks["bf16_tflops"], 4),
        "frac_of_sustained_peak": round(work / (ms / 1e3) / 1e12 / peaks["bf16_tflops_sustained"], 4),
        "work_flops_per_step": work, "rows_taking_part": case.n_part,
        "tiles_skipped_frac": round(st["skipped"] / max(st["tiles"], 1), 4),
        "peak_extra_hbm_bytes": peak_extra,
        "l2": "inputs larger than L2" if not flush else "inputs fit in L2: a 258 MB buffer is written between steps",
        "clocks": clocks.summary(),
        "phases": phase_report(phases, steps, gemm_phase_flops(case, kept)),
    }


def run_e2e(case, steps, stream):
    """The public API end to end: every step copies its inputs from pinned
    host memory into HBM, runs the autograd forward and backward, and copies
    its loss back to pinned host memory; the wall clock covers every step's
    copies.  The copies run on a second stream into one of two device buffer
    sets, so step i+1's inputs travel while step i computes (a prefetching
    loader); the serial form (copy, compute, read, in turn) is reported beside
    it."""
    torch, cce, w = case.torch, case.cce, case.w
    N = w.N
    red = w.reduction
    Eh = torch.from_numpy(case.E_bits.view(np.int16)).view(torch.bfloat16).pin_memory()
    Ch = torch.from_numpy(case.C_bits.view(np.int16)).view(torch.bfloat16).pin_memory()
    xh = torch.from_numpy(case.x).pin_memory()
    bufs = [(torch.empty_like(case.E), torch.empty_like(case.C), torch.empty_like(case.xt)) for _ in range(2)]
    loss_h = torch.zeros(steps, dtype=torch.float32).pin_memory()
    copy_stream = torch.cuda.Stream(case.dev)
    copied = [torch.cuda.Event() for _ in range(2)]
    consumed = [torch.cuda.Event() for _ in range(2)]
    copy_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    comp_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]

    def e2e_copy(j, s):
        Ed, Cd, xd = bufs[j % 2]
        with torch.cuda.stream(s):
            s.wait_event(consumed[j % 2])
            copy_ev[j][0].record(s)
            Ed.copy_(Eh, non_blocking=True)
            Cd.copy_(Ch, non_blocking=True)
            xd.copy_(xh, non_blocking=True)
            copy_ev[j][1].record(s)
            copied[j % 2].record(s)

    def e2e_compute(j):
        Ed, Cd, xd = bufs[j % 2]
        stream.wait_event(copied[j % 2])
        comp_ev[j][0].record(stream)
        Ed.requires_grad_(True)
        Cd.requires_grad_(True)
        if case.single:
            loss = cce.fused_linear_cross_entropy(Ed, Cd, xd, -100, red, case.eps)
        else:
            loss = cce.linear_cross_entropy(Ed, Cd, xd, -100, red, case.eps, vocab_sort=case.sort,
                                            max_staging_bytes=case.budget)
        loss.backward()
        loss_h[j].copy_(loss.detach().reshape(()), non_blocking=True)
        comp_ev[j][1].record(stream)
        consumed[j % 2].record(stream)
        Ed.requires_grad_(False)
        Cd.requires_grad_(False)
        Ed.grad = None
        Cd.grad = None

    def e2e_run(overlap):
        loss_h.zero_()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        if overlap:
            e2e_copy(0, copy_stream)
            for j in range(steps):
                if j + 1 < steps:
                    e2e_copy(j + 1, copy_stream)
                e2e_compute(j)
        else:
            for j in range(steps):
                e2e_copy(j, stream)
                e2e_compute(j)
        t_host = time.perf_counter() - t0
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
        if not bool(torch.isfinite(loss_h).all()) or float(loss_h.min()) != float(loss_h.max()):
            raise RuntimeError(f"end-to-end losses differ across steps: {loss_h.tolist()}")
        dev_ms = sum(a.elapsed_time(b) for a, b in comp_ev) / steps
        h2d_ms = sum(a.elapsed_time(b) for a, b in copy_ev) / steps
        return N * steps / dt, 1e3 * t_host / steps, dev_ms, h2d_ms

    e2e_run(True)
    e2e_serial, _, _, h2d_serial_ms = e2e_run(False)
    e2e_value, host_ms, dev_ms, h2d_ms = e2e_run(True)
    out = {"value": e2e_value, "unit": UNIT,
           "h2d_bytes_per_step": Eh.numel() * 2 + Ch.numel() * 2 + xh.numel() * 8, "d2h_bytes_per_step": 4,
           "steps": steps, "api": ("fused_linear_cross_entropy" if case.single else "linear_cross_entropy")
           + " + backward (autograd Function over the C ABI)",
           "overlap": "inputs of step i+1 copied on a second stream while step i computes (two buffer sets)",
           # wall time of the host loop per step: the host blocks once the launch
           # queue is full, so this follows the GPU whenever the GPU sets the pace
           "serial_value": e2e_serial, "host_loop_ms_per_step": round(host_ms, 3),
           "compute_stream_ms_per_step": round(dev_ms, 3), "h2d_ms_per_step": round(h2d_ms, 3),
           "h2d_ms_per_step_serial": round(h2d_serial_ms, 3)}
    del Eh, Ch, bufs
    cce.raise_pending_errors()
    return out


def per_config_cases(headline, headline_filter, headline_single, headline_skip=True):
    """(workload, filter mode, single call, forward skips ignored rows) of
    every workload and filter mode except the headline, in the headline's
    mode; with a two-call headline, also the single call on the long-context
    batch and that batch with the forward over every row."""
    out = []
    for name in W.CONFIG_ORDER:
        for f in W.CONFIGS[name].filter_modes:
            if (name, f) != (headline, headline_filter):
                out.append((name, f, headline_single, headline_skip))
    if not headline_single:
        out.append(("long", "on", True, True))
        out.append(("long", "on", False, not headline_skip))
    return out


def run_gpu(args, rank, world, local_rank):
    import torch
    import linear_cross_entropy_gb300 as cce

    dist = None
    if world > 1:
        import torch.distributed as dist
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    single = args.mode == "single"
    budget = int(args.g_budget_mib) << 20
    case = Case(cce, torch, dev, args.config, args.filter, bool(args.vocab_sort), bool(args.skip_ignored), single,
                budget)
    w = case.w
    N, D, V = w.N, w.D, w.V
    stream = torch.cuda.current_stream(dev)
    uuid = getattr(torch.cuda.get_device_properties(dev), "uuid", None)
    gpu_id = f"GPU-{uuid}" if uuid is not None else str(local_rank)
    peaks, peak_src = load_peaks()

    for _ in range(args.warmup):
        case.step()
    torch.cuda.synchronize()
    st, peak_extra = case.stats_step()
    kept = 1.0 - st["skipped"] / max(st["tiles"], 1)

    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    launches0 = cce.kernel_launch_count()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(gpu_id) as clocks, cce.Profiler():
        ev0.record(stream)
        for _ in range(args.steps):
            case.step()
        ev1.record(stream)
        torch.cuda.synchronize()
    phases = cce.Profiler.read()
    launches = cce.kernel_launch_count() - launches0
    elapsed = ev0.elapsed_time(ev1)
    if int(case.err.item()) != 0:
        raise RuntimeError(f"device error word {int(case.err.item())} set during the timed steps")
    elapsed_max = reduce_max(elapsed, dist, dev)
    if dist:
        dist.barrier()
    agg = aggregate([elapsed_max] * world, N, args.steps)

    e2e = None if args.quick else run_e2e(case, max(3, min(args.steps, 30)), stream)

    # Roofline of the dominant GEMM phase, timed live by the library's CUDA
    # events on the launching stream: its algorithmic flops (over the rows
    # that take part and, for dE / dC, the filter tiles kept) per launch over
    # its average launch time, against the measured burst bf16 peak (the
    # sustained one beside it).
    flops = gemm_phase_flops(case, kept)
    phase_rep = phase_report(phases, args.steps, flops)
    dom = max(GEMM_PHASES, key=lambda p: phases.ms.get(p, 0.0))
    achieved = phase_rep[dom]["tflops"]
    launches_dom = phases.launches[dom] / args.steps
    roofline = {"bound": "tensor", "kernel": dom, "achieved": round(achieved, 1), "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_tflops"], 4),
                "peak_kind": f"burst bf16 ({peak_src})",
                "frac_of_sustained_peak": round(achieved / peaks["bf16_tflops_sustained"], 4),
                "sustained_peak": peaks["bf16_tflops_sustained"],
                "traffic": recorded_traffic(dom, args.config + ("-single" if single else "")),
                "algorithmic_flops_per_launch": flops[dom] / launches_dom,
                "launches_per_step": launches_dom,
                "avg_launch_ms": phases.ms[dom] / phases.launches[dom]}
    n_fwd = case.n_part if (case.skip or single) else N
    work = work_flops(n_fwd, case.n_part, D, V, kept, single)
    total_flops = 8.0 * N * D * V
    ms = agg["ms_per_step"]
    page = PAGE_TOKENS_PER_S.get(args.config)
    out = {
        "metric": METRIC, "value": round(agg["value"], 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": round(agg["value"] / page[0], 2) if page else None,
        "vs_baseline_basis": page[1] if page else None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{WORKLOAD_NAMES[args.config]} N={N} D={D} V={V}", "N": N, "D": D, "V": V,
                   "reduction": w.reduction, "filter_eps": case.eps, "vocab_sort": case.sort,
                   "ignore_frac": w.ignore_frac,
                   "mode": "single call (cce_loss_and_grad)" if single else "two calls (cce_forward + cce_backward)",
                   "forward_skips_ignored_rows": case.skip or single,
                   "g_staging_budget_bytes": budget if budget else "default (512 MiB)",
                   "g_chunk_cols": None if single else cce.backward_chunk_cols(N, V, budget),
                   "l2": f"inputs larger than L2 (C is {C_MB(case)} MB, E {E_MB(case)} MB)",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        # the pages' metric: 8 N D V over all N tokens, whatever the filter or
        # the ignored rows save
        "tflops_8NDV": round(total_flops / (ms / 1e3) / 1e12, 1),
        # the work actually done: ignored rows compacted away in the backward,
        # filtered tiles skipped
        "achieved_tflops": round(work / (ms / 1e3) / 1e12, 1),
        "frac_of_burst_peak": round(work / (ms / 1e3) / 1e12 / peaks["bf16_tflops"], 4),
        "rows_taking_part": case.n_part,
        "tiles_skipped_frac": round(st["skipped"] / max(st["tiles"], 1), 4),
        "peak_extra_hbm_bytes": int(peak_extra),
        "roofline": roofline, "phases": phase_rep, "e2e": e2e, "gpu_launches": int(launches),
        "clocks": clocks.summary(),
    }
    inputs = (case.w, case.E_bits, case.C_bits, case.x)
    keep_inputs = (case.E_bits, case.C_bits, case.x)
    case_skip = case.skip
    del case
    torch.cuda.empty_cache()

    if not args.quick and rank == 0:
        table = []
        for name, fmode, sgl, skp in per_config_cases(args.config, args.filter, single, case_skip):
            c = Case(cce, torch, dev, name, fmode, False, skp, sgl and W.CONFIGS[name].reduction != "none",
                     budget, inputs=keep_inputs if name == args.config else None)
            r = measure_case(c, min(args.steps, 20), 3, stream, peaks, gpu_id)
            r["mode"] = "single call (cce_loss_and_grad)" if c.single else "two calls (cce_forward + cce_backward)"
            r["forward_skips_ignored_rows"] = bool(c.skip or c.single)
            table.append(r)
            del c
            torch.cuda.empty_cache()
        out["per_config"] = table
    return out, inputs


def C_MB(case):
    return f"{case.C.numel() * 2 / 1e6:.0f}"


def E_MB(case):
    return f"{case.E.numel() * 2 / 1e6:.0f}"


W_FILTER_EPS = 2.0 ** -12


def run_reference(args):
    """The fp64 oracle on the host cores: each step one bounded sample."""
    import oracle
    w = W.ALL_CONFIGS[args.config]
    E_bits, C_bits, x = W.make_inputs(w)
    rate, sample, cores = oracle_sample_rate(w, E_bits, C_bits, x, target_s=6.0)
    k = max(1, int(round(rate * 3.0)))  # ~3 s per step
    C = oracle.widen_bf16(C_bits)
    E = oracle.widen_bf16(E_bits[:k])
    rows = np.arange(k)
    for _ in range(args.warmup):
        oracle.fwd_bwd_rows(E, C, x, rows, reduction=w.reduction)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.fwd_bwd_rows(E, C, x, rows, reduction=w.reduction)
    dt = time.perf_counter() - t0
    value = k * args.steps / dt
    desc = (f"each step: fp64 oracle forward+backward of the first {k} tokens of the workload as a standalone "
            f"batch (V={w.V}, D={w.D})")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{WORKLOAD_NAMES[args.config]} N={w.N} D={w.D} V={w.V}", "N": w.N, "D": w.D,
                   "V": w.V, "reduction": w.reduction},
        "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc},
        "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("gb300", "reference"), default="gb300")
    ap.add_argument("--config", choices=tuple(W.ALL_CONFIGS), default=DEFAULT_CONFIG)
    ap.add_argument("--filter", choices=("on", "off"), default=None)
    ap.add_argument("--vocab-sort", action="store_true",
                    help="filter over the vocabulary sorted by average logit")
    ap.add_argument("--all-rows-forward", action="store_true",
                    help="two-call mode: the forward computes the LSE of every row, ignored rows too (default: "
                         "it compacts away the rows that take part in no loss first, CCE_FWD_SKIP_IGNORED)")
    ap.add_argument("--mode", choices=("two-call", "single"), default="two-call",
                    help="two-call: cce_forward + cce_backward; single: cce_loss_and_grad")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--quick", action="store_true",
                    help="the headline step only: no end-to-end run, no other configs, no CPU baseline "
                         "(for profiler runs)")
    ap.add_argument("--g-budget-mib", type=int, default=0,
                    help="two-call mode: bound of the backward's G-hat chunk buffer in MiB (0: the default)")
    args = ap.parse_args(argv)
    args.skip_ignored = not args.all_rows_forward
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.filter is None:
        args.filter = W.ALL_CONFIGS[args.config].filter_modes[0]
    if args.mode == "single" and (args.vocab_sort or W.ALL_CONFIGS[args.config].reduction == "none"):
        ap.error("--mode single takes neither --vocab-sort nor a workload with reduction 'none'")
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args)), flush=True)
        return 0

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    out, inputs = run_gpu(args, rank, world, local_rank)
    if rank == 0:
        if not (args.no_cpu_baseline or args.quick):
            w, E_bits, C_bits, x = inputs
            rate, sample, cores = oracle_sample_rate(w, E_bits, C_bits, x)
            out["cpu_baseline"] = {"value": round(rate, 3), "unit": UNIT, "cores": cores, "kind": "oracle",
                                   "sample": sample}
        else:
            out["cpu_baseline"] = None
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
