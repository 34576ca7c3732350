"""Benchmark: attention forward + backward TFLOP/s on one GB300 (or N replicas).

One step = one forward (fa_fwd) and one backward (fa_bwd_preprocess,
fa_bwd_dkdv, fa_bwd_dq) over one batch of the workload, inputs resident in
device memory. FLOPs are algorithmic and counted over allowed (query, key)
pairs P: forward 4 d P (two contractions), backward 10 d P (five), so a step
is 14 d P. Kernels that recompute work (the dQ kernel recomputes S and dP)
get no credit for it.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                       [--impl ours|reference]
Under torchrun every rank runs the same workload on its own GPU (the path
shards by heads and batches; there is no data-path collective) and rank 0
prints one JSON line with the whole-job throughput.

``--workload decode_16k`` measures the forward-only short-query kernel
(fa_decode) instead: one step is one decode call, and the metric is the
algorithmic HBM bytes it must move per second (K/V cache rows each sequence
sees, Q, O, lse) against the measured copy bandwidth.
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from io_aware_exact_07_gb300 import inputs  # noqa: E402

METRIC = "attention fwd+bwd TFLOP/s (bf16) and % of GB300 dense BF16 tensor peak"
UNIT = "TFLOP/s"
# The largest single-GPU workload of the suite, and one of those the forward /
# backward tensor-core targets (N >= 4K) apply to; the others run with --workload.
DEFAULT_WORKLOAD = "long_16k_d128"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KERNELS = ("fwd", "bwd_preprocess", "bwd_dkdv", "bwd_dq")
# algorithmic flops per allowed pair for each tensor-core kernel (per unit of d)
KERNEL_FLOPS_PER_PAIR_D = {"fwd": 4, "bwd_dkdv": 8, "bwd_dq": 6, "bwd": 10}


# --------------------------------------------------------------------- work model

def allowed_pairs(w: inputs.Workload, seqlens) -> int:
    """Exact number of allowed (query, key) pairs over all heads."""
    N, T = w.N, 128
    nb = math.ceil(N / T)
    mask = None
    if w.butterfly:
        i = np.arange(nb)[:, None]
        j = np.arange(nb)[None, :]
        x = i ^ j
        mask = (x == 0) | ((x & (x - 1)) == 0)
    lens = [N] * w.B if seqlens is None else [min(max(int(s), 0), N) for s in seqlens]
    rows = np.arange(N)
    wl, wr = w.window
    # per row, the visible keys form [lo, hi) before the block mask
    lo_r = np.zeros(N, dtype=np.int64) if wl < 0 else np.maximum(rows - wl, 0)
    hi_r = rows + 1 if w.causal else np.full(N, N, dtype=np.int64)
    if wr >= 0:
        hi_r = np.minimum(hi_r, rows + wr + 1)
    total = 0
    for L in lens:
        if mask is None:  # dense, causal, padded and / or windowed
            total += int(np.clip(np.minimum(hi_r, L) - lo_r, 0, None).sum())
            continue
        cnt = 0
        for qt in range(nb):
            r = rows[qt * T:(qt + 1) * T]
            for kt in range(nb):
                if not mask[qt, kt]:
                    continue
                lo, hi = kt * T, min((kt + 1) * T, L)
                if hi <= lo:
                    continue
                hi_t = np.minimum(hi, hi_r[qt * T:(qt + 1) * T])
                lo_t = np.maximum(lo, lo_r[qt * T:(qt + 1) * T])
                cnt += int(np.clip(hi_t - lo_t, 0, None).sum())
        total += cnt
    return total * w.H


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except Exception:
        return FALLBACK_PEAKS, "fallback"


# Sources each timed kernel is built from: a committed DRAM-traffic figure is
# used only while these files are unchanged since it was captured.
KERNEL_SOURCES = {
    "fwd": ("fa_fwd.cu", "fa_fwd128.cu", "fa_kernels.h"),
    "bwd_dkdv": ("fa_bwd.cu", "fa_bwd_split.cu", "fa_kernels.h"),
    "bwd_dq": ("fa_bwd_split.cu", "fa_kernels.h"),
    "bwd_preprocess": ("fa_bwd.cu", "fa_kernels.h"),
    "decode": ("fa_decode.cu", "fa_decode.h"),
    "fwd_fp8": ("fa_fwd_fp8.cu", "fa_fp8.h"),
}
COMMON_SOURCES = ("fa_common.cuh", "sm103_ptx.cuh")


def kernel_source_hash(kernel=None):
    """sha256 (16 hex digits) of the CUDA sources a kernel is built from (all of
    them when the kernel is not listed)."""
    csrc = os.path.join(ROOT, "io_aware_exact_07_gb300", "csrc")
    names = sorted(os.listdir(csrc)) if kernel not in KERNEL_SOURCES else \
        sorted(KERNEL_SOURCES[kernel] + COMMON_SOURCES)
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, workload: str):
    """Per-launch DRAM bytes from a committed ncu summary, if it matches the current source."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
        e = t[workload][kernel]
        if e.get("source_hash") != kernel_source_hash(kernel):
            return None
        return float(e["bytes_per_launch"])
    except Exception:
        return None


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running.

    The sampler starts `lead_s` before the timed region so that it is already
    producing samples when the region begins (nvidia-smi takes a while to start),
    and only the samples whose timestamps fall inside the region are summarised
    (all of them if none does, e.g. for a region shorter than the interval)."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, lead_s: float = 0.3):
        self.index = index
        self.lead_s = lead_s
        self.proc = None
        self.t_begin = self.t_end = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(self.lead_s)
        except Exception:
            self.proc = None
        self.t_begin = datetime.datetime.now()
        return self

    def __exit__(self, *a):
        self.t_end = datetime.datetime.now()
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        rows = []
        for ln in getattr(self, "lines", []):
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f")
            except ValueError:
                ts = None
            try:
                sm, mx = float(f[2]), float(f[3])
            except ValueError:
                continue
            rows.append((ts, sm, mx, [n for n, v in zip(names, f[6:10]) if v.lower() == "active"]))
        inside = [r for r in rows if r[0] is not None and self.t_begin is not None
                  and self.t_begin <= r[0] <= self.t_end]
        window = "timed region"
        if not inside:
            inside, window = rows, "whole sampler run (no sample inside the timed region)"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        reasons = sorted({n for r in inside for n in r[3]})
        return {"sm_mhz": statistics.median(r[1] for r in inside),
                "sm_max_mhz": max(r[2] for r in inside), "reasons": reasons,
                "samples": len(inside), "window": window}


# -------------------------------------------------------------------- our arm

class Step:
    """Device buffers and the four library calls of one fwd+bwd step."""

    def __init__(self, w, x, dev):
        import io_aware_exact_07_gb300 as fa
        self.fa = fa
        self.w = w
        self.q, self.k, self.v, self.do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
        self.sl = None if x["seqlens"] is None else x["seqlens"].to(dev)
        self.bm = None
        if w.butterfly:
            self.bm = fa.fa_butterfly_mask(math.ceil(w.N / 128)).to(dev)
        B, H, N, d = w.B, w.H, w.N, w.d
        # grouped K/V heads and sliding windows go through fa_fwd_window /
        # fa_bwd_window, timed as fwd and the whole backward (the per-stage
        # entry points take neither)
        self.whole = w.kv_heads != H or tuple(w.window) != (-1, -1)
        self.kernels = ("fwd", "bwd") if self.whole else KERNELS
        self.o = torch.empty_like(self.q)
        self.lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
        self.dq = torch.empty_like(self.q)
        self.dk, self.dv = torch.empty_like(self.k), torch.empty_like(self.v)
        self.ws_bytes = fa.fa_bwd_workspace_size(B, H, N, d)
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=dev)
        self.opts = dict(causal=w.causal, dropout_p=w.dropout_p, seed=0, offset=0,
                         block_mask=self.bm, seqlens_k=self.sl)

    def run(self, events=None):
        fa, w = self.fa, self.w
        B, H, N, d, s = w.B, w.H, w.N, w.d, w.scale
        o = self.opts
        ev = events or [None] * 5
        if self.whole:
            Hkv = w.kv_heads
            win = dict(window_left=w.window[0], window_right=w.window[1])
            if ev[0] is not None:
                ev[0].record()
            st = fa.fa_fwd_window(self.q, self.k, self.v, self.o, self.lse, B, H, Hkv, N, d, s,
                                  **win, **o)
            if ev[1] is not None:
                ev[1].record()
            st |= fa.fa_bwd_window(self.q, self.k, self.v, self.o, self.do, self.lse, self.dq,
                                   self.dk, self.dv, B, H, Hkv, N, d, s, workspace=self.ws,
                                   workspace_bytes=self.ws_bytes, **win, **o)
            if ev[2] is not None:
                ev[2].record()
            if st != 0:
                raise RuntimeError(f"library call failed with status {st}")
            return
        if ev[0] is not None:
            ev[0].record()
        st = fa.fa_fwd(self.q, self.k, self.v, self.o, self.lse, B, H, N, d, s, **o)
        if ev[1] is not None:
            ev[1].record()
        st |= fa.fa_bwd_preprocess(self.o, self.do, B, H, N, d, self.ws, self.ws_bytes)
        if ev[2] is not None:
            ev[2].record()
        st |= fa.fa_bwd_dkdv(self.q, self.k, self.v, self.do, self.lse, self.dk, self.dv, B, H,
                             N, d, s, workspace=self.ws, workspace_bytes=self.ws_bytes, **o)
        if ev[3] is not None:
            ev[3].record()
        st |= fa.fa_bwd_dq(self.q, self.k, self.v, self.do, self.lse, self.dq, B, H, N, d, s,
                           workspace=self.ws, workspace_bytes=self.ws_bytes, **o)
        if ev[4] is not None:
            ev[4].record()
        if st != 0:
            raise RuntimeError(f"library call failed with status {st}")


def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
        pg = dist
    return world, rank, local, pg


def whole_job_value(flops_step: float, steps: int, world: int, elapsed_max: float) -> float:
    """TFLOP/s of the whole job: every rank ran `steps` steps of `flops_step`
    (weak scaling), and the slowest rank's time bounds the job."""
    return flops_step * steps * world / elapsed_max / 1e12


def barrier(pg):
    if pg is not None:
        pg.barrier()


def max_over_ranks(pg, value: float) -> float:
    if pg is None:
        return value
    t = torch.tensor([value], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def cpu_baseline(w, x, seqlens, budget_s=15.0):
    """Time the fp64 oracle (fwd + bwd) on a bounded sample of heads."""
    import oracle
    heads_all = [(b, h) for b in range(w.B) for h in range(w.H)]
    G = w.H // w.kv_heads  # query heads per K/V head
    sl_np = None if seqlens is None else seqlens.numpy()
    bm = None
    if w.butterfly:
        bm = oracle.butterfly(math.ceil(w.N / 128))

    def run(heads):
        f64 = lambda t: np.stack([t[b, h].double().numpy() for b, h in heads])
        f64kv = lambda t: np.stack([t[b, h // G].double().numpy() for b, h in heads])
        q, do = f64(x["q"]), f64(x["do"])
        k, v = f64kv(x["k"]), f64kv(x["v"])
        t0 = time.perf_counter()
        kw = dict(causal=w.causal, dropout_p=w.dropout_p, seed=0, offset=0, block_mask=bm,
                  seqlens_k=sl_np, heads=heads, H=w.H, window_left=w.window[0],
                  window_right=w.window[1])
        oracle.fwd(q, k, v, w.scale, **kw)
        oracle.bwd(q, k, v, do, w.scale, **kw)
        return time.perf_counter() - t0

    t1 = run(heads_all[:1])
    n = int(max(1, min(len(heads_all), budget_s / max(t1, 1e-6))))
    sample = heads_all[:n]
    t = run(sample) if n > 1 else t1
    # allowed pairs of the sampled heads
    per_b = {}
    for b, h in sample:
        per_b[b] = per_b.get(b, 0) + 1
    pairs = 0
    for b, cnt in per_b.items():
        wb = inputs.Workload("s", 1, cnt, w.N, w.d, causal=w.causal, butterfly=w.butterfly,
                             window=w.window)
        pairs += allowed_pairs(wb, None if seqlens is None else [int(seqlens[b])])
    flops = 14.0 * w.d * pairs
    cores = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    return {"value": flops / t / 1e12, "unit": UNIT, "cores": cores, "kind": "oracle", "cpu_model": cpu_model(),
            "sample": f"{n} of {w.B * w.H} heads of {w.name}, fwd+bwd in fp64, {t:.1f} s",
            "seconds": t}


def cpu_model() -> str:
    """The host CPU's model name (for the CPU-baseline line), or the machine type."""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu model")):
                    return line.split(":", 1)[1].strip()
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.machine()


def measure_e2e(step, x, pg, stream, n_steps, w=None, dev=None):
    """Same step through the public calls with host buffers: every step copies
    its inputs from pinned host memory and reads all its results (O, lse, dQ,
    dK, dV) back to pinned host memory, all inside the timed region. The
    copies are pipelined as a training loop would run them: step i + 1's
    inputs go in on one stream while step i computes on another, and step i's
    results come back on a third, with two sets of device buffers so that no
    buffer is overwritten while in use (events order every reuse)."""
    ins, outs = ("q", "k", "v", "do"), ("o", "lse", "dq", "dk", "dv")
    steps = [step, Step(w, x, dev)] if w is not None else [step, step]
    host_in = {n: x[n].pin_memory() for n in ins}
    host_out = [{n: torch.empty(getattr(step, n).shape, dtype=getattr(step, n).dtype,
                                pin_memory=True) for n in outs} for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out[0].values())
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    in_done, comp_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    used = [False, False]

    def one(i):
        b = i % 2
        st = steps[b]
        with torch.cuda.stream(s_in):
            if used[b]:
                s_in.wait_event(comp_done[b])      # the compute that last read these inputs
            for n in ins:
                getattr(st, n).copy_(host_in[n], non_blocking=True)
            in_done[b].record(s_in)
        stream.wait_event(in_done[b])
        if used[b]:
            stream.wait_event(out_done[b])         # the results of two steps ago are read back
        with torch.cuda.stream(stream):
            st.run()
        comp_done[b].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(comp_done[b])
            for n in outs:
                host_out[b][n].copy_(getattr(st, n), non_blocking=True)
            out_done[b].record(s_out)
        used[b] = True

    for i in range(2):
        one(i)
    torch.cuda.synchronize()
    barrier(pg)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for i in range(n_steps):
        one(i)
    e1.record(s_out)  # the last step's results are on the host once this completes
    torch.cuda.synchronize()
    return {"seconds": max_over_ranks(pg, e0.elapsed_time(e1) / 1e3), "h2d": h2d, "d2h": d2h,
            "steps": n_steps}


def run_ours(args, w):
    world, rank, local, pg = dist_setup(args.gpus)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    x = inputs.draw(w, with_grad=True)
    seqlens = x["seqlens"]
    step = Step(w, x, dev)
    pairs = allowed_pairs(w, None if seqlens is None else seqlens.tolist())
    flops_step = 14.0 * w.d * pairs
    stream = torch.cuda.current_stream()

    for _ in range(args.warmup):
        step.run()
    torch.cuda.synchronize()
    # status word: a device-side timeout would be reported here
    assert step.fa.fa_device_status() == 0, "device-side error during warm-up"

    # ---- device-resident timed region, per-kernel events
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(pg)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        start.record(stream)
        for i in range(args.steps):
            step.run(evs[i])
        end.record(stream)
        torch.cuda.synchronize()
    barrier(pg)
    elapsed = start.elapsed_time(end) / 1e3
    elapsed = max_over_ranks(pg, elapsed)
    per_kernel = {k: [] for k in step.kernels}
    for e in evs:
        for j, k in enumerate(step.kernels):
            per_kernel[k].append(e[j].elapsed_time(e[j + 1]) / 1e3)
    kstats = {k: statistics.mean(v) for k, v in per_kernel.items()}
    assert step.fa.fa_device_status() == 0, "device-side error during the timed region"

    # ---- end to end: pinned host inputs in, results out, every step
    e2e = None
    if not args.no_e2e:
        e2e = measure_e2e(step, x, pg, stream, max(3, min(args.steps, 20)), w, dev)

    if rank != 0:
        if pg is not None:
            pg.destroy_process_group()
        return None

    peaks, peak_src = load_peaks()
    peak_sus = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    peak_burst = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    total_k = sum(kstats.values())
    dominant = max(kstats, key=lambda k: kstats[k])
    if dominant in KERNEL_FLOPS_PER_PAIR_D:
        # the kernel runs a few milliseconds at a time: its denominator is the
        # burst peak; the fraction of the sustained (power-capped) one is kept beside it
        ach = KERNEL_FLOPS_PER_PAIR_D[dominant] * w.d * pairs / kstats[dominant] / 1e12
        roof = {"bound": "tensor", "achieved": ach, "peak": peak_burst, "unit": "TFLOP/s",
                "frac": ach / peak_burst, "frac_of_sustained": ach / peak_sus}
    else:
        rows = w.B * w.H * w.N
        byts = 2 * rows * w.d * 2 + rows * 4
        ach = byts / kstats[dominant] / 1e9
        roof = {"bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm}
    roof["kernel"] = dominant
    roof["peak_source"] = f"{peak_src} ({'bf16_tflops' if roof['bound'] == 'tensor' else 'hbm_gbs'})"
    roof["traffic"] = ncu_traffic(dominant, w.name)
    value = whole_job_value(flops_step, args.steps, world, elapsed)
    fwd_t, bwd_t = kstats["fwd"], total_k - kstats["fwd"]
    fwd_tf = 4 * w.d * pairs / fwd_t / 1e12
    bwd_tf = 10 * w.d * pairs / bwd_t / 1e12
    result = {
        "metric": METRIC,
        "value": value,
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": elapsed / args.steps * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 Q, K, V, dO; no dataset)",
        "config": {"workload": w.name, "description": w.description, "B": w.B, "H": w.H,
                   "H_kv": w.kv_heads, "window": list(w.window),
                   "N": w.N, "d": w.d, "causal": w.causal, "dropout_p": w.dropout_p,
                   "key_padding": w.padding, "block_mask": "butterfly" if w.butterfly else None,
                   "allowed_pairs": pairs, "flops_per_step": flops_step,
                   "l2": "inputs larger than L2 (no flush)" if 4 * w.B * w.H * w.N * w.d * 2 > 129e6
                   else "inputs smaller than L2",
                   "parallelism": f"replicas x{world} (heads are independent; no collective)"},
        "pct_of_peak": {"burst": 100 * value / world / peak_burst,
                        "sustained": 100 * value / world / peak_sus},
        "breakdown": {"fwd_ms": fwd_t * 1e3, "bwd_ms": bwd_t * 1e3, "fwd_tflops": fwd_tf,
                      "bwd_tflops": bwd_tf,
                      "fwd_pct_burst_peak": 100 * fwd_tf / peak_burst,
                      "bwd_pct_burst_peak": 100 * bwd_tf / peak_burst,
                      "kernels_ms": {k: v * 1e3 for k, v in kstats.items()},
                      "kernel_share": {k: v / total_k for k, v in kstats.items()}},
        "roofline": roof,
        "e2e": None if e2e is None else {
            "value": flops_step * e2e["steps"] * world / e2e["seconds"] / 1e12, "unit": UNIT,
            "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
            "steps": e2e["steps"],
            "copies": "pipelined: step i+1's inputs in and step i-1's results out during step i"},
        "gpu_launches": len(KERNELS) * args.steps,
        "clocks": clk.summary(),
    }
    if not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(w, x, seqlens)
        result["cpu_baseline"].pop("seconds", None)
    if pg is not None:
        pg.destroy_process_group()
    return result


# -------------------------------------------------------------- reference arm

def run_reference(args, w):
    """The fp64 CPU oracle timed on the host cores, one bounded sample per step."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return None
    import oracle
    x = inputs.draw(w, with_grad=True)
    seqlens = x["seqlens"]
    sl_np = None if seqlens is None else seqlens.numpy()
    bm = oracle.butterfly(math.ceil(w.N / 128)) if w.butterfly else None
    heads = [(0, 0)]
    f64 = lambda t: np.stack([t[b, h].double().numpy() for b, h in heads])
    q, k, v, do = (f64(x[n]) for n in ("q", "k", "v", "do"))  # head 0 uses K/V head 0
    kw = dict(causal=w.causal, dropout_p=w.dropout_p, seed=0, offset=0, block_mask=bm,
              seqlens_k=sl_np, heads=heads, H=w.H, window_left=w.window[0],
              window_right=w.window[1])
    wb = inputs.Workload("s", 1, 1, w.N, w.d, causal=w.causal, butterfly=w.butterfly,
                         window=w.window)
    pairs = allowed_pairs(wb, None if seqlens is None else [int(seqlens[0])])
    flops = 14.0 * w.d * pairs

    def one():
        oracle.fwd(q, k, v, w.scale, **kw)
        oracle.bwd(q, k, v, do, w.scale, **kw)

    for _ in range(args.warmup):
        one()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one()
    t = time.perf_counter() - t0
    value = flops * args.steps / t / 1e12
    cores = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    sample = f"head (0, 0) of {w.name} per step, fwd+bwd in fp64"
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": t / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded N(0,1), same inputs)",
        "config": {"workload": w.name, "description": w.description, "allowed_pairs": pairs,
                   "flops_per_step": flops},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "cpu_model": cpu_model(),
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


# ------------------------------------------------------------ decode workload

DECODE_METRIC = "decode attention (fa_decode): algorithmic HBM GB/s"


def decode_bytes(w, seqlens, heads=None):
    """Bytes fa_decode must move: the visible K/V cache rows of every K/V head
    (bf16 K and V), Q read, O written (bf16) and lse (fp32). heads: optional
    list of (b, K/V head) groups to count instead of all."""
    G = w.H // w.Hkv
    groups = heads if heads is not None else [(b, j) for b in range(w.B) for j in range(w.Hkv)]
    total = 0
    for b, _ in groups:
        L = w.Nk if seqlens is None else min(max(int(seqlens[b]), 0), w.Nk)
        total += 2 * L * w.d * 2 + G * w.Nq * (2 * w.d * 2 + 4)
    return total


def run_decode(args, w):
    world, rank, local, pg = dist_setup(args.gpus)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    import io_aware_exact_07_gb300 as fa
    x = inputs.draw_decode(w)
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    sl = None if x["seqlens"] is None else x["seqlens"].to(dev)
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.Nq), dtype=torch.float32, device=dev)
    ws_bytes = fa.fa_decode_workspace_size(w.B, w.H, w.Hkv, w.Nq, w.Nk, w.d, 0)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    byts = decode_bytes(w, None if x["seqlens"] is None else x["seqlens"].tolist())

    def call():
        st = fa.fa_decode(q, k, v, o, lse, w.B, w.H, w.Hkv, w.Nq, w.Nk, w.d, w.scale, w.causal,
                          sl, 0, ws, ws_bytes)
        if st != 0:
            raise RuntimeError(f"fa_decode failed with status {st}")

    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0, "device-side error during warm-up"
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(pg)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        start.record(stream)
        for e0, e1 in evs:
            e0.record(stream)
            call()
            e1.record(stream)
        end.record(stream)
        torch.cuda.synchronize()
    barrier(pg)
    elapsed = max_over_ranks(pg, start.elapsed_time(end) / 1e3)
    t_call = statistics.mean(e0.elapsed_time(e1) / 1e3 for e0, e1 in evs)
    assert fa.fa_device_status() == 0, "device-side error during the timed region"

    e2e = None
    if not args.no_e2e:
        # per step: the new query rows in from pinned host memory, O and lse out;
        # the K/V cache is device-resident state, as in serving
        hq = x["q"].pin_memory()
        ho = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
        hl = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)
        n = max(3, min(args.steps, 50))

        def one():
            q.copy_(hq, non_blocking=True)
            call()
            ho.copy_(o, non_blocking=True)
            hl.copy_(lse, non_blocking=True)

        one()
        torch.cuda.synchronize()
        barrier(pg)
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for _ in range(n):
            one()
        a1.record(stream)
        torch.cuda.synchronize()
        secs = max_over_ranks(pg, a0.elapsed_time(a1) / 1e3)
        e2e = {"value": byts * n * world / secs / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": hq.numel() * hq.element_size(),
               "d2h_bytes_per_step": ho.numel() * ho.element_size() + hl.numel() * hl.element_size(),
               "steps": n}
    if rank != 0:
        if pg is not None:
            pg.destroy_process_group()
        return None
    peaks, peak_src = load_peaks()
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    value = byts * args.steps * world / elapsed / 1e9
    ach = byts / t_call / 1e9
    launches = 2 if ws_bytes > 0 else 1
    result = {
        "metric": DECODE_METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": elapsed / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 Q, K/V cache; no dataset)",
        "config": {"workload": w.name, "description": w.description, "B": w.B, "H": w.H,
                   "H_kv": w.Hkv, "Nq": w.Nq, "Nk": w.Nk, "d": w.d, "causal": w.causal,
                   "cache_lengths": w.lengths, "bytes_per_step": byts,
                   "tokens_per_s": w.B * w.Nq * args.steps * world / elapsed,
                   "l2": "K/V cache larger than L2 (no flush)",
                   "parallelism": f"replicas x{world} (no collective)"},
        "roofline": {"bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s",
                     "frac": ach / hbm, "traffic": ncu_traffic("decode", w.name),
                     "kernel": "fa_decode call (main kernel + combine)",
                     "peak_source": f"{peak_src} (hbm_gbs)"},
        "e2e": e2e,
        "gpu_launches": launches * args.steps,
        "clocks": clk.summary(),
    }
    if not args.no_cpu_baseline:
        result["cpu_baseline"] = decode_cpu_baseline(w, x)
        result["cpu_baseline"].pop("seconds", None)
    if pg is not None:
        pg.destroy_process_group()
    return result


def decode_cpu_baseline(w, x, budget_s=12.0):
    """The fp64 oracle's fwd_decode timed on whole K/V groups (all G query heads
    of a K/V head), as many as fit the time budget."""
    import oracle
    G = w.H // w.Hkv
    f64 = {n: x[n].double().numpy() for n in ("q", "k", "v")}
    sl = None if x["seqlens"] is None else x["seqlens"].numpy()
    groups = [(b, j) for b in range(w.B) for j in range(w.Hkv)]

    def run(gs):
        heads = [(b, j * G + g) for b, j in gs for g in range(G)]
        t0 = time.perf_counter()
        oracle.fwd_decode(f64["q"], f64["k"], f64["v"], w.scale, causal=w.causal, seqlens_k=sl,
                          heads=heads)
        return time.perf_counter() - t0

    t1 = run(groups[:1])
    n = int(max(1, min(len(groups), budget_s / max(t1, 1e-6))))
    t = run(groups[:n]) if n > 1 else t1
    reps = 1
    if n == len(groups) and budget_s > 0:
        # the whole workload is fast: repeat it so the timing spans a few seconds
        reps = int(max(1, min(50, 2.0 / max(t, 1e-6))))
        if reps > 1:
            t = sum(run(groups) for _ in range(reps))
    byts = decode_bytes(w, sl, groups[:n]) * reps
    # numpy's matrix-vector products run in its BLAS, which may use every core
    cores = int(os.environ.get("OPENBLAS_NUM_THREADS", os.environ.get("OMP_NUM_THREADS",
                                                                      os.cpu_count() or 1)))
    return {"value": byts / t / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle", "cpu_model": cpu_model(),
            "sample": f"{n} of {len(groups)} K/V groups of {w.name} (all their query heads)"
                      f"{f' x{reps}' if reps > 1 else ''}, fp64 numpy (BLAS threads up to "
                      f"{cores}), {t:.1f} s", "seconds": t}


def run_decode_reference(args, w):
    """The fp64 oracle's fwd_decode on the host, one K/V group per step."""
    if int(os.environ.get("RANK", "0")) != 0:
        return None
    x = inputs.draw_decode(w)
    cb = None
    for _ in range(args.warmup):
        decode_cpu_baseline(w, x, budget_s=0.0)
    secs = 0.0
    for _ in range(args.steps):
        cb = decode_cpu_baseline(w, x, budget_s=0.0)  # one group per step
        secs += cb["seconds"]
    byts = decode_bytes(w, None if x["seqlens"] is None else x["seqlens"].numpy(), [(0, 0)])
    value = byts * args.steps / secs / 1e9
    sample = f"K/V group (0, 0) of {w.name} (all its query heads) per step, fp64 numpy"
    return {
        "impl": "reference", "metric": DECODE_METRIC, "value": value, "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded N(0,1), same inputs)",
        "config": {"workload": w.name, "description": w.description, "bytes_per_step": byts},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cb["cores"], "kind": "oracle", "cpu_model": cpu_model(),
                         "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


# --------------------------------------------------------------- FP8 workload

FP8_METRIC = "attention fwd TFLOP/s (FP8 e4m3 operands, fp32 accumulation)"


def run_fp8(args, w):
    """FP8 forward on the causal decoder shape: bf16 inputs quantised once by
    fa_fp8_quantize (timed separately), then fa_fwd_fp8 timed per step."""
    world, rank, local, pg = dist_setup(args.gpus)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    import io_aware_exact_07_gb300 as fa
    x = inputs.draw(w, with_grad=False)
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    signs = inputs.rotation_signs(w.d, seed=0).to(dev)
    B, H, N, d = w.B, w.H, w.N, w.d
    Np = fa.fa_fp8_vt_stride(N)
    z = dict(q8=torch.empty((B, H, N, d), dtype=torch.uint8, device=dev),
             k8=torch.empty((B, H, N, d), dtype=torch.uint8, device=dev),
             vt8=torch.empty((B, H, d, Np), dtype=torch.uint8, device=dev),
             s_q=torch.empty((B, H), dtype=torch.float32, device=dev),
             s_k=torch.empty((B, H), dtype=torch.float32, device=dev),
             s_v=torch.empty((B, H, d), dtype=torch.float32, device=dev))
    wsb = fa.fa_fp8_workspace_size(B, H, d)
    ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
    o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)

    def quant():
        st = fa.fa_fp8_quantize(q, k, v, signs, B, H, N, d, z["q8"], z["k8"], z["vt8"], z["s_q"],
                                z["s_k"], z["s_v"], ws, wsb)
        if st != 0:
            raise RuntimeError(f"fa_fp8_quantize failed with status {st}")

    def fwd():
        st = fa.fa_fwd_fp8(z["q8"], z["k8"], z["vt8"], z["s_q"], z["s_k"], z["s_v"], o, lse, B,
                           H, N, d, w.scale, w.causal)
        if st != 0:
            raise RuntimeError(f"fa_fwd_fp8 failed with status {st}")

    pairs = allowed_pairs(w, None)
    flops = 4.0 * w.d * pairs
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        quant()
        fwd()
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0, "device-side error during warm-up"
    q0, q1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    q0.record(stream)
    for _ in range(10):
        quant()
    q1.record(stream)
    torch.cuda.synchronize()
    t_quant = q0.elapsed_time(q1) / 10 / 1e3
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(pg)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        start.record(stream)
        for _ in range(args.steps):
            fwd()
        end.record(stream)
        torch.cuda.synchronize()
    barrier(pg)
    elapsed = max_over_ranks(pg, start.elapsed_time(end) / 1e3)
    assert fa.fa_device_status() == 0, "device-side error during the timed region"
    e2e = None
    if not args.no_e2e:
        # per step: bf16 Q, K, V in from pinned host memory, quantise, forward, O and lse out,
        # pipelined over two buffer sets as in measure_e2e
        hq, hk, hv = (x[n].pin_memory() for n in ("q", "k", "v"))
        sets = []
        for b_ in range(2):
            if b_ == 0:
                bufs = dict(q=q, k=k, v=v, z=z, o=o, lse=lse)
            else:
                bufs = dict(q=torch.empty_like(q), k=torch.empty_like(k), v=torch.empty_like(v),
                            z={n_: torch.empty_like(t) for n_, t in z.items()},
                            o=torch.empty_like(o), lse=torch.empty_like(lse))
            bufs["ho"] = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
            bufs["hl"] = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)
            sets.append(bufs)
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        in_done = [torch.cuda.Event() for _ in range(2)]
        comp_done = [torch.cuda.Event() for _ in range(2)]
        out_done = [torch.cuda.Event() for _ in range(2)]
        used = [False, False]

        def one(i):
            b_ = i % 2
            st = sets[b_]
            with torch.cuda.stream(s_in):
                if used[b_]:
                    s_in.wait_event(comp_done[b_])
                st["q"].copy_(hq, non_blocking=True)
                st["k"].copy_(hk, non_blocking=True)
                st["v"].copy_(hv, non_blocking=True)
                in_done[b_].record(s_in)
            stream.wait_event(in_done[b_])
            if used[b_]:
                stream.wait_event(out_done[b_])
            zz = st["z"]
            a_ = fa.fa_fp8_quantize(st["q"], st["k"], st["v"], signs, B, H, N, d, zz["q8"],
                                    zz["k8"], zz["vt8"], zz["s_q"], zz["s_k"], zz["s_v"], ws, wsb)
            a_ |= fa.fa_fwd_fp8(zz["q8"], zz["k8"], zz["vt8"], zz["s_q"], zz["s_k"], zz["s_v"],
                                st["o"], st["lse"], B, H, N, d, w.scale, w.causal)
            if a_ != 0:
                raise RuntimeError("FP8 step failed")
            comp_done[b_].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(comp_done[b_])
                st["ho"].copy_(st["o"], non_blocking=True)
                st["hl"].copy_(st["lse"], non_blocking=True)
                out_done[b_].record(s_out)
            used[b_] = True

        for i in range(2):
            one(i)
        torch.cuda.synchronize()
        n = max(3, min(args.steps, 20))
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(s_in)
        for i in range(n):
            one(i)
        a1.record(s_out)
        torch.cuda.synchronize()
        secs = max_over_ranks(pg, a0.elapsed_time(a1) / 1e3)
        e2e = {"value": flops * n * world / secs / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": 3 * q.numel() * 2,
               "d2h_bytes_per_step": o.numel() * 2 + lse.numel() * 4, "steps": n,
               "copies": "pipelined: step i+1's inputs in and step i-1's results out during step i"}
    if rank != 0:
        if pg is not None:
            pg.destroy_process_group()
        return None
    peaks, peak_src = load_peaks()
    # FP8 dense peak: the measured bf16 peak times the nominal FP8 / bf16 ratio (2)
    peak8 = 2.0 * float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    t_step = elapsed / args.steps
    value = flops * args.steps * world / elapsed / 1e12
    qbytes = 2 * 3 * B * H * N * d * 2 + 3 * B * H * N * d  # bf16 read by both passes, e4m3 written
    result = {
        "metric": FP8_METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_step * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3",
        "data": "synthetic (seeded N(0,1) bf16 Q, K, V quantised by the library; no dataset)",
        "config": {"workload": w.name, "description": w.description, "B": B, "H": H, "N": N,
                   "d": d, "causal": w.causal, "allowed_pairs": pairs, "flops_per_step": flops,
                   "l2": "inputs larger than L2 (no flush)",
                   "parallelism": f"replicas x{world} (no collective)"},
        "breakdown": {"fwd_ms": t_step * 1e3, "quantise_ms": t_quant * 1e3,
                      "quantise_gbs": qbytes / t_quant / 1e9},
        "roofline": {"bound": "tensor", "achieved": value / world, "peak": peak8,
                     "unit": "TFLOP/s", "frac": value / world / peak8,
                     "traffic": ncu_traffic("fwd_fp8", w.name),
                     "kernel": "fa_fwd_fp8_kernel",
                     "peak_source": f"{peak_src} (bf16_tflops x 2, the nominal FP8 ratio)"},
        "e2e": e2e,
        "gpu_launches": args.steps,
        "clocks": clk.summary(),
    }
    if not args.no_cpu_baseline:
        import oracle
        z_cpu = {n_: t.cpu() for n_, t in z.items()}
        t0 = time.perf_counter()
        heads = 0
        v8 = z_cpu["vt8"][..., :N].transpose(2, 3).contiguous()
        while time.perf_counter() - t0 < 10.0 and heads < B * H:
            b, h = divmod(heads, H)
            sl = lambda t: t[b:b + 1, h:h + 1].numpy()
            oracle.fwd_fp8(sl(z_cpu["q8"]), sl(z_cpu["k8"]), sl(v8), sl(z_cpu["s_q"]).astype(np.float64),
                           sl(z_cpu["s_k"]).astype(np.float64), sl(z_cpu["s_v"]).astype(np.float64),
                           w.scale, causal=w.causal)
            heads += 1
        secs = time.perf_counter() - t0
        cores = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
        result["cpu_baseline"] = {"value": flops / (B * H) * heads / secs / 1e12, "unit": "TFLOP/s",
                                  "cores": cores, "kind": "oracle", "cpu_model": cpu_model(),
                                  "sample": f"{heads} of {B * H} heads of {w.name}, fp64, {secs:.1f} s"}
    if pg is not None:
        pg.destroy_process_group()
    return result


def run_fp8_reference(args, w):
    """The fp64 oracle's FP8 forward (exact attention of the dequantised
    inputs) on the host, head (0, 0) per step."""
    if int(os.environ.get("RANK", "0")) != 0:
        return None
    import oracle
    x = inputs.draw(inputs.Workload("s", 1, 1, w.N, w.d, causal=w.causal), with_grad=False)
    f64 = lambda t: t.double().numpy()
    signs = inputs.rotation_signs(w.d, seed=0).double().numpy()
    q8, k8, v8, sq, sk, sv = oracle.quantize_fp8(f64(x["q"]), f64(x["k"]), f64(x["v"]), signs)
    for _ in range(args.warmup):
        oracle.fwd_fp8(q8, k8, v8, sq, sk, sv, w.scale, causal=w.causal)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.fwd_fp8(q8, k8, v8, sq, sk, sv, w.scale, causal=w.causal)
    secs = time.perf_counter() - t0
    flops = 4.0 * w.d * allowed_pairs(inputs.Workload("s", 1, 1, w.N, w.d, causal=w.causal), None)
    value = flops * args.steps / secs / 1e12
    cores = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    return {
        "impl": "reference", "metric": FP8_METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded N(0,1), same recipe)",
        "config": {"workload": w.name, "description": w.description},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "cpu_model": cpu_model(),
                         "sample": f"one head of {w.name} per step, fp64"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=sorted(inputs.ALL) + [inputs.DECODE.name, inputs.FP8_CAUSAL.name])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer measurement")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)  # at least three untimed warm-up steps
    if args.workload == inputs.FP8_CAUSAL.name:
        w = inputs.FP8_CAUSAL
        res = run_fp8_reference(args, w) if args.impl == "reference" else run_fp8(args, w)
    elif args.workload == inputs.DECODE.name:
        w = inputs.DECODE
        res = run_decode_reference(args, w) if args.impl == "reference" else run_decode(args, w)
    else:
        w = inputs.ALL[args.workload]
        res = run_reference(args, w) if args.impl == "reference" else run_ours(args, w)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
