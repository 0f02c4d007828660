#!/usr/bin/env python3
"""Benchmark: attention forward TFLOP/s and row-softmax GB/s on GB300.

One step = one call of the fused attention forward (the tensor-core kernel)
on the causal bf16 workload B=2, H=32, N=4096, d=128 (Q, K, V ~ N(0,1) rounded
to bf16; 192 MiB of Q/K/V, larger than the 129 MB L2), through the C ABI.
The row softmax (fp32, 4096 x N, the HBM-resident lengths) is timed in the
same run with L2 flushed before every repetition and reported under
"softmax" (all five row lengths, each with its regime); the other attention
configurations (fp32 single head, bf16 d=64 non-causal, bf16 varlen causal)
under "configs"; split-KV attention on a decode-like shape (256 queries, 32768 keys)
under "splitkv"; the attention backward on the headline workload under
"bwd" and the FP8 forward under "fp8".  Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Multi-GPU (torchrun, one process per GPU): every rank runs its own replica of
the workload (weak scaling, no collective on the data path); the time is the
max over ranks and the value counts the work of all ranks.
``--impl reference`` times the fp64 CPU oracle on the host cores instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = ("attention fwd TFLOP/s and % BF16 peak; softmax GB/s and % HBM peak (1×GB300)")
HEADLINE = "attn_bf16_causal_b2h32n4096d128"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KERNEL_SOURCE = os.path.join(ROOT, "online_softmax_06_gb300", "csrc", "attn_bf16.cu")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "attn_bf16_causal_b2h32n4096d128.md")


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(
        k for k, w in workloads.WORKLOADS.items() if w.dtype == "bf16"))
    ap.add_argument("--softmax-n", default="32,128,1024,4096,32768",
                    help="comma-separated row lengths for the softmax leg ('' to skip)")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the legs of the other attention configurations")
    ap.add_argument("--softmax-reps", type=int, default=20)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-splitkv", action="store_true", help="skip the split-KV leg")
    ap.add_argument("--no-bwd", action="store_true", help="skip the backward leg")
    ap.add_argument("--no-fp8", action="store_true", help="skip the FP8 forward leg")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle baseline sample")
    return ap.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash() -> str:
    with open(KERNEL_SOURCE, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def recorded_traffic():
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source (else None)."""
    try:
        text = open(TRAFFIC_FILE, encoding="utf-8").read()
    except OSError:
        return None
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)\s*\(kernel source sha256\[:16\]\s*"
                  r"([0-9a-f]+)\)", text)
    if not m or m.group(2) != kernel_source_hash():
        return None
    return float(m.group(1))


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.windows = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def mark(self, t0: float, t1: float):
        self.windows.append((t0, t1))

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        time.sleep(0.05)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                frac = float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                rows.append((ts + frac, float(parts[1]), float(parts[2]), parts[4:8]))
            except (ValueError, IndexError):
                continue
        inside = [r for r in rows if any(a - 0.03 <= r[0] <= b + 0.03 for a, b in self.windows)]
        use = inside if inside else rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in use for i, v in enumerate(r[3]) if v == "Active"})
        return {"sm_mhz": statistics.median(r[1] for r in use) if use else None,
                "sm_max_mhz": max(r[2] for r in use) if use else None,
                "reasons": reasons, "samples": len(use),
                "samples_in_timed_region": len(inside)}


# ---------------------------------------------------------------------------
# oracle on the host cores (cpu_baseline and --impl reference)
# ---------------------------------------------------------------------------
def oracle_sample(w, n_rows: int, seed: int):
    """A bounded, deterministic sample of the workload's query rows for the
    oracle, and the algorithmic flops of those rows (4 * visible keys * d)."""
    tok, head = workloads.sample_rows(w.total, w.H, n_rows, seed=seed)
    cu = w.cu_seqlens()
    seq = np.searchsorted(cu, tok, side="right") - 1
    pos = tok - cu[seq]
    L = (cu[seq + 1] - cu[seq]).astype(np.int64)
    vis = (pos + 1) if w.causal else L
    return tok, head, float(np.sum(4.0 * vis * w.d))


def time_oracle(w, Qp, Kp, Vp, n_rows: int, seed: int):
    import oracle
    tok, head, flops = oracle_sample(w, n_rows, seed)
    t0 = time.perf_counter()
    oracle.attention_rows(Qp, Kp, Vp, w.cu_seqlens(), w.scale, w.causal, tok, head)
    return time.perf_counter() - t0, flops


def packed_f32(w):
    Q, K, V = w.inputs()
    Q, K, V = (t.float().numpy().reshape(w.total, w.H, w.d) for t in (Q, K, V))
    return Q, K, V


def cpu_baseline(w, seconds: float):
    import oracle
    oracle.load()                                            # built and loaded before timing
    Qp, Kp, Vp = packed_f32(w)
    time_oracle(w, Qp, Kp, Vp, 64, seed=0)                   # warm-up (threads, caches)
    dt, _ = time_oracle(w, Qp, Kp, Vp, 64, seed=1)          # calibration
    per_row = max(dt / 64, 1e-6)
    n = int(min(max(seconds / per_row, 256), w.total * w.H))
    dt, flops = time_oracle(w, Qp, Kp, Vp, n, seed=2)
    cores = oracle.num_threads()
    out = {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
           "sample": f"{n} (token, head) query rows of {w.name} drawn uniformly with seed 2 "
                     f"(fp64, {dt:.1f} s); flops = 4 * visible keys * d per row"}
    # per-core speed: every query row of the first sequence's first head on one thread
    L0 = int(w.cu_seqlens()[1])
    tok = np.arange(L0, dtype=np.int64)
    head = np.zeros(L0, dtype=np.int64)
    vis = (tok + 1) if w.causal else np.full(L0, L0)
    flops1 = float(np.sum(4.0 * vis * w.d))
    oracle.set_num_threads(1)
    try:
        t0 = time.perf_counter()
        oracle.attention_rows(Qp, Kp, Vp, w.cu_seqlens(), w.scale, w.causal, tok, head)
        dt1 = time.perf_counter() - t0
    finally:
        oracle.set_num_threads(cores)
    out["one_thread"] = {"value": flops1 / dt1 / 1e12, "unit": "TFLOP/s", "cores": 1,
                         "sample": f"all {L0} query rows of (sequence 0, head 0) ({dt1:.1f} s)"}
    return out


def run_reference(args, rank: int):
    if rank != 0:
        return 0
    import oracle
    oracle.load()                                            # built and loaded before timing
    w = workloads.WORKLOADS[args.workload]
    Qp, Kp, Vp = packed_f32(w)
    time_oracle(w, Qp, Kp, Vp, 64, seed=0)                   # warm-up (threads, caches)
    dt, _ = time_oracle(w, Qp, Kp, Vp, 64, seed=1)
    per_row = max(dt / 64, 1e-6)
    # each step is a bounded sample sized so the whole run stays within minutes
    budget = 150.0 / max(args.steps + args.warmup, 1)
    n = int(min(max(budget / per_row, 64), w.total * w.H))
    for s in range(args.warmup):
        time_oracle(w, Qp, Kp, Vp, n, seed=100 + s)
    tot_t, tot_f = 0.0, 0.0
    for s in range(args.steps):
        dt, fl = time_oracle(w, Qp, Kp, Vp, n, seed=1000 + s)
        tot_t += dt
        tot_f += fl
    value = tot_f / tot_t / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000 * tot_t / max(args.steps, 1), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.num_threads(),
                             "kind": "oracle",
                             "sample": f"{n} sampled query rows of {w.name} per step"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def workload_config(w):
    return {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": w.causal,
            "varlen_lengths": list(w.lengths) or None,
            "flops_per_step": w.flops(),
            "l2": "inputs larger than L2 (Q/K/V %.0f MiB vs 129 MB L2)" %
                  (3 * w.total * w.H * w.d * 2 / 2**20),
            "parallelism": "replicas (weak scaling, no collective)"}


# ---------------------------------------------------------------------------
# GPU legs
# ---------------------------------------------------------------------------
def time_attention(fa, w, dev, steps, warmup, dist, clocks):
    import torch
    Q, K, V = w.inputs()
    q, k, v = (t.to(dev) for t in (Q, K, V))
    o = torch.empty_like(q)
    lse_shape = (w.H, w.total) if w.varlen else (w.B, w.H, w.N)
    lse = torch.empty(lse_shape, dtype=torch.float32, device=dev)
    cu = torch.from_numpy(w.cu_seqlens()).to(dev) if w.varlen else None
    stream = torch.cuda.current_stream(dev)
    fa.fa_set_stream(stream.cuda_stream)
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr())

    def launch():
        if w.varlen:
            rc = fa.fa_attention_fwd_varlen(*args, w.B, w.H, w.N, w.total, w.d, w.scale,
                                            int(w.causal), cu.data_ptr())
        else:
            rc = fa.fa_attention_fwd(*args, w.B, w.H, w.N, w.d, w.scale, int(w.causal), None)
        if rc != 0:
            raise RuntimeError(f"attention launch failed: {fa.strerror(rc)}")

    for _ in range(warmup):
        launch()
    torch.cuda.synchronize(dev)
    if dist:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    e0.record(stream)
    for _ in range(steps):
        launch()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    clocks.mark(t0, time.time())
    if dist:
        dist.barrier()
    ms = e0.elapsed_time(e1)
    dev_err = fa.fa_get_device_error()
    if dev_err != 0:
        raise RuntimeError(f"device error word {dev_err:#x}")
    return ms, steps


def time_config(fa, w, dev, reps, peaks, clocks):
    """One more attention configuration, timed like the headline (CUDA events
    over back-to-back launches on the library stream, after warm-up): the
    d = 64 non-causal and the varlen causal workloads on the tensor-core
    kernel, and the fp32 single-head workload on the CUDA-core kernel (a
    correctness path: 16.8 MFLOP, one launch's latency)."""
    import torch
    if w.dtype == "f32":
        Q, K, V = w.inputs()
        q, k, v = (torch.from_numpy(t).to(dev) for t in (Q, K, V))
        o = torch.empty_like(q)
        lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
        stream = torch.cuda.current_stream(dev)
        fa.fa_set_stream(stream.cuda_stream)

        def launch():
            rc = fa.fa_attention_fwd_f32(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                         lse.data_ptr(), w.B, w.H, w.N, w.d, w.scale,
                                         int(w.causal), None)
            if rc != 0:
                raise RuntimeError(fa.strerror(rc))
        for _ in range(3):
            launch()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0 = time.time()
        e0.record(stream)
        for _ in range(reps):
            launch()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        clocks.mark(t0, time.time())
        ms = e0.elapsed_time(e1) / reps
        tf = w.flops() / (ms / 1e3) / 1e12
        return {"ms": ms, "TFLOP_per_s": tf, "dtype": "f32", "bound": "latency",
                "kernel": "attn_fwd_f32_kernel", "flops_per_launch": w.flops(),
                "note": "fp32 CUDA-core path for fp32 accuracy; one small launch, so the "
                        "time is launch and latency, not a roofline"}
    ms, steps = time_attention(fa, w, dev, reps, 3, None, clocks)
    ms /= steps
    tf = w.flops() / (ms / 1e3) / 1e12
    return {"ms": ms, "TFLOP_per_s": tf, "frac_of_bf16_peak": tf / peaks["bf16_tflops"],
            "dtype": "bf16", "bound": "tensor", "kernel": f"attn_fwd_bf16_kernel<{w.d}>",
            "flops_per_launch": w.flops(),
            "l2": "inputs larger than L2 (Q/K/V %.0f MiB); %d back-to-back launches"
                  % (3 * w.total * w.H * w.d * 2 / 2**20, reps)}


def time_e2e(fa, w, dev, steps, warmup):
    """Same metric through the C ABI with host buffers: every step takes Q, K, V
    from pinned host memory and leaves O and lse in pinned host memory.  Dense
    workloads call fa_attention_fwd_host (the library copies head group by
    head group and overlaps the copies with the kernels); packed batches copy
    with torch around fa_attention_fwd_varlen."""
    import torch
    Q, K, V = w.inputs()
    hq, hk, hv = (t.pin_memory() for t in (Q, K, V))
    lse_shape = (w.H, w.total) if w.varlen else (w.B, w.H, w.N)
    ho = torch.empty_like(Q).pin_memory()
    hl = torch.empty(lse_shape, dtype=torch.float32).pin_memory()
    stream = torch.cuda.current_stream(dev)
    fa.fa_set_stream(stream.cuda_stream)
    if w.varlen:
        q, k, v = (torch.empty_like(t, device=dev) for t in (Q, K, V))
        o = torch.empty_like(q)
        lse = torch.empty(lse_shape, dtype=torch.float32, device=dev)
        cu = torch.from_numpy(w.cu_seqlens()).to(dev)
        args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr())

        def step():
            q.copy_(hq, non_blocking=True)
            k.copy_(hk, non_blocking=True)
            v.copy_(hv, non_blocking=True)
            rc = fa.fa_attention_fwd_varlen(*args, w.B, w.H, w.N, w.total, w.d, w.scale,
                                            int(w.causal), cu.data_ptr())
            if rc != 0:
                raise RuntimeError(fa.strerror(rc))
            ho.copy_(o, non_blocking=True)
            hl.copy_(lse, non_blocking=True)
        api = "fa_attention_fwd_varlen (torch copies around it)"
    else:
        nbytes = fa.fa_attention_host_workspace_bytes(w.B, w.H, w.N, w.d)
        ws = torch.empty(int(nbytes), dtype=torch.uint8, device=dev)
        args = (hq.data_ptr(), hk.data_ptr(), hv.data_ptr(), ho.data_ptr(), hl.data_ptr(),
                w.B, w.H, w.N, w.d, w.scale, int(w.causal), ws.data_ptr(), int(nbytes))

        def step():
            rc = fa.fa_attention_fwd_host(*args)
            if rc != 0:
                raise RuntimeError(fa.strerror(rc))
        api = "fa_attention_fwd_host"

    for _ in range(warmup):
        step()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1)
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
    d2h = ho.numel() * ho.element_size() + hl.numel() * hl.element_size()
    return {"value": w.flops() * steps / (ms / 1e3) / 1e12, "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": ms / steps, "api": api}


def time_softmax(fa, dev, Ns, reps, peaks, clocks):
    """Row softmax 4096 x N, each rep timed alone with CUDA events, median reported.

    Before every rep the L2 is flushed by writing a 512 MiB buffer (4x the L2)
    and then reading it back, so x is cold and the L2 holds clean lines: the
    kernel is not charged for writing back the flush's dirty lines.  The
    write-only flush (dirty L2) and the warm (no flush) figures are reported
    beside it."""
    import torch
    stream = torch.cuda.current_stream(dev)
    fa.fa_set_stream(stream.cuda_stream)
    flush = torch.empty(512 * 2**20 // 4, dtype=torch.float32, device=dev)
    out = {}

    def timed_reps(rows, N, x, y, read_back):
        times = []
        for _ in range(reps):
            flush.zero_()
            if read_back:
                flush.sum()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            rc = fa.fa_softmax_rows(x.data_ptr(), y.data_ptr(), rows, N)
            e1.record(stream)
            if rc != 0:
                raise RuntimeError(fa.strerror(rc))
            torch.cuda.synchronize(dev)
            times.append(e0.elapsed_time(e1))
        return statistics.median(times)

    for N in Ns:
        x = torch.from_numpy(workloads.softmax_workload(N)).to(dev)
        y = torch.empty_like(x)
        rows = x.shape[0]
        for _ in range(3):
            fa.fa_softmax_rows(x.data_ptr(), y.data_ptr(), rows, N)
        t0 = time.time()
        ms = timed_reps(rows, N, x, y, True)
        ms_dirty = timed_reps(rows, N, x, y, False)
        clocks.mark(t0, time.time())
        # warm (no flush) for context
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            fa.fa_softmax_rows(x.data_ptr(), y.data_ptr(), rows, N)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        warm_ms = e0.elapsed_time(e1) / reps
        nbytes = 8.0 * rows * N
        gbs = nbytes / (ms / 1e3) / 1e9
        if nbytes >= 2 * 129e6:
            regime = "HBM-bound (input and output larger than the 129 MB L2)"
        elif nbytes >= 16 * 2**20:
            regime = ("input read cold from HBM, output (%.0f MiB) fits in L2 and is written "
                      "back after the kernel: partly L2-bound" % (nbytes / 2 / 2**20))
        else:
            regime = ("latency-bound: %.1f MiB in and out, launch and one-wave latency "
                      "dominate; the GB/s figure is not an HBM roofline fraction"
                      % (nbytes / 2 / 2**20))
        out[str(N)] = {"rows": rows, "N": N, "ms": ms, "GB_per_s": gbs,
                       "frac_of_hbm": gbs / peaks["hbm_gbs"], "regime": regime,
                       "bytes_per_launch": nbytes,
                       "l2": "flushed before each rep (512 MiB written, then read back)",
                       "dirty_l2_GB_per_s": nbytes / (ms_dirty / 1e3) / 1e9,
                       "warm_GB_per_s": nbytes / (warm_ms / 1e3) / 1e9}
        del x, y
    return out


def time_splitkv(fa, dev, reps, peaks, clocks):
    """Split-KV attention (tensor-core kernel per key split + combine kernel) on
    the decode-like workload: 256 new queries, 32768 keys, 16 heads, causal.

    K and V (256 MiB) exceed the L2, so back-to-back calls re-read them from
    HBM.  At this shape the HBM floor (every Q, K, V, O byte once: 270 MB) is
    above the tensor floor (68.5 GFLOP), so both fractions are reported and the
    bound is HBM.  The one-split figure (same kernel, 16 CTAs) is beside it."""
    import torch
    w = workloads.SPLITKV_WORKLOADS["attn_bf16_splitkv_b1h16nq256nk32768d128_causal"]
    Q, K, V = w.inputs()
    q, k, v = (t.to(dev) for t in (Q, K, V))
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.Nq), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    fa.fa_set_stream(stream.cuda_stream)
    splits = fa.fa_splitkv_num_splits(w.B, w.H, w.Nq, w.Nk, w.d)
    if splits < 1:
        raise RuntimeError(fa.strerror(splits))
    o_acc = torch.empty((splits, w.B, w.Nq, w.H, w.d), dtype=torch.float32, device=dev)
    l_acc = torch.empty((splits, w.B, w.H, w.Nq), dtype=torch.float32, device=dev)

    def timed(n_splits):
        def launch():
            rc = fa.fa_attention_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                             o.data_ptr(), lse.data_ptr(), w.B, w.H, w.Nq,
                                             w.Nk, w.d, w.scale, int(w.causal), n_splits,
                                             o_acc.data_ptr(), l_acc.data_ptr())
            if rc != 0:
                raise RuntimeError(fa.strerror(rc))
        for _ in range(3):
            launch()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            launch()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / reps

    t0 = time.time()
    ms = timed(splits)
    ms1 = timed(1)
    clocks.mark(t0, time.time())
    dev_err = fa.fa_get_device_error()
    if dev_err != 0:
        raise RuntimeError(f"device error word {dev_err:#x}")
    flops = w.flops()
    nbytes = 2.0 * (q.numel() + k.numel() + v.numel() + o.numel()) + 4.0 * lse.numel()
    partial_bytes = 2.0 * 4.0 * (o_acc.numel() + l_acc.numel())
    tf = flops / (ms / 1e3) / 1e12
    gbs = nbytes / (ms / 1e3) / 1e9
    return {"workload": w.name, "B": w.B, "H": w.H, "Nq": w.Nq, "Nk": w.Nk, "d": w.d,
            "causal": w.causal, "splits": splits, "launches_per_call": 2 if splits > 1 else 1,
            "ms": ms, "TFLOP_per_s": tf, "frac_of_bf16_peak": tf / peaks["bf16_tflops"],
            "algorithmic_bytes": nbytes, "GB_per_s": gbs, "frac_of_hbm": gbs / peaks["hbm_gbs"],
            "bound": "hbm", "partial_bytes_written_and_read": partial_bytes,
            "flops_per_call": flops, "one_split_ms": ms1,
            "one_split_TFLOP_per_s": flops / (ms1 / 1e3) / 1e12,
            "l2": "K/V 256 MiB, larger than L2; %d back-to-back calls" % reps}


def time_bwd(fa, w, dev, reps, peaks, clocks):
    """Attention backward on the headline workload, both forms: the one-pass
    call (fa_attention_bwd_atomic: D and zeroing, one pass over the key tiles
    with dQ summed by fp32 atomic adds, the dQ conversion) and the
    deterministic two-pass call (fa_attention_bwd: dQ/D kernel, dK/dV
    kernel).  O and lse come from one forward call outside the timed region;
    dO ~ N(0, 1) in bf16.  Algorithmic work = 2.5 x the forward's (the five
    products S, dP, dV, dK, dQ of 2 N^2 d each against the forward's two);
    the two-pass form runs seven, recomputing S and dP for dQ."""
    import torch
    if w.varlen:
        return None
    Q, K, V = w.inputs()
    q, k, v = (t.to(dev) for t in (Q, K, V))
    rng = np.random.default_rng(w.seed + 77)
    do = torch.from_numpy(rng.standard_normal(q.shape, dtype=np.float32)).to(torch.bfloat16).to(dev)
    stream = torch.cuda.current_stream(dev)
    fa.fa_set_stream(stream.cuda_stream)
    o, lse = fa.attention_fwd(q, k, v, causal=w.causal)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    dbuf = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    args = [t.data_ptr() for t in (q, k, v, o, do, lse, dq, dk, dv, dbuf)]
    ws_bytes = fa.fa_attention_bwd_atomic_workspace_bytes(w.B, w.H, w.N, w.d)
    ws = torch.empty((max(ws_bytes, 4) // 4,), dtype=torch.float32, device=dev)

    def two_pass():
        rc = fa.fa_attention_bwd(*args, w.B, w.H, w.N, w.d, w.scale, int(w.causal))
        if rc != 0:
            raise RuntimeError(fa.strerror(rc))

    def one_pass():
        rc = fa.fa_attention_bwd_atomic(*args, w.B, w.H, w.N, w.d, w.scale, int(w.causal),
                                        ws.data_ptr(), ws_bytes)
        if rc != 0:
            raise RuntimeError(fa.strerror(rc))

    def timed(launch):
        for _ in range(3):
            launch()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0 = time.time()
        e0.record(stream)
        for _ in range(reps):
            launch()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        clocks.mark(t0, time.time())
        dev_err = fa.fa_get_device_error()
        if dev_err != 0:
            raise RuntimeError(f"device error word {dev_err:#x}")
        return e0.elapsed_time(e1) / reps

    flops = 2.5 * w.flops()
    out = {"workload": w.name, "bound": "tensor", "algorithmic_flops_per_call": flops,
           "l2": "inputs larger than L2 (Q/K/V/O/dO 320 MiB); %d back-to-back calls" % reps}
    ms2 = timed(two_pass)
    det = {"api": "fa_attention_bwd", "ms": ms2, "TFLOP_per_s": flops / (ms2 / 1e3) / 1e12,
           "executed_flops_per_call": 3.5 * w.flops(), "launches_per_call": 2}
    det["frac_of_bf16_peak"] = det["TFLOP_per_s"] / peaks["bf16_tflops"]
    if w.d == 128:
        ms1 = timed(one_pass)
        tf = flops / (ms1 / 1e3) / 1e12
        out.update({"api": "fa_attention_bwd_atomic", "ms": ms1, "TFLOP_per_s": tf,
                    "frac_of_bf16_peak": tf / peaks["bf16_tflops"],
                    "executed_flops_per_call": flops, "launches_per_call": 3,
                    "deterministic": det})
    else:
        out.update(det)
    return out


def time_fp8(fa, w, dev, reps, peaks, clocks):
    """FP8 forward on the headline workload: the whole call (rotation and
    blockwise e4m3 quantisation of Q, K, V, then the e4m3 tensor-core kernel)
    and the attention kernel alone (the quantised tensors reused).  Peak: the
    measured bf16 peak x 2, the nominal e4m3 / bf16 ratio (4.5 / 2.25
    PFLOP/s dense)."""
    import torch
    if w.varlen or w.d != 128:
        return None
    Q, K, V = w.inputs()
    q, k, v = (t.to(dev) for t in (Q, K, V))
    rng = np.random.default_rng(w.seed + 88)
    signs = torch.from_numpy(rng.choice([-1.0, 1.0], size=w.d).astype(np.float32)).to(dev)
    stream = torch.cuda.current_stream(dev)
    fa.fa_set_stream(stream.cuda_stream)
    nbytes = fa.fa_attention_fp8_workspace_bytes(w.B, w.H, w.N, w.d)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)

    def launch():
        rc = fa.fa_attention_fwd_fp8(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                     lse.data_ptr(), w.B, w.H, w.N, w.d, w.scale, int(w.causal),
                                     signs.data_ptr(), ws.data_ptr(), nbytes)
        if rc != 0:
            raise RuntimeError(fa.strerror(rc))

    for _ in range(3):
        launch()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    e0.record(stream)
    for _ in range(reps):
        launch()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    clocks.mark(t0, time.time())
    dev_err = fa.fa_get_device_error()
    if dev_err != 0:
        raise RuntimeError(f"device error word {dev_err:#x}")
    ms = e0.elapsed_time(e1) / reps
    flops = w.flops()
    tf = flops / (ms / 1e3) / 1e12
    peak = 2.0 * peaks["bf16_tflops"]
    return {"workload": w.name, "ms_per_call": ms, "TFLOP_per_s": tf,
            "frac_of_fp8_peak": tf / peak, "fp8_peak_TFLOP_per_s": peak,
            "peak_source": "measured bf16 dense x 2 (nominal e4m3/bf16 ratio)",
            "launches_per_call": 3, "flops_per_call": flops,
            "l2": "inputs larger than L2; %d back-to-back calls" % reps}


def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, rank)

    import torch
    import online_softmax_06_gb300 as fa
    fa.build()
    fa.lib()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as tdist
        tdist.init_process_group("nccl", device_id=dev)
        dist = tdist
    peaks, peak_src = load_peaks()
    w = workloads.WORKLOADS[args.workload]
    clocks = ClockSampler(local_rank)
    try:
        ms, steps = time_attention(fa, w, dev, args.steps, args.warmup, dist, clocks)
        ms_t = torch.tensor([ms], dtype=torch.float64, device=dev)
        if dist:
            dist.all_reduce(ms_t, op=dist.ReduceOp.MAX)
        ms_max = float(ms_t.item())
        softmax = {}
        if args.softmax_n and rank == 0:
            Ns = [int(s) for s in args.softmax_n.split(",") if s]
            softmax = time_softmax(fa, dev, Ns, args.softmax_reps, peaks, clocks)
        splitkv = None
        if not args.no_splitkv and rank == 0:
            splitkv = time_splitkv(fa, dev, 50, peaks, clocks)
        bwd = None
        if not args.no_bwd and rank == 0:
            bwd = time_bwd(fa, w, dev, 20, peaks, clocks)
        fp8 = None
        if not args.no_fp8 and rank == 0:
            fp8 = time_fp8(fa, w, dev, 50, peaks, clocks)
        configs = None
        if not args.no_configs and rank == 0:
            configs = {}
            for name, wc in workloads.WORKLOADS.items():
                if name == w.name:
                    continue
                configs[name] = time_config(fa, wc, dev, 50 if wc.dtype == "f32" else 30,
                                            peaks, clocks)
    finally:
        clk = clocks.stop()
    e2e = None
    if not args.no_e2e:
        e2e = time_e2e(fa, w, dev, max(3, min(args.steps, 50)), 2)
    flops = w.flops()
    value = world * flops * steps / (ms_max / 1e3) / 1e12
    per_launch_s = (ms / 1e3) / steps
    achieved = flops / per_launch_s / 1e12
    peak = peaks["bf16_tflops"]
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": steps,
        "warmup": args.warmup, "ms_per_step": ms_max / steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(w),
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak,
                     # the committed DRAM capture covers the headline workload
                     "traffic": recorded_traffic() if w.name == HEADLINE else None,
                     "peak_source": f"{peak_src} bf16 dense (burst)",
                     "kernel": f"attn_fwd_bf16_kernel<{w.d}>",
                     "algorithmic_flops_per_launch": flops},
        "gpu_launches": steps,
        "clocks": clk,
        "softmax": softmax,
        "splitkv": splitkv,
        "bwd": bwd,
        "fp8": fp8,
        "configs": configs,
        "e2e": e2e,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
