#!/usr/bin/env python
"""Benchmark of fused LM-head scoring (libfusedlogp) on GB300.

A step is one fused log-prob + entropy call over the forward-scoring workload
(T = 4096 scored rows, H = 4096, V = 151,936, bf16, temperature 0.7): the
tensor-core logit tiles, the FP32 online log-sum-exp/entropy fold and the
split merge.  Inputs are resident in HBM; the 1.24 GB weight is larger than
L2 and is streamed from HBM every step, so no L2 flush is needed.

Prints ONE JSON line (rank 0):
  value       scored tokens/s over all ranks (device-timed, CUDA events)
  roofline    achieved TFLOP/s of the tensor-core kernel (2 n V H flops per
              launch / its event-timed duration) against the measured bf16
              peak in MEASURED_PEAKS.json; DRAM traffic from the committed
              ncu summary when it matches the current kernel sources
  e2e         the same metric through the public API with the step's inputs
              copied from pinned host memory and the results read back
  cpu_baseline the float64 oracle on a bounded row sample on the host cores
  memory      the allocator's peak over one call beside the workspace and
              the [n, V] FP32 logits the fused path never forms
  workloads   the other workloads (long packed fp16, KL, backward) measured
              the same way, when available

--impl reference times the float64 CPU oracle (the reference arm of this
build: the pages ship no runnable implementation) on the same workload.

Multi-GPU: the path has no exchange step; under torchrun each rank scores its
own replica of the workload (weak scaling) and the time is the max over ranks.
"""
import argparse
import hashlib
import json
import math
import os
import platform
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "scored tokens/s and TFLOP/s (% of GB300 dense BF16 peak), fused logp+entropy"
UNIT = "scored tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# Nominal dense rate of tcgen05.mma kind::mxf8f6f4 (E4M3 x E2M1 with E8M0
# block scales) over kind::f16 with bf16 operands: 4.5 against 2.25 PFLOP/s.
MX_OVER_BF16 = 2.0


def own_peak(P, arith, sustained=False):
    """Peak of the arithmetic a kernel runs, in bf16-equivalent TFLOP/s (the
    flops counted are 2nVH per head), from the measured bf16 figure.
    arith: "bf16"; "mx" (every MMA block-scaled); "bf16+mx" (half the flops,
    the student's, in bf16 and half, the teacher's, block-scaled, which the
    tensor pipe runs one after the other)."""
    b = P["bf16_tflops_sustained" if sustained else "bf16_tflops"]
    return {"bf16": b, "mx": MX_OVER_BF16 * b,
            "bf16+mx": 2.0 / (1.0 / b + 1.0 / (MX_OVER_BF16 * b))}[arith]


PEAK_KIND = {
    "bf16": "bf16 dense, burst, %s",
    "mx": "kind::mxf8f6f4 dense (E4M3 x E2M1), burst: %s bf16 x 2, the nominal fp8:bf16 ratio",
    "bf16+mx": ("student bf16 + teacher kind::mxf8f6f4, burst: %s bf16 x 4/3 (half the flops "
                "at twice the rate)"),
}
DTYPE = {"mx": "e4m3 x e2m1 (MX block-scaled), f32 accumulate",
         "bf16+mx": "bf16 student + e4m3 x e2m1 (MX block-scaled) teacher, f32 accumulate"}
FWD_KERNEL_SOURCES = ["ptx.cuh", "schedule.h", "vocab_pipeline.cuh", "kernels_fwd.cu", "launch.h",
                      "lse_epilogue.cuh", "support.cuh"]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "vocab_pipeline_forward-scoring.txt")


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=300)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", type=int, default=1)
    p.add_argument("--no-extra", action="store_true", help="skip the other workloads")
    p.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    p.add_argument("--no-e2e", action="store_true", help="skip the end-to-end loop")
    p.add_argument("--cpu-seconds", type=float, default=12.0)
    p.add_argument("--T", type=int, default=None,
                   help="replace the workload's row count (same H, V, recipe): small profiling cases")
    p.add_argument("--head", choices=["bf16", "mx"], default="bf16",
                   help="forward workloads: the head in bf16, or in MXFP4 on the block-scaled "
                        "tensor cores with the scored rows in MXFP8 (head quantised before timing)")
    p.add_argument("--teacher", choices=["bf16", "mxfp4", "mx"], default="bf16",
                   help="KL workloads: the teacher head in bf16, in MXFP4 decoded to bf16 next to "
                        "the tensor cores, or (mx) MXFP4 on the block-scaled tensor cores with the "
                        "teacher rows in MXFP8 (heads quantised before timing)")
    p.add_argument("--support-j", type=int, default=None,
                   help="forward workloads: restrict each row to a sampling support keeping each "
                        "token with probability 2^-J (targets kept)")
    return p.parse_args()


# ---------------------------------------------------------------- utilities
def dist_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    return ws, int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0"))


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        d["source"] = "measured"
        return d
    d = dict(FALLBACK_PEAKS)
    d["source"] = "fallback"
    return d


def kernel_sources_sha():
    h = hashlib.sha256()
    for fn in FWD_KERNEL_SOURCES:
        with open(os.path.join(ROOT, "entropy_tcgen05_vocab_gb300", "csrc", fn), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic():
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources."""
    if not os.path.exists(TRAFFIC_FILE):
        return None, "no ncu summary"
    kv = {}
    for ln in open(TRAFFIC_FILE):
        if ":" in ln and not ln.startswith("#"):
            k, v = ln.split(":", 1)
            kv[k.strip()] = v.strip()
    if kv.get("kernel_sources_sha256") != kernel_sources_sha():
        return None, "kernel changed since the ncu capture"
    try:
        return int(kv["dram_bytes_per_launch"]), os.path.relpath(TRAFFIC_FILE, ROOT)
    except (KeyError, ValueError):
        return None, "no dram_bytes_per_launch"


REASON_BITS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
               0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
               0x100: "display_clock_setting"}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 100 ms."""

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.out = tempfile.TemporaryFile(mode="w+")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index),
                 "--query-gpu=timestamp,clocks.sm,clocks.max.sm,clocks_event_reasons.active,power.draw",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        self.proc.wait()
        self.out.seek(0)
        rows = []
        for ln in self.out.read().splitlines():
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) != 5:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                ts += float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                pw = float(parts[4]) if parts[4] not in ("[N/A]", "N/A") else float("nan")
                rows.append((float(parts[1]), float(parts[2]), int(parts[3], 16), ts, pw))
            except (ValueError, IndexError):
                continue
        if not rows:
            return None
        # samples inside the timed region (fall back to all non-idle samples)
        inside = [r for r in rows if self.t0 is not None and self.t0 - 0.05 <= r[3] <= self.t1 + 0.05]
        busy = inside or [r for r in rows if r[2] & 0x1 == 0] or rows
        mhz = sorted(r[0] for r in busy)
        reasons = set()
        for r in busy:
            for bit, name in REASON_BITS.items():
                if r[2] & bit and name != "gpu_idle":
                    reasons.add(name)
        pw = sorted(r[4] for r in busy if r[4] == r[4])
        return {"sm_mhz": mhz[len(mhz) // 2], "sm_max_mhz": max(r[1] for r in rows),
                "reasons": sorted(reasons), "samples": len(busy),
                "in_timed_region": bool(inside),
                "power_w": pw[len(pw) // 2] if pw else None}


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(x, world, device):
    """Max of a per-rank float over the process group (nccl on GPUs, gloo on CPU)."""
    if world == 1:
        return x
    if torch.distributed.get_backend() != "nccl":
        device = torch.device("cpu")
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def compact(**kv):
    """A workload's figures, rounded to 4 significant digits."""
    return {k: (float("%.4g" % v) if isinstance(v, float) else v) for k, v in kv.items()}


def job_throughput(units_per_rank, steps, ms_max, world):
    """Whole-job units/s: every rank scores its own replica; the job takes as
    long as its slowest rank."""
    return world * units_per_rank * steps / (ms_max / 1e3)


# ---------------------------------------------------------------- workloads
def describe(d):
    w = d["workload"]
    return {"workload": "%s (T=%d, H=%d, V=%d, %s, tau=%g)" % (w.name, w.T, w.H, w.V, w.dtype, w.tau),
            "T": w.T, "H": w.H, "V": w.V, "n_rows": d["n"], "dtype": w.dtype,
            "temperature": w.tau, "row_selection": w.rows,
            "l2": "inputs larger than L2: W is %.2f GB and is streamed from HBM every step"
                  % (w.V * w.H * 2 / 1e9)}


def flops_per_call(d):
    w = d["workload"]
    mult = {"fwd": 2, "kl": 4, "bwd": 6}[w.kind]
    return mult * d["n"] * w.V * w.H


def call_once(flp, d, ws, stats=None):
    w = d["workload"]
    if w.kind == "fwd":
        if d.get("mx_head") is not None:
            return flp.logprob_entropy_mx(d["h"], d["mx_head"], w.V, d["targets"], d["row_idx"],
                                          d["tau"], workspace=ws)
        return flp.logprob_entropy(d["h"], d["W"], d["targets"], d["row_idx"], d["tau"],
                                   workspace=ws, support=d.get("support"))
    if w.kind == "kl":
        if d.get("mx") is not None:
            return flp.kl_divergence_mxfp4(d["h_s"], d["W_s"], d["h_t"], *d["mx"], d["row_idx"],
                                           workspace=ws)
        if d.get("mx_head") is not None:
            return flp.kl_divergence_mx(d["h_s"], d["W_s"], d["h_t"], d["mx_head"], d["row_idx"],
                                        workspace=ws)
        return flp.kl_divergence(d["h_s"], d["W_s"], d["h_t"], d["W_t"], d["row_idx"],
                                 workspace=ws)
    lse, ez = stats
    return flp.backward(d["h"], d["W"], d["targets"], d["row_idx"], d["tau"], d["g1"], d["g2"],
                        lse, ez, workspace=ws)


def memory_footprint(flp, d, ws, device):
    """Peak of torch's allocator over one call with the workspace passed in
    (outside the timed region), beside the workspace and the [n, V] FP32
    logits that the fused path never forms."""
    w = d["workload"]
    stats = None
    if w.kind == "bwd":
        _, _, lse, ez = flp.logprob_entropy(d["h"], d["W"], d["targets"], d["row_idx"], d["tau"],
                                            return_stats=True)
        stats = (lse, ez)
    torch.cuda.synchronize(device)
    free0 = torch.cuda.mem_get_info(device)[0]
    torch.cuda.reset_peak_memory_stats(device)
    base = torch.cuda.memory_allocated(device)
    out = call_once(flp, d, ws, stats)
    torch.cuda.synchronize(device)
    peak = torch.cuda.max_memory_allocated(device) - base
    outs = out if isinstance(out, tuple) else (out,)
    out_bytes = sum(t.numel() * t.element_size() for t in outs if t is not None)
    del out, outs
    torch.cuda.synchronize(device)
    return {"peak_alloc_delta_bytes": int(peak), "output_bytes": int(out_bytes),
            "workspace_bytes": int(ws.numel()),
            "logits_fp32_bytes_not_formed": int(d["n"]) * int(w.V) * 4,
            "free_memory_unchanged": bool(torch.cuda.mem_get_info(device)[0] >= free0 - (2 << 20))}


def op_of(d):
    if d["workload"].kind == "kl" and d.get("mx_head") is not None:
        return 3     # the block-scaled KL's workspace (it holds the MXFP8 teacher rows)
    if d["workload"].kind == "fwd" and d.get("mx_head") is not None:
        return 4     # the block-scaled forward's (it holds the MXFP8 scored rows)
    return {"fwd": 0, "kl": 1, "bwd": 2}[d["workload"].kind]


def launches_per_call(d):
    w = d["workload"]
    gather = 1 if d["row_idx"] is not None else 0
    if w.kind == "fwd":
        if d.get("mx_head") is not None:
            return 2               # MXFP8 quantiser (it gathers) + the block-scaled pipeline
        return gather + 1          # (gather) + the fused scoring kernel
    if w.kind == "kl":
        if d.get("mx_head") is not None:   # (gather of h_s) + MXFP8 quantiser + pipeline
            return gather + 2
        return 2 * gather + 1
    # backward with the statistics supplied: per row chunk, the gradient pass
    # and the dh and dW GEMMs, plus the sum of the dh GEMM's split tail tiles
    # when its last wave is split (counted as planned for the first chunk)
    import entropy_tcgen05_vocab_gb300 as flp
    shape = flp.make_shape(w.T, w.H, w.V, d["n"], d["h"].dtype)
    sms = torch.cuda.get_device_properties(d["h"].device).multi_processor_count
    pl = flp.plan(shape, flp.OP_BACKWARD, sms)
    per_chunk = 3 + (1 if pl["dh_split"] > 1 else 0)
    return gather + per_chunk * len(flp.row_chunks(d["n"], pl["chunk_rows"]))


def time_calls(fn, steps, device, warmup=3):
    """Device time (ms, CUDA events on the current stream) of `steps` calls of fn."""
    for _ in range(warmup):
        fn()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(device)
    a.record()
    for _ in range(steps):
        fn()
    b.record()
    torch.cuda.synchronize(device)
    return a.elapsed_time(b)


def time_device(flp, d, steps, warmup, world, device, sampler=None):
    """Device time of `steps` calls (CUDA events) and of their tensor-core kernels."""
    w = d["workload"]
    shape = flp.make_shape(w.T, w.H, w.V, d["n"], d["h"].dtype if "h" in d else d["h_s"].dtype)
    ws = torch.empty(flp.workspace_size(shape, op_of(d)), dtype=torch.uint8, device=device)
    stats = None
    if w.kind == "bwd":
        _, _, lse, ez = flp.logprob_entropy(d["h"], d["W"], d["targets"], d["row_idx"], d["tau"],
                                            return_stats=True)
        stats = (lse, ez)
    for _ in range(warmup):
        call_once(flp, d, ws, stats)
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for a, b in kev:          # create the events before they are handed to the library
        a.record()
        b.record()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(device)
    barrier(world)
    torch.cuda.synchronize(device)
    if sampler:
        sampler.mark("t0")
    t0.record()
    for a, b in kev:
        flp.set_kernel_events(a, b)
        call_once(flp, d, ws, stats)
    t1.record()
    torch.cuda.synchronize(device)
    barrier(world)
    torch.cuda.synchronize(device)
    if sampler:
        sampler.mark("t1")
    total_ms = t0.elapsed_time(t1)
    kernel_ms = [a.elapsed_time(b) for a, b in kev]
    status = flp.read_device_status(ws)
    if any(status.values()):
        raise RuntimeError("device status after timing: %s" % status)
    return total_ms, float(np.mean(kernel_ms)), ws


def time_e2e(flp, d, ws, steps, world, device):
    """Through the public API with every step's inputs copied from pinned host
    memory (hidden rows, targets, row selection) and its results read back;
    the weight is a resident model parameter.  The copy of step i+1's inputs
    runs on a second stream into the other of two device buffers while step i
    computes (the usual double-buffered input pipeline); all copies of all
    steps are inside the timed region."""
    h_pin = d["h"].cpu().pin_memory()
    t_pin = d["targets"].cpu().pin_memory()
    r_pin = None if d["row_idx"] is None else d["row_idx"].cpu().pin_memory()
    bufs = [(torch.empty_like(d["h"]), torch.empty_like(d["targets"]),
             None if r_pin is None else torch.empty_like(d["row_idx"])) for _ in range(2)]
    n = d["n"]
    lp_pin = torch.empty(n, dtype=torch.float32).pin_memory()
    en_pin = torch.empty(n, dtype=torch.float32).pin_memory()
    h2d = h_pin.numel() * h_pin.element_size() + t_pin.numel() * 8 + (0 if r_pin is None else r_pin.numel() * 8)
    d2h = 2 * n * 4
    compute = torch.cuda.current_stream(device)
    copy = torch.cuda.Stream(device)
    ready = [torch.cuda.Event() for _ in range(2)]
    free = [torch.cuda.Event() for _ in range(2)]

    def load(i):
        hb, tb, rb = bufs[i % 2]
        with torch.cuda.stream(copy):
            copy.wait_event(free[i % 2])
            hb.copy_(h_pin, non_blocking=True)
            tb.copy_(t_pin, non_blocking=True)
            if r_pin is not None:
                rb.copy_(r_pin, non_blocking=True)
            ready[i % 2].record(copy)

    def run(i, last):
        hb, tb, rb = bufs[i % 2]
        compute.wait_event(ready[i % 2])
        if not last:
            load(i + 1)
        if d.get("mx_head") is not None:
            logp, ent = flp.logprob_entropy_mx(hb, d["mx_head"], d["workload"].V, tb, rb,
                                               d["tau"], workspace=ws)
        else:
            logp, ent = flp.logprob_entropy(hb, d["W"], tb, rb, d["tau"], workspace=ws)
        free[i % 2].record(compute)
        lp_pin.copy_(logp, non_blocking=True)
        en_pin.copy_(ent, non_blocking=True)

    for e in free:
        e.record(compute)
    for i in range(3):
        if i == 0:
            load(0)
        run(i, i == 2)
    torch.cuda.synchronize(device)
    barrier(world)
    for e in free:
        e.record(compute)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(compute)
    copy.wait_event(t0)
    load(0)
    for i in range(steps):
        run(i, i == steps - 1)
    t1.record(compute)
    torch.cuda.synchronize(device)
    barrier(world)
    return t0.elapsed_time(t1), h2d, d2h


def cpu_oracle_rate(d, seconds, calib_rows=2):
    """Oracle rows per second on a bounded sample of the workload's rows."""
    from oracle import coracle
    w = d["workload"]
    h, W = d["h"].cpu(), d["W"].cpu()
    tg = d["targets"].cpu().numpy()
    rows_all = np.arange(w.T) if d["row_idx"] is None else d["row_idx"].cpu().numpy()
    t = time.perf_counter()
    coracle.logprob_entropy(h, W, tg, rows_all[:calib_rows], d["tau"], w.dtype)
    per_row = max((time.perf_counter() - t) / calib_rows, 1e-6)
    k = int(max(1, min(len(rows_all), seconds / per_row)))
    pos = np.linspace(0, len(rows_all) - 1, k).astype(np.int64)
    t = time.perf_counter()
    coracle.logprob_entropy(h, W, tg, rows_all[pos], d["tau"], w.dtype)
    dt = time.perf_counter() - t
    return k / dt, k, dt, coracle.num_threads()


def numpy_oracle_rate(d, seconds):
    """Rows per second of the NumPy float64 restatement (BLAS matmul) on a
    row sample, inputs decoded to float64 beforehand: an optimistic CPU
    figure beside the C oracle's."""
    from oracle import ref
    w = d["workload"]
    rows_all = np.arange(w.T) if d["row_idx"] is None else d["row_idx"].cpu().numpy()
    Wd = ref.decode(d["W"].cpu(), w.dtype)
    k = 256
    hd = ref.decode(d["h"][torch.from_numpy(rows_all[:k]).to(d["h"].device)].cpu(), w.dtype)
    t = time.perf_counter()
    ref.row_stats(hd[:32], Wd, None, d["tau"])
    per_row = max((time.perf_counter() - t) / 32, 1e-6)
    k = int(max(32, min(k, seconds / per_row)))
    t = time.perf_counter()
    ref.row_stats(hd[:k], Wd, None, d["tau"])
    dt = time.perf_counter() - t
    return k / dt, k, dt


def cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.startswith("Model name:"):
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return platform.machine()


# ---------------------------------------------------------------- arms
def run_ours(args):
    import entropy_tcgen05_vocab_gb300 as flp
    import workloads

    world, rank, local = dist_info()
    if world > 1:
        torch.distributed.init_process_group("nccl")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    flp.build()
    flp.lib()
    P = peaks()

    w0 = workloads.WORKLOADS[args.workload]
    d = workloads.make(w0 if args.T is None else w0.scaled(T=args.T), device=device)
    variant = {}
    if args.teacher == "mxfp4" and w0.kind == "kl":
        d["mx"] = flp.mxfp4_quantize(d["W_t"])
        variant["teacher_head"] = "MXFP4 (E2M1 + E8M0 per 32), quantised before timing"
    if args.teacher == "mx" and w0.kind == "kl":
        d["mx_head"] = flp.mx_head_quantize(d["W_t"])
        variant["teacher_head"] = ("MXFP4 (E2M1 + E8M0 per 32), quantised before timing, on the "
                                   "block-scaled tensor cores; teacher rows quantised to MXFP8 "
                                   "inside each call")
    if args.head == "mx" and w0.kind == "fwd":
        d["mx_head"] = flp.mx_head_quantize(d["W"])
        variant["head"] = ("MXFP4 (E2M1 + E8M0 per 32), quantised before timing, on the "
                           "block-scaled tensor cores; scored rows quantised to MXFP8 inside "
                           "each call")
    if args.support_j is not None and w0.kind == "fwd":
        d["support"] = torch.from_numpy(workloads.support_words(
            d["workload"].T, d["workload"].V, args.support_j, d["workload"].seed,
            targets=d["targets"].cpu().numpy())).to(device)
        variant["support"] = "each token kept with probability 2^-%d, targets kept" % args.support_j
    headline = w0.kind == "fwd" and args.workload == 1 and args.T is None and not variant
    arith = ("mx" if w0.kind == "fwd" and args.head == "mx" else
             "bf16+mx" if w0.kind == "kl" and args.teacher == "mx" else "bf16")
    sampler = ClockSampler(device.index) if rank == 0 else None
    if sampler:
        sampler.start()
    total_ms, kernel_ms, ws = time_device(flp, d, args.steps, args.warmup, world, device, sampler)
    clocks = sampler.stop() if sampler else None
    total_ms = max_over_ranks(total_ms, world, device)
    n = d["n"]
    value = job_throughput(n, args.steps, total_ms, world)
    fl = flops_per_call(d)
    achieved = fl / (kernel_ms / 1e3) / 1e12
    traffic, traffic_src = recorded_traffic() if headline else (None, "not the headline kernel")

    e2e = None
    if not args.no_e2e and w0.kind == "fwd":
        e2e_steps = min(args.steps, 100)
        e2e_ms, h2d, d2h = time_e2e(flp, d, ws, e2e_steps, world, device)
        e2e_ms = max_over_ranks(e2e_ms, world, device)
        e2e = {"value": world * n * e2e_steps / (e2e_ms / 1e3), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e2e_ms / e2e_steps, "resident": "W (model weight)",
               "pipeline": "inputs of step i+1 copied on a second stream while step i computes"}

    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": DTYPE.get(arith, d["workload"].dtype),
        "data": "synthetic (seeded; shapes and distributions of the pages' workloads)",
        "config": dict(describe(d), parallelism="replicas" if world > 1 else "single GPU",
                       **variant),
        "tflops": world * fl * args.steps / (total_ms / 1e3) / 1e12,
        "pct_of_bf16_peak": 100.0 * fl * args.steps / (total_ms / 1e3) / 1e12 / P["bf16_tflops"],
        "kernel_ms": kernel_ms,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": own_peak(P, arith),
                     "unit": "TFLOP/s", "frac": achieved / own_peak(P, arith), "traffic": traffic,
                     "kernel": {"fwd": ("mx_fwd_pipeline_kernel<LseEpi<1,false>>"
                                        if "head" in variant else
                                        "vocab_pipeline_kernel<256,4,2,LseEpi<1,%s>,2,1,8,true>"
                                        % ("true" if "support" in variant else "false")),
                                "kl": ("mx_kl_pipeline_kernel<KlEpiT<224,16>>"
                                       if args.teacher == "mx" else
                                       "vocab_pipeline_kernel<256,3,2,KlEpi,2,1,%s>"
                                       % ("4,false,true" if "teacher_head" in variant else "8")),
                                "bwd": "grad pass + dh and dW GEMMs"}[w0.kind],
                     "peak_kind": PEAK_KIND[arith] % P["source"],
                     "frac_of_sustained": achieved / own_peak(P, arith, sustained=True),
                     "algorithmic_flops_per_launch": fl,
                     "traffic_source": traffic_src},
        "e2e": e2e,
        "clocks": clocks,
        "gpu_launches": launches_per_call(d) * args.steps,
        "memory": memory_footprint(flp, d, ws, device),
    }

    configs = {}   # each extra workload's configuration, reported apart from its figures
    if not args.no_extra:
        extra = {}
        for wid in (2, 3, 4):
            if wid == args.workload:
                continue
            try:
                dx = workloads.make(wid, device=device)
                steps = 20
                tms, kms, _ = time_device(flp, dx, steps, 3, world, device)
                tms = max_over_ranks(tms, world, device)
                flx = flops_per_call(dx)
                configs[dx["workload"].name] = dict(describe(dx), steps=steps,
                                                    algorithmic_flops_per_call=flx)
                extra[dx["workload"].name] = compact(
                    n_rows=dx["n"], scored_tokens_per_s=world * dx["n"] * steps / (tms / 1e3),
                    ms_per_step=tms / steps, kernel_ms=kms,
                    tflops=flx / (tms / steps / 1e3) / 1e12,
                    pct_of_bf16_peak=100 * flx / (tms / steps / 1e3) / 1e12 / P["bf16_tflops"])
                del dx
            except Exception as e:  # a workload whose op is not available is reported, not fatal
                extra[workloads.WORKLOADS[wid].name] = {"unavailable": str(e).splitlines()[0][:200]}
            torch.cuda.empty_cache()
        # K-candidate scoring (4 target tokens per row) and a sampling support
        # (about 1/32 of the tokens per row, targets kept) on the main workload's
        # inputs, each timed in blocks of 10 calls interleaved (ABBA) with blocks
        # of the plain call, so both see the same clocks.
        if d["workload"].kind == "fwd":
            w = d["workload"]
            shape = flp.make_shape(w.T, w.H, w.V, n, d["h"].dtype)
            wsk = torch.empty(flp.workspace_size(shape, 0), dtype=torch.uint8, device=device)

            def plain():
                flp.logprob_entropy(d["h"], d["W"], d["targets"], d["row_idx"], d["tau"],
                                    workspace=wsk)

            def variant_line(name, fn, note, arith_v="bf16"):
                try:
                    # blocks of 10 calls in ABBA order, so a drift of the clock over
                    # the run (heating towards the power cap) weighs on both alike
                    t_var = t_plain = 0.0
                    for order in ((plain, fn), (fn, plain), (plain, fn), (fn, plain)):
                        for f in order:
                            t = time_calls(f, 10, device)
                            if f is fn:
                                t_var += t
                            else:
                                t_plain += t
                    t_var = max_over_ranks(t_var, world, device)
                    t_plain = max_over_ranks(t_plain, world, device)
                    configs[name] = dict(describe(d), steps=40, **note)
                    extra[name] = compact(
                        n_rows=n, scored_tokens_per_s=job_throughput(n, 40, t_var, world),
                        ms_per_step=t_var / 40, tflops=fl / (t_var / 40 / 1e3) / 1e12,
                        pct_of_bf16_peak=100 * fl / (t_var / 40 / 1e3) / 1e12 / P["bf16_tflops"],
                        plain_ms_same_clocks=t_plain / 40)
                    if arith_v != "bf16":
                        extra[name]["pct_of_own_peak"] = float("%.4g" % (
                            100 * fl / (t_var / 40 / 1e3) / 1e12 / own_peak(P, arith_v)))
                except Exception as e:  # reported, not fatal
                    extra[name] = {"unavailable": str(e)[:200]}

            K = 4
            g = torch.Generator(device=device)
            g.manual_seed(w.seed * 100 + 30)
            tk = torch.randint(0, w.V, (w.T, K), generator=g, device=device)
            tk[:, 0] = d["targets"]
            variant_line(w.name + "-k4-candidates",
                         lambda: flp.logprob_entropy_k(d["h"], d["W"], tk, d["row_idx"], d["tau"],
                                                       workspace=wsk),
                         {"candidates_per_row": K})
            sup = torch.from_numpy(workloads.support_words(
                w.T, w.V, 5, w.seed, targets=d["targets"].cpu().numpy())).to(device)
            variant_line(w.name + "-sampling-support",
                         lambda: flp.logprob_entropy(d["h"], d["W"], d["targets"], d["row_idx"],
                                                     d["tau"], workspace=wsk, support=sup),
                         {"support": "each token kept with probability 1/32, targets kept"})
            del sup, tk
            # scoring with the head in MXFP4 and the rows in MXFP8 on the
            # block-scaled tensor cores (the forward of a model that needs no
            # backward, e.g. the reference policy's log-probs)
            try:
                mxh = flp.mx_head_quantize(d["W"])
                wsm = torch.empty(flp.workspace_size(shape, flp.OP_LOGPROB_ENTROPY_MX),
                                  dtype=torch.uint8, device=device)
                variant_line(w.name + "-mx-head",
                             lambda: flp.logprob_entropy_mx(d["h"], mxh, w.V, d["targets"],
                                                            d["row_idx"], d["tau"], workspace=wsm),
                             {"head": "MXFP4 head (%.3f GB against %.3f GB in bf16) x MXFP8 rows "
                                      "on the block-scaled tensor cores (tcgen05.mma "
                                      "kind::mxf8f6f4)"
                                      % (mxh.numel() / 1e9, w.V * w.H * 2 / 1e9),
                              "own_peak": PEAK_KIND["mx"] % P["source"]}, "mx")
                del mxh, wsm
            except Exception as e:  # reported, not fatal
                extra[w.name + "-mx-head"] = {"unavailable": str(e)[:200]}
        # distillation KL with the teacher head in MXFP4 (4.25 bits per weight):
        # decoded to bf16 next to the tensor cores, and on the block-scaled
        # tensor cores with the teacher rows in MXFP8; each interleaved (ABBA)
        # with the bf16 teacher head on the same inputs
        try:
            dk = workloads.make(3, device=device)
            wk = dk["workload"]
            packed, scales = flp.mxfp4_quantize(dk["W_t"])
            head = flp.mx_head_quantize(dk["W_t"])
            shape = flp.make_shape(wk.T, wk.H, wk.V, dk["n"], dk["h"].dtype)
            wsk = torch.empty(max(flp.workspace_size(shape, flp.OP_KL),
                                  flp.workspace_size(shape, flp.OP_KL_MX)),
                              dtype=torch.uint8, device=device)
            flk = flops_per_call(dk)
            bf16_gb = wk.V * wk.H * 2 / 1e9

            def bf16_teacher():
                flp.kl_divergence(dk["h_s"], dk["W_s"], dk["h_t"], dk["W_t"], None, workspace=wsk)

            variants = (  # (suffix, call, note, arithmetic of the MMAs)
                ("-mxfp4-teacher",
                 lambda: flp.kl_divergence_mxfp4(dk["h_s"], dk["W_s"], dk["h_t"], packed, scales,
                                                 None, workspace=wsk),
                 "MXFP4 (E2M1, E8M0 per 32) decoded to bf16 in shared memory, %.3f GB against "
                 "%.3f GB in bf16" % (packed.numel() / 1e9 + scales.numel() / 1e9, bf16_gb),
                 "bf16"),
                ("-mx-teacher",
                 lambda: flp.kl_divergence_mx(dk["h_s"], dk["W_s"], dk["h_t"], head, None,
                                              workspace=wsk),
                 "MXFP4 head (%.3f GB against %.3f GB in bf16) x MXFP8 teacher rows on the "
                 "block-scaled tensor cores (tcgen05.mma kind::mxf8f6f4)"
                 % (head.numel() / 1e9, bf16_gb), "bf16+mx"),
            )
            for suffix, fn, note, arith_v in variants:
                t_mx = t_bf = 0.0
                for order in ((bf16_teacher, fn), (fn, bf16_teacher)):  # ABBA
                    for f in order:
                        t = time_calls(f, 10, device)
                        if f is fn:
                            t_mx += t
                        else:
                            t_bf += t
                t_mx = max_over_ranks(t_mx, world, device)
                t_bf = max_over_ranks(t_bf, world, device)
                configs[wk.name + suffix] = dict(describe(dk), steps=20, teacher_head=note)
                if arith_v != "bf16":
                    configs[wk.name + suffix]["own_peak"] = PEAK_KIND[arith_v] % P["source"]
                extra[wk.name + suffix] = compact(
                    n_rows=dk["n"], scored_tokens_per_s=job_throughput(dk["n"], 20, t_mx, world),
                    ms_per_step=t_mx / 20, tflops=flk / (t_mx / 20 / 1e3) / 1e12,
                    pct_of_bf16_peak=100 * flk / (t_mx / 20 / 1e3) / 1e12 / P["bf16_tflops"],
                    plain_ms_same_clocks=t_bf / 20)
                if arith_v != "bf16":
                    extra[wk.name + suffix]["pct_of_own_peak"] = float("%.4g" % (
                        100 * flk / (t_mx / 20 / 1e3) / 1e12 / own_peak(P, arith_v)))
            del dk, packed, scales, head, wsk
        except Exception as e:  # reported, not fatal
            extra[workloads.WORKLOADS[3].name + "-mx-teacher"] = {"unavailable": str(e)[:200]}
        torch.cuda.empty_cache()
        out["workload_configs"] = configs

    if rank == 0 and world == 1 and not args.no_cpu:
        rate, k, dt, cores = cpu_oracle_rate(d, args.cpu_seconds)
        out["cpu_baseline"] = {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle",
                               "sample": "%d of %d rows of the same workload (float64 C oracle, "
                                         "%.1f s)" % (k, n, dt),
                               "host_cpus": len(os.sched_getaffinity(0)), "cpu_model": cpu_model()}
        try:
            nrate, nk, ndt = numpy_oracle_rate(d, args.cpu_seconds / 2)
            out["cpu_baseline"]["numpy_blas"] = {
                "value": nrate, "unit": UNIT,
                "sample": "%d rows, per-row statistics by the NumPy float64 oracle (BLAS matmul) "
                          "on inputs decoded beforehand, %.1f s" % (nk, ndt)}
        except MemoryError as e:  # reported, not fatal
            out["cpu_baseline"]["numpy_blas"] = {"unavailable": str(e)[:200]}
    if not args.no_extra:
        # last on the line, short entries: the figures of every workload stay
        # in view when only the end of the output is kept
        out["workloads"] = extra
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(out), flush=True)


def run_reference(args):
    world, rank, local = dist_info()
    if rank != 0:
        return
    import workloads
    from oracle import coracle

    device = torch.device("cuda", local) if torch.cuda.is_available() else torch.device("cpu")
    d = workloads.make(args.workload, device=device)
    w = d["workload"]
    h, W = d["h"].cpu(), d["W"].cpu()
    tg = d["targets"].cpu().numpy()
    rows_all = np.arange(w.T) if d["row_idx"] is None else d["row_idx"].cpu().numpy()
    # size each step so the whole run stays within about two minutes
    t = time.perf_counter()
    coracle.logprob_entropy(h, W, tg, rows_all[:1], d["tau"], w.dtype)
    per_row = max(time.perf_counter() - t, 1e-6)
    k = int(max(1, min(64, 120.0 / (args.steps + args.warmup) / per_row)))
    rng = np.random.default_rng(0)

    def step():
        pos = np.sort(rng.choice(len(rows_all), size=k, replace=False))
        coracle.logprob_entropy(h, W, tg, rows_all[pos], d["tau"], w.dtype)

    for _ in range(args.warmup):
        step()
    t = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t
    value = k * args.steps / dt
    cores = coracle.num_threads()
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded; shapes and distributions of the pages' workloads)",
        "config": describe(d),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": "%d random rows of %d per step (float64 C oracle)" % (k, d["n"]),
                         "host_cpus": len(os.sched_getaffinity(0)), "cpu_model": cpu_model()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
