"""Benchmark of the fused MXFP8 SwiGLU MLP on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload m16] [--no-sweep]

One step = one call of the hot path (quantise x, gate/up block-scaled GEMM,
SiLU(g) * u, requantise, down GEMM) on one batch of M tokens of the workload.
The headline workload is m16 (M = 16, H = 2560, I = 9728, one layer).  Weights
are rotated over enough quantised copies that every call streams its weights
from HBM (the copies together exceed twice the 129 MB L2).  Rank 0 prints ONE
JSON line.

Multi-GPU: replicas only -- every rank runs its own copy of the workload, no
collective on the data path; the ranks only meet at the timing barrier and the
max-over-ranks of the elapsed time.

--impl reference times the CPU oracle (fp64, the test infrastructure) on the
host cores instead, on the same workload, metric and unit.
"""
from __future__ import annotations

import argparse
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

METRIC = "MXFP8 SwiGLU MLP tokens/s and HBM GB/s (% roofline) at M=1/16/64/128"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0


# DRAM bytes per launch of the fused kernel (dram__bytes_read.sum +
# dram__bytes_write.sum, mean of the captured launches) from ncu captures, by
# workload: the sha256 prefix of the kernel sources they were taken on (the
# number is reported only while those sources are unchanged), the bytes, the
# launch form captured and the summary under profiles/.
NCU_TRAFFIC = {
    "m16": {"sha": "bda093efa9298a67", "bytes": 80.59e6, "source": "profiles/mx_persistent_kernel_m16_memory.md",
            "form": "gate/up split over all blocks (--knob PAIRS=0); the timed default splits gate/up tiles by "
                    "2-block clusters, same weight stream"},
    "m128": {"sha": "bda093efa9298a67", "bytes": 164.39e6, "source": "profiles/mx_persistent_kernel_m128_memory.md",
             "form": "the default (no cluster split at M > 32)"},
}
KERNEL_SOURCES = ("mx_kernels.cu", "mx_internal.h", "mx_mxfp8.cuh", "sm103.cuh", "mx_device.cuh")


def kernel_sources_hash():
    import hashlib

    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "mxfp8_swiglu_mlp_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload):
    rec = NCU_TRAFFIC.get(workload)
    if rec is None or rec["sha"] != kernel_sources_hash():
        return None, None
    return rec["bytes"], "%s; launch form: %s" % (rec["source"], rec["form"])


def fp8_peak_tflops():
    """Dense FP8 tensor peak: the measured bf16 GEMM rate x 2 (the nominal
    FP8 : bf16 ratio of the tensor cores), else the nominal 4.5 PFLOP/s."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return 2.0 * float(json.load(f)["bf16_tflops"]), "measured bf16 x 2"
    except Exception:
        return 4500.0, "nominal"


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def algorithmic_bytes(M, H, I):
    """Codes + scales of the three weight matrices, x read, y written."""
    return 3 * H * I + 3 * H * I // 32 + 2 * M * H + 2 * M * H


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clock / throttle-reason samples with host timestamps."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.samples = []
        self.proc = None
        self.dev = device_index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        rows = []
        for ts, line in self.samples:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append((ts, float(parts[0]), float(parts[1]), parts[3:]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        inside = [r for r in rows if t0 <= r[0] <= t1]
        if not inside:  # timed region shorter than the sampling period: nearest samples
            inside = sorted(rows, key=lambda r: min(abs(r[0] - t0), abs(r[0] - t1)))[:3]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in inside:
            flags = r[3][1:5]
            for n, v in zip(names, flags):
                if v.strip().lower() in ("active", "1"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": sorted(reasons), "samples": len(inside)}


# ---------------------------------------------------------------- GPU workload
class MlpBench:
    def __init__(self, fs, wl, M, device, seed_layers=None, use_numpy=False):
        import numpy as np
        import torch

        from workloads import inputs

        self.fs, self.M, self.H, self.I = fs, M, wl.H, wl.I
        per_layer = wl.weight_bytes
        n_layers = wl.layers
        copies = max(n_layers, -(-2 * L2_BYTES // per_layer) + 1)
        self.weights = []
        for c in range(copies):
            layer = c % n_layers
            if use_numpy:
                wg, wu, wd = (torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).to(device).view(torch.bfloat16)
                              for b in inputs.make_layer(wl, layer))
            else:
                wg, wu, wd = inputs.make_layer_torch(wl, layer, device)
            self.weights.append(fs.prepare_mlp_weights(wg, wu, wd))
            del wg, wu, wd
        if use_numpy:
            xb = inputs.make_activations(wl, M)
            self.x = torch.from_numpy(np.ascontiguousarray(xb).view(np.int16)).to(device).view(torch.bfloat16)
        else:
            self.x = inputs.make_activations_torch(wl, M, device)
        self.y = torch.empty((M, self.H), dtype=torch.bfloat16, device=device)
        gb = inputs.make_norm_gain(wl)
        self.gamma = torch.from_numpy(np.ascontiguousarray(gb).view(np.int16)).to(device).view(torch.bfloat16)
        self.ws = fs.Workspace(M, self.H, self.I, device=device)
        self.copies = copies
        torch.cuda.synchronize()

    def call(self, i, fused=True, stream=None, x=None, y=None):
        """fused: True (single launch), False (three launches) or "block"
        (RMSNorm + MLP + residual, fsops_mxfp8_swiglu_mlp_block)."""
        w = self.weights[i % self.copies]
        if fused == "block":
            from workloads import inputs

            self.fs.fsops_mxfp8_swiglu_mlp_block(self.x if x is None else x, self.gamma, inputs.NORM_EPS, True,
                                                 w.gateup_codes, w.down_codes, w.scales, self.y if y is None else y,
                                                 self.M, self.H, self.I, stream)
            return
        f = self.fs.fsops_mxfp8_swiglu_mlp if fused else self.fs.fsops_mxfp8_swiglu_mlp_unfused
        f(self.x if x is None else x, w.gateup_codes, w.down_codes, w.scales, self.y if y is None else y,
          self.M, self.H, self.I, stream)

    def capture(self, nsteps, fused, stream, start=0):
        import torch

        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(nsteps):
                self.call(start + i, fused, stream)
        return g

    def timed(self, steps, fused, warmup, stream, chunk=256):
        """Device time of exactly `steps` calls (graph replays), in seconds."""
        import torch

        chunk = max(self.copies, (min(chunk, steps) // self.copies) * self.copies) if steps >= self.copies else steps
        with torch.cuda.stream(stream):
            for i in range(warmup):
                self.call(i, fused, stream)
            g_main = self.capture(chunk, fused, stream) if steps >= chunk else None
            rem = steps - (steps // chunk) * chunk if g_main is not None else steps
            g_rem = self.capture(rem, fused, stream) if rem > 0 else None
            g_main and g_main.replay()
            g_rem and g_rem.replay()
            stream.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            t_host0 = time.time()
            e0.record(stream)
            for _ in range(steps // chunk if g_main is not None else 0):
                g_main.replay()
            if g_rem is not None:
                g_rem.replay()
            e1.record(stream)
            e1.synchronize()
            t_host1 = time.time()
        return e0.elapsed_time(e1) / 1e3, (t_host0, t_host1)

    def timed_same(self, steps, stream):
        """Per-call device time of `steps` fused calls on the first weight copy."""
        import torch

        with torch.cuda.stream(stream):
            for _ in range(5):
                self.call(0, True, stream)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for _ in range(steps):
                    self.call(0, True, stream)
            g.replay()
            stream.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g.replay()
            e1.record(stream)
            e1.synchronize()
        return e0.elapsed_time(e1) / 1e3 / steps

    def per_launch(self, n, stream):
        """Mean duration of single fused launches, each bracketed by events on its stream."""
        import torch

        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        with torch.cuda.stream(stream):
            for i, (a, b) in enumerate(evs):
                a.record(stream)
                self.call(i, True, stream)
                b.record(stream)
        stream.synchronize()
        return statistics.mean(a.elapsed_time(b) for a, b in evs) / 1e3

    def e2e(self, steps, warmup, stream, chunk=256):
        """Through the public API with host buffers: every step copies x from
        pinned host memory to the device, makes the call and copies y back to
        pinned host memory.  The copies run on a second stream into and out
        of two device buffers each, so that step i + 1's x and step i's y
        move while the calls run back to back (as a decode server overlaps
        its transfers); the steps run as CUDA-graph replays of `chunk` steps,
        else eagerly if the copies cannot be captured.  Returns (seconds,
        H2D bytes, D2H bytes, how the steps ran)."""
        import torch

        x_host = torch.empty_like(self.x, device="cpu").pin_memory()
        x_host.copy_(self.x.cpu())
        y_host = torch.empty_like(self.y, device="cpu").pin_memory()
        x_dev = [torch.empty_like(self.x) for _ in range(2)]
        y_dev = [torch.empty_like(self.y) for _ in range(2)]
        cs = torch.cuda.Stream(device=self.x.device)

        def run(start, n):
            # copy stream: H2D(start), then per step i: H2D(i + 1), wait for
            # call i, D2H(i); compute stream: per step i: wait for H2D(i),
            # call i.  Buffer i % 2 is rewritten only after call i - 2 and
            # D2H(i - 2), both ordered before H2D(i) on the copy stream.
            cs.wait_stream(stream)
            with torch.cuda.stream(cs):
                x_dev[start % 2].copy_(x_host, non_blocking=True)
            e_h = torch.cuda.Event()
            e_h.record(cs)
            for k in range(n):
                i = start + k
                stream.wait_event(e_h)
                self.call(i, True, stream, x=x_dev[i % 2], y=y_dev[i % 2])
                e_k = torch.cuda.Event()
                e_k.record(stream)
                with torch.cuda.stream(cs):
                    if k + 1 < n:
                        x_dev[(i + 1) % 2].copy_(x_host, non_blocking=True)
                    e_h = torch.cuda.Event()
                    e_h.record(cs)
                    cs.wait_event(e_k)
                    y_host.copy_(y_dev[i % 2], non_blocking=True)
            stream.wait_stream(cs)

        def capture(n):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                run(0, n)
            return g

        chunk = max(self.copies, (min(chunk, steps) // self.copies) * self.copies) if steps >= self.copies else steps
        mode = "CUDA graph replays of %d steps, copies on a second stream" % chunk
        with torch.cuda.stream(stream):
            run(0, warmup)
            try:
                g_main = capture(chunk) if steps >= chunk else None
                rem = steps - (steps // chunk) * chunk if g_main is not None else steps
                g_rem = capture(rem) if rem > 0 else None
                g_main and g_main.replay()
                g_rem and g_rem.replay()
            except RuntimeError:
                g_main = g_rem = None
                mode = "eager, copies on a second stream"
            stream.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            if mode.startswith("eager"):
                run(0, steps)
            else:
                for _ in range(steps // chunk if g_main is not None else 0):
                    g_main.replay()
                if g_rem is not None:
                    g_rem.replay()
            e1.record(stream)
            e1.synchronize()
        nbytes = self.x.numel() * 2
        return e0.elapsed_time(e1) / 1e3, nbytes, self.y.numel() * 2, mode


def max_over_ranks(dt, world, device=None):
    """The job's time: the slowest rank's (a MAX all-reduce, then a barrier);
    every rank gets it.  One rank: dt itself."""
    if world <= 1:
        return dt
    import torch

    t = torch.tensor([dt], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    torch.distributed.barrier()
    return float(t.item())


def job_tokens_per_s(world, tokens_per_step, steps, dt):
    """Whole-job throughput: every replica processes its own batch of
    tokens_per_step tokens per step (weak scaling), timed by the slowest."""
    return world * tokens_per_step * steps / dt


def run_ours(args, rank, world, local_rank):
    import torch

    import mxfp8_swiglu_mlp_gb300 as fs
    from workloads import inputs

    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    stream = torch.cuda.Stream(device=device)
    hbm_peak, peak_kind = peaks()
    wl = inputs.WORKLOADS[args.workload]
    if args.layers:
        import dataclasses

        wl = dataclasses.replace(wl, layers=args.layers)
    M, H, I = wl.M, wl.H, wl.I
    B = algorithmic_bytes(M, H, I)

    bench = MlpBench(fs, wl, M, device, use_numpy=False)
    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    dt, (h0, h1) = bench.timed(args.steps, not args.unfused, args.warmup, stream)
    dt = max_over_ranks(dt, world, device)
    time.sleep(0.1)
    sampler.stop()
    clocks = sampler.summary(h0, h1)

    t_launch = bench.per_launch(min(args.steps, 200), stream)
    ms_per_step = dt / args.steps * 1e3
    value = job_tokens_per_s(world, M, args.steps, dt)
    # the dominant (and, fused, the only) kernel of a step: its average
    # duration over the timed region is the region's time over its launches
    t_kernel = dt / args.steps / (3 if args.unfused else 1)
    achieved = B / (dt / args.steps) / 1e9

    n_e2e = min(args.steps, 5000)
    e2e_t, h2d, d2h, e2e_mode = bench.e2e(n_e2e, args.warmup, stream)
    e2e_val = job_tokens_per_s(world, M, n_e2e, max_over_ranks(e2e_t, world, device))

    traffic, traffic_src = ncu_traffic(wl.name)
    out = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3 (fp32 accumulate)", "data": "synthetic",
        "config": {"workload": "%s: %s MXFP8 SwiGLU MLP, M=%d, H=%d, I=%d, one layer per step" %
                               (wl.name, "three-launch" if args.unfused else "fused", M, H, I),
                   "M": M, "H": H, "I": I, "weight_copies_rotated": bench.copies,
                   "l2": "inputs larger than L2: %d rotated weight copies, %.0f MB" %
                         (bench.copies, bench.copies * wl.weight_bytes / 1e6),
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "timing": "CUDA graph replays of exactly `steps` calls, CUDA events on the launching stream"},
        "weight_GBps": round(value / world / M * wl.weight_bytes / 1e9, 1),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(achieved / hbm_peak, 4), "traffic": traffic, "traffic_source": traffic_src,
                     "peak_kind": peak_kind + " (MEASURED_PEAKS.json hbm_gbs, copy bandwidth)",
                     "kernel": decode_kernel_name(fs, M, H, I) + (" (three-launch path)" if args.unfused else ""),
                     "bytes_per_launch": B,
                     "achieved_from": "bytes_per_launch / (timed region / steps): CUDA events around the "
                                      "graph replays of the timed region",
                     "kernel_us_in_timed_region": round(t_kernel * 1e6, 3),
                     "single_launch_us_event_bracketed": round(t_launch * 1e6, 3),
                     "single_launch_frac": round(B / t_launch / 1e9 / hbm_peak, 4)},
        "e2e": {"value": round(e2e_val, 1), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "api": "fsops_mxfp8_swiglu_mlp via ctypes, pinned host buffers; every step H2D x, the call, D2H y "
                       "(%s)" % e2e_mode},
        "gpu_launches": args.steps * (3 if args.unfused else 1),
        "clocks": {k: clocks[k] for k in ("sm_mhz", "sm_max_mhz", "reasons")},
    }
    if rank == 0 and not args.no_sweep:
        out["sweep"] = sweep(fs, device, stream, hbm_peak, args)
        out["sweep_c5"] = sweep_c5(fs, device, stream, hbm_peak)
        out["blockscale_gemm"] = blockscale_gemm(fs, stream, hbm_peak)
        out["prefill_gemm"] = prefill_gemm(fs, stream)
        out["attention_decode"] = attention_decode(fs, stream, hbm_peak)
    if rank == 0 and not args.no_cpu:
        out["cpu_baseline"] = cpu_baseline(wl)
    del bench
    return out


def sweep(fs, device, stream, hbm_peak, args):
    """Fused and three-launch numbers at M = 1, 16, 64, 128 (the metric's points)."""
    import torch

    from workloads import inputs

    res = {}
    for name in ("m1", "m16", "m64", "m128"):
        wl = inputs.WORKLOADS[name]
        b = MlpBench(fs, wl, wl.M, device)
        B = algorithmic_bytes(wl.M, wl.H, wl.I)
        n = max(64, min(4096, int(0.25 / (B / hbm_peak / 1e9 * 1.5))))
        n = (n // b.copies + 1) * b.copies
        entry = {"M": wl.M, "H": wl.H, "I": wl.I, "layers": wl.layers, "copies": b.copies, "steps": n}
        for fused in (True, False):
            dt, _ = b.timed(n, fused, 5, stream)
            t = dt / n
            key = "fused" if fused else "unfused_3_launches"
            entry[key] = {"tokens_per_s": round(wl.M / t, 1), "us_per_call": round(t * 1e6, 3),
                          "GBps": round(B / t / 1e9, 1), "frac_hbm": round(B / t / 1e9 / hbm_peak, 4)}
        # the decoder block around it: one launch, RMSNorm in the MLP kernel's
        # quantisation prologue, + x in the bf16 store
        dt, _ = b.timed(n, "block", 5, stream)
        entry["block_rmsnorm_residual"] = {"us_per_call": round(dt / n * 1e6, 3),
                                           "tokens_per_s": round(wl.M / (dt / n), 1), "launches": 1}
        tl = b.per_launch(min(n, 200), stream)
        entry["fused"]["launch_us"] = round(tl * 1e6, 3)
        entry["fused"]["launch_frac_hbm"] = round(B / tl / 1e9 / hbm_peak, 4)
        fl = 2.0 * wl.M * 3 * wl.H * wl.I
        entry["fused"]["tensor_TFLOPs"] = round(fl / tl / 1e12, 1)
        tf = fl / (entry["fused"]["us_per_call"] * 1e-6) / 1e12
        entry["fused"]["frac_fp8_tensor"] = round(tf / fp8_peak_tflops()[0], 4)
        # labelled separately: the same weight copy every call, L2-warm where it fits (m1, m16)
        tw = b.timed_same(max(64, n // 4), stream)
        entry["fused_l2_warm"] = {"us_per_call": round(tw * 1e6, 3), "tokens_per_s": round(wl.M / tw, 1),
                                  "note": "one weight copy reused every call; L2-resident only if it fits 129 MB"}
        res[name] = entry
        del b
        torch.cuda.empty_cache()
    return res


def decode_kernel_name(fs, M, H=4096, I=12288):
    """The kernel the fused MLP call runs for M tokens (the library's default plan)."""
    if M <= 16 and H >= 256 and I // 128 < 76:
        return "mx_slice_kernel (fused MLP, one launch, 2-block clusters)"
    return "mx_persistent_kernel (fused MLP, one launch)" if M <= 128 else "mx_gemm_tiled_kernel (3 launches)"


def gemm_bytes(M, N, K):
    """Algorithmic bytes of one GEMM call: B codes + scales, bf16 A in, bf16 C out."""
    return N * K + N * K // 32 + 2 * M * K + 2 * M * N


def sweep_c5(fs, device, stream, hbm_peak, Ms=None):
    """The H = 5120, I = 17408 sweep over M in {1, 2, 4, 8, 16, 32, 64, 128}
    (16 distinct layers, 1% all-zero 32-blocks): the standalone GEMM entry
    point on the gate/up (N = 2I, K = H) and down (N = H, K = I) shapes, and
    the fused and three-launch MLP, each timed as CUDA-graph replays that
    rotate over the 16 layers (4.4 GB of weights, far beyond L2)."""
    import torch

    from workloads import inputs

    wl = inputs.WORKLOADS["sweep"]
    H, I, L = wl.H, wl.I, wl.layers
    layers = []
    for layer in range(L):
        wg, wu, wd = inputs.make_layer_torch(wl, layer, device)
        layers.append(fs.prepare_mlp_weights(wg, wu, wd))
        del wg, wu, wd
    torch.cuda.synchronize()
    res = {"H": H, "I": I, "layers": L, "weight_bytes_per_layer": wl.weight_bytes,
           "timing": "CUDA graph replays rotating over the 16 layers; us per call"}
    Ms = Ms or wl.M_sweep
    for M in Ms:
        x = inputs.make_activations_torch(wl, M, device)
        h_in = inputs.make_activations_torch(inputs.Workload("h", M, I, H, 1, wl.seed + 1), M, device)
        y = torch.empty(M, H, dtype=torch.bfloat16, device=device)
        cgu = torch.empty(M, 2 * I, dtype=torch.bfloat16, device=device)
        ws = fs.Workspace(M, H, I, device=device)
        gws_n = max(fs.fsops_gemm_workspace_bytes(M, 2 * I, H), fs.fsops_gemm_workspace_bytes(M, H, I))
        gws = torch.zeros(gws_n, dtype=torch.uint8, device=device)
        s = stream.cuda_stream
        calls = {
            "gemm_gateup": (lambda w: fs.fsops_mxfp8_gemm(x, w.gateup_codes, w.gateup_scales, cgu, M, 2 * I, H, gws,
                                                          gws_n, stream=s), gemm_bytes(M, 2 * I, H), 2.0 * M * 2 * I * H),
            "gemm_down": (lambda w: fs.fsops_mxfp8_gemm(h_in, w.down_codes, w.down_scales, y, M, H, I, gws, gws_n,
                                                        stream=s), gemm_bytes(M, H, I), 2.0 * M * H * I),
            "mlp_fused": (lambda w: fs.fsops_mxfp8_swiglu_mlp(x, w.gateup_codes, w.down_codes, w.scales, y, M, H, I,
                                                              stream=s), algorithmic_bytes(M, H, I),
                          2.0 * M * 3 * H * I),
            "mlp_unfused_3_launches": (lambda w: fs.fsops_mxfp8_swiglu_mlp_unfused(
                x, w.gateup_codes, w.down_codes, w.scales, y, M, H, I, stream=s), algorithmic_bytes(M, H, I),
                2.0 * M * 3 * H * I),
        }
        entry = {}
        for name, (fn, nbytes, flops) in calls.items():
            n = 4 * L
            with torch.cuda.stream(stream):
                for i in range(3):
                    fn(layers[i % L])
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    for i in range(n):
                        fn(layers[i % L])
                g.replay()
                stream.synchronize()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for _ in range(3):
                    g.replay()
                e1.record(stream)
                e1.synchronize()
            t = e0.elapsed_time(e1) / 1e3 / (3 * n)
            entry[name] = {"us_per_call": round(t * 1e6, 3), "GBps": round(nbytes / t / 1e9, 1),
                           "frac_hbm": round(nbytes / t / 1e9 / hbm_peak, 4),
                           "TFLOPs": round(flops / t / 1e12, 1)}
            if name.startswith("mlp"):
                entry[name]["tokens_per_s"] = round(M / t, 1)
            del g
        res["M%d" % M] = entry
        del x, h_in, y, cgu, ws, gws
        torch.cuda.empty_cache()
    del layers
    torch.cuda.empty_cache()
    return res


def blockscale_gemm(fs, stream, hbm_peak):
    """The 128 x 128 block-scaled FP8 GEMM (fsops_fp8_blockscale_gemm) on the
    H = 5120, I = 17408 decode shapes (gate/up N = 34816, K = 5120; down
    N = 5120, K = 17408) at M = 1, 16, 128, with pre-quantised A, rotating
    over enough weight copies to exceed L2; the MXFP8 GEMM
    (fsops_mxfp8_gemm_ex, pre-quantised A) on the same shapes beside it."""
    import torch

    res = {"timing": "CUDA graph replays rotating over weight copies (> 2x L2); us per call"}
    g = torch.Generator(device="cuda").manual_seed(5)
    for name, (N, K) in (("gateup", (34816, 5120)), ("down", (5120, 17408))):
        w = (torch.randn(N, K, device="cuda", generator=g) / K ** 0.5).to(torch.bfloat16)
        copies = max(2, -(-2 * L2_BYTES // (N * K)) + 1)
        bs_w = [fs.quantize_blockscale(w, 128) for _ in range(copies)]
        mx_w = [fs.quantize_weight(w) for _ in range(copies)]
        del w
        for M in (1, 16, 128):
            a = torch.randn(M, K, device="cuda", generator=g).to(torch.bfloat16)
            ac, asc = fs.quantize_blockscale(a, 1)
            mc, msc = fs.quantize_weight(a)
            c = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
            n_bs = fs.fsops_blockscale_gemm_workspace_bytes(M, N, K)
            ws_bs = torch.zeros(n_bs + 256, dtype=torch.uint8, device="cuda")
            p_bs = ws_bs.data_ptr() + (-ws_bs.data_ptr()) % 256
            n_mx = fs.fsops_gemm_workspace_bytes(M, N, K)
            ws_mx = torch.zeros(n_mx, dtype=torch.uint8, device="cuda")
            s = stream.cuda_stream
            calls = {
                "blockscale": (lambda i: fs.fsops_fp8_blockscale_gemm(ac, asc, bs_w[i % copies][0], bs_w[i % copies][1], c,
                                                                      fs.DTYPE_BF16, M, N, K, p_bs, n_bs, stream=s),
                               N * K + (N // 128) * (K // 128) * 4 + M * K + M * (K // 128) * 4 + 2 * M * N),
                "mxfp8": (lambda i: fs.fsops_mxfp8_gemm_ex(mc, msc, fs.DTYPE_MXFP8, mx_w[i % copies][0], mx_w[i % copies][1],
                                                           c, fs.DTYPE_BF16, M, N, K, ws_mx, n_mx, stream=s),
                          N * K + N * K // 32 + M * K + M * K // 32 + 2 * M * N),
            }
            entry = {}
            for kind, (fn, nbytes) in calls.items():
                n = 8 * copies
                with torch.cuda.stream(stream):
                    for i in range(3):
                        fn(i)
                    gr = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(gr, stream=stream):
                        for i in range(n):
                            fn(i)
                    gr.replay()
                    stream.synchronize()
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    for _ in range(3):
                        gr.replay()
                    e1.record(stream)
                    e1.synchronize()
                t = e0.elapsed_time(e1) / 1e3 / (3 * n)
                entry[kind] = {"us_per_call": round(t * 1e6, 3), "GBps": round(nbytes / t / 1e9, 1),
                               "frac_hbm": round(nbytes / t / 1e9 / hbm_peak, 4),
                               "TFLOPs": round(2.0 * M * N * K / t / 1e12, 1)}
                del gr
            res["%s_N%d_K%d_M%d" % (name, N, K, M)] = entry
            del a, ac, asc, mc, msc, c, ws_bs, ws_mx
        del bs_w, mx_w
        torch.cuda.empty_cache()
    return res


def prefill_gemm(fs, stream, only=None):
    """The GEMM API above 128 rows (whole 128 x 256 tiles): the m16 MLP's
    gate/up and down projections at M = 4096, bf16 A (quantised by its own
    launch) and pre-quantised A; tensor-bound, so TFLOP/s against the FP8
    peak.  torch's FP8 GEMM with one scale per tensor (cuBLAS, no 1x32 block
    scales) is timed beside it for context."""
    import torch

    peak, peak_kind = fp8_peak_tflops()
    res = {"fp8_peak_tflops": round(peak, 1), "peak_kind": peak_kind}

    def timeit(fn, n=30):
        with torch.cuda.stream(stream):
            for _ in range(3):
                fn()
            stream.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(n):
                fn()
            e1.record(stream)
            e1.synchronize()
        return e0.elapsed_time(e1) / 1e3 / n

    g = torch.Generator(device="cuda").manual_seed(7)
    shapes = (("gateup_m4096", (4096, 19456, 2560)), ("down_m4096", (4096, 2560, 9728)),
              ("square_1024", (1024, 1024, 1024)), ("square_4096", (4096, 4096, 4096)),
              ("square_8192", (8192, 8192, 8192)), ("square_16384", (16384, 16384, 16384)))
    for name, (M, N, K) in shapes:
        if only and name not in only:
            continue
        a = torch.randn(M, K, device="cuda", generator=g).to(torch.bfloat16)
        w = (torch.randn(N, K, device="cuda", generator=g) / K ** 0.5).to(torch.bfloat16)
        bc, bs = fs.quantize_weight(w)
        ac, asc = fs.quantize_weight(a)
        ws_n = fs.fsops_gemm_workspace_bytes(M, N, K)
        ws = torch.zeros(ws_n, dtype=torch.uint8, device="cuda")
        c = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
        s = stream.cuda_stream
        reps = 30 if M * N * K <= 8192 ** 3 else 8
        t_bf16 = timeit(lambda: fs.fsops_mxfp8_gemm(a, bc, bs, c, M, N, K, ws, ws_n, stream=s), reps)
        t_pre = timeit(lambda: fs.fsops_mxfp8_gemm_ex(ac, asc, fs.DTYPE_MXFP8, bc, bs, c, fs.DTYPE_BF16, M, N, K, ws,
                                                      ws_n, stream=s), reps)
        fl = 2.0 * M * N * K
        entry = {"M": M, "N": N, "K": K,
                 "bf16_a_us": round(t_bf16 * 1e6, 2), "bf16_a_tflops": round(fl / t_bf16 / 1e12, 1),
                 "mxfp8_a_us": round(t_pre * 1e6, 2), "mxfp8_a_tflops": round(fl / t_pre / 1e12, 1),
                 "frac_fp8_tensor": round(fl / t_pre / 1e12 / peak, 4)}
        try:
            a8, w8 = a.to(torch.float8_e4m3fn), w.to(torch.float8_e4m3fn)
            one = torch.ones((), device="cuda")
            t_s = timeit(lambda: torch._scaled_mm(a8, w8.t(), scale_a=one, scale_b=one, out_dtype=torch.bfloat16),
                         reps)
            entry["cublas_fp8_per_tensor_us"] = round(t_s * 1e6, 2)
            del a8, w8
        except Exception:  # not every torch build exposes it
            entry["cublas_fp8_per_tensor_us"] = None
        # torch's MXFP8 GEMM (cuBLAS block-scaled) on the same codes and scales:
        # its block-scale layout is the same 128 x 4 tiling, so the buffers
        # pass as they are; the outputs must agree
        try:
            MT, KS = (M + 127) // 128, K // 128
            sa = asc.view(torch.float8_e8m0fnu).reshape(MT * 128, KS * 4)
            sb = bs.view(torch.float8_e8m0fnu).reshape(N, KS * 4)
            a8, b8 = ac.view(torch.float8_e4m3fn), bc.view(torch.float8_e4m3fn)
            ref = torch._scaled_mm(a8, b8.t(), scale_a=sa, scale_b=sb, out_dtype=torch.bfloat16)
            fs.fsops_mxfp8_gemm_ex(ac, asc, fs.DTYPE_MXFP8, bc, bs, c, fs.DTYPE_BF16, M, N, K, ws, ws_n, stream=s)
            stream.synchronize()
            finite = bool(torch.isfinite(ref).all())
            diff = ((ref.float() - c.float()).norm() / ref.float().norm()).item() if finite else None
            t_mx = timeit(lambda: torch._scaled_mm(a8, b8.t(), scale_a=sa, scale_b=sb, out_dtype=torch.bfloat16),
                          reps)
            entry["cublas_mxfp8_us"] = round(t_mx * 1e6, 2)
            entry["cublas_mxfp8_output_finite"] = finite
            entry["cublas_mxfp8_rel_l2_vs_ours"] = None if diff is None else float("%.3g" % diff)
            del ref
        except Exception as e:  # older torch / cuBLAS without MX block scaling
            entry["cublas_mxfp8_us"] = None
            entry["cublas_mxfp8_error"] = str(e).splitlines()[0][:160] if str(e) else type(e).__name__
        res[name] = entry
        del a, w, bc, bs, ac, asc, ws, c
        torch.cuda.empty_cache()
    if only:
        return res
    # the whole MLP of the m16 layer at 4096 tokens: x quantisation, the gate/up
    # GEMM with the SwiGLU + requantisation epilogue, the down GEMM; and the
    # three-launch ablation (gate/up to fp32 in HBM, SwiGLU-quantise, down)
    M, H, I = 4096, 2560, 9728
    x = torch.randn(M, H, device="cuda", generator=g).to(torch.bfloat16)
    wg, wu = [(torch.randn(I, H, device="cuda", generator=g) / H ** 0.5).to(torch.bfloat16) for _ in range(2)]
    wd = (torch.randn(H, I, device="cuda", generator=g) / I ** 0.5).to(torch.bfloat16)
    mw = fs.prepare_mlp_weights(wg, wu, wd)
    del wg, wu, wd
    mws = fs.Workspace(M, H, I)
    y = torch.empty(M, H, dtype=torch.bfloat16, device="cuda")
    s = stream.cuda_stream
    t_f = timeit(lambda: fs.fsops_mxfp8_swiglu_mlp(x, mw.gateup_codes, mw.down_codes, mw.scales, y, M, H, I, stream=s))
    t_u = timeit(lambda: fs.fsops_mxfp8_swiglu_mlp_unfused(x, mw.gateup_codes, mw.down_codes, mw.scales, y, M, H, I,
                                                           stream=s))
    fl = 2.0 * M * 3 * H * I
    res["mlp_m4096"] = {"M": M, "H": H, "I": I, "launches": 3,
                        "us": round(t_f * 1e6, 2), "tokens_per_s": round(M / t_f, 1),
                        "tflops": round(fl / t_f / 1e12, 1), "frac_fp8_tensor": round(fl / t_f / 1e12 / peak, 4),
                        "unfused_us": round(t_u * 1e6, 2)}
    del x, mw, mws, y
    torch.cuda.empty_cache()
    return res


def attention_decode(fs, stream, hbm_peak):
    """Paged decode attention over the MXFP8 KV cache, a64 workload (Qwen3-4B
    attention geometry, 64 sequences of 2k-6k tokens, 16-token pages): µs
    per call and the cache bytes read per call against the HBM peak."""
    import math

    import numpy as np
    import torch

    from workloads import inputs

    wl = inputs.ATTN_WORKLOADS["a64"]
    d = inputs.make_attention(wl)
    npages = d["k"].shape[0]
    rows = npages * wl.Hkv * wl.P
    cache = []
    for name in ("k", "v"):
        x = torch.from_numpy(np.ascontiguousarray(d[name]).view(np.int16).reshape(rows, wl.D)).cuda()
        codes = torch.empty(rows, wl.D, dtype=torch.uint8, device="cuda")
        scales = torch.empty(rows * wl.D // 32, dtype=torch.uint8, device="cuda")
        fs.fsops_quantize_mxfp8(x, rows, wl.D, wl.D, codes, scales, fs.SCALES_ROWMAJOR)
        cache += [codes, scales]
        del x
    q = torch.from_numpy(np.ascontiguousarray(d["q"]).view(np.int16)).cuda()
    table = torch.from_numpy(d["block_table"]).cuda()
    lens = torch.from_numpy(d["seq_lens"]).cuda()
    max_pages = d["block_table"].shape[1]
    ws_n = fs.fsops_paged_attention_workspace_bytes(wl.B, wl.Hq, wl.Hkv, wl.D, wl.P, max_pages)
    ws = torch.zeros(ws_n + 256, dtype=torch.uint8, device="cuda")
    ws_ptr = ws.data_ptr() + (-ws.data_ptr()) % 256
    out = torch.empty(wl.B, wl.Hq, wl.D, dtype=torch.bfloat16, device="cuda")
    s = stream.cuda_stream

    def call():
        fs.fsops_mxfp8_paged_decode_attention(q, cache[0], cache[1], cache[2], cache[3], npages, table, max_pages,
                                              lens, out, wl.B, wl.Hq, wl.Hkv, wl.D, wl.P, 1.0 / math.sqrt(wl.D),
                                              ws_ptr, ws_n, stream=s)

    with torch.cuda.stream(stream):
        for _ in range(3):
            call()
        stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(20):
            call()
        e1.record(stream)
        e1.synchronize()
    t = e0.elapsed_time(e1) / 1e3 / 20
    tokens = int(d["seq_lens"].sum())
    kv = tokens * wl.Hkv * 2 * (wl.D + wl.D // 32)
    status = fs.fsops_read_kernel_status(ws_ptr)
    res = {"workload": "a64: B=%d, Hq=%d, Hkv=%d, D=%d, page %d, lengths %d-%d (%d tokens)" %
                       (wl.B, wl.Hq, wl.Hkv, wl.D, wl.P, wl.len_lo, wl.len_hi, tokens),
           "us": round(t * 1e6, 2), "kv_bytes": kv, "GBps": round(kv / t / 1e9, 1),
           "frac_hbm": round(kv / t / 1e9 / hbm_peak, 4), "launches": 2, "status": status}
    del cache, q, table, lens, ws, out
    torch.cuda.empty_cache()
    return res


def cpu_baseline(wl):
    """The oracle as it stands, timed on this host on one full layer of the workload."""
    import numpy as np

    import oracle
    from workloads import inputs

    x = inputs.make_activations(wl)
    wg, wu, wd = inputs.make_layer(wl, 0)
    qw = oracle.quantize_weights(wg, wu, wd)
    t0 = time.time()
    reps = 0
    while True:
        oracle.swiglu_mlp(x, qw)
        reps += 1
        if time.time() - t0 > 8.0 or reps >= 20:
            break
    dt = (time.time() - t0) / reps
    return {"value": round(wl.M / dt, 3), "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": "%d full %s layer(s) (M=%d tokens each): x quantisation, weight dequantisation, "
                      "fp64 GEMMs, SiLU, requantisation; %.2f s per layer" % (reps, wl.name, wl.M, dt)}


def _slice_layer(qw, I, s):
    """Oracle inputs for the first s intermediate features of a layer."""
    return {"gateup_codes": __import__("numpy").concatenate([qw["gateup_codes"][:s], qw["gateup_codes"][I:I + s]]),
            "gateup_scales": __import__("numpy").concatenate([qw["gateup_scales"][:s], qw["gateup_scales"][I:I + s]]),
            "down_codes": qw["down_codes"][:, :s].copy(), "down_scales": qw["down_scales"][:, :s // 32].copy()}


def run_reference(args, rank, world):
    """The CPU oracle as the reference arm (rank 0 only).

    Each step is a bounded sample of the workload: a full layer if K + W full
    layers fit in about two minutes, otherwise the layer restricted to its
    first s intermediate features (s a multiple of 128), with tokens/s scaled
    by s / I (the fraction of the layer's work a step does)."""
    import oracle
    from workloads import inputs

    if rank != 0:
        return None
    wl = inputs.WORKLOADS[args.workload]
    x = inputs.make_activations(wl)
    wg, wu, wd = inputs.make_layer(wl, 0)
    qw = oracle.quantize_weights(wg, wu, wd)
    t0 = time.time()
    oracle.swiglu_mlp(x, qw)
    t_full = time.time() - t0
    budget = 120.0
    s = wl.I
    if (args.steps + args.warmup) * t_full > budget:
        s = int(wl.I * budget / ((args.steps + args.warmup) * t_full)) // 128 * 128
        s = max(128, min(wl.I, s))
    sample = qw if s == wl.I else _slice_layer(qw, wl.I, s)
    for _ in range(args.warmup):
        oracle.swiglu_mlp(x, sample)
    t0 = time.time()
    for _ in range(args.steps):
        oracle.swiglu_mlp(x, sample)
    dt = time.time() - t0
    value = wl.M * (s / wl.I) * args.steps / dt
    desc = ("one full %s layer" % wl.name) if s == wl.I else (
        "the %s layer restricted to its first %d of %d intermediate features (tokens/s scaled by %d/%d)" %
        (wl.name, s, wl.I, s, wl.I))
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "%s: MXFP8 SwiGLU MLP, M=%d, H=%d, I=%d, one layer per step" % (wl.name, wl.M, wl.H,
                                                                                              wl.I),
                   "M": wl.M, "H": wl.H, "I": wl.I},
        "cpu_baseline": {"value": round(value, 4), "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
                         "sample": "each step: " + desc + " through the fp64 oracle"},
        "e2e": {"value": round(value, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    # defaults: 20000 steps and 20 warm-up calls for the GPU arm (about half a
    # second of timed work at m16); 20 and 5 for the CPU oracle arm, whose
    # every call costs at least ~50 ms whatever its sample
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="m16")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--layers", type=int, default=0,
                    help="distinct weight layers of the workload (0: its own count); profiling runs use fewer")
    ap.add_argument("--unfused", action="store_true", help="time the three-launch path as the main loop")
    ap.add_argument("--prefill-only", action="store_true",
                    help="print only the prefill GEMM / MLP section (a short run for profiling the tiled kernel)")
    ap.add_argument("--attention-only", action="store_true",
                    help="print only the paged decode attention section")
    ap.add_argument("--blockscale-only", action="store_true",
                    help="print only the 128 x 128 block-scaled GEMM section")
    ap.add_argument("--knob", action="append", default=[],
                    help="NAME=VALUE plan knob of the library (fsops_debug_set_knob), e.g. PAIRS=0 for the launch form "
                         "an ncu capture uses; repeatable")
    ap.add_argument("--prefill-shapes", default="",
                    help="comma-separated subset of the prefill section's GEMM shapes (default: all)")
    args = ap.parse_args()
    if args.steps is None:
        args.steps = 20 if args.impl == "reference" else 20000
    if args.warmup is None:
        args.warmup = 5 if args.impl == "reference" else 20
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    if args.knob and args.impl == "ours":
        import mxfp8_swiglu_mlp_gb300 as fs

        for kv in args.knob:
            k, v = kv.split("=")
            fs.fsops_debug_set_knob(k.strip(), int(v))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        out = run_reference(args, rank, world)
        if out is not None:
            print(json.dumps(out), flush=True)
        return
    if args.attention_only:
        import torch

        import mxfp8_swiglu_mlp_gb300 as fs

        torch.cuda.set_device(local_rank)
        print(json.dumps({"attention_decode": attention_decode(fs, torch.cuda.Stream(), peaks()[0])}), flush=True)
        return
    if args.blockscale_only:
        import torch

        import mxfp8_swiglu_mlp_gb300 as fs

        torch.cuda.set_device(local_rank)
        print(json.dumps({"blockscale_gemm": blockscale_gemm(fs, torch.cuda.Stream(), peaks()[0])}), flush=True)
        return
    if args.prefill_only:
        import torch

        import mxfp8_swiglu_mlp_gb300 as fs

        torch.cuda.set_device(local_rank)
        only = [x for x in args.prefill_shapes.split(",") if x]
        print(json.dumps({"prefill_gemm": prefill_gemm(fs, torch.cuda.Stream(), only)}), flush=True)
        return
    if world > 1:
        import torch

        torch.distributed.init_process_group("nccl")
    out = run_ours(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch

        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
