"""Throughput benchmark of the GB300 mixed-precision GEMM (one JSON line).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME]

A step is one pass of the hot path over one batch of synthetic input: by
default the three GEMMs of a transformer layer at 8192 tokens (BF16 inputs,
weights stored N x K, FP32 accumulation, BF16 output):
    8192 x 4096 x 4096, 8192 x 14336 x 4096, 8192 x 4096 x 14336.
Throughput is 2*M*N*K per GEMM summed over the step, divided by the
device-timed step (CUDA events on the launching stream, W warm-up steps,
barrier + synchronize around K timed steps, max over ranks).  Every step
touches about 1 GB of operands, far more than the 129 MB L2, so no L2 flush is
needed between steps.

Also reported:
  roofline     -- the dominant kernel's achieved TFLOP/s (algorithmic flops per
                  launch / mean launch duration from events around each launch)
                  against the measured dense BF16 peak in MEASURED_PEAKS.json;
                  `traffic` is the DRAM bytes per launch from the committed ncu
                  summary when it was taken on the current kernel sources;
  e2e          -- the same metric through the C ABI with host (pinned) buffers:
                  each step copies its inputs host->device and the outputs back;
  cpu_baseline -- the CPU oracle (plain FP64 triple loop, all host cores) timed
                  on a bounded sample of the same workload (rank 0, N = 1);
  clocks       -- nvidia-smi SM clocks and throttle reasons sampled during the
                  timed region;
  sustained    -- (default workload) the same step back to back for about two
                  seconds, at the power cap, against the measured sustained
                  BF16 peak, with its own clocks;
  skinny       -- (default workload) the skinny decode GEMM 64 x 16384 x 8192
                  (FP16, weights N x K) back to back: GB/s against the
                  measured HBM copy bandwidth, with its own clocks;
  context      -- (default workload) cuBLAS via torch.matmul on this GPU:
                  BF16, FP16 and TF32 8192^3 rates and the step's three shapes
                  (denominator checks, not part of the measurement).
--impl reference times the CPU oracle as the comparison arm (the pages ship
no runnable implementation); it runs on rank 0 only.

--workload conv* times the implicit-GEMM convolution (CATLASS page, section
5.1): a step is one conv2d_fprop call; the metric is TFLOP/s
(2 N P Q K R S C / t) against the dense BF16 peak.

--workload softmax_* times the row softmax instead (SGEMM tutorial page,
section 2): a step is one softmax_rows call over the whole matrix; the metric
is GB/s (X read once + Y written once, per unit time) against the measured
HBM copy bandwidth; e2e copies X up and Y back every step.
With N > 1 (torchrun, one rank per GPU) every rank runs the same step on its
own GPU: replicas, no collective on the data path (weak scaling).
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
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "GEMM TFLOP/s (2MNK/t) at 1 GB300; % of dense tensor peak or HBM roofline"
LAYER = ["linear_8192x4096x4096_bf16", "linear_8192x14336x4096_bf16",
         "linear_8192x4096x14336_bf16"]
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# every file the timed kernels compile from, and the host planner whose
# raster and L2 policies set their DRAM traffic: a committed traffic figure
# is reported only while these hash to the build it was captured on
KERNEL_SOURCES = ["mixed_precision_dense_sm_gb300/csrc/gemm_tc.cuh",
                  "mixed_precision_dense_sm_gb300/csrc/api.cu",
                  "mixed_precision_dense_sm_gb300/csrc/ptx.cuh",
                  "mixed_precision_dense_sm_gb300/csrc/epilogue_ops.cuh",
                  "mixed_precision_dense_sm_gb300/csrc/kern_inst.cuh"]
SOFTMAX_SOURCES = ["mixed_precision_dense_sm_gb300/csrc/softmax_kern.cuh",
                   "mixed_precision_dense_sm_gb300/csrc/softmax_tma.cuh",
                   "mixed_precision_dense_sm_gb300/csrc/softmax_inst.cuh",
                   "mixed_precision_dense_sm_gb300/csrc/softmax_launch.h",
                   "mixed_precision_dense_sm_gb300/csrc/softmax.cu",
                   "mixed_precision_dense_sm_gb300/csrc/ptx.cuh"]
SOFTMAX_METRIC = "softmax GB/s (X read once + Y written once, per second) at 1 GB300; % of HBM"
CONV_METRIC = "conv2d TFLOP/s (2 N P Q K R S C / t) at 1 GB300; % of dense tensor peak"


def kernel_hash(sources=None) -> str:
    h = hashlib.sha256()
    for f in (sources or KERNEL_SOURCES):
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK), "fallback"


def committed_traffic(workload: str, sources=None):
    """DRAM bytes per launch from profiles/traffic.json, if taken on these sources."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(workload)
    if not e or e.get("kernel_hash") != kernel_hash(sources):
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi SM clock / throttle-reason samples during the timed region."""

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
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append((time.time(), ln.strip()))

    def stop(self, window=None):
        """Summarise the samples that arrived inside `window` (host wall-clock
        start/end of the timed region); when fewer than 3 did, the samples of
        the warm-up and the timed region together."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        lines, which = self.lines, "warmup+timed"
        if window is not None:
            inside = [x for x in self.lines if window[0] <= x[0] <= window[1] + 0.15]
            if len(inside) >= 3:
                lines, which = inside, "timed"
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for _, ln in lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
                power.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm), "window": which,
                "sm_mhz_min": min(sm) if sm else None,
                "power_w_median": statistics.median(power) if power else None}


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """The largest of every rank's x (the slowest rank's time decides)."""
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_step: float, steps: int, world: int, max_ms: float) -> float:
    """Replicas: every rank runs the same step, so the job does world x the
    work in the slowest rank's time."""
    return world * flops_per_step * steps / (max_ms * 1e-3) / 1e12


def workload_list(name: str):
    if name == "transformer_layer":
        return [workloads.WORKLOADS[n] for n in LAYER]
    return [workloads.WORKLOADS[name]]


def describe(name: str, ws):
    if name == "transformer_layer":
        return ("transformer linear layers at 8192 tokens, BF16 activations N(0,1) and "
                "N x K weights N(0,0.02), FP32 accumulate, BF16 out: "
                "8192x4096x4096 + 8192x14336x4096 + 8192x4096x14336 (M x N x K) per step")
    w = ws[0]
    return f"{w.name}: {w.M}x{w.N}x{w.K} {w.transA}{w.transB}"


# ------------------------------------------------------------------ CPU oracle

class OracleSampler:
    """Times the CPU oracle (all host cores) on a bounded sample of the step:
    `n` seeded output elements of each GEMM, each one a full K-long dot
    product evaluated by the oracle's sampled entry point."""

    def __init__(self, ws, seed=1):
        import numpy as np
        import oracle
        self.orc = oracle.get()
        self.threads = self.orc.max_threads()
        self.ws = ws
        self.inputs = []
        rng = np.random.default_rng(seed)
        for w in ws:
            inp = workloads.make_inputs(w)
            codes = (workloads.as_codes(inp.A), workloads.as_codes(inp.B),
                     None if inp.C is None else workloads.as_codes(inp.C))
            pos = (rng.integers(0, w.M, 1 << 20), rng.integers(0, w.N, 1 << 20))
            self.inputs.append((inp, codes, pos))

    def run(self, n):
        """Oracle seconds and flops for n sampled outputs of each GEMM."""
        total_t, flops = 0.0, 0.0
        for w, (inp, (A, B, C), (rows, cols)) in zip(self.ws, self.inputs):
            t = time.perf_counter()
            self.orc.gemm_sampled(w.transA, w.transB, w.M, w.N, w.K, w.alpha, A, inp.lda, B,
                                  inp.ldb, w.beta, C, inp.ldc, w.ab_dtype, w.c_dtype,
                                  rows[:n], cols[:n], nthreads=self.threads)
            total_t += time.perf_counter() - t
            flops += 2.0 * n * w.K
        return flops, total_t

    def run_rows(self, rows):
        """The oracle's full-matrix entry point on the first `rows` rows of each
        GEMM (it decodes op(A) and op(B) once per call, then runs the triple
        loop).  Returns (flops, seconds)."""
        import numpy as np
        total_t, flops = 0.0, 0.0
        for w, (inp, (A, B, C), _) in zip(self.ws, self.inputs):
            r = min(rows, w.M)
            if w.transA in "Nn":
                a_rows, a_ld = A[:r], inp.lda
            else:
                a_rows, a_ld = np.ascontiguousarray(A[:, :r]), r
            t = time.perf_counter()
            self.orc.gemm(w.transA, w.transB, r, w.N, w.K, w.alpha, a_rows, a_ld, B, inp.ldb,
                          0.0, None, w.N, w.ab_dtype, w.c_dtype, nthreads=self.threads)
            total_t += time.perf_counter() - t
            flops += 2.0 * r * w.N * w.K
        return flops, total_t

    def calibrate(self, target_s):
        """Sample size (per GEMM) that takes about target_s seconds."""
        n, t = 64, 0.0
        while n < (1 << 20):
            _, t = self.run(n)
            if t >= target_s / 8:
                break
            n = min(n * 4, 1 << 20)
        if t > 0:
            n = int(min(1 << 20, max(16, n * target_s / t)))
        return n

    def calibrate_rows(self, target_s):
        """Row count for run_rows that takes about target_s seconds."""
        max_rows = min(w.M for w in self.ws)
        rows, t = 4, 0.0
        while rows < max_rows:
            _, t = self.run_rows(rows)
            if t >= target_s / 4:
                break
            rows = min(rows * 4, max_rows)
        if t > 0 and rows < max_rows:
            rows = int(min(max_rows, max(4, rows * target_s / t)))
        return rows


# ------------------------------------------------------------------ GPU arm

def run_ours(args):
    import mixed_precision_dense_sm_gb300 as lib
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    ws = workload_list(args.workload)
    if (args.epilogue or args.layernorm) and args.workload != "transformer_layer":
        raise SystemExit("--epilogue / --layernorm apply to the transformer_layer workload")
    fused = args.epilogue or args.layernorm
    g = lib.Gemm()
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream

    bufs = []
    epis = []
    for j, w in enumerate(ws):
        if fused:
            # transformer MLP block: bias on every GEMM, GELU after the
            # up-projection, the residual added (beta = 1) after the down one
            w = dataclasses.replace(w, beta=1.0, c_dist="N1") if j == 2 else w
            ws[j] = w
        inp = workloads.make_inputs(w)
        A, B = inp.A.cuda(), inp.B.cuda()
        cdt = workloads.TORCH_DTYPE[w.c_dtype]
        C = (inp.C.cuda() if inp.C is not None
             else torch.zeros((w.M, inp.ldc), dtype=cdt, device="cuda"))
        bufs.append((w, inp, A, B, C))
        if fused:
            gen = torch.Generator().manual_seed(100 + j)
            bias = (0.02 * torch.randn(w.N, generator=gen)).to(cdt).cuda()
            act = lib.ACT_GELU if j == 1 else lib.ACT_NONE
            if args.layernorm and j == 2:
                # post-LN block: LayerNorm(x + W2 h + b2) over the 4096 columns,
                # gamma = 1 + 0.1 N(0,1), shift = 0.1 N(0,1) in BF16
                gamma = (1.0 + 0.1 * torch.randn(w.N, generator=gen)).to(cdt).cuda()
                shift = (0.1 * torch.randn(w.N, generator=gen)).to(cdt).cuda()
                epis.append(("ln", bias, gamma, shift))
            else:
                epis.append(("ex", bias, act))
        else:
            epis.append(None)
    del inp

    plans = []
    for (w, inp, A, B, C) in bufs:
        st, p = lib.gemm_plan_query(w.transA, w.transB, w.M, w.N, w.K, w.alpha, A.data_ptr(),
                                    inp.lda, B.data_ptr(), inp.ldb, w.beta, C.data_ptr(), inp.ldc,
                                    (w.ab_dtype, w.ab_dtype, w.c_dtype),
                                    num_sms=torch.cuda.get_device_properties(local).multi_processor_count)
        plans.append(p)
    # one gemm_tc_kernel launch per call, plus a pack pre-pass per operand
    # that needs one (the stream-K finish runs inside the GEMM kernel), plus
    # the LayerNorm row pass where rows span several tiles
    ln_rows = [0] * len(bufs)
    for i, (w, inp, A, B, C) in enumerate(bufs):
        if epis[i] is not None and epis[i][0] == "ln":
            bias, gamma, shift = epis[i][1:]
            st, q = lib.gemm_layernorm_plan_query(
                w.transA, w.transB, w.M, w.N, w.K, w.alpha, A.data_ptr(), inp.lda, B.data_ptr(),
                inp.ldb, w.beta, C.data_ptr(), inp.ldc, (w.ab_dtype, w.ab_dtype, w.c_dtype),
                bias=bias.data_ptr(), bias_dtype=lib.dtype_code(bias.dtype),
                gamma=gamma.data_ptr(), shift=shift.data_ptr(),
                ln_dtype=lib.dtype_code(gamma.dtype),
                num_sms=torch.cuda.get_device_properties(local).multi_processor_count)
            plans[i] = q
            ln_rows[i] = 0 if q["ln_fused"] else 1
    launches_per_step = sum(1 + p["pack_a"] + p["pack_b"] + r for p, r in zip(plans, ln_rows))
    gemm_only = all(p["pack_a"] == 0 and p["pack_b"] == 0 for p in plans) and not any(ln_rows)

    def launch(i, A, B, C, s):
        """The step's call i through the C ABI on stream s (the plain GEMM, the
        fused bias/activation epilogue, or LayerNorm after the linear layer)."""
        w, inp = bufs[i][0], bufs[i][1]
        dts = (w.ab_dtype, w.ab_dtype, w.c_dtype)
        e = epis[i]
        if e is None:
            st = lib.gemm_run(g.h, w.transA, w.transB, w.M, w.N, w.K, w.alpha, A.data_ptr(),
                              inp.lda, B.data_ptr(), inp.ldb, w.beta, C.data_ptr(), inp.ldc, dts, s)
        elif e[0] == "ex":
            bias, act = e[1], e[2]
            st = lib.gemm_run_ex(g.h, w.transA, w.transB, w.M, w.N, w.K, w.alpha, A.data_ptr(),
                                 inp.lda, B.data_ptr(), inp.ldb, w.beta, C.data_ptr(), inp.ldc,
                                 dts, bias.data_ptr(), lib.dtype_code(bias.dtype), act, s)
        else:
            bias, gamma, shift = e[1:]
            st = lib.gemm_run_layernorm(
                g.h, w.transA, w.transB, w.M, w.N, w.K, w.alpha, A.data_ptr(), inp.lda,
                B.data_ptr(), inp.ldb, w.beta, C.data_ptr(), inp.ldc, dts, bias.data_ptr(),
                lib.dtype_code(bias.dtype), gamma.data_ptr(), shift.data_ptr(),
                lib.dtype_code(gamma.dtype), 1e-5, s)
        if st != 0:
            raise lib.GemmError(st, "gemm_run")

    def step(events=None):
        for i, (w, inp, A, B, C) in enumerate(bufs):
            if events is not None:
                events[i][0].record(stream)
            launch(i, A, B, C, sh)
            if events is not None:
                events[i][1].record(stream)

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)                      # nvidia-smi start-up
    for _ in range(args.warmup):
        step()
    g.sync()

    # timed region: K steps.  When every launch of the step is the GEMM
    # kernel, events bracket the region only: an event between two launches
    # would stop the next kernel's set-up from overlapping the previous
    # kernel's tail (programmatic dependent launch), so per-launch events
    # would time a slower program than the one a caller runs.  Otherwise
    # (pack pre-passes in the step) events around each GEMM launch attribute
    # the time to the kernel.
    ev = None if gemm_only else [
        [[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)]
         for _ in bufs] for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    w0 = time.time()
    t_start.record(stream)
    for k in range(args.steps):
        step(None if ev is None else ev[k])
    t_end.record(stream)
    torch.cuda.synchronize()
    w1 = time.time()
    clk = clocks.stop((w0, w1))
    barrier(world)
    g.sync()
    ms_total = t_start.elapsed_time(t_end)
    ms_total = max_over_ranks(ms_total, world)
    ms_step = ms_total / args.steps
    flops_step = sum(w.flops() for w in ws)
    value = whole_job_tflops(flops_step, args.steps, world, ms_total)

    # dominant kernel: gemm_tc_kernel, the one launch of each call.  Its
    # average launch duration is the timed region over its launches when the
    # step launches nothing else, else the mean of the per-launch events.
    # A separate pass after the timed region times each shape with events
    # around every launch (the per-shape breakdown; those events stop the
    # launch overlap, so these figures are a little slower).
    if ev is None:
        region_ms_per_step = ms_total / args.steps
        ev_shape = [[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)]
                    for _ in range(len(bufs) * min(args.steps, 50))]
        for k in range(min(args.steps, 50)):
            step(ev_shape[k * len(bufs):(k + 1) * len(bufs)])
        torch.cuda.synchronize()
        shape_ms = [statistics.fmean(ev_shape[k * len(bufs) + i][0].elapsed_time(
                        ev_shape[k * len(bufs) + i][1]) for k in range(min(args.steps, 50)))
                    for i in range(len(bufs))]
        launch_scale = region_ms_per_step / sum(shape_ms)
        launch_ms = [t * launch_scale for t in shape_ms]          # sums to the region's step
        launch_src = ("timed region / launches (events at the region's ends only); per shape "
                      "split in proportion to a separate pass with events around each launch")
    else:
        launch_ms = [statistics.fmean(ev[k][i][0].elapsed_time(ev[k][i][1])
                                      for k in range(args.steps)) for i in range(len(bufs))]
        shape_ms = launch_ms
        launch_src = "events around each GEMM launch inside the timed region"
        if any(ln_rows):
            launch_src = ("events around each call inside the timed region; the LayerNorm "
                          "call's time includes its row pass")
    achieved = sum(w.flops() for w in ws) / (sum(launch_ms) * 1e-3) / 1e12
    peaks, peak_src = load_peaks()
    bound = "tensor"
    # A timed region of back-to-back launches longer than half a second runs
    # at the power cap: the sustained peak is the matching denominator.
    long_region = ms_total > 500.0
    peak = peaks["bf16_tflops_sustained"] if long_region else peaks["bf16_tflops"]
    # FP32 inputs run kind::tf32.  Its dense rate is measured here, on this
    # GPU: cuBLAS's FP32 8192^3 GEMM with TF32 allowed (burst, best of 10),
    # as a ratio to cuBLAS's BF16 rate timed the same way; the measured BF16
    # peaks scaled by that ratio are the TF32 burst / sustained peaks.
    tf32 = all(w.ab_dtype == workloads.DT_F32 for w in ws)
    dscale, tf32_ctx = 1.0, None
    if tf32:
        tf32_ctx = cublas_dense_rates(("bf16", "tf32"))
        dscale = tf32_ctx["tf32_8192cubed_tflops"] / tf32_ctx["bf16_8192cubed_tflops"]
    peak = peak * dscale
    ws_names = [w.name for w in ws]
    if all(w.M <= 64 for w in ws):       # skinny: HBM-bound
        bound = "hbm"
        gbs = sum(w.algorithmic_bytes() for w in ws) / (sum(launch_ms) * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 4)}
    else:
        roof = {"bound": bound, "achieved": round(achieved, 1), "peak": peak, "unit": "TFLOP/s",
                "frac": round(achieved / peak, 4),
                "peak_kind": "sustained (timed region %.0f ms at the power cap)" % ms_total
                if long_region else "burst",
                "frac_of_burst": round(achieved / (peaks["bf16_tflops"] * dscale), 4),
                "frac_of_sustained": round(achieved / (peaks["bf16_tflops_sustained"] * dscale), 4)}
        if tf32:
            roof["peak_kind"] += ("; TF32 = measured BF16 x %.4f, the cuBLAS TF32 / BF16 8192^3 "
                                  "rate ratio measured in this run" % dscale)
            roof["tf32_context"] = tf32_ctx
    traffic = [committed_traffic(n) for n in ws_names]
    roof["traffic"] = (sum(traffic) / len(traffic)) if all(t is not None for t in traffic) else None
    roof["peak_source"] = f"{peak_src} ({'MEASURED_PEAKS.json' if peak_src == 'measured' else 'recipe fallback'})"
    roof["kernel"] = "gemm_tc_kernel" + (" (+ ln_rows_stats_kernel in the LayerNorm call)"
                                         if any(ln_rows) else "")
    roof["launch_ms"] = [round(x, 4) for x in launch_ms]
    roof["launch_ms_source"] = launch_src
    roof["per_launch_tflops"] = [round(w.flops() / (t * 1e-3) / 1e12, 1)
                                 for w, t in zip(ws, launch_ms)]
    roof["per_shape_events_ms"] = [round(x, 4) for x in shape_ms]

    # e2e: host buffers through the C ABI; copies inside the timed region
    e2e = run_e2e(lib, g, bufs, stream, args, world, launch)

    # Default line only: the same step at the power cap, the skinny decode
    # GEMM against the HBM roofline, and cuBLAS denominators as context.
    extra = {}
    if args.workload == "transformer_layer" and not fused and not args.no_extra:
        peaks_m, _ = load_peaks()
        extra["sustained"] = run_sustained(step, stream, ms_step, flops_step, peaks_m, local,
                                           world, launches_per_step)
        extra["skinny"] = run_skinny_leg(lib, g, local, world, peaks_m)
        extra["context"] = run_context(bufs, local, peaks_m)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        smp = OracleSampler(ws)
        n = smp.calibrate(12.0)
        f, t = smp.run(n)
        rows = smp.calibrate_rows(8.0)
        fr, tr = smp.run_rows(rows)
        cpu = {"value": round(f / t / 1e12, 6), "unit": "TFLOP/s", "cores": smp.threads,
               "kind": "oracle",
               "sample": f"{n} seeded output elements of each GEMM of the step, each a full "
                         f"K-long dot product: {f / 1e9:.2f} GFLOP in {t:.1f} s" + (
                             " (the fused epilogue's per-element work is not in the sample)"
                             if fused else ""),
               "full_matrix_entry_point": {
                   "value": round(fr / tr / 1e12, 6), "unit": "TFLOP/s",
                   "sample": f"first {rows} rows of each GEMM (decode once, then the triple "
                             f"loop): {fr / 1e9:.1f} GFLOP in {tr:.1f} s"}}

    out = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "tf32" if tf32 else ("f16" if all(w.ab_dtype == workloads.DT_F16 for w in ws)
                                      else "bf16"),
        "data": "synthetic",
        "config": {"workload": describe(args.workload, ws) + (
                       "; fused epilogues: bias, bias + GELU, bias + residual (beta = 1) + "
                       "LayerNorm over the 4096 columns (BF16 gamma, shift; eps 1e-5)"
                       if args.layernorm else
                       "; fused epilogues: bias, bias + GELU, bias + residual (beta = 1)"
                       if args.epilogue else ""), "shapes": ws_names,
                   "l2": "no flush: each step touches "
                         f"{sum(w.algorithmic_bytes() for w in ws) / 1e9:.2f} GB > 129 MB L2",
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "paths": [p["path_name"] for p in plans]},
        "roofline": roof, "e2e": e2e, "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
    }
    out.update(extra)
    if cpu is not None:
        out["cpu_baseline"] = cpu
    g.close()
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def timed_region(fn, n, stream, local, world):
    """n back-to-back calls of fn() between two events on `stream`, with a
    barrier + synchronize on both sides and nvidia-smi clocks sampled
    meanwhile.  Returns (ms over the region, max over ranks; clocks)."""
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    w0 = time.time()
    e0.record(stream)
    for _ in range(n):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    w1 = time.time()
    clk = clocks.stop((w0, w1))
    barrier(world)
    return max_over_ranks(e0.elapsed_time(e1), world), clk


def run_sustained(step, stream, ms_step, flops_step, peaks, local, world, launches_per_step):
    """The layer step back to back for about two seconds: long enough to run
    at the power cap, so the measured sustained cuBLAS figure is the matching
    denominator."""
    n = max(50, int(2000.0 / max(ms_step, 1e-3)))
    ms, clk = timed_region(step, n, stream, local, world)
    value = world * flops_step * n / (ms * 1e-3) / 1e12
    peak = peaks["bf16_tflops_sustained"]
    return {"value": round(value, 2), "unit": "TFLOP/s", "steps": n, "region_ms": round(ms, 1),
            "ms_per_step": round(ms / n, 4), "peak": peak,
            "peak_kind": "sustained (bf16_tflops_sustained, cuBLAS back to back at the power cap)",
            "frac": round(value / world / peak, 4), "gpu_launches": launches_per_step * n,
            "clocks": clk}


def run_skinny_leg(lib, g, local, world, peaks, calls=200, warmup=20):
    """The skinny decode GEMM (64 x 16384 x 8192 FP16, weights stored N x K)
    through gemm_run, back to back: bytes moved (A + B read once, C written
    once) per second against the measured HBM copy bandwidth.  The 268 MB of
    weights exceed the 129 MB L2, so each call streams them from HBM."""
    w = workloads.WORKLOADS["skinny_64x16384x8192_f16"]
    inp = workloads.make_inputs(w)
    A, B = inp.A.cuda(), inp.B.cuda()
    C = torch.zeros((w.M, inp.ldc), dtype=workloads.TORCH_DTYPE[w.c_dtype], device="cuda")
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream
    dts = (w.ab_dtype, w.ab_dtype, w.c_dtype)

    def call():
        st = lib.gemm_run(g.h, w.transA, w.transB, w.M, w.N, w.K, w.alpha, A.data_ptr(), inp.lda,
                          B.data_ptr(), inp.ldb, w.beta, C.data_ptr(), inp.ldc, dts, sh)
        if st != 0:
            raise lib.GemmError(st, "gemm_run")

    for _ in range(warmup):
        call()
    g.sync()
    ms, clk = timed_region(call, calls, stream, local, world)
    g.sync()
    us = ms * 1e3 / calls
    gbs = w.algorithmic_bytes() / (us * 1e-6) / 1e9
    st, plan = lib.gemm_plan_query(w.transA, w.transB, w.M, w.N, w.K, w.alpha, A.data_ptr(),
                                   inp.lda, B.data_ptr(), inp.ldb, w.beta, C.data_ptr(), inp.ldc,
                                   dts, num_sms=torch.cuda.get_device_properties(local)
                                   .multi_processor_count)
    return {"workload": f"{w.name}: {w.M}x{w.N}x{w.K} {w.transA}{w.transB}, X N(0,1), "
                        "W N(0,0.02) stored N x K, FP16 in, FP32 accumulate, FP16 out",
            "bound": "hbm", "achieved": round(gbs * world, 1), "unit": "GB/s",
            "peak": peaks["hbm_gbs"], "frac": round(gbs / peaks["hbm_gbs"], 4),
            "us_per_call": round(us, 2), "tflops": round(world * w.flops() / (us * 1e-6) / 1e12, 1),
            "calls": calls, "path": plan["path_name"] if st == 0 else None,
            "bytes_per_call": w.algorithmic_bytes(), "gpu_launches": calls, "clocks": clk}


def best_ms(fn, reps=10):
    """Best of `reps` calls of fn() timed one by one with CUDA events."""
    fn()
    torch.cuda.synchronize()
    best = float("inf")
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1))
    return best


def cublas_dense_rates(kinds=("bf16", "f16", "tf32"), n=8192, reps=10):
    """cuBLAS (torch.matmul) n^3 GEMM rates on this GPU, burst (best of
    `reps`): BF16, FP16, and FP32 with TF32 allowed."""
    gen = torch.Generator(device="cuda").manual_seed(0)
    dts = {"bf16": torch.bfloat16, "f16": torch.float16, "tf32": torch.float32}
    out = {"source": "torch.matmul (cuBLAS), best of %d, burst" % reps}
    tf32_prev = torch.backends.cuda.matmul.allow_tf32
    try:
        for name in kinds:
            a = torch.randn((n, n), device="cuda", generator=gen).to(dts[name])
            b = torch.randn((n, n), device="cuda", generator=gen).to(dts[name])
            torch.backends.cuda.matmul.allow_tf32 = (name == "tf32")
            ms = best_ms(lambda: torch.matmul(a, b), reps)
            out[f"{name}_8192cubed_tflops"] = round(2.0 * n ** 3 / (ms * 1e-3) / 1e12, 1)
            del a, b
    finally:
        torch.backends.cuda.matmul.allow_tf32 = tf32_prev
    return out


def run_context(bufs, local, peaks, reps=10):
    """cuBLAS (torch.matmul) timings on this GPU, for context only: the dense
    8192^3 rates of BF16, FP16 and FP32 with TF32 allowed (best of `reps`
    calls, burst), and the step's three layer shapes in BF16."""
    out = cublas_dense_rates(reps=reps)
    b16 = out["bf16_8192cubed_tflops"]
    out["f16_over_bf16"] = round(out["f16_8192cubed_tflops"] / b16, 4)
    out["tf32_over_bf16"] = round(out["tf32_8192cubed_tflops"] / b16, 4)
    out["bf16_tflops_measured_peak"] = peaks.get("bf16_tflops")
    shapes = {}
    for (w, inp, A, B, C) in bufs:
        x, wt = A[:, :w.K], B[:, :w.K]
        ms = best_ms(lambda: torch.matmul(x, wt.t()), reps)
        shapes[w.name] = {"cublas_us": round(ms * 1e3, 1),
                          "cublas_tflops": round(w.flops() / (ms * 1e-3) / 1e12, 1)}
    out["layer_shapes"] = shapes
    return out


def run_e2e(lib, g, bufs, stream, args, world, launch):
    """Same step with inputs in pinned host memory: H2D copies, the GEMMs,
    D2H of every output, all inside the timed region.  Three streams pipeline
    the step: the inputs of GEMM i+1 go up and the output of GEMM i-1 comes
    back while GEMM i runs; events order the reuse of each device buffer
    across steps (A and B are refilled only after the GEMM that read them, C
    -- when beta != 0 uploads it -- only after its copy-back, and a GEMM
    overwrites C only after the previous step's copy-back of it)."""
    host = []
    h2d = d2h = 0
    for (w, inp, A, B, C) in bufs:
        hA, hB = inp.A.pin_memory(), inp.B.pin_memory()
        hC = torch.empty(C.shape, dtype=C.dtype).pin_memory()
        hCin = C.cpu().pin_memory() if w.beta != 0 else None
        host.append((hA, hB, hC, hCin))
        h2d += hA.numel() * hA.element_size() + hB.numel() * hB.element_size()
        if hCin is not None:
            h2d += hCin.numel() * hCin.element_size()
        d2h += hC.numel() * hC.element_size()
    s_up, s_mm, s_down = torch.cuda.Stream(), stream, torch.cuda.Stream()
    n = len(bufs)
    ev_in = [torch.cuda.Event() for _ in range(n)]      # inputs of GEMM i on the device
    ev_mm = [torch.cuda.Event() for _ in range(n)]      # GEMM i finished
    ev_out = [torch.cuda.Event() for _ in range(n)]     # C_i copied back
    for e in ev_mm + ev_out:
        e.record(s_mm)

    def step():
        for i, ((w, inp, A, B, C), (hA, hB, hC, hCin)) in enumerate(zip(bufs, host)):
            s_up.wait_event(ev_mm[i])           # previous step's GEMM i has read A, B (and C)
            if hCin is not None:
                s_up.wait_event(ev_out[i])      # C_i is refilled only once it has been copied back
            with torch.cuda.stream(s_up):
                A.copy_(hA, non_blocking=True)
                B.copy_(hB, non_blocking=True)
                if hCin is not None:
                    C.copy_(hCin, non_blocking=True)
            ev_in[i].record(s_up)
            s_mm.wait_event(ev_in[i])
            s_mm.wait_event(ev_out[i])
            launch(i, A, B, C, s_mm.cuda_stream)
            ev_mm[i].record(s_mm)
            s_down.wait_event(ev_mm[i])
            with torch.cuda.stream(s_down):
                hC.copy_(C, non_blocking=True)
            ev_out[i].record(s_down)

    for _ in range(min(args.warmup, 3)):
        step()
    steps = max(3, min(args.steps, 20))
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_up)
    for _ in range(steps):
        step()
    s_up.wait_event(ev_out[-1])
    for e in ev_out:
        s_up.wait_event(e)
    e1.record(s_up)
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1), world)
    flops = sum(w.flops() for (w, *_rest) in bufs)
    return {"value": round(world * flops * steps / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "ms_per_step": round(ms / steps, 4),
            "h2d_d2h_gbs": round((h2d + d2h) * steps / (ms * 1e-3) / 1e9, 1)}


# ------------------------------------------------------------------ softmax

def softmax_inputs(name):
    w = workloads.SOFTMAX_WORKLOADS[name]
    return w, workloads.make_softmax_input(w)


class SoftmaxOracleSampler:
    """Times the CPU oracle's softmax on seeded rows of the workload."""

    def __init__(self, w, Xs):
        import oracle
        self.o = oracle.get()
        self.w, self.Xs = w, Xs
        self.codes = workloads.as_codes(Xs)
        self.threads = self.o.max_threads()
        self.rng = __import__("numpy").random.default_rng(0)

    def run(self, nrows):
        ids = self.rng.integers(0, self.w.rows, nrows)
        ldx, _ = self.w.lds()
        t0 = time.perf_counter()
        self.o.softmax(self.codes, self.w.rows, self.w.cols, ldx, self.w.x_dtype, row_ids=ids)
        t = time.perf_counter() - t0
        ex = 4 if self.w.x_dtype == workloads.DT_F32 else 2
        ey = 4 if self.w.y_dtype == workloads.DT_F32 else 2
        return nrows * self.w.cols * (ex + ey), t

    def calibrate(self, seconds):
        n = 1
        while True:
            _, t = self.run(n)
            if t > seconds / 8 or n >= self.w.rows:
                break
            n = min(self.w.rows, n * 4)
        _, t = self.run(n)
        return max(1, min(self.w.rows * 4, int(n * seconds / max(t, 1e-6))))


def run_softmax(args):
    import mixed_precision_dense_sm_gb300 as lib
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    w, Xs = softmax_inputs(args.workload)
    ldx, ldy = w.lds()
    X = Xs.cuda()
    Y = torch.empty((w.rows, ldy), dtype=workloads.TORCH_DTYPE[w.y_dtype], device="cuda")
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream
    sms = torch.cuda.get_device_properties(local).multi_processor_count
    st, plan = lib.softmax_plan_query(w.rows, w.cols, X.data_ptr(), ldx, w.x_dtype, Y.data_ptr(),
                                      ldy, w.y_dtype, num_sms=sms)
    assert st == 0
    nbytes = w.algorithmic_bytes()

    def step(Xd=X, Yd=Y, s=sh):
        st = lib.softmax_rows(w.rows, w.cols, Xd.data_ptr(), ldx, w.x_dtype, Yd.data_ptr(), ldy,
                              w.y_dtype, s)
        if st != 0:
            raise lib.GemmError(st, "softmax_rows")

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    w0 = time.time()
    t_start.record(stream)
    for _ in range(args.steps):
        step()
    t_end.record(stream)
    torch.cuda.synchronize()
    w1 = time.time()
    clk = clocks.stop((w0, w1))
    barrier(world)
    ms = max_over_ranks(t_start.elapsed_time(t_end), world)
    ms_step = ms / args.steps
    value = world * nbytes * args.steps / (ms * 1e-3) / 1e9
    peaks, peak_src = load_peaks()
    # one kernel launch per step: the average launch is the timed region / steps
    achieved = nbytes / (ms_step * 1e-3) / 1e9
    roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
            "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
            "traffic": committed_traffic(w.name, SOFTMAX_SOURCES),
            "peak_source": f"{peak_src} ({'MEASURED_PEAKS.json' if peak_src == 'measured' else 'recipe fallback'})",
            "kernel": "softmax_kernel", "launch_ms": round(ms_step, 4),
            "launch_ms_source": "timed region / launches (events at the region's ends only)",
            "algorithmic_bytes_per_launch": nbytes, "plan_hbm_bytes": plan["hbm_bytes"]}

    # e2e: X up from pinned host memory, the softmax, Y back, every step
    hX = Xs.pin_memory()
    hY = torch.empty(Y.shape, dtype=Y.dtype).pin_memory()
    e_steps = max(3, min(args.steps, 20))
    for _ in range(2):
        X.copy_(hX, non_blocking=True)
        step()
        hY.copy_(Y, non_blocking=True)
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e_steps):
        X.copy_(hX, non_blocking=True)
        step()
        hY.copy_(Y, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    ems = max_over_ranks(e0.elapsed_time(e1), world)
    h2d = hX.numel() * hX.element_size()
    d2h = hY.numel() * hY.element_size()
    e2e = {"value": round(world * nbytes * e_steps / (ems * 1e-3) / 1e9, 1), "unit": "GB/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e_steps,
           "ms_per_step": round(ems / e_steps, 4)}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        smp = SoftmaxOracleSampler(w, Xs)
        n = smp.calibrate(10.0)
        b, t = smp.run(n)
        cpu = {"value": round(b / t / 1e9, 4), "unit": "GB/s", "cores": smp.threads,
               "kind": "oracle",
               "sample": f"{n} seeded rows of {w.cols} elements (binary64 max, exp, sum, "
                         f"divide): {b / 1e9:.3f} GB of X + Y in {t:.1f} s"}
    out = {
        "metric": SOFTMAX_METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": workloads.DT_NAME[w.x_dtype], "data": "synthetic",
        "config": {"workload": f"{w.name}: row softmax of {w.rows} x {w.cols} "
                               f"{workloads.DT_NAME[w.x_dtype]} -> {workloads.DT_NAME[w.y_dtype]}, "
                               f"logits {w.dist}" + (f", {w.mask} mask" if w.mask else ""),
                   "plan": plan,
                   "l2": f"no flush: each step touches {nbytes / 1e9:.2f} GB > 129 MB L2"
                         if nbytes > 2.6e8 else "each step touches less than 2x the L2",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": roof, "e2e": e2e, "gpu_launches": args.steps, "clocks": clk,
    }
    if cpu is not None:
        out["cpu_baseline"] = cpu
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_softmax_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    w, Xs = softmax_inputs(args.workload)
    smp = SoftmaxOracleSampler(w, Xs)
    per_step = max(0.05, min(5.0, 150.0 / max(1, args.steps + args.warmup)))
    n = smp.calibrate(per_step)
    times, b = [], 0
    for k in range(args.warmup + args.steps):
        b, t = smp.run(n)
        if k >= args.warmup:
            times.append(t)
    t = sum(times)
    value = b * len(times) / t / 1e9
    sample = f"{n} seeded rows of {w.cols} elements per step ({b / 1e9:.4f} GB of X + Y)"
    out = {"metric": SOFTMAX_METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(1e3 * t / len(times), 2), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "impl": "reference", "config": {"workload": w.name},
           "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": smp.threads,
                            "kind": "oracle", "sample": sample},
           "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


# -------------------------------------------------------------- convolution

class ConvOracleSampler:
    """Times the CPU oracle's convolution at seeded output pixels."""

    def __init__(self, w, x, wt):
        import numpy as np
        import oracle
        self.o = oracle.get()
        self.w = w
        self.xc, self.wc = workloads.as_codes(x), workloads.as_codes(wt)
        self.threads = self.o.max_threads()
        self.rng = np.random.default_rng(0)
        M, _, _ = w.gemm_mnk()
        self.M = M

    def run(self, n):
        w = self.w
        rows = self.rng.integers(0, self.M, n)
        t0 = time.perf_counter()
        self.o.conv2d_sampled(w.N, w.H, w.W, w.C, w.K, w.R, w.S, w.pad[0], w.pad[1], w.stride[0],
                              w.stride[1], w.dil[0], w.dil[1], 1.0, self.xc, self.wc, 0.0, None,
                              w.x_dtype, w.y_dtype, rows)
        t = time.perf_counter() - t0
        _, N, K = w.gemm_mnk()
        return 2.0 * n * N * K, t

    def calibrate(self, seconds):
        n = 8
        while True:
            _, t = self.run(n)
            if t > seconds / 8 or n >= self.M:
                break
            n = min(self.M, n * 4)
        _, t = self.run(n)
        return max(1, int(n * seconds / max(t, 1e-6)))


def run_conv(args):
    import mixed_precision_dense_sm_gb300 as lib
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    w = workloads.CONV_WORKLOADS[args.workload]
    x, wt = workloads.make_conv_inputs(w)
    M, Ng, Kg = w.gemm_mnk()
    X, Wd = x.cuda(), wt.cuda()
    Y = torch.empty((M, w.K), dtype=workloads.TORCH_DTYPE[w.y_dtype], device="cuda")
    g = lib.Gemm()
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream
    dts = (w.x_dtype, w.x_dtype, w.y_dtype)
    sms = torch.cuda.get_device_properties(local).multi_processor_count
    st, plan = lib.conv2d_plan_query(w.N, w.H, w.W, w.C, w.K, w.R, w.S, w.pad, w.stride, w.dil,
                                     1.0, X.data_ptr(), Wd.data_ptr(), 0.0, Y.data_ptr(), dts,
                                     num_sms=sms)
    assert st == 0

    def step(Xd=X, Wdd=Wd, Yd=Y, s=sh):
        st = lib.conv2d_fprop(g.h, w.N, w.H, w.W, w.C, w.K, w.R, w.S, w.pad, w.stride, w.dil, 1.0,
                              Xd.data_ptr(), Wdd.data_ptr(), 0.0, Yd.data_ptr(), dts, stream=s)
        if st != 0:
            raise lib.GemmError(st, "conv2d_fprop")

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    for _ in range(args.warmup):
        step()
    g.sync()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    w0 = time.time()
    t_start.record(stream)
    for _ in range(args.steps):
        step()
    t_end.record(stream)
    torch.cuda.synchronize()
    w1 = time.time()
    clk = clocks.stop((w0, w1))
    barrier(world)
    g.sync()
    ms = max_over_ranks(t_start.elapsed_time(t_end), world)
    ms_step = ms / args.steps
    value = world * w.flops() * args.steps / (ms * 1e-3) / 1e12
    peaks, peak_src = load_peaks()
    long_region = ms > 500.0
    peak = peaks["bf16_tflops_sustained"] if long_region else peaks["bf16_tflops"]
    achieved = w.flops() / (ms_step * 1e-3) / 1e12
    roof = {"bound": "tensor", "achieved": round(achieved, 1), "peak": peak, "unit": "TFLOP/s",
            "frac": round(achieved / peak, 4),
            "peak_kind": "sustained (timed region %.0f ms at the power cap)" % ms if long_region
            else "burst",
            "traffic": committed_traffic(w.name),
            "peak_source": f"{peak_src} ({'MEASURED_PEAKS.json' if peak_src == 'measured' else 'recipe fallback'})",
            "kernel": "gemm_tc_kernel (im2col A operand)", "launch_ms": round(ms_step, 4),
            "launch_ms_source": "timed region / launches (events at the region's ends only)"}
    # e2e: X and Wt up from pinned host memory, the convolution, Y back
    hX, hW = x.pin_memory(), wt.pin_memory()
    hY = torch.empty(Y.shape, dtype=Y.dtype).pin_memory()
    e_steps = max(3, min(args.steps, 20))
    for _ in range(2):
        X.copy_(hX, non_blocking=True)
        Wd.copy_(hW, non_blocking=True)
        step()
        hY.copy_(Y, non_blocking=True)
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e_steps):
        X.copy_(hX, non_blocking=True)
        Wd.copy_(hW, non_blocking=True)
        step()
        hY.copy_(Y, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    ems = max_over_ranks(e0.elapsed_time(e1), world)
    e2e = {"value": round(world * w.flops() * e_steps / (ems * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
           "h2d_bytes_per_step": hX.numel() * hX.element_size() + hW.numel() * hW.element_size(),
           "d2h_bytes_per_step": hY.numel() * hY.element_size(), "steps": e_steps,
           "ms_per_step": round(ems / e_steps, 4)}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        smp = ConvOracleSampler(w, x, wt)
        n = smp.calibrate(10.0)
        f, t = smp.run(n)
        cpu = {"value": round(f / t / 1e12, 6), "unit": "TFLOP/s", "cores": smp.threads,
               "kind": "oracle",
               "sample": f"{n} seeded output pixels, all {w.K} channels, each a full "
                         f"{Kg}-term sum: {f / 1e9:.2f} GFLOP in {t:.1f} s"}
    P, Q = w.out_hw()
    out = {
        "metric": CONV_METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": workloads.DT_NAME[w.x_dtype], "data": "synthetic",
        "config": {"workload": f"{w.name}: N={w.N} H={w.H} W={w.W} C={w.C} K={w.K} R={w.R} "
                               f"S={w.S} pad={w.pad} stride={w.stride} dilation={w.dil} -> "
                               f"P={P} Q={Q}; GEMM {M} x {Ng} x {Kg}",
                   "plan": plan, "parallelism": "replicas" if world > 1 else "single GPU",
                   "l2": "no flush between steps"},
        "roofline": roof, "e2e": e2e, "gpu_launches": args.steps, "clocks": clk,
    }
    if cpu is not None:
        out["cpu_baseline"] = cpu
    if rank == 0:
        print(json.dumps(out), flush=True)
    g.close()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_conv_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    w = workloads.CONV_WORKLOADS[args.workload]
    x, wt = workloads.make_conv_inputs(w)
    smp = ConvOracleSampler(w, x, wt)
    per_step = max(0.05, min(5.0, 150.0 / max(1, args.steps + args.warmup)))
    n = smp.calibrate(per_step)
    times, f = [], 0.0
    for k in range(args.warmup + args.steps):
        f, t = smp.run(n)
        if k >= args.warmup:
            times.append(t)
    t = sum(times)
    value = f * len(times) / t / 1e12
    out = {"metric": CONV_METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(1e3 * t / len(times), 2), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "impl": "reference", "config": {"workload": w.name},
           "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": smp.threads,
                            "kind": "oracle",
                            "sample": f"{n} seeded output pixels per step ({f / 1e9:.3f} GFLOP)"},
           "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


# ------------------------------------------------------------ reference arm

def run_reference(args):
    """The comparison arm: the CPU oracle, timed on the host cores.  Each step
    is a bounded sample of the step's GEMMs, sized so that the whole run of
    warm-up and timed steps takes about two and a half minutes."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    ws = workload_list(args.workload)
    smp = OracleSampler(ws)
    per_step = max(0.05, min(5.0, 150.0 / max(1, args.steps + args.warmup)))
    n = smp.calibrate(per_step)
    times, f = [], 0.0
    for k in range(args.warmup + args.steps):
        f, t = smp.run(n)
        if k >= args.warmup:
            times.append(t)
    t = sum(times)
    value = f * len(times) / t / 1e12
    sample = (f"{n} seeded output elements of each GEMM of the step per step, each a full "
              f"K-long dot product ({f / 1e9:.3f} GFLOP per step)")
    out = {"metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(1e3 * t / len(times), 2), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "impl": "reference",
           "config": {"workload": describe(args.workload, ws), "shapes": [w.name for w in ws]},
           "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": smp.threads,
                            "kind": "oracle", "sample": sample},
           "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=800)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="transformer_layer",
                    choices=["transformer_layer"] + list(workloads.WORKLOADS) +
                    list(workloads.SOFTMAX_WORKLOADS) + list(workloads.CONV_WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the sustained, skinny and cuBLAS-context legs of the default line")
    ap.add_argument("--epilogue", action="store_true",
                    help="fused epilogues of a transformer MLP block: bias on every GEMM, "
                         "GELU after the up-projection, residual add after the down-projection")
    ap.add_argument("--layernorm", action="store_true",
                    help="as --epilogue, with LayerNorm after the down-projection's residual "
                         "add (a post-LN transformer block)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        ap.error("--warmup must be >= 3")
    softmax = args.workload in workloads.SOFTMAX_WORKLOADS
    conv = args.workload in workloads.CONV_WORKLOADS
    if (softmax or conv) and (args.epilogue or args.layernorm):
        ap.error("--epilogue / --layernorm apply to the transformer_layer workload")
    if args.impl == "reference":
        (run_softmax_reference if softmax else run_conv_reference if conv else run_reference)(args)
    else:
        (run_softmax if softmax else run_conv if conv else run_ours)(args)


if __name__ == "__main__":
    main()
