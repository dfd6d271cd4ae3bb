#!/usr/bin/env python
"""Benchmark of the FP8 block-scaled GEMM hot path on GB300.

One step = the whole hot path over one batch of the dense prefill workload:
for each of the two prefill shapes (M, N, K) = (4096, 7168, 16384) and
(4096, 4096, 4096): quantise the FP32 activations per 1x128 tile
(fp8_quant_1x128) and run the block-scaled GEMM (fp8gemm_dense) against
weights quantised per 128x128 tile beforehand (the offline step, untimed).
Inputs are synthetic (A ~ N(0,1) with 1 % outlier columns x50, B ~ N(0,0.02)),
drawn and kept on the device; L2 is flushed before every timed step (a
256 MB write, then a 256 MB read so that no dirty line of the flush is
written back inside the timed interval); each step is timed with CUDA events
on the launching stream, with no event between its kernels (an event there
would end a kernel's programmatic overlap with the one before it); the
roofline kernel is timed in a second pass of the same steps.  With
`--gemm-form batch` the two GEMMs run as one fp8gemm_dense_batch launch; the
form not chosen is timed as whole steps under `configs`.

Printed: one JSON line (rank 0).  `value` is TFLOP/s over all ranks;
`roofline` describes the GEMM kernel; `e2e` repeats the step through the
public API with host (pinned) inputs and outputs, copies included;
`cpu_baseline` times the CPU oracle on a bounded sample; `configs` adds
measurements of the other workloads (correctness case, decode shapes, MoE
contiguous and masked, the quantiser) against their own rooflines.

`--impl reference` times the CPU oracle as the reference arm instead.
Multi-GPU (torchrun): every rank runs the same workload on its own GPU
(replicas; no collective on the data path).
"""

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

PREFILL_SHAPES = [(4096, 7168, 16384), (4096, 4096, 4096)]
METRIC = "FP8 block-scaled GEMM TFLOPS & GB/s, % of GB300 roofline (dense/grouped)"
UNIT = "TFLOP/s"
WORKLOAD = ("dense prefill FP8 e4m3 GEMM, 1x128 A / 128x128 B FP32 scales, BF16 out: "
            "quantise A + GEMM for (M,N,K) = (4096,7168,16384) and (4096,4096,4096)")
FLUSH_BYTES = 256 << 20


class L2Flush:
    """Evicts the 129 MB L2 between timed intervals: writes one buffer twice
    the L2's size, then reads another.  The read leaves L2 holding clean lines
    of that buffer only, so the timed kernel neither hits on its inputs nor
    pays for writing back the flush's dirty lines (up to 14.5 us on an
    HBM-bound kernel of about 100 us)."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.r = torch.ones(FLUSH_BYTES // 8, dtype=torch.int64, device=dev)
        self.out = torch.empty((), dtype=torch.int64, device=dev)

    def __call__(self, i):
        import torch
        self.w.fill_(i & 0xFF)
        torch.sum(self.r, dim=0, out=self.out)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16": p["bf16_tflops"],
                "bf16_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16": 1900.0, "bf16_sustained": 1700.0, "source": "fallback"}


def fp8_peak(peaks, sustained=True):
    # FP8 dense tensor rate = 2 x BF16 (nominal 4.5 vs 2.25 PFLOP/s)
    return 2.0 * (peaks["bf16_sustained"] if sustained else peaks["bf16"])


# ----------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples (every 10 ms) of SM clock, power and throttle
    reasons.  `window(t0, t1)` marks the timed interval (host epoch seconds);
    the summary is taken over the samples stamped inside it, or over all of
    them when none fell inside (a very short interval)."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.file = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "10"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def window(self, t0, t1):
        self.t0, self.t1 = t0, t1

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        text = self.file.read()
        self.file.close()
        os.unlink(self.file.name)
        out = self.summarise(text, self.t0, self.t1)
        out["source"] = "nvidia-smi, 10 ms"
        return out

    @classmethod
    def summarise(cls, text, t0=None, t1=None):
        """Median SM clock, max clock and active reasons of the CSV rows in
        [t0, t1] (every row when t0 is None or no row falls inside)."""
        from datetime import datetime
        rows = []
        for line in text.splitlines():
            r = [x.strip() for x in line.split(",")]
            try:
                ts = datetime.strptime(r[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(r[2]), float(r[3]),
                             [name for name, v in zip(cls.REASONS, r[6:10])
                              if v.lower() == "active"]))
            except (ValueError, IndexError):
                continue
        return summarise_clock_rows(rows, t0, t1)


def summarise_clock_rows(rows, t0=None, t1=None):
    """rows: (host epoch s, SM MHz, max SM MHz, [active reason names]).
    Median SM clock, max clock and reasons of the rows in [t0, t1] (every row
    when t0 is None or no row falls inside)."""
    inside = [x for x in rows if t0 is not None and t0 <= x[0] <= t1]
    use = inside or rows
    reasons = set()
    for _, _, _, names in use:
        reasons.update(names)
    return {"sm_mhz": statistics.median(x[1] for x in use) if use else None,
            "sm_max_mhz": max(x[2] for x in use) if use else None,
            "samples": len(inside), "samples_total": len(rows),
            "window_ms": round((t1 - t0) * 1e3, 1) if t0 is not None else None,
            "reasons": sorted(reasons)}


class NvmlClockSampler:
    """The same record read from NVML (the driver's management library,
    read-only queries) by a host thread every millisecond, so that even a
    timed interval of a few milliseconds holds several samples.  start()
    returns False where the library cannot be loaded (the caller then uses
    ClockSampler)."""
    BITS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown",
            0x4: "sw_power_cap"}

    def __init__(self, gpu_index, period_s=0.001):
        self.gpu = gpu_index
        self.period = period_s
        self.rows = []
        self.t0 = self.t1 = None
        self._stop = None
        self._thread = None

    def start(self):
        import ctypes
        import threading
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return False
            h = ctypes.c_void_p()
            if nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.gpu), ctypes.byref(h)) != 0:
                return False
            reasons_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, ctypes.c_int(1), ctypes.byref(mx)) != 0:
                return False
        except (OSError, AttributeError):
            return False
        self._nv, self._h, self._reasons_fn, self._max = nv, h, reasons_fn, float(mx.value)
        self._stop = threading.Event()
        self._thread = threading.Thread(target=self._run, daemon=True)
        self._thread.start()
        return True

    def _run(self):
        import ctypes
        clk, bits = ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop.is_set():
            t = time.time()
            if (self._nv.nvmlDeviceGetClockInfo(self._h, ctypes.c_int(1), ctypes.byref(clk)) == 0 and
                    self._reasons_fn(self._h, ctypes.byref(bits)) == 0):
                names = [n for b, n in self.BITS.items() if bits.value & b]
                self.rows.append((t, float(clk.value), self._max, names))
            time.sleep(self.period)

    def window(self, t0, t1):
        self.t0, self.t1 = t0, t1

    def stop(self):
        self._stop.set()
        self._thread.join(timeout=5)
        self._nv.nvmlShutdown()
        out = summarise_clock_rows(self.rows, self.t0, self.t1)
        out["source"] = "nvml, 1 ms"
        return out


# ------------------------------------------------------------- GPU arm
def max_over_ranks(x, world):
    """The slowest rank's value (replicas are timed separately; the job is as
    slow as its slowest GPU).  Works on NCCL (CUDA tensor) and gloo (CPU)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_tflops(flops_per_rank_step, ms_per_step, world):
    """Whole-job throughput: every rank does the same step (weak scaling)."""
    return world * flops_per_rank_step / (ms_per_step * 1e-3) / 1e12


def gemm_bytes(M, N, K, e_active=1, rows=None):
    """Algorithmic bytes of one block-scaled GEMM: A and its scales for the
    real rows, B and its scales for the active experts, D for the real rows."""
    rows = M if rows is None else rows
    Kb = -(-K // 128)  # a partial last K block carries a scale too
    Nb = -(-N // 128)
    return rows * K + 4 * rows * Kb + e_active * (N * K + 4 * Nb * Kb) + 2 * rows * N


def run_gpu(args, rank, world):
    import torch

    from fp8_fine_grained_e4m3_gb300 import binding as b
    from fp8_fine_grained_e4m3_gb300 import synthetic

    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
    dev = torch.device("cuda", torch.cuda.current_device())
    peaks = load_peaks()
    stream = torch.cuda.current_stream()

    # ---- inputs resident in HBM; weights quantised once (offline step)
    cases = []
    for i, (M, N, K) in enumerate(PREFILL_SHAPES):
        X, W = synthetic.dense_operands_device(M, N, K, kind="prefill", seed=i, device=dev)
        B8, sB = b.fp8_quant_128x128(W)
        del W
        A8 = torch.empty((M, K), dtype=torch.uint8, device=dev)
        sA = torch.empty((M, K // 128), dtype=torch.float32, device=dev)
        D = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        cases.append(dict(M=M, N=N, K=K, X=X, A8=A8, sA=sA, B8=B8, sB=sB, D=D))
    flush = L2Flush(dev)
    flops_step = sum(2.0 * c["M"] * c["N"] * c["K"] for c in cases)

    batched = args.gemm_form == "batch"
    batch = [(c["A8"], c["sA"], c["B8"], c["sB"], c["D"]) for c in cases]

    def step(gemm_events=None, batched=batched):
        # both quantisers first: while they run, the host enqueues the GEMMs,
        # so the device never waits on the host inside a step.  Then the GEMMs:
        # by default one call per shape, the dominant one (cases[0]) last;
        # with --gemm-form batch, both shapes in one launch
        # (fp8gemm_dense_batch: the short tiles of 4096^3 fill the last round
        # of the long ones).  gemm_events (the roofline pass only) bracket the batched
        # launch, or the dominant single call: an event between two kernels
        # ends the programmatic overlap of the second with the first, which
        # is why the steps that give ms_per_step carry no such events
        for c in cases:
            b.fp8_quant_1x128(c["X"], Q=c["A8"], sX=c["sA"])
        if batched:
            if gemm_events is not None:
                gemm_events[0].record(stream)
            b.fp8gemm_dense_batch(batch)
            if gemm_events is not None:
                gemm_events[1].record(stream)
            return
        for c in cases[1:] + cases[:1]:
            timed = gemm_events is not None and c is cases[0]
            if timed:
                gemm_events[0].record(stream)
            b.fp8gemm_dense(c["A8"], c["sA"], c["B8"], c["sB"], D=c["D"])
            if timed:
                gemm_events[1].record(stream)

    for i in range(args.warmup):
        flush(i)
        step()
    torch.cuda.synchronize()
    if b.fp8gemm_get_device_status() != b.OK:
        raise RuntimeError("device status set during warm-up")

    K_steps = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K_steps)]
    gev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(K_steps)]
    gev_step = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(K_steps)]
    clocks = NvmlClockSampler(torch.cuda.current_device())
    if not clocks.start():
        clocks = ClockSampler(torch.cuda.current_device())
        clocks.start()
    time.sleep(0.3)
    launches0 = b.num_kernel_launches()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_begin = time.time()
    for i in range(K_steps):
        flush(i)  # L2 flush, outside the timed interval
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    clocks.window(t_begin, time.time())
    if world > 1:
        torch.distributed.barrier()
    launches = b.num_kernel_launches() - launches0
    # the roofline pass: the same K steps again, with events around the
    # dominant GEMM launch (they cost that launch its programmatic overlap
    # with the kernel before it; these steps' times are reported beside)
    for i in range(K_steps):
        flush(i)
        gev_step[i][0].record(stream)
        step(gev[i])
        gev_step[i][1].record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()  # summarised over the timed interval (the first pass)
    status = b.fp8gemm_get_device_status()
    if status != b.OK:
        raise RuntimeError(f"device status {status} after the timed region")

    step_ms = [s.elapsed_time(e) for s, e in ev]
    ms_per_step = sum(step_ms) / K_steps
    gemm_ms = sum(g[0].elapsed_time(g[1]) for g in gev) / K_steps  # the timed GEMM launch
    roof_step_ms = sum(g[0].elapsed_time(g[1]) for g in gev_step) / K_steps
    ms_per_step = max_over_ranks(ms_per_step, world)
    value = aggregate_tflops(flops_step, ms_per_step, world)

    # roofline of the dominant kernel: the tensor-core GEMM launch -- the
    # 4096x7168x16384 call (about 70 % of the step), or with --gemm-form
    # batch the launch that runs both prefill shapes (about 85 %)
    timed_shapes = PREFILL_SHAPES if batched else PREFILL_SHAPES[:1]
    gemm_flops = sum(2.0 * M * N * K for M, N, K in timed_shapes)
    achieved = gemm_flops / (gemm_ms * 1e-3) / 1e12
    # each step is short (sub-ms) and starts after an L2 flush at full clock:
    # the burst figure is the denominator; the sustained one is listed beside
    peak = fp8_peak(peaks, sustained=False)
    kernel = ("gemm_tc_kernel<BN=256, batched> (fp8gemm_dense_batch): 4096x7168x16384 and "
              "4096x4096x4096 in one launch" if batched else
              "gemm_tc_kernel<BN=256> (fp8gemm_dense, M > 64), M=4096 N=7168 K=16384")
    traffic_key = "gemm_tc_batch_prefill_pair" if batched else "gemm_tc_dense_4096x7168x16384"
    roofline = {"kernel": kernel,
                "bound": "tensor", "achieved": round(achieved, 1), "peak": round(peak, 1),
                "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                "peak_source": (f"{peaks['source']} bf16 burst x 2 (FP8/BF16 nominal ratio): "
                                "the kernel is timed in sub-ms steps after an L2 flush"),
                "frac_of_sustained_peak": round(achieved / fp8_peak(peaks, True), 4),
                "measured_fp8_tflops": measure_library_fp8(*PREFILL_SHAPES[0], flush),
                "traffic": traffic_from_profiles(traffic_key),
                "algorithmic_bytes": sum(gemm_bytes(*shp) for shp in timed_shapes),
                "gemm_us": round(1e3 * gemm_ms, 2),
                "timing": ("CUDA events around the GEMM launch in a second pass of the same "
                           f"{K_steps} steps (those steps: {roof_step_ms:.4f} ms each, against "
                           f"{ms_per_step:.4f} without the GEMM events)")}

    # ---- the other form of the step's GEMMs, whole steps only (no event
    # between its kernels, so every programmatic overlap stays), and that
    # form's GEMM launch(es) alone with L2 flushed
    other = None
    if not args.no_extras:
        other = measure_other_form(step, not batched, batch, cases, flush, flops_step, peaks,
                                   max(5, min(K_steps, 50)))

    # ---- end to end through the public API with host buffers
    e2e = measure_e2e(args, cases, flops_step, world)

    out = {"metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
           "steps": K_steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
           "dtype": "e4m3 (FP8 products, FP32 accumulate, BF16 out)", "data": "synthetic",
           "config": {"workload": WORKLOAD,
                      "l2": ("flushed before every timed step: a 256 MB device write, then a "
                             "256 MB read (no dirty flush lines written back while timed)"),
                      "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                      "gemm_form": ("both shapes in one fp8gemm_dense_batch launch" if batched
                                    else "one fp8gemm_dense call per shape"),
                      "timing": "CUDA events around each whole step on the launching stream"},
           "roofline": roofline, "e2e": e2e, "gpu_launches": int(launches),
           "clocks": clk, "impl": "gb300"}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(budget_s=args.cpu_seconds)
    if rank == 0 and not args.no_extras:
        for c in cases:
            del c["X"]
        del cases
        torch.cuda.empty_cache()
        out["configs"] = measure_configs(peaks, dev)
        out["configs"][other["name"]] = other
    return out


def measure_other_form(step, batched, batch, cases, flush, flops_step, peaks, n):
    """The prefill step with the GEMM form the main measurement did not use:
    mean time of n whole steps (L2 flushed before each, events around the
    step only), and the GEMM launch(es) of that form timed alone."""
    import torch

    from fp8_fine_grained_e4m3_gb300 import binding as b
    stream = torch.cuda.current_stream()
    for i in range(3):
        flush(i)
        step(batched=batched)
    ts = []
    for i in range(n):
        flush(i)
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        step(batched=batched)
        e.record(stream)
        e.synchronize()
        ts.append(s.elapsed_time(e))
    ms = sum(ts) / n
    if batched:
        gemm = lambda: b.fp8gemm_dense_batch(batch)  # noqa: E731
    else:
        def gemm():
            for c in cases:
                b.fp8gemm_dense(c["A8"], c["sA"], c["B8"], c["sB"], D=c["D"])
    g_ms = time_launch(gemm, flush)
    g_tflops = flops_step / (g_ms * 1e-3) / 1e12
    peak = fp8_peak(peaks, sustained=False)
    return {"name": "prefill_step_batched_gemm" if batched else "prefill_step_single_gemms",
            "ms_per_step": round(ms, 4), "tflops": round(flops_step / (ms * 1e-3) / 1e12, 1),
            "gemm_us": round(1e3 * g_ms, 2), "gemm_tflops": round(g_tflops, 1),
            "gemm_frac": round(g_tflops / peak, 4),
            "form": ("both shapes in one fp8gemm_dense_batch launch" if batched else
                     "one fp8gemm_dense call per shape"),
            "timing": "whole steps (quantisers + GEMMs), L2 flushed before each; the GEMMs "
                      "alone by time_launch"}


def gemm_parts(M, N, chunks, sms):
    """Row parts for an M x N output whose activations land in `chunks` row
    blocks: the most (a divisor of `chunks`) that still leave every part at
    least a wave of whole 128 x 256 tiles over `sms` SMs, else 1."""
    return max(p for p in range(1, chunks + 1)
               if p == 1 or (chunks % p == 0 and (M // p) // 128 * -(-N // 256) >= sms))


def measure_e2e(args, cases, flops_step, world, chunks=4):
    """The step through the public API with pinned host input and output,
    every copy inside the timed interval (CUDA events around the whole step):
    H2D of each shape's X in `chunks` row blocks on a copy stream, the 1x128
    quantiser on each block as soon as it has landed, the GEMM in row parts
    (each as soon as its rows are quantised; rows are independent, so D is the
    same as one call's), and the D2H of each part on a second copy stream --
    so copies overlap kernels and the two copy directions run at once.  A
    shape takes as many parts (dividing `chunks`) as still leave each part at
    least a wave of whole 128 x 256 tiles: a smaller part would take the
    split-tile form, whose K order, and so its rounding, differs from one
    call's.  Steps do not overlap: each ends when its last D2H has landed."""
    import torch

    from fp8_fine_grained_e4m3_gb300 import binding as b
    cur = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    hosts = []
    h2d = d2h = 0
    for c in cases:
        Xh = torch.empty(c["X"].shape, dtype=torch.float32, pin_memory=True)
        Xh.copy_(c["X"])
        Dh = torch.empty(c["D"].shape, dtype=torch.bfloat16, pin_memory=True)
        hosts.append((Xh, Dh))
        h2d += Xh.numel() * 4
        d2h += Dh.numel() * 2
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    n_parts = [gemm_parts(*c["D"].shape, chunks, sms) for c in cases]
    n = max(3, min(args.steps, 20))
    times = []
    for i in range(n + 2):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(cur)
        s_in.wait_event(s)
        s_out.wait_event(s)
        landed = []
        with torch.cuda.stream(s_in):
            for c, (Xh, _) in zip(cases, hosts):
                M = Xh.shape[0]
                evs = []
                for j in range(chunks):
                    r0, r1 = j * M // chunks, (j + 1) * M // chunks
                    c["X"][r0:r1].copy_(Xh[r0:r1], non_blocking=True)
                    ev = torch.cuda.Event()
                    ev.record(s_in)
                    evs.append((r0, r1, ev))
                landed.append(evs)
        last = None
        for c, (_, Dh), evs, parts in zip(cases, hosts, landed, n_parts):
            per = chunks // parts
            for q in range(parts):
                for r0, r1, ev in evs[q * per:(q + 1) * per]:
                    cur.wait_event(ev)
                    b.fp8_quant_1x128(c["X"][r0:r1], Q=c["A8"][r0:r1], sX=c["sA"][r0:r1])
                g0, g1 = evs[q * per][0], evs[(q + 1) * per - 1][1]
                b.fp8gemm_dense(c["A8"][g0:g1], c["sA"][g0:g1], c["B8"], c["sB"],
                                D=c["D"][g0:g1])
                done = torch.cuda.Event()
                done.record(cur)
                s_out.wait_event(done)
                with torch.cuda.stream(s_out):
                    Dh[g0:g1].copy_(c["D"][g0:g1], non_blocking=True)
                    last = torch.cuda.Event()
                    last.record(s_out)
        cur.wait_event(last)
        e.record(cur)
        e.synchronize()
        if i >= 2:
            times.append(s.elapsed_time(e))
    ms = sum(times) / len(times)
    # the result of the timed path equals one-call results
    ref = [(c["D"].clone()) for c in cases]
    for c, r in zip(cases, ref):
        b.fp8gemm_dense(c["A8"], c["sA"], c["B8"], c["sB"], D=c["D"])
        if not torch.equal(c["D"], r):
            raise RuntimeError("row-block GEMMs differ from the one-call result")
    return {"value": round(world * flops_step / (ms * 1e-3) / 1e12, 2), "unit": UNIT,
            "ms_per_step": round(ms, 3), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": n, "overlap": f"H2D in {chunks} row blocks per shape, quantiser per block, "
                                   f"GEMM in {'/'.join(map(str, n_parts))} row blocks, D2H of "
                                   "each on a second copy stream"}


def time_launch(fn, flush, n=20, warm=3):
    """Mean device time (ms) of fn() over n launches, L2 flushed before each."""
    import torch
    stream = torch.cuda.current_stream()
    for i in range(warm):
        fn()
    ts = []
    for i in range(n):
        flush(i)
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        fn()
        e.record(stream)
        ts.append((s, e))
    torch.cuda.synchronize()
    return sum(s.elapsed_time(e) for s, e in ts) / n


def time_graph(fns, reps=4):
    """Mean device time (ms) per call of the closures in `fns`, captured once
    each into a CUDA graph (in order) and replayed `reps` times."""
    import torch
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):  # first calls (workspace, attributes) before capture
        for fn in fns:
            fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for fn in fns:
            fn()
    g.replay()
    torch.cuda.synchronize()
    st, en = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    st.record()
    for _ in range(reps):
        g.replay()
    en.record()
    torch.cuda.synchronize()
    return st.elapsed_time(en) / (reps * len(fns))


def measure_library_fp8(M, N, K, flush, n=10):
    """Context for the FP8 peak: cuBLAS's per-tensor-scaled FP8 GEMM
    (torch._scaled_mm, one scale per operand, so no per-block promotion) on
    the same shape, timed like the GEMM here (L2 flushed, CUDA events).  It is
    not part of the hot path; None where the call is unavailable."""
    import torch
    try:
        a = torch.randn(M, K, device="cuda").to(torch.float8_e4m3fn)
        b = torch.randn(N, K, device="cuda").to(torch.float8_e4m3fn)
        one = torch.tensor(1.0, device="cuda")

        def f():
            return torch._scaled_mm(a, b.t(), scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
        for _ in range(3):
            f()
        torch.cuda.synchronize()
        ts = []
        stream = torch.cuda.current_stream()
        for i in range(n):
            flush(i)
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record(stream)
            f()
            e.record(stream)
            ts.append((s, e))
        torch.cuda.synchronize()
        ms = sum(s.elapsed_time(e) for s, e in ts) / n
        del a, b
        return {"tflops": round(2.0 * M * N * K / (ms * 1e-3) / 1e12, 1), "us": round(1e3 * ms, 1),
                "what": "cuBLAS per-tensor FP8 (torch._scaled_mm), same shape, no block scales"}
    except Exception as exc:  # pragma: no cover - depends on the torch build
        return {"unavailable": f"{type(exc).__name__}: {exc}"[:200]}


def _roof(flops, nbytes, ms, peaks, sustained=False):
    t_c = flops / (fp8_peak(peaks, sustained) * 1e12)
    t_m = nbytes / (peaks["hbm_gbs"] * 1e9)
    t = ms * 1e-3
    return {"us": round(ms * 1e3, 2), "tflops": round(flops / t / 1e12, 1),
            "gbs": round(nbytes / t / 1e9, 1), "bound": "tensor" if t_c > t_m else "hbm",
            "roofline_frac": round(max(t_c, t_m) / t, 4)}


def measure_configs(peaks, dev):
    """The other workloads, each timed alone (L2 flushed) against its own
    roofline max(FLOP / FP8 peak, bytes / HBM peak), burst peaks."""
    import numpy as np
    import torch

    from fp8_fine_grained_e4m3_gb300 import binding as b
    from fp8_fine_grained_e4m3_gb300 import synthetic
    flush = L2Flush(dev)
    res = {}

    def dense_case(M, N, K, kind, seed):
        X, W = synthetic.dense_operands_device(M, N, K, kind=kind, seed=seed, device=dev)
        A8, sA = b.fp8_quant_1x128(X)
        B8, sB = b.fp8_quant_128x128(W)
        del X, W
        D = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        return A8, sA, B8, sB, D

    A8, sA, B8, sB, D = dense_case(128, 256, 512, "normal", 0)
    ms = time_launch(lambda: b.fp8gemm_dense(A8, sA, B8, sB, D=D), flush)
    res["dense_128x256x512"] = _roof(2 * 128 * 256 * 512, gemm_bytes(128, 256, 512), ms, peaks)

    # a few hundred rows: every tile fits in one wave, so each tile's K blocks
    # are shared by a cluster of CTAs (split instance)
    for (M, N, K) in ((128, 4096, 7168), (384, 4096, 7168)):
        A8, sA, B8, sB, D = dense_case(M, N, K, "prefill", M)
        ms = time_launch(lambda: b.fp8gemm_dense(A8, sA, B8, sB, D=D), flush)
        r = _roof(2 * M * N * K, gemm_bytes(M, N, K), ms, peaks)
        r["note"] = "tiles split along K over thread-block clusters"
        res[f"dense_split_{M}x{N}x{K}"] = r

    for M in (1, 16, 64):
        for (N, K) in ((7168, 2048), (2048, 7168)):
            # 24 weight copies (> 2x L2 in total) used in turn, launched back to
            # back from a CUDA graph, so each launch reads its weights from HBM
            # and no host launch overhead sits between launches
            A8, sA, B8, sB, D = dense_case(M, N, K, "decode", M)
            copies = [(B8.clone(), sB.clone()) for _ in range(24)]
            fns = [(lambda Bc=Bc, sBc=sBc: b.fp8gemm_dense(A8, sA, Bc, sBc, D=D))
                   for Bc, sBc in copies]
            ms = time_graph(fns, reps=4)
            r = _roof(2 * M * N * K, gemm_bytes(M, N, K), ms, peaks)
            r["timing"] = "CUDA graph, 24 rotating weight copies"
            res[f"decode_{M}x{N}x{K}"] = r
            # From FP32 activations: fp8gemm_dense_quant_a (the quantiser, then
            # the GEMM as its programmatic dependent)
            X, _ = synthetic.dense_operands_device(M, 8, K, kind="decode", seed=M, device=dev)
            fns_q = [(lambda Bc=Bc, sBc=sBc: b.fp8gemm_dense_quant_a(X, Bc, sBc, D=D))
                     for Bc, sBc in copies]
            nb = gemm_bytes(M, N, K) - M * K - 4 * M * (K // 128) + 4 * M * K
            ms_q = time_graph(fns_q, reps=4)
            l0 = b.num_kernel_launches()
            fns_q[0]()
            n_launch = b.num_kernel_launches() - l0
            how = ("1 launch, quantised on load" if n_launch == 1
                   else f"quantiser + GEMM, {n_launch} launches")
            r = _roof(2 * M * N * K, nb, ms_q, peaks)
            r["timing"] = f"CUDA graph, 24 rotating weight copies; {how}"
            res[f"decode_quant_a_{M}x{N}x{K}"] = r
            # Constant weights declared read-only (FP8GEMM_FLAG_B_READ_ONLY):
            # each GEMM stages its first weight tiles while the one before
            # it finishes
            fns_ro = [(lambda Bc=Bc, sBc=sBc: b.fp8gemm_dense_ex(A8, sA, "e4m3", Bc, sBc, "e4m3",
                                                                 D=D, flags=b.FLAG_B_READ_ONLY))
                      for Bc, sBc in copies]
            ms_ro = time_graph(fns_ro, reps=4)
            r = _roof(2 * M * N * K, gemm_bytes(M, N, K), ms_ro, peaks)
            r["timing"] = "CUDA graph, 24 rotating weight copies; weights declared read-only"
            res[f"decode_ro_{M}x{N}x{K}"] = r
            fns_qro = [(lambda Bc=Bc, sBc=sBc: b.fp8gemm_dense_quant_a(X, Bc, sBc, D=D,
                                                                       flags=b.FLAG_B_READ_ONLY))
                       for Bc, sBc in copies]
            ms_qro = time_graph(fns_qro, reps=4)
            r = _roof(2 * M * N * K, nb, ms_qro, peaks)
            r["timing"] = (f"CUDA graph, 24 rotating weight copies; {how}; weights declared "
                           "read-only (staged before the dependency wait)")
            res[f"decode_quant_a_ro_{M}x{N}x{K}"] = r
            del copies, fns, fns_q, fns_ro, fns_qro, X

    # mixed formats: e5m2 A (a gradient) against e4m3 B, large and decode shapes
    for (M, N, K) in ((4096, 7168, 16384), (16, 7168, 2048)):
        X, W = synthetic.dense_operands_device(M, N, K, kind="prefill", seed=1, device=dev)
        A8, sA = b.fp8_quant_1x128_fmt(X, "e5m2")
        B8, sB = b.fp8_quant_128x128(W)
        del X, W
        D = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        if M <= 64:
            copies = [(B8.clone(), sB.clone()) for _ in range(24)]
            fns = [(lambda Bc=Bc, sBc=sBc: b.fp8gemm_dense_fmt(A8, sA, "e5m2", Bc, sBc, "e4m3",
                                                                 D=D))
                   for Bc, sBc in copies]
            ms = time_graph(fns, reps=4)
            del copies, fns
        else:
            ms = time_launch(lambda: b.fp8gemm_dense_fmt(A8, sA, "e5m2", B8, sB, "e4m3", D=D),
                             flush)
        res[f"dense_e5m2xe4m3_{M}x{N}x{K}"] = _roof(2 * M * N * K, gemm_bytes(M, N, K), ms, peaks)
        del A8, sA, B8, sB, D

    # quantiser on the large prefill activations
    X, _ = synthetic.dense_operands_device(4096, 8, 16384, kind="prefill", seed=0, device=dev)
    Q = torch.empty(X.shape, dtype=torch.uint8, device=dev)
    S = torch.empty((4096, 128), dtype=torch.float32, device=dev)
    ms = time_launch(lambda: b.fp8_quant_1x128(X, Q=Q, sX=S), flush)
    nb = X.numel() * 5 + S.numel() * 4
    res["quant_1x128_4096x16384"] = {"us": round(ms * 1e3, 2),
                                     "gbs": round(nb / (ms * 1e-3) / 1e9, 1),
                                     "bound": "hbm",
                                     "roofline_frac": round(nb / (peaks["hbm_gbs"] * 1e9) /
                                                            (ms * 1e-3), 4)}
    # the same with the saturation counter
    cnt = torch.zeros(1, dtype=torch.int64, device=dev)
    ms = time_launch(lambda: b.fp8_quant_1x128_fmt(X, "e4m3", Q=Q, sX=S, sat_count=cnt), flush)
    res["quant_1x128_count_4096x16384"] = {"us": round(ms * 1e3, 2),
                                           "gbs": round(nb / (ms * 1e-3) / 1e9, 1),
                                           "bound": "hbm",
                                           "roofline_frac": round(nb / (peaks["hbm_gbs"] * 1e9) /
                                                                  (ms * 1e-3), 4),
                                           "note": "fp8_quant_1x128_ex with a saturation counter"}
    del X, Q, S

    # weight quantiser (the offline step) on the prefill B, 7168 x 16384
    _, W = synthetic.dense_operands_device(8, 7168, 16384, kind="prefill", seed=0, device=dev)
    QW = torch.empty(W.shape, dtype=torch.uint8, device=dev)
    SW = torch.empty((56, 128), dtype=torch.float32, device=dev)
    ms = time_launch(lambda: b.fp8_quant_128x128(W, Q=QW, sW=SW), flush)
    nb = W.numel() * 5 + SW.numel() * 4
    res["quant_128x128_7168x16384"] = {"us": round(ms * 1e3, 2),
                                       "gbs": round(nb / (ms * 1e-3) / 1e9, 1),
                                       "bound": "hbm",
                                       "roofline_frac": round(nb / (peaks["hbm_gbs"] * 1e9) /
                                                              (ms * 1e-3), 4)}
    del W, QW, SW, cnt

    # MoE contiguous: 32 experts, 8192 Zipf(1.1) tokens, N=4096, K=7168
    E, T, N, K = 32, 8192, 4096, 7168
    lay = synthetic.contiguous_layout(synthetic.zipf_counts(E, T, seed=0))
    X = synthetic.contiguous_activations_device(lay, K, seed=0, device=dev)
    A8, sA = b.fp8_quant_1x128(X)
    del X
    W = synthetic.expert_weights_device(E, N, K, seed=0, device=dev)
    B8, sB = b.fp8_quant_128x128(W)
    del W
    mi = torch.from_numpy(lay.m_indices).to(dev)
    D = torch.empty((lay.M_pad, N), dtype=torch.bfloat16, device=dev)
    ms = time_launch(lambda: b.fp8gemm_grouped_contiguous(A8, sA, B8, sB, mi, D=D), flush)
    rows = int(lay.counts.sum())
    e_act = int((lay.counts > 0).sum())
    nbytes = gemm_bytes(rows, N, K, e_active=e_act, rows=rows) + 4 * lay.M_pad
    r = _roof(2.0 * rows * N * K, nbytes, ms, peaks)
    r["note"] = "padding rows not credited"
    res["moe_contiguous_E32_T8192_N4096_K7168"] = r
    # the same layer as one batched launch, each expert's unpadded rows one
    # entry (for a caller that knows the counts on the host), captured once
    # in a CUDA graph so that the 32 entries' host-side checks stay outside
    # the timed interval
    ents = [(A8[o:o + c], sA[o:o + c], B8[e], sB[e], D[o:o + c])
            for e, (o, c) in enumerate(zip(lay.offsets.tolist(), lay.counts.tolist())) if c > 0]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        b.fp8gemm_dense_batch(ents)  # the stream's tile counters
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        b.fp8gemm_dense_batch(ents)
    ms = time_launch(graph.replay, flush)
    r = _roof(2.0 * rows * N * K, gemm_bytes(rows, N, K, e_active=e_act, rows=rows), ms, peaks)
    r["note"] = ("fp8gemm_dense_batch, one entry per expert (unpadded rows), largest and "
                 "smallest experts alternating; CUDA graph replay")
    res["moe_contiguous_as_batch_E32_T8192_N4096_K7168"] = r
    del graph, ents
    del A8, sA, B8, sB, D
    torch.cuda.empty_cache()

    # MoE masked: 16 experts, A [16, 256, 7168] Student-t, masked_m ~ U[0, 256]
    E, M_max, N, K = 16, 256, 4096, 7168
    mm = synthetic.masked_counts(E, M_max, seed=0)
    X = synthetic.masked_activations_device(E, M_max, K, seed=0, device=dev)
    A8, sA = b.fp8_quant_1x128(X)
    del X
    W = synthetic.expert_weights_device(E, N, K, seed=1, device=dev)
    B8, sB = b.fp8_quant_128x128(W)
    del W
    mmd = torch.from_numpy(mm).to(dev)
    D = torch.empty((E, M_max, N), dtype=torch.bfloat16, device=dev)
    ms = time_launch(lambda: b.fp8gemm_grouped_masked(A8, sA, B8, sB, mmd, D=D), flush)
    rows = int(mm.sum())
    e_act = int((mm > 0).sum())
    nbytes = gemm_bytes(rows, N, K, e_active=e_act, rows=rows) + 4 * E
    r = _roof(2.0 * rows * N * K, nbytes, ms, peaks)
    r["note"] = f"sum(masked_m) = {rows}; masked-out rows not credited"
    res["moe_masked_E16_M256_N4096_K7168"] = r
    del A8, sA, B8, sB, D
    torch.cuda.empty_cache()

    # Batched decode from a device problem table: 16 problems (one per
    # expert), M_e ~ U{1..16} tokens, N=4096, K=7168; the masked grouped
    # kernel on the same operands beside it
    E, M_max, N, K = 16, 16, 4096, 7168
    mm = (synthetic.masked_counts(E, M_max - 1, seed=3) + 1).astype(np.int32)
    X = synthetic.masked_activations_device(E, M_max, K, seed=3, device=dev)
    A8, sA = b.fp8_quant_1x128(X)
    del X
    W = synthetic.expert_weights_device(E, N, K, seed=4, device=dev)
    B8, sB = b.fp8_quant_128x128(W)
    del W
    D = torch.empty((E, M_max, N), dtype=torch.bfloat16, device=dev)
    probs = [(A8[e, :mm[e]], sA[e, :mm[e]], B8[e], sB[e], D[e, :mm[e]]) for e in range(E)]
    table = b.problem_table(probs)
    ms_t = time_launch(lambda: b.fp8gemm_grouped_table(table, E, M_max), flush)
    mmd = torch.from_numpy(mm).to(dev)
    ms_m = time_launch(lambda: b.fp8gemm_grouped_masked(A8, sA, B8, sB, mmd, D=D), flush)
    rows = int(mm.sum())
    nbytes = gemm_bytes(rows, N, K, e_active=E, rows=rows) + 56 * E
    r = _roof(2.0 * rows * N * K, nbytes, ms_t, peaks)
    r["note"] = f"sum(M_e) = {rows}; fp8gemm_grouped_masked on the same operands: {ms_m * 1e3:.2f} us"
    res["table_E16_M1-16_N4096_K7168"] = r
    del A8, sA, B8, sB, D, table, probs
    torch.cuda.empty_cache()
    if b.fp8gemm_get_device_status() != b.OK:
        raise RuntimeError("device status set while measuring the other workloads")
    return res


KERNEL_SOURCES = ["gemm_tc.cu", "ptx.cuh", "common.cuh"]


def kernel_source_hash(files=KERNEL_SOURCES):
    import hashlib
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "fp8_fine_grained_e4m3_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_from_profiles(key):
    """DRAM bytes (read + write) per launch from the committed ncu summary
    profiles/traffic.json -- only if it was taken on the current kernel
    source (same hash); None otherwise."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        t = json.load(f).get(key)
    if not t or t.get("source_hash") != kernel_source_hash(t.get("sources", KERNEL_SOURCES)):
        return None
    return t["dram_bytes_per_launch"]


# ------------------------------------------------------------ CPU oracle
def _oracle_sample(rows, cols, seed=0):
    """Inputs for the oracle timing: the prefill shapes restricted to `rows`
    rows of A and `cols` rows of B (whole 128-row scale tiles), same K and
    same value recipe; B is quantised here (untimed, like the offline step)."""
    import numpy as np

    from fp8_fine_grained_e4m3_gb300 import synthetic
    from oracle import quant as oq
    out = []
    for i, (M, N, K) in enumerate(PREFILL_SHAPES):
        X, W = synthetic.dense_operands(rows, cols, K, kind="prefill", seed=seed + i)
        Bq, sB = oq.quant_128x128_fast(W)
        out.append((X, Bq, sB, K))
    return out


def _oracle_step(sample):
    from oracle import gemm as og
    from oracle import quant as oq
    flops = 0.0
    for X, Bq, sB, K in sample:
        A, sA = oq.quant_1x128(X)
        og.gemm_dense(A, sA, Bq, sB)
        flops += 2.0 * X.shape[0] * Bq.shape[0] * K
    return flops


def cpu_baseline(budget_s=15.0):
    """The oracle (quantise A rows + FP64 block-scaled GEMM), as it stands,
    on a sample of the step: 16 rows of A x 1024 rows of B per prefill shape,
    repeated for about `budget_s` seconds of host time."""
    sample = _oracle_sample(16, 1024)
    t0 = time.perf_counter()
    flops = 0.0
    reps = 0
    while True:
        flops += _oracle_step(sample)
        reps += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return {"value": flops / dt / 1e12, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
            "sample": (f"{reps} x [16 rows of A x 1024 rows of B, full K] per prefill shape "
                       f"(quantise A rows + FP64 block-scaled GEMM), {dt:.1f} s")}


def run_reference(args, rank, world):
    """Reference arm: the CPU oracle timed on the host cores, one bounded
    sample (4 rows of A x 128 rows of B per prefill shape) per step."""
    if rank != 0:
        return None
    sample = _oracle_sample(4, 128, seed=1)
    for _ in range(args.warmup):
        _oracle_step(sample)
    t0 = time.perf_counter()
    flops = 0.0
    for _ in range(args.steps):
        flops += _oracle_step(sample)
    dt = time.perf_counter() - t0
    value = flops / dt / 1e12
    return {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * dt / args.steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": WORKLOAD, "sample": "4 rows of A x 128 rows of B per shape"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": os.cpu_count(),
                             "kind": "oracle",
                             "sample": "4 rows of A x 128 rows of B, full K, per prefill shape"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def run_kernel_case(name, reps):
    """Launch one kernel of the path `reps` times on a fixed case, nothing
    else timed or printed: the target of the ncu captures."""
    import torch

    from fp8_fine_grained_e4m3_gb300 import binding as b
    from fp8_fine_grained_e4m3_gb300 import synthetic
    dev = torch.device("cuda", 0)
    shapes = {"gemm_prefill": (4096, 7168, 16384), "gemm_square": (4096, 4096, 4096),
              "gemm_decode64": (64, 7168, 2048), "gemm_decode1": (1, 7168, 2048),
              "gemm_split": (128, 4096, 7168), "quant": (4096, 8, 16384)}
    if name == "gemm_prefill_batch":  # both prefill shapes in one batched launch
        ops = []
        for i, (M, N, K) in enumerate(PREFILL_SHAPES):
            X, W = synthetic.dense_operands_device(M, N, K, kind="prefill", seed=i, device=dev)
            A8, sA = b.fp8_quant_1x128(X)
            B8, sB = b.fp8_quant_128x128(W)
            del X, W
            ops.append((A8, sA, B8, sB, torch.empty((M, N), dtype=torch.bfloat16, device=dev)))
        fn = lambda: b.fp8gemm_dense_batch(ops)  # noqa: E731
    elif name in shapes:
        M, N, K = shapes[name]
        X, W = synthetic.dense_operands_device(M, N, K, kind="prefill", seed=0, device=dev)
        A8, sA = b.fp8_quant_1x128(X)
        B8, sB = b.fp8_quant_128x128(W)
        D = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        if name == "quant":
            fn = lambda: b.fp8_quant_1x128(X, Q=A8, sX=sA)  # noqa: E731
        else:
            del X, W
            fn = lambda: b.fp8gemm_dense(A8, sA, B8, sB, D=D)  # noqa: E731
    elif name == "quant_w":  # the 128x128 weight quantiser on 7168 x 16384
        W = synthetic.expert_weights_device(1, 7168, 16384, seed=0, device=dev)[0]
        QW = torch.empty(W.shape, dtype=torch.uint8, device=dev)
        SW = torch.empty((56, 128), dtype=torch.float32, device=dev)
        fn = lambda: b.fp8_quant_128x128(W, Q=QW, sW=SW)  # noqa: E731
    elif name == "table":
        E, M_max, N, K = 16, 16, 4096, 7168
        mm = (synthetic.masked_counts(E, M_max - 1, seed=3) + 1).astype("int32")
        X = synthetic.masked_activations_device(E, M_max, K, seed=3, device=dev)
        A8, sA = b.fp8_quant_1x128(X)
        del X
        B8, sB = b.fp8_quant_128x128(synthetic.expert_weights_device(E, N, K, seed=4, device=dev))
        D = torch.empty((E, M_max, N), dtype=torch.bfloat16, device=dev)
        table = b.problem_table([(A8[e, :mm[e]], sA[e, :mm[e]], B8[e], sB[e], D[e, :mm[e]])
                                 for e in range(E)])
        fn = lambda: b.fp8gemm_grouped_table(table, E, M_max)  # noqa: E731
    elif name in ("contiguous", "masked"):
        if name == "contiguous":
            E, N, K = 32, 4096, 7168
            lay = synthetic.contiguous_layout(synthetic.zipf_counts(E, 8192, seed=0))
            X = synthetic.contiguous_activations_device(lay, K, seed=0, device=dev)
            info = torch.from_numpy(lay.m_indices).to(dev)
            D = torch.empty((lay.M_pad, N), dtype=torch.bfloat16, device=dev)
        else:
            E, N, K = 16, 4096, 7168
            X = synthetic.masked_activations_device(E, 256, K, seed=0, device=dev)
            info = torch.from_numpy(synthetic.masked_counts(E, 256, seed=0)).to(dev)
            D = torch.empty((E, 256, N), dtype=torch.bfloat16, device=dev)
        A8, sA = b.fp8_quant_1x128(X)
        del X
        B8, sB = b.fp8_quant_128x128(synthetic.expert_weights_device(E, N, K, device=dev))
        if name == "contiguous":
            fn = lambda: b.fp8gemm_grouped_contiguous(A8, sA, B8, sB, info, D=D)  # noqa: E731
        else:
            fn = lambda: b.fp8gemm_grouped_masked(A8, sA, B8, sB, info, D=D)  # noqa: E731
    else:
        raise SystemExit(f"unknown kernel case {name}")
    torch.cuda.synchronize()
    torch.cuda.empty_cache()  # keep the device footprint small for profilers
    for _ in range(reps):
        fn()
    torch.cuda.synchronize()
    st = b.fp8gemm_get_device_status()
    print(json.dumps({"kernel_case": name, "reps": reps, "status": st}))
    if st != b.OK:
        raise SystemExit(1)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--kernel-case", default=None,
                    help="launch one kernel case --reps times (profiling target) and exit")
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--gemm-form", choices=["single", "batch"], default="single",
                    help="the step's GEMMs: both shapes in one batched launch (the roofline "
                         "kernel), or one call per shape (the 4096x7168x16384 call the roofline "
                         "kernel)")
    ap.add_argument("--no-extras", action="store_true", help="skip the other workloads")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    if args.kernel_case:
        run_kernel_case(args.kernel_case, args.reps)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        out = run_reference(args, rank, world)
        if out is not None:
            print(json.dumps(out), flush=True)
        return
    if world > 1:
        import torch
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        torch.distributed.init_process_group("nccl")
    out = run_gpu(args, rank, world)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
