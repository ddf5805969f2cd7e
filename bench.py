#!/usr/bin/env python3
"""Benchmark of the mixed-precision tensor-core GEMM on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME]

A step is one call of the library's GEMM (the whole hot path) on one batch of
synthetic input already resident in HBM.  Default workload: the 8192^3 FP16 ->
FP32 GEMM (A, B uniform[-1,1] rounded to FP16, beta = 0, seed 1).  Prints one
JSON line (rank 0).  Under torchrun (--gpus N > 1) every rank runs an
independent replica ("replicas only": the GEMM has no exchange step), timing is
bracketed by a barrier and a device synchronisation and the max over ranks is
taken; value = all ranks' FLOPs / that time.

--impl reference times the CPU oracle (the plain FP64 C implementation under
oracle/), as it stands, on this host's cores, on bounded samples of the same
workload, and prints the same line with "impl": "reference".
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GEMM TFLOP/s and % of dense tensor peak (FP16→FP32, 8192³) on 1 GB300"
UNIT = "TFLOP/s"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def load_peaks(root: str = ROOT):
    p = os.path.join(root, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def traffic_record(kernel: str, workload: str, root: str = ROOT):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the
    current kernel source (its source digest must match), else None."""
    import hashlib
    p = os.path.join(root, "profiles", "dram_traffic.txt")
    if not os.path.exists(p):
        return None
    h = hashlib.sha256()
    csrc = os.path.join(root, "mixed_precision_tensor_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    digest = h.hexdigest()[:16]
    with open(p) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            kv = dict(x.split("=", 1) for x in line.split())
            if kv.get("kernel") == kernel and kv.get("workload") == workload and \
                    kv.get("source_sha") == digest:
                return float(kv["dram_bytes_per_launch"])
    return None


# NVML (read-only queries) through ctypes: the GPU machine has the driver's libnvidia-ml but
# no Python NVML package.  Nothing here sets a clock, a limit or any other GPU setting.
NVML_CLOCK_SM = 1
# nvmlClocksEventReasons bits (throttle reasons) that the JSON line reports by name
REASON_BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
               "hw_thermal_slowdown": 0x40, "hw_power_brake_slowdown": 0x80}


class Nvml:
    """One GPU's SM clock, maximum SM clock, power draw and clock-event reasons.

    ``lib`` is the loaded NVML library (a ctypes CDLL) or anything with the same
    functions (the CPU tests pass a fake).  ``uuid`` picks the GPU the CUDA device is
    (NVML numbers every GPU of the machine, CUDA only the visible ones); ``index`` is
    the fallback."""

    def __init__(self, lib, uuid=None, index=0):
        import ctypes
        self.lib = lib
        self.c = ctypes
        if lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        self.dev = ctypes.c_void_p()
        rc = 1
        if uuid:
            rc = lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.dev))
        if rc != 0:
            rc = lib.nvmlDeviceGetHandleByIndex_v2(index, ctypes.byref(self.dev))
        if rc != 0:
            raise RuntimeError("no NVML handle for the device")
        fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None)
        self.reasons_fn = fn if fn is not None else lib.nvmlDeviceGetCurrentClocksThrottleReasons

    @classmethod
    def open(cls, uuid=None, index=0):
        import ctypes
        return cls(ctypes.CDLL("libnvidia-ml.so.1"), uuid, index)

    def sample(self):
        """(sm_mhz, sm_max_mhz, power_w, reason_bits); None for a field that failed."""
        c = self.c
        sm, smax, mw, rs = c.c_uint(), c.c_uint(), c.c_uint(), c.c_ulonglong()
        ok_sm = self.lib.nvmlDeviceGetClockInfo(self.dev, NVML_CLOCK_SM, c.byref(sm)) == 0
        ok_max = self.lib.nvmlDeviceGetMaxClockInfo(self.dev, NVML_CLOCK_SM, c.byref(smax)) == 0
        ok_pw = self.lib.nvmlDeviceGetPowerUsage(self.dev, c.byref(mw)) == 0
        ok_rs = self.reasons_fn(self.dev, c.byref(rs)) == 0
        return (float(sm.value) if ok_sm else None, float(smax.value) if ok_max else None,
                mw.value / 1000.0 if ok_pw else None, int(rs.value) if ok_rs else None)


class ClockSampler:
    """Samples an Nvml source on a background thread every ``period_s`` (1 ms) and
    summarises the samples that fall inside a timed region (perf_counter times)."""

    def __init__(self, nvml, period_s=0.001):
        import threading
        self.nvml = nvml
        self.period = period_s
        self.samples = []                     # (t, sm, smax, power_w, reasons)
        self._stop = threading.Event()
        self._thread = threading.Thread(target=self._run, daemon=True)

    def _run(self):
        while not self._stop.is_set():
            t = time.perf_counter()
            try:
                self.samples.append((t,) + tuple(self.nvml.sample()))
            except Exception:
                pass
            self._stop.wait(self.period)

    def start(self):
        self._thread.start()
        return self

    def stop(self):
        self._stop.set()
        self._thread.join(timeout=2)

    def region(self, t0, t1):
        return summarise_samples(list(self.samples), t0, t1)


def summarise_samples(samples, t0, t1):
    """Clock record of the timed region [t0, t1]: median SM clock, maximum SM clock,
    largest power draw and the clock-event reasons seen in the samples taken inside it.
    With no sample inside, the clock is unknown (None), never borrowed from outside."""
    during = [r for r in samples if t0 <= r[0] <= t1 and r[1] is not None]
    if not during:
        return {"sm_mhz": None, "sm_max_mhz": None, "samples_in_timed_region": 0,
                "reasons": [], "source": "nvml"}
    reasons = set()
    for r in during:
        if r[4] is not None:
            reasons.update(nm for nm, bit in REASON_BITS.items() if r[4] & bit)
    maxes = [r[2] for r in during if r[2] is not None]
    powers = [r[3] for r in during if r[3] is not None]
    return {"sm_mhz": statistics.median(r[1] for r in during),
            "sm_max_mhz": max(maxes) if maxes else None,
            "power_w_max": max(powers) if powers else None,
            "samples_in_timed_region": len(during),
            "reasons": sorted(reasons), "source": "nvml"}


def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl"
        try:
            import torch
            if not torch.cuda.is_available():
                backend = "gloo"
        except Exception:
            backend = "gloo"
        dist.init_process_group(backend=backend)
    return world, rank, local


def max_over_ranks(x: float, world: int) -> float:
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if torch.cuda.is_available() and \
        dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# --------------------------------------------------------------- CPU oracle
def oracle_blocks(w, A, B, rows_per_block, count, seed):
    """Sampled output blocks (rows_per_block x 128, full k) of the row-major D."""
    from mixed_precision_tensor_gb300 import workloads as wl
    tiles = wl.sample_tiles(w.m, w.n, count=count, tile=128, seed=seed)
    return [(i0, min(i0 + rows_per_block, i1), j0, j1) for (i0, i1, j0, j1) in tiles]


def time_oracle(w, A, B, C, blocks, nthreads):
    import numpy as np

    import oracle
    codes = {"f16": oracle.F16, "bf16": oracle.BF16, "f32": oracle.F32, "e4m3": oracle.F8E4M3,
             "e5m2": oracle.F8E5M2}

    def rawv(x):
        return x.view(np.uint16) if x.dtype == np.float16 else x
    flops = 0.0
    t0 = time.perf_counter()
    for (i0, i1, j0, j1) in blocks:
        # the column-major call the library gets: gemm(N, N, n, m, k, B, n, A, k, C, n)
        oracle.gemm(oracle.OP_N, oracle.OP_N, w.n, w.m, w.k, w.alpha,
                    rawv(B[0]).reshape(-1), codes[w.in_type], w.n,
                    rawv(A[0]).reshape(-1), codes[w.in_type], w.k,
                    w.beta, None if C is None else rawv(C[0]).reshape(-1), codes[w.out_type],
                    w.n, tf32=(w.in_type == "f32" and w.compute != "3xtf32"),
                    rows=(j0, j1), cols=(i0, i1),
                    nthreads=nthreads, want_r=False, want_abs=False)
        flops += 2.0 * (i1 - i0) * (j1 - j0) * w.k
    return time.perf_counter() - t0, flops


def cpu_baseline(w, A, B, C, budget_s=12.0):
    """The oracle timed on this host's cores on a bounded sample of the workload."""
    nthreads = os.cpu_count() or 1
    blk = oracle_blocks(w, A, B, 128, 4, seed=w.seed)
    dt1, fl1 = time_oracle(w, A, B, C, blk, nthreads)
    count = max(4, min(1024, int(budget_s / max(dt1 / len(blk), 1e-6))))
    blocks = oracle_blocks(w, A, B, 128, count, seed=w.seed)
    dt, fl = time_oracle(w, A, B, C, blocks, nthreads)
    return {"value": fl / dt / 1e12, "unit": UNIT, "cores": nthreads, "kind": "oracle",
            "sample": f"{len(blocks)} seeded 128x128 output tiles of the {w.m}x{w.n}x{w.k} "
                      f"GEMM{' (batch entry 0 of %d)' % w.batch if w.batch > 1 else ''}, "
                      f"full k each ({fl:.3e} FLOP in {dt:.2f} s)",
            # the whole workload at the sampled rate (extrapolated, not measured)
            "extrapolated_full_s": w.flops / (fl / dt)}


# ------------------------------------------------------------------ main arms
def run_reference(args, w):
    world, rank, _ = int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")), 0
    if rank != 0:
        return 0
    from mixed_precision_tensor_gb300 import workloads as wl
    import oracle
    oracle.build()
    A, B, C = wl.draw(w)
    nthreads = os.cpu_count() or 1
    # Size one step so the whole run stays within about two minutes.
    probe = oracle_blocks(w, A, B, 16, 1, seed=w.seed)
    dtp, _ = time_oracle(w, A, B, C, probe, nthreads)
    per_step_budget = 120.0 / max(1, args.steps + args.warmup)
    rows = 128
    while rows > 8 and dtp * rows / 16 > per_step_budget:
        rows //= 2
    blocks = oracle_blocks(w, A, B, rows, 1, seed=w.seed)
    for _ in range(args.warmup):
        time_oracle(w, A, B, C, blocks, nthreads)
    tot_t, tot_f = 0.0, 0.0
    for _ in range(args.steps):
        dt, fl = time_oracle(w, A, B, C, blocks, nthreads)
        tot_t += dt
        tot_f += fl
    value = tot_f / tot_t / 1e12
    sample = (f"each step: one {rows}x128 output block of the {w.m}x{w.n}x{w.k} GEMM, "
              f"full k ({tot_f / args.steps:.3e} FLOP)")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": tot_t / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "m": w.m, "n": w.n, "k": w.k,
                       "in": w.in_type, "out": w.out_type, "batch": w.batch},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": nthreads,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def roofline_entry(w, kernel_ms, peaks, peak_src, traffic):
    """The JSON line's roofline object for workload ``w`` whose step took ``kernel_ms``.

    Bound: tensor when the arithmetic intensity (FLOP per algorithmic byte) is at or above
    the ridge of the measured peaks (~284 FLOP/B), else HBM.  A contraction's peak is the
    measured dense BF16 rate scaled by the nominal ratio of its own kind: TF32 half, FP8
    twice, and the three-product TF32 split a third of TF32 (three products per useful
    one)."""
    bound = "hbm" if w.flops / max(1, w.algorithmic_bytes()) < 284 else "tensor"
    if bound == "tensor":
        peak = float(peaks["bf16_tflops"])        # FP16 and BF16 share the dense rate
        if w.in_type == "f32":
            peak = peak / 2.0                     # TF32 dense rate: half of FP16/BF16
        if w.in_type in ("e4m3", "e5m2"):
            peak = peak * 2.0                     # FP8 dense rate: twice FP16/BF16
        if w.compute == "3xtf32":
            peak = peak / 3.0                     # three TF32 products per useful product
        achieved = w.flops / (kernel_ms * 1e-3) / 1e12
        unit = "TFLOP/s"
    else:
        peak = float(peaks["hbm_gbs"])
        achieved = w.algorithmic_bytes() / (kernel_ms * 1e-3) / 1e9
        unit = "GB/s"
    return {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
            "frac": achieved / peak, "traffic": traffic,
            "peak_source": f"{peak_src} ({'bf16_tflops' if bound == 'tensor' else 'hbm_gbs'})",
            # context: the same ratio against cuBLAS's sustained (power-capped) rate, the
            # regime a long run of back-to-back calls ends in
            "frac_of_sustained": (achieved / (peak * float(
                peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
                / float(peaks["bf16_tflops"])) if bound == "tensor" else None)}


def _device_tensors(w, dev):
    """Workload ``w``'s seeded inputs on the device: (A, B, C0 or None, out, host draws)."""
    import numpy as np
    import torch

    from mixed_precision_tensor_gb300 import workloads as wl
    A, B, C = wl.draw(w)
    tdt = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}
    squeeze = w.batch == 1
    views = {"bf16": torch.bfloat16, "e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}

    def host(x):
        a = np.ascontiguousarray(x[0] if squeeze else x)
        return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a)

    def to_dev(x, t):
        tt = host(x).to(dev)
        return tt.view(views[t]) if t in views else tt
    dA, dB = to_dev(A, w.in_type), to_dev(B, w.in_type)
    oshape = (w.m, w.n) if squeeze else (w.batch, w.m, w.n)
    dC0 = to_dev(C, w.out_type) if C is not None else None
    dC = dC0.clone() if dC0 is not None else torch.empty(oshape, dtype=tdt[w.out_type],
                                                         device=dev)
    return dA, dB, dC, (A, B, C, host, views, oshape, tdt)


def time_steps(step, stream, steps, warmup, flush, world, sampler, counter=None,
               before=None):
    """W untimed warm-up steps, then exactly K timed steps on ``stream`` bracketed by a
    barrier and a device synchronisation.  With ``flush`` (inputs that fit in L2) each
    step is an L2 flush then the call, timed by its own pair of CUDA events; without, the
    K calls run back to back between one pair of events (events between them would stop a
    call from starting while the previous one drains), and the per-step time is the
    region's over K.  The clock record covers the timed region; ``counter`` (the library's
    launch counter) is read around it.  Returns (per-step kernel ms, region ms, clocks,
    launches in the timed region)."""
    import torch
    with torch.cuda.stream(stream):
        for _ in range(max(3, warmup)):
            step()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    g0 = torch.cuda.Event(enable_timing=True)
    g1 = torch.cuda.Event(enable_timing=True)
    if before is not None:
        before()
    barrier(world)
    torch.cuda.synchronize()
    n0 = counter() if counter else 0
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        g0.record(stream)
        for i in range(steps):
            if flush is not None:
                flush.zero_()
                starts[i].record(stream)
                step()
                ends[i].record(stream)
            else:
                step()
        g1.record(stream)
    torch.cuda.synchronize()
    t1 = time.perf_counter()
    launches = (counter() - n0) if counter else 0
    barrier(world)
    region_ms = g0.elapsed_time(g1)
    kernel_ms = (sum(a.elapsed_time(b) for a, b in zip(starts, ends)) / steps
                 if flush is not None else region_ms / steps)
    clocks = sampler.region(t0, t1) if sampler is not None else None
    return kernel_ms, region_ms, clocks, launches


def per_clk_flops(w):
    """Dense FLOP per clock per SM of the workload's MMA kind (the rate ncu's tensor-pipe
    utilisation treats as 100%): 8192 for kind::f16, half for kind::tf32, twice for FP8;
    the three-product TF32 split delivers a third of the TF32 rate as useful FLOPs."""
    if w.in_type == "f32":
        return 4096 // 3 if w.compute == "3xtf32" else 4096
    return 16384 if w.in_type in ("e4m3", "e5m2") else 8192


def at_clock_entry(w, tflops, clocks, sms, kernel_mhz=None):
    """The workload's dense tensor peak at the SM clock of its timed region, and the
    fraction reached.  The clock is the one the GEMM kernel itself measured (its SM
    cycles over its nanoseconds, ``kernel_mhz``) when given, else the median of the NVML
    samples inside the region; None with neither."""
    mhz, src = None, None
    if kernel_mhz:
        mhz, src = kernel_mhz, "kernel clock64 / globaltimer"
    elif clocks and clocks.get("sm_mhz"):
        mhz, src = clocks["sm_mhz"], "nvml samples in the timed region"
    if mhz is None:
        return None
    pk = sms * per_clk_flops(w) * mhz * 1e6 / 1e12
    return {"sm_mhz": mhz, "clock_source": src, "sms": sms,
            "flop_per_clk_per_sm": per_clk_flops(w), "peak_tflops": pk, "frac": tflops / pk}


# The other workloads of the run, each timed in the same process with the same steps and
# warm-up as the headline: the four other synthetic workloads, then the FP8 and
# three-product TF32 variants of the survey's next rows.
SIDE_WORKLOADS = ["fp16_gemm_256", "bf16_proj_16384x4096x4096", "tf32_gemm_4096x4096x16384",
                  "fp16_batched_512x256", "fp8e4m3_gemm_8192", "fp32_3xtf32_4096x4096x16384"]


def run_ours(args, w):
    import torch

    import mixed_precision_tensor_gb300 as tcg
    from mixed_precision_tensor_gb300 import workloads as wl

    world, rank, local = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    tcg.load_library()
    peaks, peak_src = load_peaks()
    props = torch.cuda.get_device_properties(dev)
    sms = props.multi_processor_count
    sampler = None
    try:
        uuid = getattr(props, "uuid", None)
        sampler = ClockSampler(Nvml.open(f"GPU-{uuid}" if uuid else None, local)).start()
    except Exception as e:            # no NVML: the clock record says so
        log(f"clock sampling unavailable: {e}")
    stream = torch.cuda.Stream(device=dev)
    h = tcg.Handle(stream)

    def measure(wk):
        """Time workload ``wk`` (device-resident inputs); returns its record and tensors."""
        dA, dB, dC, extra = _device_tensors(wk, dev)
        A, B, C = extra[0], extra[1], extra[2]
        in_bytes = A.nbytes + B.nbytes + (C.nbytes if C is not None else 0)
        flush = (torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
                 if in_bytes <= L2_BYTES else None)
        tf32 = wk.in_type == "f32"

        def step():
            tcg.gemm_rowmajor(h, dA, dB, dC, alpha=wk.alpha, beta=wk.beta, tf32=tf32,
                              split3=wk.compute == "3xtf32")
        kernel_ms, region_ms, clocks, launches = time_steps(
            step, stream, args.steps, args.warmup, flush, world, sampler,
            counter=lambda: tcg.tcg_launch_count(h.h),
            before=lambda: tcg.check(tcg.tcg_set_clock_probe(h.h, 1), "clock probe"))
        st, cyc, ns = tcg.tcg_read_clock_probe(h.h)
        tcg.check(st, "clock probe")
        tcg.check(tcg.tcg_set_clock_probe(h.h, 0), "clock probe")
        kernel_mhz = cyc / ns * 1e3 if ns else None
        if clocks is not None:
            clocks["sm_mhz_kernel"] = kernel_mhz
        tcg.check(tcg.tcg_get_device_error(h.h), f"{wk.name}: timed region")
        step_ms = kernel_ms if flush is not None else region_ms / args.steps
        step_ms = max_over_ranks(step_ms, world)
        rec = {"ms_per_step": step_ms, "us_per_call": step_ms * 1e3,
               "tflops": wk.flops * world / (step_ms * 1e-3) / 1e12,
               "gpu_launches": launches, "clocks": clocks,
               "l2": ("inputs larger than L2" if flush is None else
                      "L2 flushed between steps (write of a 258 MiB buffer)")}
        rec["roofline"] = roofline_entry(wk, kernel_ms, peaks, peak_src,
                                         traffic_record("tcg_gemm_kernel", wk.name))
        rec["tensor_peak_at_clock"] = at_clock_entry(wk, rec["tflops"] / world, clocks, sms,
                                                     kernel_mhz)
        if rec["roofline"]["bound"] == "hbm":
            rec["hbm_gbs"] = rec["roofline"]["achieved"]
        return rec, (dA, dB, dC, extra)

    head, (dA, dB, dC, extra) = measure(w)
    A, B, C, host, views, oshape, tdt = extra
    tf32 = w.in_type == "f32"
    value = head["tflops"]

    # End to end through the C ABI's host-buffer call (tcg_gemm_ex_host /
    # tcg_gemm_strided_batched_host): pinned host inputs, the copies in, the GEMM and the
    # copy of D back into host memory all inside the timed region; the library pipelines
    # the copies against the product.  Each call returns when D is in host memory.
    def pinned(x, t):
        tt = host(x).pin_memory()
        return tt.view(views[t]) if t in views else tt
    hA, hB = pinned(A, w.in_type), pinned(B, w.in_type)
    hD = (pinned(C, w.out_type) if C is not None else
          torch.zeros(oshape, dtype=torch.int16 if w.out_type == "bf16" else tdt[w.out_type]
                      ).pin_memory())
    if w.out_type == "bf16" and hD.dtype == torch.int16:
        hD = hD.view(torch.bfloat16)
    e2e_steps = max(3, min(20, args.steps // 10))
    h2d = hA.nbytes + hB.nbytes + (hD.nbytes if C is not None else 0)
    d2h = hD.nbytes

    def e2e_step():
        tcg.gemm_rowmajor(h, hA, hB, hD, alpha=w.alpha, beta=w.beta, tf32=tf32,
                          split3=w.compute == "3xtf32", host=True)

    e2e_step()                                  # grows the handle's staging buffers
    torch.cuda.synchronize()
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    e2e_ms = max_over_ranks((time.perf_counter() - t0) * 1e3 / e2e_steps, world)
    e2e_value = w.flops * world / (e2e_ms * 1e-3) / 1e12
    tcg.check(tcg.tcg_get_device_error(h.h), "e2e")
    del hA, hB, hD, dA, dB, dC, extra

    roof = head["roofline"]
    bound, peak = roof["bound"], roof["peak"]
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": head["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": {"f16": "f16", "bf16": "bf16", "f32": "tf32", "e4m3": "e4m3",
                  "e5m2": "e5m2"}[w.in_type] +
                 ("x3" if w.compute == "3xtf32" else ""),
        "data": "synthetic",
        "config": {"workload": w.name, "m": w.m, "n": w.n, "k": w.k, "batch": w.batch,
                   "in": w.in_type, "accumulate": "f32", "out": w.out_type,
                   "alpha": w.alpha, "beta": w.beta, "seed": w.seed, "l2": head["l2"],
                   "input_bytes": A.nbytes + B.nbytes + (C.nbytes if C is not None else 0),
                   "parallelism": f"replicas x{world}"},
        # the headline's fraction of the dense tensor peak: against the measured cuBLAS
        # burst rate (pct_of_peak, roofline.frac) and against SMs x FLOP/clk x the SM clock
        # sampled in the timed region (tensor_peak_at_clock)
        "pct_of_peak": 100.0 * value / world / (peak if bound == "tensor" else float(
            peaks["bf16_tflops"])),
        "tensor_peak_at_clock": head["tensor_peak_at_clock"],
        "roofline": roof,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": head["gpu_launches"],
        "clocks": head["clocks"],
    }
    if not args.only_headline:
        side = {}
        for name in SIDE_WORKLOADS:
            if name == w.name:
                continue
            wk = wl.WORKLOADS[name]
            rec, tensors = measure(wk)
            rec["config"] = {"m": wk.m, "n": wk.n, "k": wk.k, "batch": wk.batch,
                             "in": wk.in_type, "out": wk.out_type, "alpha": wk.alpha,
                             "beta": wk.beta, "seed": wk.seed,
                             "compute": wk.compute or "default"}
            if rank == 0 and world == 1 and not args.no_cpu_baseline:
                # the oracle on a small sample of this workload (~1.5 s of host time)
                rec["cpu_baseline"] = cpu_baseline(wk, *tensors[3][:3], budget_s=1.5)
            side[name] = rec
            del tensors
            torch.cuda.empty_cache()
        line["workloads"] = side
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, A, B, C)
    if sampler is not None:
        sampler.stop()
    h.close()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=None)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only-headline", action="store_true",
                    help="time the chosen workload only (no 'workloads' object)")
    args = ap.parse_args()
    from mixed_precision_tensor_gb300 import workloads as wl
    w = wl.WORKLOADS[args.workload or wl.HEADLINE]
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
