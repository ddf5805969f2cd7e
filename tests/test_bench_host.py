"""Host logic of bench.py that decides what the JSON line may claim, without a GPU:
the clock summary from NVML samples (the timed region only; throttle reasons; a fake
NVML library stands in for the driver's),
the DRAM-traffic record (reported only while the kernel sources match the digest it
was measured on) and the choice between measured and fallback peaks."""
import hashlib
import json
import os

import bench

def test_clock_summary_uses_the_timed_region_only():
    cap, hwt = bench.REASON_BITS["sw_power_cap"], bench.REASON_BITS["hw_thermal_slowdown"]
    samples = [(9.0, 2070.0, 2070.0, 300.0, hwt),          # before the region: ignored
               (10.1, 1400.0, 2070.0, 1300.0, cap),
               (10.2, 1500.0, 2070.0, 1350.0, 0),
               (10.3, 1450.0, 2070.0, 1390.0, cap | 0x1),   # idle bit: not reported
               (10.4, None, None, None, None),             # a failed query: skipped
               (15.0, 900.0, 2070.0, 100.0, bench.REASON_BITS["hw_slowdown"])]   # after
    s = bench.summarise_samples(samples, 10.0, 11.0)
    assert s["sm_mhz"] == 1450 and s["sm_max_mhz"] == 2070
    assert s["samples_in_timed_region"] == 3 and s["power_w_max"] == 1390.0
    assert s["reasons"] == ["sw_power_cap"]


def test_clock_summary_never_borrows_samples_from_outside_the_region():
    samples = [(float(i), 1000.0 + 100 * i, 2070.0, 500.0, 0) for i in range(5)]
    s = bench.summarise_samples(samples, 100.0, 101.0)
    assert s["samples_in_timed_region"] == 0 and s["sm_mhz"] is None
    assert bench.at_clock_entry(bench_workload(), 1000.0, s, 152) is None
    assert bench.summarise_samples([], 0.0, 1.0)["sm_mhz"] is None


def bench_workload(name="fp16_gemm_8192"):
    from mixed_precision_tensor_gb300 import workloads as wl
    return wl.WORKLOADS[name]


class _FakeNvml:
    """The NVML functions bench.Nvml calls, answering like a GPU at 1500 of 2070 MHz under
    the power cap; records every call, and has no function that sets anything."""

    def __init__(self):
        self.calls = []

    def _set(self, ref, v):
        ref._obj.value = v

    def nvmlInit_v2(self):
        self.calls.append("init")
        return 0

    def nvmlDeviceGetHandleByUUID(self, uuid, ref):
        self.calls.append(("uuid", uuid))
        return 0 if uuid == b"GPU-abc" else 13

    def nvmlDeviceGetHandleByIndex_v2(self, i, ref):
        self.calls.append(("index", i))
        return 0

    def nvmlDeviceGetClockInfo(self, dev, kind, ref):
        assert kind == bench.NVML_CLOCK_SM
        self._set(ref, 1500)
        return 0

    def nvmlDeviceGetMaxClockInfo(self, dev, kind, ref):
        self._set(ref, 2070)
        return 0

    def nvmlDeviceGetPowerUsage(self, dev, ref):
        self._set(ref, 1391000)
        return 0

    def nvmlDeviceGetCurrentClocksEventReasons(self, dev, ref):
        self._set(ref, bench.REASON_BITS["sw_power_cap"])
        return 0


def test_nvml_sampling_against_a_fake_library():
    lib = _FakeNvml()
    n = bench.Nvml(lib, uuid="GPU-abc", index=3)
    assert ("uuid", b"GPU-abc") in lib.calls and ("index", 3) not in lib.calls
    assert n.sample() == (1500.0, 2070.0, 1391.0, bench.REASON_BITS["sw_power_cap"])
    n2 = bench.Nvml(lib, uuid="GPU-other", index=3)            # unknown UUID: the index
    assert ("index", 3) in lib.calls and n2.sample()[0] == 1500.0
    sampler = bench.ClockSampler(n, period_s=0.0005).start()
    import time
    t0 = time.perf_counter()
    time.sleep(0.03)
    t1 = time.perf_counter()
    sampler.stop()
    s = sampler.region(t0, t1)
    assert s["samples_in_timed_region"] >= 5
    assert s["sm_mhz"] == 1500.0 and s["reasons"] == ["sw_power_cap"]
    e = bench.at_clock_entry(bench_workload(), 1500.0, s, 152)
    assert e["peak_tflops"] == 152 * 8192 * 1500e6 / 1e12
    assert abs(e["frac"] - 1500.0 / e["peak_tflops"]) < 1e-12
    assert e["clock_source"].startswith("nvml")
    # the kernel's own clock measurement takes precedence over the NVML samples
    e = bench.at_clock_entry(bench_workload("tf32_gemm_4096x4096x16384"), 900.0, s, 152,
                             kernel_mhz=1800.0)
    assert e["sm_mhz"] == 1800.0 and e["clock_source"].startswith("kernel")
    assert e["peak_tflops"] == 152 * 4096 * 1800e6 / 1e12


def _tree(tmp_path, sources, records):
    csrc = tmp_path / "mixed_precision_tensor_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for name, text in sources.items():
        (csrc / name).write_text(text)
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "dram_traffic.txt").write_text(
        "# comment\n\n" + "\n".join(records) + "\n")
    return csrc


def _digest(sources):
    h = hashlib.sha256()
    for name in sorted(sources):
        h.update(sources[name].encode())
    return h.hexdigest()[:16]


def test_traffic_is_reported_only_for_the_measured_sources(tmp_path):
    src = {"b.cu": "kernel B\n", "a.h": "header A\n"}
    d = _digest(src)
    csrc = _tree(tmp_path, src, [
        f"kernel=k workload=w1 source_sha={d} dram_bytes_per_launch=1234",
        "kernel=k workload=w2 source_sha=0000000000000000 dram_bytes_per_launch=99"])
    root = str(tmp_path)
    assert bench.traffic_record("k", "w1", root) == 1234.0
    assert bench.traffic_record("k", "w2", root) is None        # measured on other sources
    assert bench.traffic_record("k", "w3", root) is None        # never measured
    assert bench.traffic_record("other", "w1", root) is None
    (csrc / "b.cu").write_text("kernel B, changed\n")            # the kernel changed since
    assert bench.traffic_record("k", "w1", root) is None
    (csrc / "b.cu").write_text("kernel B\n")
    assert bench.traffic_record("k", "w1", root) == 1234.0
    os.remove(tmp_path / "profiles" / "dram_traffic.txt")
    assert bench.traffic_record("k", "w1", root) is None


def test_committed_traffic_records_are_well_formed():
    """Every committed record names a kernel, a known workload, a 16-hex-digit source
    digest and a positive byte count (whether the digest is current is the bench's
    business: a stale record is reported as null, not as a number)."""
    from mixed_precision_tensor_gb300 import workloads as wl
    path = os.path.join(bench.ROOT, "profiles", "dram_traffic.txt")
    recs = [dict(x.split("=", 1) for x in line.split())
            for line in open(path) if line.strip() and not line.startswith("#")]
    assert recs
    for r in recs:
        assert set(r) == {"kernel", "workload", "source_sha", "dram_bytes_per_launch"}
        assert r["workload"] in wl.WORKLOADS
        assert len(r["source_sha"]) == 16 and int(r["source_sha"], 16) >= 0
        assert float(r["dram_bytes_per_launch"]) > 0


def test_peaks_measured_or_fallback(tmp_path):
    peaks, src = bench.load_peaks(str(tmp_path))
    assert src == "fallback" and peaks == bench.FALLBACK_PEAKS
    peaks["hbm_gbs"] = 1.0                                       # a copy, not the constant
    assert bench.FALLBACK_PEAKS["hbm_gbs"] != 1.0
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6500.0}))
    peaks, src = bench.load_peaks(str(tmp_path))
    assert src == "measured" and peaks["hbm_gbs"] == 6500.0


def test_roofline_bound_peak_and_fractions():
    """Bound by arithmetic intensity; each contraction against its own dense peak (BF16
    measured rate x the nominal ratio of its kind); HBM-bound work against the copy rate."""
    import pytest
    from mixed_precision_tensor_gb300 import workloads as wl
    peaks = {"hbm_gbs": 6000.0, "bf16_tflops": 2000.0, "bf16_tflops_sustained": 1500.0}
    W = wl.WORKLOADS

    def at(w, tflops):                      # step time at which w runs at `tflops`
        return w.flops / (tflops * 1e12) * 1e3

    c2 = W["fp16_gemm_8192"]
    r = bench.roofline_entry(c2, at(c2, 1000.0), peaks, "measured", 123.0)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s" and r["traffic"] == 123.0
    assert r["peak"] == 2000.0 and r["achieved"] == pytest.approx(1000.0)
    assert r["frac"] == pytest.approx(0.5)
    assert r["frac_of_sustained"] == pytest.approx(1000.0 / 1500.0)
    assert r["peak_source"] == "measured (bf16_tflops)"
    for name, peak in (("tf32_gemm_4096x4096x16384", 1000.0), ("fp8e4m3_gemm_8192", 4000.0),
                       ("fp32_3xtf32_4096x4096x16384", 2000.0 / 2.0 / 3.0),  # TF32 / 3
                       ("bf16_proj_16384x4096x4096", 2000.0)):
        r = bench.roofline_entry(W[name], 1.0, peaks, "measured", None)
        assert r["bound"] == "tensor" and r["peak"] == pytest.approx(peak), name
    # 512 x 256^3 FP16 -> FP16, beta != 0: A, B, C read and D written once, 2 bytes each
    c5 = W["fp16_batched_512x256"]
    assert c5.algorithmic_bytes() == 4 * 512 * 256 * 256 * 2
    ms = c5.algorithmic_bytes() / 3000e9 * 1e3                    # 3000 GB/s
    r = bench.roofline_entry(c5, ms, peaks, "fallback", None)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] == 6000.0
    assert r["achieved"] == pytest.approx(3000.0) and r["frac"] == pytest.approx(0.5)
    assert r["frac_of_sustained"] is None and r["peak_source"] == "fallback (hbm_gbs)"
