"""Host logic of bench.py that decides what the JSON line may claim, without a GPU:
the clock summary from nvidia-smi samples (the timed region only; throttle reasons),
the DRAM-traffic record (reported only while the kernel sources match the digest it
was measured on) and the choice between measured and fallback peaks."""
import datetime as dt
import hashlib
import json
import os

import bench

FMT = "%Y/%m/%d %H:%M:%S.%f"


def _line(t, sm, smax=2070, hw="Not Active", hwt="Not Active", swt="Not Active",
          cap="Not Active"):
    return ", ".join([t.strftime(FMT)[:-3], "0", str(sm), str(smax), "900.0",
                      "0x0000000000000000", hw, hwt, swt, cap])


def test_clock_summary_uses_the_timed_region_only():
    t0 = dt.datetime(2026, 1, 1, 12, 0, 0)
    lines = [_line(t0 - dt.timedelta(seconds=1), 2070, hwt="Active"),   # before: ignored
             "garbage line", "",
             _line(t0 + dt.timedelta(milliseconds=100), 1400, cap="Active"),
             _line(t0 + dt.timedelta(milliseconds=200), 1500),
             _line(t0 + dt.timedelta(milliseconds=300), 1450, cap="Active"),
             _line(t0 + dt.timedelta(seconds=5), 900, hw="Active")]          # after: ignored
    s = bench.summarise_clocks("\n".join(lines), t0, t0 + dt.timedelta(seconds=1))
    assert s["sm_mhz"] == 1450 and s["sm_max_mhz"] == 2070
    assert s["samples"] == 3 and s["samples_in_timed_region"] == 3
    assert s["reasons"] == ["sw_power_cap"]


def test_clock_summary_falls_back_to_the_last_samples():
    t0 = dt.datetime(2026, 1, 1, 12, 0, 0)
    lines = [_line(t0 + dt.timedelta(seconds=i), 1000 + 100 * i,
                   swt="Active" if i == 4 else "Not Active") for i in range(5)]
    # a region that no sample falls in: the last three samples stand in, flagged as such
    s = bench.summarise_clocks("\n".join(lines), t0 - dt.timedelta(hours=1),
                               t0 - dt.timedelta(minutes=59))
    assert s["samples_in_timed_region"] == 0 and s["samples"] == 3
    assert s["sm_mhz"] == 1300 and s["reasons"] == ["sw_thermal_slowdown"]
    assert bench.summarise_clocks("", t0, t0) is None


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
