"""The benchmark's host-side arithmetic without a GPU: algorithmic bytes and
flops, the roofline's bound and fractions, the DRAM-traffic record's gating on
the kernel source, and the clock-sample summaries that decide whether a
number is kept."""
import json

import pytest

import bench

PEAKS = {"hbm_gbs": 6707.2, "bf16_tflops": 1941.9, "bf16_tflops_sustained": 1734.6,
         "source": "measured"}


def test_algorithmic_bytes_and_flops():
    B, d, V = 64, 4096, 151936
    by, fl = bench.algorithmic(B, d, V)
    # W once, H once, the ids (int64), per-row temperature (fp32) and seed (u64)
    assert by == V * d * 2 + B * d * 2 + B * 8 + B * 4 + B * 8
    assert fl == 2.0 * B * V * d
    by_m, _ = bench.algorithmic(B, d, V, mask=True, tiles=True, seeds=False)
    nt = (V + 127) // 128
    assert by_m == V * d * 2 + B * d * 2 + B * 8 + B * 4 + B * ((V + 31) // 32) * 4 + B * nt * 12


def test_roofline_bound_switches_at_the_crossover():
    d, V = 4096, 151936
    # crossover batch: 2 B V d / F = (V d 2) / BW  =>  B = F / BW (bytes of H aside)
    cross = PEAKS["bf16_tflops"] * 1e12 / (PEAKS["hbm_gbs"] * 1e9)
    lo = bench.roofline(int(cross) - 20, d, V, 200.0, PEAKS)
    hi = bench.roofline(int(cross) + 20, d, V, 400.0, PEAKS)
    assert lo["bound"] == "hbm" and lo["unit"] == "GB/s" and "frac_of_sustained" not in lo
    assert hi["bound"] == "tensor" and hi["unit"] == "TFLOP/s"
    assert hi["frac_of_sustained"] > hi["frac"]


def test_roofline_fraction_is_achieved_over_peak():
    B, d, V = 64, 4096, 151936
    by, _ = bench.algorithmic(B, d, V)
    us = by / (PEAKS["hbm_gbs"] * 1e9) * 1e6  # exactly at the peak
    rf = bench.roofline(B, d, V, us, PEAKS, traffic=123)
    assert rf["frac"] == pytest.approx(1.0, abs=1e-4)
    assert rf["achieved"] == pytest.approx(PEAKS["hbm_gbs"], rel=1e-4)
    assert rf["traffic"] == 123 and rf["algorithmic_bytes"] == by
    assert rf["peak_source"] == "measured"
    rf2 = bench.roofline(B, d, V, 2 * us, PEAKS)
    assert rf2["frac"] == pytest.approx(0.5, abs=1e-4)


def test_traffic_record_only_for_the_current_kernel_source(tmp_path, monkeypatch):
    src = tmp_path / "lm_head_gumbel_gb300" / "csrc"
    src.mkdir(parents=True)
    for name in ("fs_kernels.cuh", "fs_ptx.cuh", "fs_noise.cuh"):
        (src / name).write_text(f"// {name}\n")
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    sha = bench.kernel_source_hash()
    rec = {"source_sha": sha, "launches": {"qwen3-8b/B=64": {"dram_bytes_per_launch": 1234}}}
    path = tmp_path / "profiles" / "stage1_traffic.json"
    path.write_text(json.dumps(rec))
    assert bench.measured_traffic("qwen3-8b", 64) == 1234
    assert bench.measured_traffic("qwen3-8b", 512) is None  # not captured
    (src / "fs_kernels.cuh").write_text("// changed\n")      # the kernel changed since
    assert bench.kernel_source_hash() != sha
    assert bench.measured_traffic("qwen3-8b", 64) is None


def _row(t, sm, reasons=()):
    r = {"t": t, "sm": sm, "sm_max": 2070.0, "power": "1000.0", "active": "0x0",
         "hw_slowdown": "Not Active", "hw_thermal_slowdown": "Not Active",
         "sw_thermal_slowdown": "Not Active", "sw_power_cap": "Not Active"}
    for k in reasons:
        r[k] = "Active"
    return r


def test_clock_summary_inside_the_window():
    rows = [_row(0.0, 900.0), _row(1.0, 2000.0), _row(1.1, 1990.0, ["sw_power_cap"]),
            _row(1.2, 2010.0), _row(5.0, 800.0, ["hw_slowdown"])]
    c = bench.ClockSampler.summarize(rows, 0.95, 1.25)
    assert c["sm_mhz"] == 2000.0 and c["samples"] == 3 and c["window"] == "timed region"
    assert c["reasons"] == ["sw_power_cap"]  # the hw_slowdown sample lies outside
    assert c["sm_max_mhz"] == 2070.0


def test_clock_summary_falls_back_to_the_whole_phase():
    rows = [_row(0.0, 1900.0), _row(10.0, 1950.0, ["hw_thermal_slowdown"])]
    c = bench.ClockSampler.summarize(rows, 5.0, 5.1)  # no sample in a short window
    assert c["window"] == "measurement phase" and c["samples"] == 2
    assert c["reasons"] == ["hw_thermal_slowdown"]
    assert bench.ClockSampler.summarize([], 0.0, 1.0) is None


def test_workload_descriptions_name_the_configuration():
    from lm_head_gumbel_gb300 import workloads as wl
    s = bench.describe(wl.WORKLOADS["qwen3-8b"], 64)
    assert "d=4096" in s and "V=151936" in s and "B=64" in s and "per-row seeds" in s
    s = bench.describe(wl.WORKLOADS["llama3-8b-mask"], 128)
    assert "mask" in s and "x4" in s and "LSE" in s


def test_default_run_times_every_workload():
    """The default run's headline head plus its other workloads cover every
    workload of the benchmark set, each with its own batch sizes and a
    description and L2 note taken from its definition."""
    from lm_head_gumbel_gb300 import workloads as wl
    assert set(bench.OTHER_WORKLOADS) == set(wl.WORKLOADS)
    for name in bench.OTHER_WORKLOADS:
        w = wl.WORKLOADS[name]
        text = bench.describe(w, "/".join(str(b) for b in w.batches))
        assert f"d={w.d}" in text and f"V={w.V}" in text
        note = bench.l2_note(w.V, w.d)
        assert ("fits in L2" in note) == (w.V * w.d * 2 <= bench.L2_BYTES)
    assert "fits in L2" in bench.l2_note(4096, 256)       # the tiny head: warm
    assert "exceed L2" in bench.l2_note(151936, 4096)     # the Qwen3-8B head: cold


def test_traffic_record_covers_every_timed_point():
    """The committed DRAM-traffic record has an entry for every (workload,
    batch) the default run times -- the headline head's sweep and every other
    workload's batches -- each a plausible multiple of the point's algorithmic
    bytes.  (Whether it was taken on the current kernel source is decided at
    run time: an older record yields `traffic: null`.)"""
    import os
    from lm_head_gumbel_gb300 import workloads as wl
    with open(os.path.join(bench.ROOT, "profiles", "stage1_traffic.json")) as f:
        rec = json.load(f)
    launches = rec["launches"]
    for name in bench.OTHER_WORKLOADS:
        w = wl.WORKLOADS[name]
        for B in w.batches:
            ent = launches.get(f"{name}/B={B}")
            assert ent is not None, (name, B)
            algo, _flops = bench.algorithmic(B, w.d, w.V, seeds=w.per_row_seeds,
                                             mask=bool(w.mask_frac), tiles=w.want_lse)
            assert 0.95 * algo <= ent["dram_bytes_per_launch"] <= 2.0 * algo, (name, B)

