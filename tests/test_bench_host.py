"""Host logic of bench.py that needs no GPU: the summary of the nvidia-smi
clock samples that goes into the bench line (median SM clock, maximum SM
clock, throttle reasons seen inside the timed region), the oracle leg
(cpu_baseline and the reference arm) timing the oracle of the measured step,
and the markdown rendering of a --table run."""
import datetime
import json
import os
import pathlib
import subprocess
import sys

import pytest

import bench

REPO = pathlib.Path(__file__).resolve().parent.parent


def _line(t, sm, mx=2070, reasons=("Not Active",) * 4):
    stamp = datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    return ", ".join([stamp, "0", str(sm), str(mx), "1100.50", "0x0000000000000000",
                      *reasons]) + "\n"


T0 = 1_800_000_000.0


def test_median_and_max_over_the_timed_region():
    lines = [_line(T0 + 0.2 * k, sm) for k, sm in enumerate([1500, 2070, 2070, 1980, 2070])]
    got = bench.summarise_clocks(lines, T0 + 0.15, T0 + 0.85)
    # samples at 0.2, 0.4, 0.6, 0.8 fall inside (0.0 is 150 ms before the start)
    assert got == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 4,
                   "in_timed_region": True}


def test_reasons_are_taken_only_inside_the_timed_region():
    hot = ("Not Active", "Active", "Not Active", "Active")      # hw_thermal, sw_power_cap
    lines = [_line(T0, 2070, reasons=("Active",) * 4),          # before the region
             _line(T0 + 1.0, 1900, reasons=hot), _line(T0 + 1.2, 1950),
             _line(T0 + 3.0, 2070, reasons=("Active",) * 4)]    # after it
    got = bench.summarise_clocks(lines, T0 + 0.95, T0 + 1.25)
    assert got["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]
    assert got["samples"] == 2 and got["in_timed_region"]
    assert got["sm_mhz"] == 1950.0


def test_every_sample_is_used_when_none_fell_inside():
    lines = [_line(T0, 1800), _line(T0 + 0.2, 1900, reasons=("Active",) + ("Not Active",) * 3)]
    got = bench.summarise_clocks(lines, T0 + 5.0, T0 + 5.01)
    assert got["samples"] == 2 and not got["in_timed_region"]
    assert got["reasons"] == ["hw_slowdown"]


def test_malformed_and_unsupported_fields_are_skipped():
    lines = ["\n", "garbage\n", _line(T0, "[N/A]"), _line(T0 + 0.1, 2070)]
    got = bench.summarise_clocks(lines, T0 - 1, T0 + 1)
    assert got["samples"] == 1 and got["sm_mhz"] == 2070.0
    assert bench.summarise_clocks(["x\n"], T0, T0 + 1) is None
    assert bench.summarise_clocks([], None, None) is None


def test_sampler_runs_a_fake_nvidia_smi_and_summarises_its_output(tmp_path, monkeypatch):
    """The sampler's process handling end to end, with a stand-in
    nvidia-smi on PATH that prints one sample every 50 ms until stopped."""
    import os
    import time

    fake = tmp_path / "nvidia-smi"
    fake.write_text(
        "#!/usr/bin/env python3\n"
        "import datetime, sys, time\n"
        "while True:\n"
        "    s = datetime.datetime.now().strftime('%Y/%m/%d %H:%M:%S.%f')[:-3]\n"
        "    print(f'{s}, 0, 1965, 2070, 900.00, 0x0, Not Active, Not Active, Not Active, "
        "Active', flush=True)\n"
        "    time.sleep(0.05)\n")
    fake.chmod(0o755)
    monkeypatch.setenv("PATH", f"{tmp_path}{os.pathsep}{os.environ['PATH']}")
    s = bench.ClockSampler("0", use_nvml=False)
    s.start()
    s.mark_start()
    time.sleep(0.4)
    s.mark_stop()
    got = s.stop()
    assert got is not None and got["in_timed_region"]
    assert got["sm_mhz"] == 1965.0 and got["sm_max_mhz"] == 2070.0
    assert got["reasons"] == ["sw_power_cap"] and got["samples"] >= 3
    assert got["source"] == "nvidia-smi -lms 20"
    assert not os.path.exists(s.path)


def test_sampler_polls_nvml_when_the_library_loads(tmp_path, monkeypatch):
    """The NVML path of the sampler against a stand-in libnvidia-ml built
    here: a 0.2 s region gets dozens of samples at the 5 ms period, and the
    event-reason bits map to the same names as nvidia-smi's columns."""
    import shutil
    import subprocess
    import time
    if not shutil.which("gcc"):
        pytest.skip("gcc needed for the stand-in library")
    src = tmp_path / "fake_nvml.c"
    src.write_text(
        "int nvmlInit_v2(void) { return 0; }\n"
        "int nvmlDeviceGetHandleByUUID(const char* u, void** h) { *h = (void*)1; return 0; }\n"
        "int nvmlDeviceGetMaxClockInfo(void* h, int t, unsigned* v) { *v = 2070; return 0; }\n"
        "int nvmlDeviceGetClockInfo(void* h, int t, unsigned* v) { *v = 1995; return 0; }\n"
        "int nvmlDeviceGetPowerUsage(void* h, unsigned* v) { *v = 812500; return 0; }\n"
        "int nvmlDeviceGetCurrentClocksEventReasons(void* h, unsigned long long* r)\n"
        "{ *r = 0x4 | 0x40; return 0; }\n")
    lib = tmp_path / "libfakenvml.so"
    subprocess.run(["gcc", "-shared", "-fPIC", "-o", str(lib), str(src)], check=True)
    monkeypatch.setattr(bench._NvmlClocks, "LIB", str(lib))
    s = bench.ClockSampler("GPU-fake")
    s.start()
    s.mark_start()
    time.sleep(0.2)
    s.mark_stop()
    got = s.stop()
    assert got["source"] == "nvml every 5 ms" and got["in_timed_region"]
    assert got["samples"] >= 10
    assert got["sm_mhz"] == 1995.0 and got["sm_max_mhz"] == 2070.0
    assert got["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]


@pytest.mark.parametrize("variant,extra", [
    ("fused", {}), ("clipped", {"max_norm": 0.5}), ("zero3", {}), ("onebit", {}),
    ("zero3_gather_units", {}), ("staged_grads", {}),
    ("compressed", {"codec": "sign", "ef": True}), ("compressed", {"codec": "int8"})])
def test_reference_arm_times_the_oracle_of_the_measured_step(variant, extra):
    """bench.py --impl reference (and the cpu_baseline of a --variant line)
    time the oracle function that defines the step the line measures, on the
    line's own config, with the thread count that function really uses."""
    import argparse
    args = argparse.Namespace(workload="uneven", variant=variant, steps=1, warmup=3,
                              codec=extra.get("codec", "int8"), ef=extra.get("ef", False),
                              max_norm=extra.get("max_norm", 1.0))
    line = bench.run_reference(args)
    cfg = line["config"]
    assert line["impl"] == "reference" and cfg["variant"] == variant
    assert cfg["R"] == 7 and cfg["M"] == 4 and line["value"] > 0
    fn = bench.ORACLE_FN[variant]
    assert line["cpu_baseline"]["sample"].startswith(fn)
    assert (line["cpu_baseline"]["cores"] > 1) == (fn == "oracle_dp_step_mt" and
                                                    (os.cpu_count() or 1) > 1)
    if variant == "compressed":
        assert cfg["codec"] == extra["codec"] and cfg["error_feedback"] == extra.get("ef", False)
    if variant == "clipped":
        assert cfg["max_norm"] == 0.5
    if variant == "onebit":
        assert cfg["freeze_step"] == 1 and cfg["align"] == 128


def test_table_oracle_rows_of_the_step_variants():
    rows = bench.oracle_variant_rows(n=1 << 14, reps=1)
    assert [r["variant"] for r in rows] == ["clipped"] + ["compressed"] * 6 + ["onebit", "zero3"]
    assert {(r.get("codec"), r.get("ef")) for r in rows if r["variant"] == "compressed"} == {
        (c, e) for c in ("fp16", "int8", "sign") for e in (False, True)}
    for r in rows:
        assert r["oracle"] == bench.ORACLE_FN[r["variant"]] and r["params_per_s"] > 0
        assert r["sample_params"] == 1 << 14 and r["oracle_threads"] == 1


def test_cpu_baseline_carries_the_all_core_and_one_core_oracle_rates():
    """The bench line's cpu_baseline times the oracle of the measured step on
    every host core and on one core, over the same prepared sample."""
    from zgen import workloads as W
    wl = W.uneven()
    cpu = bench.oracle_baseline(wl, {"variant": "fused"}, target_s=0.05, sample_elems=1 << 16)
    assert cpu["kind"] == "oracle" and cpu["unit"] == "params/s"
    assert cpu["value"] > 0 and cpu["value_1core"] > 0
    assert cpu["cores"] == (os.cpu_count() or 1) and cpu["cores_1core"] == 1
    assert cpu["sample"].startswith("oracle_dp_step_mt over the first 65,536 params")
    assert "1 thread(s)" in cpu["sample_1core"]
    # a single-core oracle (the clipped step's) is reported once
    one = bench.oracle_baseline(wl, {"variant": "clipped", "max_norm": 1.0}, target_s=0.05,
                                sample_elems=1 << 14)
    assert one["cores"] == 1 and one["value_1core"] == one["value"]


def test_render_table_writes_every_section_from_the_json_lines(tmp_path):
    """`bench.py --render-table` turns the JSON lines of a --table run into
    the markdown tables of the all-workload profile."""
    rows = [
        {"workload": "llama-3.2-1b", "R": 8, "M": 1, "N": 1235814400, "variant": "fused",
         "ms": 10.5574, "params_per_s": 1.1706e11, "bytes_per_param": 56, "GB_s": 6555.2,
         "frac_of_measured_peak": 0.9772, "l2": "inputs far larger than L2; flushed",
         "ms_clean_l2": 10.555, "frac_clean_l2": 0.9775},
        {"workload": "tiny", "R": 4, "M": 2, "N": 65536, "variant": "fused", "ms": 0.0027,
         "params_per_s": 2.4e10, "bytes_per_param": 48, "GB_s": 1168.9,
         "frac_of_measured_peak": 0.1743, "l2": "warm: inputs resident"},
        {"workload": "sweep R=4 S=1048576", "R": 4, "M": 1, "N": 4194304, "variant": "fused",
         "ms": 0.0355, "params_per_s": 1.18e11, "bytes_per_param": 40, "GB_s": 4731.8,
         "frac_of_measured_peak": 0.7054, "l2": "inputs far larger than L2; flushed",
         "ms_clean_l2": 0.0268, "frac_clean_l2": 0.935},
        {"workload": "llama-3.2-1b", "R": 8, "M": 1, "N": 1235814400, "variant": "clipped",
         "launches": 2, "ms": 12.3822, "params_per_s": 9.98e10, "bytes_per_param": 64,
         "GB_s": 6387.6, "frac_of_measured_peak": 0.9523},
        {"clocks": {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 9}},
        {"workload": "tiny", "oracle_threads": 1, "sample_params": 65536,
         "params_per_s": 3.6e7, "GB_s": 1.7},
    ]
    path = tmp_path / "table.jsonl"
    path.write_text("".join(json.dumps(r) + "\n" for r in rows) + "not json\n")
    out = subprocess.run([sys.executable, str(REPO / "bench.py"), "--render-table", str(path)],
                         capture_output=True, text=True, check=True, cwd=REPO).stdout
    assert ("| llama-3.2-1b | 8 | 1 | 1,235,814,400 | fused | > L2 | 56 | 10.5574 ms | 117.06 | "
            "6555.2 | 0.977 | 10.5550 ms | 0.978 |") in out
    assert "| tiny | 4 | 2 | 65,536 | fused | warm | 48 | 2.70 µs |" in out
    assert "| 4 | 1,048,576 | 4,194,304 | > L2 | 35.50 µs |" in out and "26.80 µs | 0.935 |" in out
    assert "| clipped | 2 | 64 | 12.3822 |" in out
    assert "median 2070 MHz of 2070, throttle reasons: none (9 samples)" in out
    assert "| tiny | 1 | 36.0 | 1.7 |" in out
