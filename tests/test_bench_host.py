"""Host logic of bench.py (no GPU): clock-sample windowing, the recorded-traffic lookup and the reference arm's config."""

import datetime
import hashlib
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _line(ts, clk, reasons=("Not Active",) * 4):
    stamp = datetime.datetime.fromtimestamp(ts).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    return ", ".join([stamp, "0", str(clk), "2070", "900.0", "0x0"] + list(reasons)) + "\n"


def test_clock_summary_keeps_only_the_timed_window(tmp_path):
    import bench
    t0 = 1_800_000_000.0
    path = tmp_path / "clocks.csv"
    with open(path, "w") as f:
        f.write(_line(t0 - 1.0, 2070))                                   # before: idle, ignored
        f.write(_line(t0 + 0.05, 1900, ("Not Active",) * 3 + ("Active",)))
        f.write(_line(t0 + 0.15, 1850, ("Not Active",) * 3 + ("Active",)))
        f.write(_line(t0 + 0.25, 1950))
        f.write(_line(t0 + 2.0, 2070, ("Active",) + ("Not Active",) * 3))  # after: ignored
        f.write("garbage line\n")
    c = bench.ClockSampler(0)
    c.path = str(path)
    c.marks = [t0, t0 + 0.3]
    out = c.summarize()
    assert out["samples"] == 3
    assert out["sm_mhz"] == 1900 and out["sm_mhz_min"] == 1850 and out["sm_max_mhz"] == 2070
    assert out["reasons"] == ["sw_power_cap"]            # hw_slowdown came after the window


def test_recorded_traffic_needs_the_captured_source(tmp_path, monkeypatch):
    import bench
    src = tmp_path / "kernel.cu"
    src.write_text("// kernel source\n")
    sha = hashlib.sha256(src.read_bytes()).hexdigest()[:16]
    (tmp_path / "profiles").mkdir()
    rec = {"w": {"source": "kernel.cu", "source_sha": sha, "dram_bytes_per_launch": 1000, "scale_to_full": 4.0}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.recorded_traffic("w") == 4000
    assert bench.recorded_traffic("other") is None
    src.write_text("// kernel source, changed\n")          # the counters no longer describe this kernel
    assert bench.recorded_traffic("w") is None


def test_reference_arm_prints_our_config(monkeypatch):
    """The reference arm reports the same config as ours (the driver compares them),
    for the default step and with the bf16-partials option.  The oracle's sample is
    cut to a few rows so the test stays fast; its config does not depend on it."""
    import numpy as np
    import bench
    import workloads
    rng = np.random.default_rng(0)
    monkeypatch.setattr(bench, "time_oracle_fraction",
                        lambda cfg, s, device=None: (0, rng.standard_normal((1, 2, 576)),
                                                     rng.standard_normal((40, 576)), 1, 40))
    for argv in (["--impl", "reference", "--steps", "1", "--warmup", "1"],
                 ["--impl", "reference", "--steps", "1", "--warmup", "1", "--partials", "bf16"],
                 ["--impl", "reference", "--steps", "1", "--warmup", "1", "--workload", "dsv3"]):
        args = bench.parse(argv)
        cfg = workloads.config(args.workload)
        out = bench.run_reference(args, cfg, 0, 1)
        assert out["impl"] == "reference"
        assert out["config"] == bench.config_dict(cfg, workloads.lengths(cfg), 1, None, args.partials)
        assert out["metric"] == bench.METRIC and out["higher_is_better"] is True
