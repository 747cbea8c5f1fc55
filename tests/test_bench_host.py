"""Host-side logic of bench.py, on the CPU: clock summaries, the roofline regime of each
workload, the traffic record's source check, the whole-job rate and the argument rules."""
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from speculative_decoding_drafter_gb300.synth import CONFIGS  # noqa: E402

PEAKS = {"hbm_gbs": 6772.9, "bf16_tflops": 1944.7}


def row(sm, mx, reasons=()):
    names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
    return [str(sm), str(mx), "900.0", "0x0"] + ["Active" if n in reasons else "Not Active" for n in names]


def test_clock_summary_median_max_and_reasons():
    rows = [row(1000, 2070), row(2070, 2070), row(2070, 2070, ["sw_power_cap"]), row(2000, 2070)]
    s = bench.ClockSampler.summarize(rows, 0)
    assert s["sm_mhz"] == 2035.0 and s["sm_max_mhz"] == 2070.0 and s["samples"] == 4
    assert s["reasons"] == ["sw_power_cap"]
    # the lead-in samples are skipped
    assert bench.ClockSampler.summarize(rows, 1)["sm_mhz"] == 2070.0
    # a thermal event is reported, malformed lines are ignored
    s = bench.ClockSampler.summarize([row(2070, 2070, ["hw_thermal_slowdown"]), ["[N/A]", "x"]], 0)
    assert s["reasons"] == ["hw_thermal_slowdown"] and s["samples"] == 1
    assert bench.ClockSampler.summarize([], 0) == {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"],
                                                   "samples": 0}


def test_clock_samples_are_taken_from_the_timed_region_only():
    import datetime

    t0 = datetime.datetime(2026, 12, 2, 10, 0, 0)
    ts = lambda ms: (t0 + datetime.timedelta(milliseconds=ms)).strftime(bench.ClockSampler.TS_FORMAT)[:-3]
    rows = [row(2070, 2070) + [ts(-40)], row(2070, 2070) + [ts(-20)], row(1800, 2070, ["sw_power_cap"]) + [ts(5)],
            row(1750, 2070, ["sw_power_cap"]) + [ts(25)], row(2070, 2070) + [ts(60)]]
    inside = bench.ClockSampler.window(rows, t0, t0 + datetime.timedelta(milliseconds=30))
    s = bench.ClockSampler.summarize(inside, 0)
    assert s["samples"] == 2 and s["sm_mhz"] == 1775.0 and s["reasons"] == ["sw_power_cap"]
    # a region shorter than the sampling period keeps the first sample after its start
    short = bench.ClockSampler.window(rows, t0 + datetime.timedelta(milliseconds=6),
                                      t0 + datetime.timedelta(milliseconds=8))
    assert len(short) == 1 and short[0][0] == "1750"
    # without marks (or without timestamps) every sample is kept
    assert bench.ClockSampler.window(rows, None, None) == rows
    bare = [r[:8] for r in rows]
    assert bench.ClockSampler.window(bare, t0, t0) == bare


def test_roofline_regime_of_each_workload():
    assert bench.roofline_bound(CONFIGS["8b_b1"], PEAKS) == "hbm"
    assert bench.roofline_bound(CONFIGS["27b_b8"], PEAKS) == "hbm"
    assert bench.roofline_bound(CONFIGS["8b_b32"], PEAKS) == "tensor"
    assert bench.roofline_bound(CONFIGS["large_vocab"], PEAKS) == "tensor"


def test_traffic_record_is_used_only_for_the_sources_it_was_taken_on(tmp_path, monkeypatch):
    rec = {"8b_b1": {"source_sha": bench.dominant_source_sha(), "dram_bytes_per_launch": 123},
           "27b_b8": {"source_sha": "0000000000000000", "dram_bytes_per_launch": 456}}
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "dominant_source_sha", lambda: rec["8b_b1"]["source_sha"])
    assert bench.recorded_traffic(CONFIGS["8b_b1"]) == 123
    assert bench.recorded_traffic(CONFIGS["27b_b8"]) is None  # taken on other sources
    assert bench.recorded_traffic(CONFIGS["tiny"]) is None  # never taken


def test_committed_traffic_record_is_consistent():
    """Each committed figure names its sources and is the sum of the bytes read and written."""
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as fh:
        rec = json.load(fh)
    for name, ent in rec.items():
        if name.startswith("_"):
            continue
        assert name in CONFIGS
        assert len(ent["source_sha"]) == 16
        assert ent["dram_bytes_per_launch"] == ent["read"] + ent["write"]


def test_whole_job_rate_is_all_ranks_over_the_slowest():
    assert bench.whole_job_rate(16, 1000, 1, 205.4) == pytest.approx(16 * 1000 / 0.2054)
    assert bench.whole_job_rate(16, 1000, 4, 210.0) == pytest.approx(4 * 16 * 1000 / 0.210)


@pytest.mark.parametrize("argv", [["--warmup", "2"], ["--steps", "0"]])
def test_timing_rules_are_enforced(argv, monkeypatch):
    monkeypatch.setattr(sys, "argv", ["bench.py"] + argv)
    with pytest.raises(SystemExit):
        bench.parse_args()


def test_defaults_finish_quickly_and_name_the_headline_workload(monkeypatch):
    monkeypatch.setattr(sys, "argv", ["bench.py"])
    a = bench.parse_args()
    # the largest single-GPU workload (1024 rows of a 262144-token vocabulary) is the headline
    assert a.gpus == 1 and a.warmup >= 3 and a.config == "large_vocab" and a.impl == "ours" and a.op == "select"


@pytest.mark.parametrize("steps,every,n", [(20, 2, 10), (10, 1, 10), (5, 1, 5), (1000, 8, 125), (80, 8, 10)])
def test_enough_lm_head_launches_are_bracketed(steps, every, n):
    assert bench.profile_every(steps) == every
    assert len(range(0, steps, bench.profile_every(steps))) == n


def test_both_arms_report_the_same_config():
    for name in CONFIGS:
        assert bench.bench_config(CONFIGS[name], 1) == bench.bench_config(CONFIGS[name], 1)
    cfg = CONFIGS["large_vocab"]
    c = bench.bench_config(cfg, 1)
    assert c["workload"].startswith("large_vocab: B=64 T=16 H=5376 V=262144 k=16 D=512")
    assert set(c) == {"workload", "l2", "parallelism"}
