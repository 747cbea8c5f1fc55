#!/usr/bin/env python3
"""Benchmark of the DFlash2 candidate-selector head on GB300.

One step = one dflash2_select call over a whole draft block: LM head with fused
top-k, gate, k x k lattice and greedy walk for every sequence of the workload
(default: the largest single-GPU workload, the large-vocabulary head at 1024 rows,
B=64 T=16 H=5376 V=262144 k=16 D=512, tensor-bound).  The same JSON line carries
the batch-1 figures of the 8B-class head (B=1 T=16 H=4096 V=151936 k=8 D=256,
HBM-bound) under "batch1", measured in the same run.  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

Multi-GPU: launched one process per GPU (torchrun); every rank runs an
independent replica of the workload (sequences shard with no exchange step),
so scaling is weak and the value is the rows of all ranks over the slowest
rank's time.  --impl reference times the CPU oracle (rank 0 only).
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from speculative_decoding_drafter_gb300.synth import CONFIGS, make_inputs  # noqa: E402

METRIC = "selector draft rows/s and µs/block; % of HBM or bf16 tensor roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
LAUNCHES_PER_STEP = 2  # LM head with fused top-k and gate; merge + lattice + walk
PROFILE_EVERY = 8  # at most every 8th LM-head launch of a timed region is bracketed by events
MIN_PROFILED = 10  # ... but at least this many launches are (every launch at 10 steps or fewer)
NOMINAL_HBM_GBS = 8000.0  # GB300 HBM3e, nominal (~8 TB/s)
BATCH1_CONFIG = "8b_b1"
BATCH1_STEPS = 400
DOMINANT_SOURCES = ["speculative_decoding_drafter_gb300/csrc/gemm_tc.cu", "speculative_decoding_drafter_gb300/csrc/ptx.cuh",
                    "speculative_decoding_drafter_gb300/csrc/topk.cuh"]


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default="large_vocab", choices=list(CONFIGS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--op", default="select", choices=["select", "conv", "topk", "walk"],
                    help="select: the selector head (default); conv: the dynamic local convolution; "
                         "topk: top-k A/B (fused epilogue vs materialised logits, ours vs torch.topk)")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the timed oracle sample")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--no-batch1", action="store_true",
                    help=f"skip the companion batch-1 measurement ({BATCH1_CONFIG}) in the select line")
    a = ap.parse_args()
    if a.warmup < 3:
        ap.error("--warmup must be at least 3")
    if a.steps < 1:
        ap.error("--steps must be at least 1")
    return a


def max_over_ranks(value: float, dist, device) -> float:
    """The largest of every rank's value (the slowest rank's time); identity without a process group."""
    if dist is None:
        return value
    import torch

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(rows_per_rank: int, steps: int, world: int, max_ms: float) -> float:
    """Rows of all ranks per second over the slowest rank's time (weak scaling: every rank runs the workload)."""
    return world * rows_per_rank * steps / (max_ms / 1e3)


def workload_name(cfg) -> str:
    return f"{cfg.name}: B={cfg.B} T={cfg.T} H={cfg.H} V={cfg.V} k={cfg.k} D={cfg.D}"


def bench_config(cfg, world: int) -> dict:
    """The `config` of the select line, identical in both arms."""
    return {"workload": workload_name(cfg),
            "l2": f"inputs larger than L2 (W_vocab {cfg.V * cfg.H * 2 / 1e9:.2f} GB vs 129 MB L2)"
            if cfg.V * cfg.H * 2 > 129e6 else "inputs fit in L2 (warm)",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


def profile_every(steps: int) -> int:
    """Stride of the bracketed LM-head launches: every PROFILE_EVERY-th, or denser so that at
    least MIN_PROFILED launches of the timed region are bracketed."""
    return max(1, min(PROFILE_EVERY, steps // MIN_PROFILED))


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            return json.load(fh), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def roofline_bound(cfg, peaks):
    t_hbm = cfg.V * cfg.H * 2 / (peaks["hbm_gbs"] * 1e9)
    t_tc = 2.0 * cfg.R * cfg.H * cfg.V / (peaks["bf16_tflops"] * 1e12)
    return "hbm" if t_hbm >= t_tc else "tensor"


def dominant_source_sha() -> str:
    h = hashlib.sha256()
    for rel in DOMINANT_SOURCES:  # the kernel's own sources
        with open(os.path.join(ROOT, rel), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(cfg):
    """DRAM bytes per LM-head launch from the committed ncu summary, if it matches this source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as fh:
        rec = json.load(fh)
    ent = rec.get(cfg.name)
    if not ent or ent.get("source_sha") != dominant_source_sha():
        return None
    return ent.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples taken while the timed region runs.

    Each sample carries nvidia-smi's timestamp; mark_start() / mark_end() bracket the timed
    region on the host clock, and window() keeps the samples inside it (a region shorter
    than the 20 ms sampling period keeps the first sample after its start)."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap,timestamp")
    TS_FORMAT = "%Y/%m/%d %H:%M:%S.%f"

    def __init__(self, device_id: str):
        self.device_id = device_id
        self.proc = None
        self.tmp = None
        self.t_start = None
        self.t_end = None

    def start(self):
        self.tmp = tempfile.NamedTemporaryFile(mode="w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", self.device_id, f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=self.tmp, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def mark_start(self):
        self.t_start = datetime.datetime.now()

    def mark_end(self):
        self.t_end = datetime.datetime.now()

    def stop(self):
        if self.proc is not None:
            time.sleep(0.05)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.tmp.flush()
        self.tmp.seek(0)
        rows = [ln.strip().split(", ") for ln in self.tmp.read().splitlines() if ln.strip()]
        self.tmp.close()
        os.unlink(self.tmp.name)
        return self.window(rows, self.t_start, self.t_end)

    @classmethod
    def window(cls, rows, t_start, t_end):
        """The samples taken between t_start and t_end (datetimes on the host clock); if none, the
        first sample after t_start; rows without a readable timestamp are kept only when no row
        has one (an nvidia-smi without the field)."""
        if t_start is None or t_end is None:
            return rows
        stamped = []
        for r in rows:
            try:
                stamped.append((datetime.datetime.strptime(r[8].strip(), cls.TS_FORMAT), r))
            except (IndexError, ValueError):
                continue
        if not stamped:
            return rows
        inside = [r for t, r in stamped if t_start <= t <= t_end]
        if inside:
            return inside
        after = [r for t, r in stamped if t >= t_start]
        return after[:1]

    @staticmethod
    def summarize(rows, t_first: int):
        """Median SM clock and the throttle reasons seen in the samples after t_first (skip the lead-in)."""
        rows = rows[t_first:] or rows
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in rows:
            try:
                sm.append(float(r[0]))
                mx.append(float(r[1]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, r[4:8]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "window": "samples taken inside the timed region"}


def device_id_for_smi(torch) -> str:
    try:
        u = str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "0").split(",")[0]
        return vis or "0"


def time_oracle_rows(cfg, x, rows_per_step: int, step: int):
    """Run the oracle on the first rows_per_step positions of one sequence; returns seconds."""
    import oracle

    b = step % cfg.B
    rows = np.arange(b * cfg.T, b * cfg.T + rows_per_step)
    t0 = time.perf_counter()
    oracle.select(x["hidden"][rows], x["W_vocab"], x["W_sel"], x["pred_cb"], x["succ_cb"], x["anchor"][b:b + 1],
                  cfg.k, rows_per_step)
    return time.perf_counter() - t0


def cpu_baseline(cfg, x, budget_s: float = 20.0):
    """The oracle, as it stands, timed on a bounded sample of the workload (whole sequences if they fit)."""
    import oracle

    t_row = time_oracle_rows(cfg, x, 1, 0)
    n_rows = int(max(1, min(cfg.T, budget_s / max(t_row, 1e-9))))
    t = time_oracle_rows(cfg, x, n_rows, 0)
    line = {"value": n_rows / t, "unit": "rows/s", "cores": oracle.threads(), "kind": "oracle",
            "sample": f"sequence 0, positions 0..{n_rows - 1} of {cfg.T} (full vocabulary, full pipeline), one run"}
    # the same oracle on one core, on as many rows as fit a quarter of the budget
    prev = oracle.set_threads(1)
    try:
        t1 = time_oracle_rows(cfg, x, 1, 0)
        n1 = int(max(1, min(cfg.T, 0.25 * budget_s / max(t1, 1e-9))))
        if n1 > 1:
            t1 = time_oracle_rows(cfg, x, n1, 0)
    finally:
        oracle.set_threads(prev)
    line["value_1_thread"] = n1 / t1
    line["sample_1_thread"] = f"sequence 0, positions 0..{n1 - 1}, one thread"
    return line


def run_reference(args, cfg, rank: int, world: int = 1):
    if rank != 0:
        return 0
    import oracle

    oracle.build()
    x = make_inputs(cfg, 0)
    t_row = time_oracle_rows(cfg, x, 1, 0)
    budget = 150.0 / (args.steps + args.warmup)
    rows_per_step = int(max(1, min(cfg.T, budget / max(t_row, 1e-9))))
    for w in range(args.warmup):
        time_oracle_rows(cfg, x, rows_per_step, w)
    total = 0.0
    for s in range(args.steps):
        total += time_oracle_rows(cfg, x, rows_per_step, s)
    value = rows_per_step * args.steps / total
    sample = (f"per step: sequence (step mod B), positions 0..{rows_per_step - 1} of {cfg.T}, full vocabulary, "
              f"full oracle pipeline")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded; stands in for the pages' GSM8K/MATH-500/HumanEval/MBPP/MT-Bench drafter states)",
        "config": bench_config(cfg, world),
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": oracle.threads(), "kind": "oracle",
                         "sample": sample, "sample_rows_per_step": rows_per_step},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def select_inputs(torch, df, cfg):
    """Device copies of a config's seeded inputs, outputs and a workspace (and the host inputs)."""
    x = make_inputs(cfg, 0)

    def dev_bf16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()

    d = {n: dev_bf16(x[n]) for n in ("hidden", "W_vocab", "W_sel", "pred_cb", "succ_cb")}
    d["anchor"] = torch.from_numpy(x["anchor"]).cuda()
    k = cfg.k
    d["lattice"] = torch.empty((cfg.R, k + k * k), dtype=torch.float32, device="cuda")
    d["draft"] = torch.empty((cfg.B, cfg.T), dtype=torch.int32, device="cuda")
    d["ws"] = df.Workspace(df.make_dims(cfg.B, cfg.T, cfg.H, cfg.V, k, cfg.D))
    return x, d


def timed_select(torch, df, cfg, d, steps: int, warmup: int, sampler=None, barrier=lambda: None):
    """Device-timed region of `steps` dflash2_select calls, back to back on one stream, after
    `warmup` untimed calls.  The LM-head launch of every profile_every(steps)-th call is
    bracketed by its own CUDA events (an event between two launches keeps the second from
    starting under the first, so the calls in between run as a drafting loop runs them).
    Returns (total ms, [LM-head us of the bracketed launches], per-step us of the windows
    between them, clock samples)."""

    def step():
        df.dflash2_select(d["hidden"], d["W_vocab"], d["W_sel"], d["pred_cb"], d["succ_cb"], d["anchor"], cfg.k,
                          cfg.T, lattice=d["lattice"], draft_ids=d["draft"], workspace=d["ws"])

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    df.dflash2_check_device_status(d["ws"])
    every = profile_every(steps)
    sampled = list(range(0, steps, every))
    eb = [torch.cuda.Event(enable_timing=True) for _ in sampled]
    ee = [torch.cuda.Event(enable_timing=True) for _ in sampled]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for ev in eb + ee:  # torch creates the CUDA event on its first record(); the library needs the handle
        ev.record()
    barrier()
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
        sampler.mark_start()
    start.record()
    for i in range(steps):
        if i % every == 0:
            df.dflash2_profile_events(eb[i // every], ee[i // every])
        elif i % every == 1:
            df.dflash2_profile_events(None, None)
        step()
    end.record()
    torch.cuda.synchronize()
    if sampler:
        sampler.mark_end()
    barrier()
    df.dflash2_profile_events(None, None)
    clock_rows = sampler.stop() if sampler else []
    df.dflash2_check_device_status(d["ws"])
    n_s = len(sampled)
    lm_us = [1e3 * eb[j].elapsed_time(ee[j]) for j in range(n_s)]
    # per-step spread: mean step of each window from one bracketed launch to the next (the last
    # window ends at the end event)
    step_us = [1e3 * eb[j].elapsed_time(eb[j + 1]) / every for j in range(n_s - 1)] + \
        [1e3 * eb[n_s - 1].elapsed_time(end) / (steps - sampled[-1])]
    return start.elapsed_time(end), lm_us, step_us, clock_rows


def percentiles(v):
    return {f"p{q}": float(np.percentile(v, q)) for q in (10, 50, 90)}


def hbm_algorithmic_bytes(cfg) -> int:
    """Per LM-head launch: W_vocab and W_sel streamed once, hidden read once, gate written
    (per vocabulary row H*2 bytes)."""
    return cfg.V * cfg.H * 2 + cfg.D * cfg.H * 2 + cfg.R * cfg.H * 2 + cfg.R * cfg.D * 4


def batch1_companion(torch, df, peaks, device_id):
    """The batch-1 (HBM-bound) workload measured in the same run, for the same JSON line."""
    cfg = CONFIGS[BATCH1_CONFIG]
    _, d = select_inputs(torch, df, cfg)
    sampler = ClockSampler(device_id)
    ms, lm_us, step_us, clock_rows = timed_select(torch, df, cfg, d, BATCH1_STEPS, 10, sampler)
    lm_mean = float(np.mean(lm_us))
    algo = hbm_algorithmic_bytes(cfg)
    gbs = algo / (lm_mean * 1e-6) / 1e9
    gbs_med = algo / (float(np.median(lm_us)) * 1e-6) / 1e9
    out = {"workload": workload_name(cfg), "steps": BATCH1_STEPS, "step_us": 1e3 * ms / BATCH1_STEPS,
           "rows_per_s": cfg.R * BATCH1_STEPS / (ms / 1e3),
           "lm_head_us": {"mean": lm_mean, "median": float(np.median(lm_us)), "launches": len(lm_us),
                          **percentiles(lm_us)},
           "step_us_percentiles": percentiles(step_us),
           "hbm": {"algorithmic_per_launch": algo, "achieved_gbs": gbs, "achieved_gbs_median_launch": gbs_med,
                   "frac_of_measured_copy": gbs / peaks["hbm_gbs"], "measured_copy_gbs": peaks["hbm_gbs"],
                   "frac_of_nominal": gbs / NOMINAL_HBM_GBS, "nominal_gbs": NOMINAL_HBM_GBS,
                   "step_frac_of_measured_copy": algo / (1e-3 * ms / BATCH1_STEPS) / 1e9 / peaks["hbm_gbs"]},
           "traffic": recorded_traffic(cfg),
           "clocks": ClockSampler.summarize(clock_rows, 0) if clock_rows else {"reasons": ["no samples"]}}
    del d
    torch.cuda.empty_cache()
    return out


def run_ours(args, cfg, rank: int, world: int):
    import torch

    from speculative_decoding_drafter_gb300 import dflash2 as df

    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    df.library()
    peaks, peak_kind = load_peaks()
    x, d = select_inputs(torch, df, cfg)
    R, k, K = cfg.R, cfg.k, args.steps

    def barrier():
        if dist is not None:
            dist.barrier()

    device_id = device_id_for_smi(torch)
    sampler = ClockSampler(device_id) if rank == 0 else None
    ms, lm_us, step_us, clock_rows = timed_select(torch, df, cfg, d, K, args.warmup, sampler, barrier)
    ms = max_over_ranks(ms, dist, "cuda")
    lm_ms = float(np.mean(lm_us)) / 1e3
    pct = {"step_us": percentiles(step_us), "lm_head_us": percentiles(lm_us)}

    # ---- end-to-end through the C ABI's host-buffer call (pinned buffers): every step copies
    # hidden and anchor in and the draft, lattice and status word out, and waits for them
    e2e = None
    if not args.no_e2e:
        h_hidden = torch.from_numpy(x["hidden"].view(np.int16)).view(torch.bfloat16).pin_memory()
        h_anchor = torch.from_numpy(x["anchor"]).pin_memory()
        h_lat = torch.empty_like(d["lattice"], device="cpu").pin_memory()
        h_draft = torch.empty_like(d["draft"], device="cpu").pin_memory()
        hws = df.HostWorkspace(df.make_dims(cfg.B, cfg.T, cfg.H, cfg.V, k, cfg.D))

        e2e_step = df.SelectHostPlan(h_hidden, d["W_vocab"], d["W_sel"], d["pred_cb"], d["succ_cb"], h_anchor, k,
                                     cfg.T, lattice_host=h_lat, draft_ids_host=h_draft, workspace=hws)

        for _ in range(args.warmup):
            e2e_step()
        barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(K):
            e2e_step()
        e_ms = max_over_ranks((time.perf_counter() - t0) * 1e3, dist, "cuda")
        h2d = h_hidden.numel() * 2 + h_anchor.numel() * 4
        d2h = h_lat.numel() * 4 + h_draft.numel() * 4 + 4
        e2e = {"value": whole_job_rate(R, K, world, e_ms), "unit": "rows/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e_ms / K, "sync": "per step (inside the call)",
               "api": "dflash2_select_host (SelectHostPlan: buffers bound once)",
               "clock": "host wall clock"}
        del hws, e2e_step

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0

    clocks = ClockSampler.summarize(clock_rows, 0) if clock_rows else {"sm_mhz": None, "sm_max_mhz": None,
                                                                        "reasons": ["no samples"], "samples": 0}
    bound = roofline_bound(cfg, peaks)
    lm_s = lm_ms / 1e3
    med_s = float(np.median(lm_us)) / 1e6
    if bound == "hbm":
        algo = hbm_algorithmic_bytes(cfg)
        achieved, peak, unit = algo / lm_s / 1e9, peaks["hbm_gbs"], "GB/s"
        extra = {"achieved_median_launch": algo / med_s / 1e9, "frac_of_nominal": achieved / NOMINAL_HBM_GBS,
                 "nominal": NOMINAL_HBM_GBS}
    else:
        algo = 2.0 * cfg.R * cfg.H * (cfg.V + cfg.D)  # logits and gate columns of the same launch
        achieved, peak, unit = algo / lm_s / 1e12, peaks["bf16_tflops"], "TFLOP/s"
        sus = peaks.get("bf16_tflops_sustained")
        extra = {"achieved_median_launch": algo / med_s / 1e12, "peak_sustained": sus,
                 "frac_of_sustained": achieved / sus if sus else None,
                 "sm_mhz_median": clocks.get("sm_mhz"),
                 "peak_note": "peak = the measured burst cuBLAS bf16 figure; the sustained figure (a seconds-long "
                              "loop at the power cap) is given beside it"}
    roof = {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit, "frac": achieved / peak,
            "traffic": recorded_traffic(cfg), "kernel": "gemm_tc_kernel (LM head + fused top-k + gate)",
            "kernel_us": lm_ms * 1e3, "kernel_us_median": float(np.median(lm_us)),
            "algorithmic_per_launch": algo,
            "peak_source": f"{peak_kind} (MEASURED_PEAKS.json)" if peak_kind == "measured" else "fallback",
            "kernel_timing": f"CUDA events around every {profile_every(K)}th LM-head launch of the timed region "
                             f"({len(lm_us)} launches, mean; median beside it); step_us percentiles are per-step "
                             f"means of the windows between them", **extra}
    # the same roofline over the whole step (every launch of the call, host gaps included)
    roof["step_frac"] = (lm_ms / (ms / K)) * roof["frac"]

    line = {
        "impl": "ours", "metric": METRIC, "value": whole_job_rate(R, K, world, ms), "unit": "rows/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": ms / K, "us_per_block": 1e3 * ms / K,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; stands in for the pages' GSM8K/MATH-500/HumanEval/MBPP/MT-Bench drafter states)",
        "config": bench_config(cfg, world),
        "roofline": roof,
        "percentiles": pct,
        "gpu_launches": LAUNCHES_PER_STEP * K,
        "clocks": clocks,
        "e2e": e2e,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg, x)
    if world == 1 and not args.no_batch1 and cfg.name != BATCH1_CONFIG:
        del d
        torch.cuda.empty_cache()
        line["batch1"] = batch1_companion(torch, df, peaks, device_id)
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


CONV_SHAPE = (1024, 16, 4096, 16)  # blocks, positions per block, channels, channels per dynamic group


def run_conv(args, rank: int, world: int):
    """The dynamic local convolution (RMS-normalised input) on B=1024 blocks of 16 rows of 4096 channels."""
    import torch

    from speculative_decoding_drafter_gb300 import dflash2 as df
    from speculative_decoding_drafter_gb300.synth import make_conv_inputs

    if rank != 0 and args.impl == "reference":
        return 0
    B, T, C, G = CONV_SHAPE
    c = make_conv_inputs(B, T, C, G, seed=0)
    name = f"dynamic_conv: B={B} T={T} C={C} G={G}, RMS-normalised input"
    peaks, peak_kind = load_peaks()
    R = B * T
    algo = R * C * 2 * 2 + B * C * 2 + R * 2 * (C // G) * 4 + 3 * C * 2  # x in, y out, x_prev, dyn, base+gamma
    if args.impl == "reference":
        import oracle

        oracle.build()
        rows = 64  # bounded sample: the first 4 blocks
        t0 = time.perf_counter()
        steps = 0
        for _ in range(args.steps):
            oracle.dynamic_conv(c["x"][:rows], c["x_prev"][:rows // T], c["base"], c["dyn"][:rows], T, G,
                                gamma=c["gamma"], eps=1e-6)
            steps += 1
        dt = time.perf_counter() - t0
        v = rows * steps / dt
        print(json.dumps({"impl": "reference", "op": "conv", "metric": "dynamic conv rows/s", "value": v,
                          "unit": "rows/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                          "ms_per_step": 1e3 * dt / steps, "higher_is_better": True, "scaling": "weak",
                          "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": {"workload": name},
                          "cpu_baseline": {"value": v, "unit": "rows/s", "cores": oracle.threads(), "kind": "oracle",
                                           "sample": f"{rows} rows per step"},
                          "e2e": {"value": v, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}))
        return 0
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))

    def dev_bf16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()

    x, xp, base, gm = dev_bf16(c["x"]), dev_bf16(c["x_prev"]), dev_bf16(c["base"]), dev_bf16(c["gamma"])
    dyn = torch.from_numpy(c["dyn"]).cuda()
    y = torch.empty_like(x)

    def step():
        df.dflash2_dynamic_conv(x, base, dyn, T, x_prev=xp, gamma=gm, eps=1e-6, G=G, out=y)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(device_id_for_smi(torch)) if rank == 0 else None
    if dist is not None:
        dist.barrier()
    if sampler:
        sampler.start()
        sampler.mark_start()
    start.record()
    for _ in range(args.steps):
        step()
    end.record()
    torch.cuda.synchronize()
    if sampler:
        sampler.mark_end()
    if dist is not None:
        dist.barrier()
    clock_rows = sampler.stop() if sampler else []
    ms = max_over_ranks(start.elapsed_time(end), dist, "cuda")
    if rank == 0:
        s_per = ms / args.steps / 1e3
        achieved = algo / s_per / 1e9
        print(json.dumps({
            "impl": "ours", "op": "conv", "metric": "dynamic conv rows/s", "value": whole_job_rate(R, args.steps, world, ms),
            "unit": "rows/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": name, "l2": f"x alone {R * C * 2 / 1e6:.0f} MB > 129 MB L2"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": achieved / peaks["hbm_gbs"], "traffic": None, "kernel": "dynamic_conv_kernel",
                         "algorithmic_per_launch": algo, "peak_source": peak_kind},
            "gpu_launches": args.steps,
            "clocks": ClockSampler.summarize(clock_rows, 0) if clock_rows else {"reasons": ["no samples"]}}), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


WALK_SHAPE = (8192, 16, 16)  # sequences, positions, candidates: a 143 MB lattice, larger than L2


def fused_walk_cost(torch, df, cfg, steps: int, warmup: int):
    """Step time of dflash2_select against dflash2_select_walk (p_min stop; and inverse-CDF sampling)
    on one config: what moving the confidence walk into the selector call costs."""
    _, d = select_inputs(torch, df, cfg)
    B, T, k = cfg.B, cfg.T, cfg.k
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([0, 47])))
    uni = torch.from_numpy(g.random((B, T), dtype=np.float32)).cuda()
    n_draft = torch.empty((B,), dtype=torch.int32, device="cuda")
    conf = torch.empty((B, T), dtype=torch.float32, device="cuda")
    common = (d["hidden"], d["W_vocab"], d["W_sel"], d["pred_cb"], d["succ_cb"], d["anchor"], k, T)

    def plain():
        df.dflash2_select(*common, lattice=d["lattice"], draft_ids=d["draft"], workspace=d["ws"])

    def pmin():
        df.dflash2_select_walk(*common, temperature=1.0, p_min=0.3, lattice=d["lattice"], draft_ids=d["draft"],
                               n_draft=n_draft, confidence=conf, workspace=d["ws"])

    def sampled():
        df.dflash2_select_walk(*common, temperature=1.0, p_min=0.3, uniforms=uni, lattice=d["lattice"],
                               draft_ids=d["draft"], n_draft=n_draft, confidence=conf, workspace=d["ws"])

    def separate():  # the plain call followed by the stand-alone sampling walk on its lattice
        plain()
        df.dflash2_walk_sample(d["lattice"], B, T, k, temperature=1.0, p_min=0.3, uniforms=uni, n_draft=n_draft,
                               confidence=conf)

    modes = {"select_us": plain, "select_walk_pmin_us": pmin, "select_walk_sampling_us": sampled,
             "select_then_walk_sample_us": separate}
    for f in modes.values():
        for _ in range(warmup):
            f()
    torch.cuda.synchronize()
    # blocks of a few back-to-back calls per mode, the modes interleaved block by block, so that a
    # clock that drifts (a long tensor-bound run settles at the power cap) weighs on every mode alike
    block = 5
    rounds = max(1, steps // block)
    ev = {m: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(rounds)]
          for m in modes}
    for i in range(rounds):
        for m, f in modes.items():
            a, b = ev[m][i]
            a.record()
            for _ in range(block):
                f()
            b.record()
    torch.cuda.synchronize()
    out = {"workload": workload_name(cfg), "steps_per_mode": rounds * block,
           "timing": f"{rounds} rounds of {block} back-to-back calls per mode, the modes interleaved"}
    for m in modes:
        out[m] = 1e3 * sum(a.elapsed_time(b) for a, b in ev[m]) / (rounds * block)
    out["fused_sampling_walk_adds_us"] = out["select_walk_sampling_us"] - out["select_us"]
    out["separate_sampling_walk_adds_us"] = out["select_then_walk_sample_us"] - out["select_us"]
    del d
    torch.cuda.empty_cache()
    return out


def run_walk(args, rank: int, world: int):
    """The walk with confidence, p_min stop and inverse-CDF sampling (and the plain greedy walk) over a
    seeded lattice of WALK_SHAPE.  One warp per sequence, T dependent row reads: latency-bound.  Also
    the cost of the same walk inside the selector call (dflash2_select_walk) on --config."""
    import torch

    from speculative_decoding_drafter_gb300 import dflash2 as df

    if rank != 0:
        return 0
    B, T, k = WALK_SHAPE
    R, W = B * T, k + k * k
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([0, 41])))
    lat = np.empty((R, W), np.float32)
    lat[:, :k] = g.integers(0, 151936, size=(R, k))
    lat[:, k:] = (1.5 * g.standard_normal((R, k * k))).astype(np.float32)
    uni = g.random((B, T), dtype=np.float32)
    tau, p_min = 1.0, 0.3
    name = f"walk: B={B} T={T} k={k}, temperature {tau}, p_min {p_min}, sampling with given uniforms"
    # bytes a walk must touch: per position the chosen predecessor row (k floats), the chosen id, the
    # uniform, and the draft and confidence it writes; plus n_draft per sequence
    algo = R * (k * 4 + 4 + 4 + 4 + 4) + B * 4
    sample_b = 256
    if args.impl == "reference":
        import oracle

        oracle.build()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            oracle.walk_sample(lat[:sample_b * T], sample_b, T, k, tau, p_min, uni[:sample_b])
        dt = time.perf_counter() - t0
        v = sample_b * args.steps / dt
        print(json.dumps({"impl": "reference", "op": "walk", "metric": "sampling walk sequences/s", "value": v,
                          "unit": "sequences/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                          "ms_per_step": 1e3 * dt / args.steps, "higher_is_better": True, "scaling": "weak",
                          "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": {"workload": name},
                          "cpu_baseline": {"value": v, "unit": "sequences/s", "cores": oracle.threads(),
                                           "kind": "oracle", "sample": f"{sample_b} sequences per step"},
                          "e2e": {"value": v, "unit": "sequences/s", "h2d_bytes_per_step": 0,
                                  "d2h_bytes_per_step": 0}}), flush=True)
        return 0
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    peaks, peak_kind = load_peaks()
    d_lat = torch.from_numpy(lat).cuda()
    d_uni = torch.from_numpy(uni).cuda()
    draft = torch.empty((B, T), dtype=torch.int32, device="cuda")
    n_draft = torch.empty((B,), dtype=torch.int32, device="cuda")
    conf = torch.empty((B, T), dtype=torch.float32, device="cuda")

    def sampled():
        df.dflash2_walk_sample(d_lat, B, T, k, temperature=tau, p_min=p_min, uniforms=d_uni, draft=draft,
                               n_draft=n_draft, confidence=conf)

    def greedy():
        df.dflash2_walk(d_lat, B, T, k, out=draft)

    # the walk touches only the rows it chooses (~10 MB), the same ones every call: flush L2 before each
    # timed launch by writing a buffer twice its size, outside the launch's own event pair
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")

    def timed(f):
        for _ in range(args.warmup):
            f()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        for a, b in ev:
            flush.zero_()
            a.record()
            f()
            b.record()
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in ev) / args.steps * 1e3

    sampler = ClockSampler(device_id_for_smi(torch))
    sampler.start()
    sampler.mark_start()
    us = timed(sampled)
    sampler.mark_end()
    clock_rows = sampler.stop()
    greedy_us = timed(greedy)
    sampled()
    torch.cuda.synchronize()
    o_draft, o_n, o_conf = oracle_walk_sample_sample(lat, uni, sample_b, T, k, tau, p_min)
    g_draft, g_n = draft.cpu().numpy()[:sample_b], n_draft.cpu().numpy()[:sample_b]
    agree = float(np.mean(np.all(g_draft == o_draft, axis=1) & (g_n == o_n)))
    achieved = algo / (us / 1e6) / 1e9
    fused = fused_walk_cost(torch, df, CONFIGS[args.config], max(args.steps, 50), args.warmup)
    print(json.dumps({
        "impl": "ours", "op": "walk", "metric": "sampling walk sequences/s", "value": B / (us / 1e6),
        "unit": "sequences/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": us / 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": name, "l2": "flushed before every timed launch (256 MB write, outside the timing)"},
        "greedy_walk_us": greedy_us, "sampling_walk_us": us, "in_select_call": fused,
        "sample_agreement_with_oracle": agree, "agreement_sample": f"first {sample_b} sequences, exact draft and n_draft",
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"], "traffic": None, "kernel": "walk_sample_kernel",
                     "algorithmic_per_launch": algo, "peak_source": peak_kind,
                     "note": "latency-bound: T dependent row reads per sequence"},
        "gpu_launches": args.steps,
        "clocks": ClockSampler.summarize(clock_rows, 0) if clock_rows else {"reasons": ["no samples"]}}), flush=True)
    return 0


def oracle_walk_sample_sample(lat, uni, nb, T, k, tau, p_min):
    """The oracle's walk on the first nb sequences (the bench's parity spot check)."""
    import oracle

    return oracle.walk_sample(lat[:nb * T], nb, T, k, tau, p_min, uni[:nb])


def run_topk(args, cfg, rank: int):
    """Top-k A/B on one config: (a) dflash2_topk vs torch.topk over the same materialised float32
    logits; (b) the fused LM head (top-k in the epilogue) vs materialising the logits and then
    taking the top-k.  Prints one JSON line (rank 0)."""
    import torch

    from speculative_decoding_drafter_gb300 import dflash2 as df

    if rank != 0:
        return 0
    if args.impl == "reference":
        # the oracle's top-k (a full sort per row) on a bounded sample of rows of seeded float32 logits
        import oracle

        oracle.build()
        rows = 4
        g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([0, 43])))
        lg = g.standard_normal((rows, cfg.V), dtype=np.float32)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            oracle.topk(lg, cfg.k)
        dt = (time.perf_counter() - t0) / args.steps
        print(json.dumps({"impl": "reference", "op": "topk", "metric": "top-k of materialised float32 logits, us per call",
                          "value": 1e6 * dt * cfg.R / rows, "unit": "us", "higher_is_better": False,
                          "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "dtype": "f32",
                          "data": "synthetic", "config": {"workload": workload_name(cfg)},
                          "cpu_baseline": {"value": 1e6 * dt * cfg.R / rows, "unit": "us", "cores": oracle.threads(),
                                           "kind": "oracle",
                                           "sample": f"{rows} rows per step, scaled to the workload's {cfg.R} rows"},
                          "e2e": {"value": 1e6 * dt * cfg.R / rows, "unit": "us", "h2d_bytes_per_step": 0,
                                  "d2h_bytes_per_step": 0}}), flush=True)
        return 0
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    peaks, peak_kind = load_peaks()
    R, V, H, k = cfg.R, cfg.V, cfg.H, cfg.k
    x = make_inputs(cfg, 0)

    def dev_bf16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()

    hidden, W = dev_bf16(x["hidden"]), dev_bf16(x["W_vocab"])
    logits = torch.empty((R, V), dtype=torch.float32, device="cuda")
    ws = df.Workspace(df.make_dims(R, 1, H, V, k, 8))
    ids = torch.empty((R, k), dtype=torch.int32, device="cuda")
    vals = torch.empty((R, k), dtype=torch.float32, device="cuda")
    df.dflash2_lm_head_logits(hidden, W, out=logits, workspace=ws)

    def timed(fn, steps):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(steps):
            fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / steps * 1e3  # us

    def graphed(fn, steps, per_graph=20):
        """Device time per call: per_graph calls captured in one CUDA graph and replayed, so that
        the host's per-call cost (Python binding, launch) does not pace the GPU."""
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for _ in range(args.warmup):
                fn()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(per_graph):
                fn()
        reps = max(1, steps // per_graph)
        g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            g.replay()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / (reps * per_graph) * 1e3  # us

    ours_eager_us = timed(lambda: df.dflash2_topk(logits, k, ids=ids, vals=vals, workspace=ws), args.steps)
    torch_eager_us = timed(lambda: torch.topk(logits, k, dim=1, largest=True, sorted=True), args.steps)
    ours_us = graphed(lambda: df.dflash2_topk(logits, k, ids=ids, vals=vals, workspace=ws), args.steps)
    torch_us = graphed(lambda: torch.topk(logits, k, dim=1, largest=True, sorted=True), args.steps)
    tv, ti = torch.topk(logits, k, dim=1, largest=True, sorted=True)
    df.dflash2_topk(logits, k, ids=ids, vals=vals, workspace=ws)
    torch.cuda.synchronize()
    same_vals = bool(torch.equal(tv, vals))
    same_sets = bool(torch.equal(torch.sort(ti.to(torch.int32), dim=1)[0], torch.sort(ids, dim=1)[0]))
    materialised_us = timed(lambda: (df.dflash2_lm_head_logits(hidden, W, out=logits, workspace=ws),
                                     df.dflash2_topk(logits, k, ids=ids, vals=vals, workspace=ws)), args.steps)
    # the fused path: the LM-head launch of dflash2_select (top-k in the epilogue; no logits in memory)
    d = {n: dev_bf16(x[n]) for n in ("W_sel", "pred_cb", "succ_cb")}
    anchor = torch.from_numpy(x["anchor"]).cuda()
    wsel = df.Workspace(df.make_dims(cfg.B, cfg.T, H, V, k, cfg.D))
    lat = torch.empty((R, k + k * k), dtype=torch.float32, device="cuda")
    dr = torch.empty((cfg.B, cfg.T), dtype=torch.int32, device="cuda")
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * args.steps)]
    for e in ev:
        e.record()
    for _ in range(args.warmup):
        df.dflash2_select(hidden, W, d["W_sel"], d["pred_cb"], d["succ_cb"], anchor, k, cfg.T, lattice=lat,
                          draft_ids=dr, workspace=wsel)
    torch.cuda.synchronize()
    for i in range(args.steps):
        df.dflash2_profile_events(ev[2 * i], ev[2 * i + 1])
        df.dflash2_select(hidden, W, d["W_sel"], d["pred_cb"], d["succ_cb"], anchor, k, cfg.T, lattice=lat,
                          draft_ids=dr, workspace=wsel)
    torch.cuda.synchronize()
    df.dflash2_profile_events(None, None)
    fused_us = sum(ev[2 * i].elapsed_time(ev[2 * i + 1]) for i in range(args.steps)) / args.steps * 1e3
    read_gbs = R * V * 4 / (ours_us * 1e-6) / 1e9
    print(json.dumps({
        "impl": "ours", "op": "topk", "metric": "top-k of materialised float32 logits, us per call",
        "value": ours_us, "unit": "us", "higher_is_better": False, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "dtype": "f32", "data": "synthetic",
        "config": {"workload": workload_name(cfg), "logits_bytes": R * V * 4},
        "timing": "device time per call: 20 calls captured in a CUDA graph, replayed (the eager figures, "
                  "one Python call per launch, include the host's per-call cost)",
        "eager_us": ours_eager_us, "torch_topk_eager_us": torch_eager_us,
        "torch_topk_us": torch_us, "speedup_vs_torch_topk": torch_us / ours_us,
        "same_values_as_torch_topk": same_vals, "same_candidate_sets_as_torch_topk": same_sets,
        "roofline": {"bound": "hbm", "achieved": read_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": read_gbs / peaks["hbm_gbs"], "kernel": "logits_topk_partial + topk_merge",
                     "peak_source": peak_kind},
        "lm_head_then_topk_us": materialised_us, "fused_lm_head_topk_gate_us": fused_us,
        "fused_saving": 1.0 - fused_us / materialised_us}), flush=True)
    return 0


def main():
    args = parse_args()
    cfg = CONFIGS[args.config]
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", str(args.gpus if args.gpus == 1 else 1)))
    if args.op == "conv":
        return run_conv(args, rank, world)
    if args.op == "topk":
        return run_topk(args, cfg, rank)
    if args.op == "walk":
        return run_walk(args, rank, world)
    if args.impl == "reference":
        return run_reference(args, cfg, rank, world)
    return run_ours(args, cfg, rank, world)


if __name__ == "__main__":
    sys.exit(main())
