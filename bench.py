#!/usr/bin/env python
"""Throughput of the exact attention backward-over-backward on GB300.

One step = one flashbob_bob call (pass 1 + pass 2) over the long-context
workload (B=1, H=4, N=65536, d=64, bf16 inputs, non-causal) with every input
already resident in device memory.  FLOPs per step follow the fixed GEMM
list of both passes: 38 N^2 d per (batch, head).

Prints one JSON line (rank 0).  ``--impl reference`` times the fp64 CPU
oracle on the host cores instead (rows and columns of the same workload).
``--entry jvp`` times flashbob_attention_jvp instead (5 GEMMs, 10 N^2 d per
head).  ``--sweep`` prints, after that line, one more line per workload of
the throughput-vs-length table (the five benchmark configurations and the
pages' causal timing shapes).
"""
from __future__ import annotations

import argparse
import json
import os
import platform
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "BoB TFLOP/s & % of GB300 bf16 tensor peak vs N (d=64); ms/call"
UNIT = "TFLOP/s"
DEFAULT_WORKLOAD = "long_B1_H4_N65536_d64"
PASS1_GEMMS, PASS2_GEMMS = 11, 8  # each 2 d flops per visible (query, key) pair
JVP_GEMMS = 5  # S, U_Q K^T, Q U_K^T, P U_V, (P o F) V
JVP_METRIC = "attention JVP TFLOP/s (5 GEMMs of 2*N^2*d per head); ms/call"
L2_BYTES = 129 * 1024 * 1024
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic_long_context.txt")
SMI_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--entry", choices=("bob", "jvp"), default="bob",
                    help="bob: flashbob_bob (the benchmark); jvp: flashbob_attention_jvp")
    ap.add_argument("--sweep", action="store_true",
                    help="also time every workload of the throughput-vs-length table")
    ap.add_argument("--sweep-oracle", action="store_true",
                    help="with --sweep: time the full fp64 oracle on the small configurations")
    ap.add_argument("--mma-costs", action="store_true",
                    help="only measure SM cycles per tcgen05.mma (M 128, K 16) for N = 16..256, "
                         "A from shared or tensor memory (flashbob_mma_cycles); one line each")
    return ap.parse_args()


def run_mma_costs(fb, torch):
    """One JSON line per MMA shape: the median of 5 runs of 4096 back-to-back
    MMAs, and the tensor-pipe efficiency N/2 / cycles (an M = 128, K = 16 MMA
    is N/2 cycles of math at the dense rate)."""
    for a_in_tmem in (False, True):
        for n in (16, 32, 48, 64, 96, 128, 192, 256):
            c = statistics.median(fb.flashbob_mma_cycles(n, a_in_tmem) for _ in range(5))
            print(json.dumps({"mma_costs": True, "m": 128, "n": n, "k": 16,
                              "a": "tmem" if a_in_tmem else "smem", "b": "smem",
                              "cycles_per_mma": round(c, 2),
                              "math_cycles": n / 2, "efficiency": round(n / 2 / c, 3)}),
                  flush=True)
    assert fb.flashbob_last_device_error() == fb.FLASHBOB_OK


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def reduce_max(x: float, world: int, device="cpu") -> float:
    """Largest value over the ranks (the job is as slow as its slowest rank)."""
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flops_per_rank_step: float, steps: int, world: int, max_ms: float) -> float:
    """Whole-job throughput: every rank processes its own units (weak
    scaling, no data exchange), divided by the slowest rank's time."""
    return world * flops_per_rank_step * steps / (max_ms * 1e-3) / 1e12


def rank_workload(w, rank: int):
    """Rank r processes its own seeded copy of the workload (independent
    (batch, head) units, the same shape on every rank)."""
    from dataclasses import replace
    return replace(w, seed=w.seed + rank)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            p = json.load(fh)
        return p, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def tensor_peak():
    """The denominator of every fraction: the burst dense-bf16 figure (a
    cuBLAS GEMM timed alone, at the clocks a sub-second timed region also
    runs at), with the sustained figure (a seconds-long loop under the power
    cap, at lower clocks) kept beside it."""
    peaks, src = measured_peaks()
    burst = float(peaks.get("bf16_tflops"))
    sustained = float(peaks.get("bf16_tflops_sustained", burst))
    clk = (peaks.get("clocks_under_load") or {}).get("sm_mhz_median")
    note = (f"bf16_tflops (burst) of {src} peaks; sustained {sustained:.1f} TFLOP/s was "
            f"measured at a median {clk} MHz" if clk else f"bf16_tflops (burst) of {src} peaks")
    return burst, sustained, note


def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as fh:
            for line in fh:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.processor() or platform.machine()


def read_traffic():
    """Per-launch DRAM bytes of the dominant kernel from the committed ncu
    summary (a line ``<kernel> dram_bytes_per_launch <int>``), else None."""
    if not os.path.exists(TRAFFIC_FILE):
        return {}
    out = {}
    with open(TRAFFIC_FILE) as fh:
        for line in fh:
            parts = line.split()
            if len(parts) == 3 and parts[1] == "dram_bytes_per_launch":
                out[parts[0]] = int(parts[2])
    return out


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    def __init__(self, uuid: str | None):
        self.proc = None
        fd, self.path = tempfile.mkstemp(prefix="flashbob_clocks_", suffix=".csv")
        os.close(fd)
        cmd = ["nvidia-smi", f"--query-gpu={SMI_FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "200"]
        if uuid:
            cmd += ["-i", uuid]
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(cmd, stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            os.unlink(self.path)
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons, power = [], [], set(), []
        with open(self.path) as fh:
            lines = fh.readlines()
        os.unlink(self.path)
        for line in lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for name, val in zip(REASONS, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "samples": len(sm), "reasons": sorted(reasons)}


def config_dict(w) -> dict:
    """The workload keys every line carries (our arm and the reference arm)."""
    return {"workload": w.name, "B": w.B, "H": w.H, "Hkv": w.kv_heads, "N": w.N,
            "Nk": w.kv_len, "d": w.d, "causal": w.causal, "tau": w.tau,
            "flop_convention": "38*N^2*d*B*H (19 GEMMs of 2*N^2*d); rectangular N*Nk for "
                               "N^2, causal the pairs j <= i"}


def oracle_sample(w, x, seconds: float, chunk: int = 16, seed: int = 7):
    """Time the oracle on a bounded sample of the workload: seeded query rows
    of head (0, 0) through ``bob_rows`` (the row outputs: L, D, alpha, E,
    d~Q, d~dO) and as many seeded key columns through ``bob_cols`` (d~K,
    d~V), alternating chunks for about ``seconds``.  ``bob_cols`` takes every
    row's scalars as input; for the timing they are the sampled rows' values
    repeated, which changes no operation.  Returns the counts and times."""
    import numpy as np

    from exact_second_order_gb300.inputs import NAMES, as_float64_numpy
    from oracle import bob as orc
    args = [as_float64_numpy(x[k][0, 0]) for k in NAMES]  # query head 0 uses key head 0
    rng = np.random.default_rng(seed)
    rows = cols = 0
    t_rows = t_cols = 0.0
    scal = None
    while t_rows + t_cols < seconds:
        t0 = time.perf_counter()
        r = orc.bob_rows(*args, w.tau, rng.choice(w.N, size=chunk, replace=False),
                         causal=w.causal)
        t_rows += time.perf_counter() - t0
        rows += chunk
        if scal is None:
            reps = -(-w.N // chunk)
            scal = {k: np.tile(r[k], reps)[:w.N] for k in ("L", "D", "alpha", "E")}
        t0 = time.perf_counter()
        orc.bob_cols(*args, w.tau, rng.choice(w.kv_len, size=chunk, replace=False),
                     causal=w.causal, scalars=scal)
        t_cols += time.perf_counter() - t0
        cols += chunk
    return {"rows": rows, "cols": cols, "t_rows": t_rows, "t_cols": t_cols}


def oracle_baseline(w, smp: dict) -> dict:
    """Throughput of the oracle sample on the BoB GEMM list: a row carries
    pass 1's 11 GEMMs over the keys it sees, a column pass 2's 8 over the
    queries that see it; plus the labelled extrapolation to one full call
    (every row and every key column of every head)."""
    per_row = 2.0 * PASS1_GEMMS * (w.pairs / w.N) * w.d
    per_col = 2.0 * PASS2_GEMMS * (w.pairs / w.kv_len) * w.d
    el = smp["t_rows"] + smp["t_cols"]
    value = (smp["rows"] * per_row + smp["cols"] * per_col) / el / 1e12
    s_row, s_col = smp["t_rows"] / smp["rows"], smp["t_cols"] / smp["cols"]
    full = w.B * (w.H * w.N * s_row + w.kv_heads * (w.H // w.kv_heads) * w.kv_len * s_col)
    return {"value": value, "unit": UNIT, "cores": os.cpu_count(), "cpu_model": cpu_model(),
            "kind": "oracle", "seconds_per_row": s_row, "seconds_per_column": s_col,
            "extrapolated_full_call_s": full,
            "sample": f"{smp['rows']} seeded rows (oracle.bob_rows) and {smp['cols']} seeded "
                      f"key columns (oracle.bob_cols) of head (0,0), fp64 numpy, {el:.1f} s; "
                      f"credited {per_row:.3e} flops per row, {per_col:.3e} per column; "
                      f"extrapolated_full_call_s = all B*H*N rows and B*H*Nk columns at the "
                      f"sampled rates (an extrapolation, not a measurement)"}


def run_reference(args, w, rank, world):
    if rank != 0:
        return
    from exact_second_order_gb300.inputs import make_inputs
    x = make_inputs(w)
    per_step = max(2.0, 60.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_sample(w, x, min(per_step, 2.0))
    tot = {"rows": 0, "cols": 0, "t_rows": 0.0, "t_cols": 0.0}
    for _ in range(args.steps):
        smp = oracle_sample(w, x, per_step)
        for k in tot:
            tot[k] += smp[k]
    base = oracle_baseline(w, tot)
    value = base["value"]
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * (tot["t_rows"] + tot["t_cols"]) / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_dict(w),
        "cpu_baseline": base,
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_jvp(args, w, dev, rank, world, local, barrier, fb, torch):
    """Time flashbob_attention_jvp on resident inputs (O, L from a
    forward-only prep outside the timed region)."""
    O, L, _ = fb.prep(dev["Q"], dev["K"], dev["V"], None, w.tau, causal=w.causal)
    Od, Ld = torch.empty_like(O), torch.empty_like(L)
    stream = torch.cuda.current_stream()

    def step():
        fb.flashbob_attention_jvp(dev["Q"], dev["K"], dev["V"], O, L, dev["UQ"], dev["UK"],
                                  dev["UV"], w.tau, Od, Ld, causal=w.causal, stream=stream)

    resident = sum(t.numel() * t.element_size() for t in (dev["Q"], dev["K"], dev["V"],
                                                          dev["UQ"], dev["UK"], dev["UV"], O, L))
    flush, l2_note = l2_flusher(torch, resident)
    for _ in range(max(3, args.warmup)):
        if flush is not None:
            flush.zero_()
        step()
    torch.cuda.synchronize()
    assert fb.flashbob_last_device_error() == fb.FLASHBOB_OK
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    sampler = ClockSampler(None)
    time.sleep(0.3)
    barrier()
    for e in evs:
        if flush is not None:
            flush.zero_()
        e[0].record(stream)
        step()
        e[1].record(stream)
    barrier()
    clocks = sampler.stop()
    assert fb.flashbob_last_device_error() == fb.FLASHBOB_OK
    if flush is not None:
        local_ms = sum(e[0].elapsed_time(e[1]) for e in evs)
    else:
        local_ms = evs[0][0].elapsed_time(evs[-1][1])
    ms = local_ms / args.steps
    total_ms = reduce_max(local_ms, world, "cuda")
    flops = JVP_GEMMS * 2.0 * w.pairs * w.d * w.B * w.H
    value = job_tflops(flops, args.steps, world, total_ms)
    peak, _, peak_note = tensor_peak()
    achieved = flops / (ms * 1e-3) / 1e12
    line = {
        "metric": JVP_METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": total_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": w.name, "entry": "flashbob_attention_jvp", "B": w.B, "H": w.H,
                   "Hkv": w.kv_heads, "N": w.N, "Nk": w.kv_len, "d": w.d, "causal": w.causal,
                   "flops_per_step_per_gpu": flops, "l2": l2_note},
        "roofline": {"kernel": "jvp", "bound": "tensor", "achieved": achieved, "peak": peak,
                     "unit": "TFLOP/s", "frac": achieved / peak, "traffic": None,
                     "peak_source": peak_note},
        "gpu_launches": args.steps,
        "clocks": clocks,
        "e2e": None,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


# The throughput-vs-length table (--sweep): the benchmark configurations at
# head dim 64 (N = 1K ... 256K) and 128, then the pages' causal timing shapes
# (B = 4, H = 12, bf16; [FBN] 实验关键数据).
SWEEP = ("gpt2_layer_B4_H12_N1024_d64", "curve_B4_H12_N2048_d64", "curve_B2_H12_N4096_d64",
         "mid_B1_H12_N8192_d64", "curve_B1_H8_N16384_d64", "curve_B1_H4_N32768_d64",
         "mid_peaked_B1_H12_N8192_d64",
         "long_B1_H4_N65536_d64", "extreme_B1_H1_N262144_d64", "extreme_B1_H1_N131072_d128",
         "causal_B4_H12_N4096_d64", "causal_B4_H12_N8192_d64", "causal_B4_H12_N16384_d64",
         "causal_B4_H12_N16384_d128", "causal_B4_H12_N32768_d128",
         "causal_B4_H12_N65536_d128", "gqa_B1_H12_Hkv4_N8192_d64", "mqa_B1_H12_Hkv1_N8192_d64",
         "rect_B1_H8_Nq4096_Nk16384_d64", "rect_B1_H8_Nq16384_Nk4096_d64")


def gpu_uuid(torch, local):
    try:
        uuid = str(torch.cuda.get_device_properties(local).uuid)
        return uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        return None


class Resident:
    """Inputs, row state and outputs of one workload in device memory, and the
    timed step: one flashbob_bob call on the current stream (both passes;
    with several head groups the library overlaps the groups' chains on its
    own streams); step_passes runs the two passes as separate calls, each
    bracketed by events, for the per-kernel times."""

    def __init__(self, w, x, fb, torch):
        self.w, self.fb = w, fb
        self.dev = {k: v.cuda() for k, v in x.items()}
        d = self.dev
        self.O, self.L, self.D = fb.prep(d["Q"], d["K"], d["V"], d["dO"], w.tau, causal=w.causal)
        self.out = fb.alloc_bob_outputs(d["Q"], K=d["K"])
        self.stream = torch.cuda.current_stream()

    def step(self, ev=None):
        w, d, o, fb, st = self.w, self.dev, self.out, self.fb, self.stream
        if ev is not None:
            ev[0].record(st)
        fb.flashbob_bob(d["Q"], d["K"], d["V"], self.O, d["dO"], self.L, self.D, d["UQ"],
                        d["UK"], d["UV"], w.tau, o["dQt"], o["dKt"], o["dVt"], o["ddOt"],
                        o["alpha"], o["E"], causal=w.causal, stream=st)
        if ev is not None:
            ev[1].record(st)

    def launches_per_step(self):
        w = self.w
        return self.fb.flashbob_bob_launches(w.B, w.H, w.kv_heads, w.N, w.kv_len, w.d,
                                             self.fb.FLASHBOB_BF16)

    def streams_per_step(self):
        w = self.w
        per_stream = 3 if w.d == 128 else 2  # d = 128: pass 1 is two launches
        return self.launches_per_step() // per_stream

    def step_passes(self, ev=None):
        w, d, o, fb, st = self.w, self.dev, self.out, self.fb, self.stream
        if ev is not None:
            ev[0].record(st)
        fb.flashbob_bob_pass1(d["Q"], d["K"], d["V"], self.O, d["dO"], self.L, self.D, d["UQ"],
                              d["UK"], d["UV"], w.tau, o["dQt"], o["ddOt"], o["alpha"], o["E"],
                              causal=w.causal, stream=st)
        if ev is not None:
            ev[1].record(st)
        fb.flashbob_bob_pass2(d["Q"], d["K"], d["V"], d["dO"], self.L, self.D, o["alpha"],
                              o["E"], d["UQ"], d["UK"], d["UV"], w.tau, o["dKt"], o["dVt"],
                              causal=w.causal, stream=st)
        if ev is not None:
            ev[2].record(st)

    def prep_ms(self, torch, reps=3):
        d, st = self.dev, self.stream
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        ev[0].record(st)
        for _ in range(reps):
            self.fb.prep(d["Q"], d["K"], d["V"], d["dO"], self.w.tau, causal=self.w.causal,
                         stream=st)
        ev[1].record(st)
        torch.cuda.synchronize()
        return ev[0].elapsed_time(ev[1]) / reps

    def input_bytes(self):
        return sum(t.numel() * t.element_size() for t in list(self.dev.values())
                   + [self.O, self.L, self.D])


def l2_flusher(torch, resident_bytes):
    """What keeps a step from finding the previous step's data in the L2:
    inputs (with the row state) of more than twice the L2 evict it by
    themselves; smaller ones get a write of twice the L2 before every timed
    step, outside that step's events.  Returns (buffer or None, note)."""
    mib = resident_bytes / 2**20
    if resident_bytes > 2 * L2_BYTES:
        return None, f"no flush: inputs {mib:.0f} MiB > 2 x L2 ({L2_BYTES / 2**20:.0f} MiB)"
    buf = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device="cuda")
    return buf, (f"L2 flushed before every step ({2 * L2_BYTES / 2**20:.0f} MiB written; "
                 f"inputs {mib:.0f} MiB <= 2 x L2); ms_per_step sums the steps' own event "
                 f"intervals")


def timed_steps(res, steps, warmup, torch, barrier, uuid, flush=None):
    """W warm-up steps, then K steps (one flashbob_bob call each) with CUDA
    events on the launching stream and nvidia-smi clocks sampled during the
    timed region; then, outside it, K steps of the two passes as separate
    calls, each pass between two events, for the per-kernel times.  With a
    ``flush`` buffer every step (and every pair of separate passes) follows a
    write of it, outside its events, and the total is the sum of the steps'
    own intervals."""
    fb = res.fb

    def flush_l2():
        if flush is not None:
            flush.zero_()

    for _ in range(max(3, warmup)):
        flush_l2()
        res.step()
    torch.cuda.synchronize()
    assert fb.flashbob_last_device_error() == fb.FLASHBOB_OK
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    sampler = ClockSampler(uuid)
    time.sleep(0.3)
    barrier()
    for i in range(steps):
        flush_l2()
        res.step(evs[i])
    barrier()
    clocks = sampler.stop()
    assert fb.flashbob_last_device_error() == fb.FLASHBOB_OK
    pev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    res.step_passes()
    for i in range(steps):
        flush_l2()
        res.step_passes(pev[i])
    torch.cuda.synchronize()
    assert fb.flashbob_last_device_error() == fb.FLASHBOB_OK
    if flush is not None:
        total_ms = sum(e[0].elapsed_time(e[1]) for e in evs)
    else:
        total_ms = evs[0][0].elapsed_time(evs[-1][1])
    return {"total_ms": total_ms,
            "median_ms": statistics.median(e[0].elapsed_time(e[1]) for e in evs),
            "p1_ms": statistics.mean(e[0].elapsed_time(e[1]) for e in pev),
            "p2_ms": statistics.mean(e[1].elapsed_time(e[2]) for e in pev),
            "passes_ms": statistics.mean(e[0].elapsed_time(e[2]) for e in pev),
            "clocks": clocks}


def roofline(w, t, peak, peak_note, traffic=None):
    """The dominant pass: its algorithmic FLOPs over its mean event time."""
    unit_flops = 2.0 * w.pairs * w.d * w.B * w.H  # one Nq x Nk x d GEMM per (b, h)
    dominant = "pass1" if t["p1_ms"] >= t["p2_ms"] else "pass2"
    dom_ms = t["p1_ms"] if dominant == "pass1" else t["p2_ms"]
    dom_flops = (PASS1_GEMMS if dominant == "pass1" else PASS2_GEMMS) * unit_flops
    achieved = dom_flops / (dom_ms * 1e-3) / 1e12
    return {"kernel": dominant, "bound": "tensor", "achieved": achieved, "peak": peak,
            "unit": "TFLOP/s", "frac": achieved / peak, "traffic": traffic,
            "peak_source": peak_note}


def run_sweep(args, fb, torch, barrier, uuid, peak, peak_note):
    """One JSON line per workload of SWEEP: TFLOP/s, ms/call, the fraction of
    the tensor peak, both passes' times and the clocks."""
    from exact_second_order_gb300.inputs import WORKLOADS, make_inputs
    for name in SWEEP:
        w = WORKLOADS[name]
        res = Resident(w, make_inputs(w), fb, torch)
        flush, l2_note = l2_flusher(torch, res.input_bytes())
        # about half a second of timed work, at least 5 steps
        res.step()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        res.step()
        torch.cuda.synchronize()
        est = max(time.perf_counter() - t0, 1e-5)
        steps = int(min(200, max(5, 0.5 / est)))
        t = timed_steps(res, steps, 3, torch, barrier, uuid, flush)
        del flush
        ms = t["total_ms"] / steps
        value = w.flops / (ms * 1e-3) / 1e12
        line = {"sweep": True, "metric": METRIC, "value": value, "unit": UNIT,
                "ms_per_step": ms, "steps": steps, "warmup": 3, "dtype": "bf16",
                "pct_of_peak": 100.0 * value / peak,
                "config": dict(config_dict(w), l2=l2_note, ms_per_call_median=t["median_ms"],
                               pass1_ms=t["p1_ms"], pass2_ms=t["p2_ms"],
                               passes_as_separate_calls_ms=t["passes_ms"],
                               head_group_streams=res.streams_per_step(),
                               prep_ms_outside_step=res.prep_ms(torch),
                               flops_per_step=w.flops),
                "roofline": roofline(w, t, peak, peak_note), "clocks": t["clocks"]}
        if args.sweep_oracle and w.N * w.kv_len * w.B * w.H <= 12 * 8192 * 8192:
            line["oracle_full"] = oracle_full_timing(w, make_inputs(w))
        print(json.dumps(line), flush=True)
        del res
        torch.cuda.empty_cache()


def oracle_full_timing(w, x):
    """The full fp64 oracle (``bob`` on every head: N x N matrices) on the
    host cores; at most two heads are run and the rest extrapolated."""
    from exact_second_order_gb300.inputs import NAMES, as_float64_numpy
    from oracle import bob as orc
    heads = [(b, h) for b in range(w.B) for h in range(w.H)]
    run = heads[:2]
    G = w.H // w.kv_heads
    t0 = time.perf_counter()
    for b, h in run:
        a = [as_float64_numpy(x[k][b, h // G if k in ("K", "V", "UK", "UV") else h])
             for k in NAMES]
        orc.bob(*a, w.tau, causal=w.causal)
    el = time.perf_counter() - t0
    return {"heads_run": len(run), "heads": len(heads), "seconds_run": el,
            "seconds_full_call": el * len(heads) / len(run),
            "note": "full_call extrapolated from the heads run" if len(run) < len(heads)
                    else "every head run", "cores": os.cpu_count(), "cpu_model": cpu_model()}


def run_e2e(args, w, x, res, fb, torch, barrier, world):
    """The benchmark step through the public C ABI (flashbob_bob) with the
    data on the host: each step uploads its inputs and row state from pinned
    host memory and downloads all six outputs.  Buffer set k % 2 serves step
    k; uploads and downloads run on two copy streams (one per direction),
    ordered against the kernels by events, so they overlap the neighbouring
    steps' kernels and each other."""
    comp = res.stream
    copy = torch.cuda.Stream()       # host -> device
    copy_out = torch.cuda.Stream()   # device -> host, so the two directions overlap
    host_in = {k: v.pin_memory() for k, v in x.items()}
    host_state = {"O": res.O.cpu().pin_memory(), "L": res.L.cpu().pin_memory(),
                  "D": res.D.cpu().pin_memory()}
    host_out = [{k: torch.empty_like(v, device="cpu").pin_memory() for k, v in res.out.items()}
                for _ in range(2)]
    sets = []
    for b in range(2):
        dev = res.dev if b == 0 else {k: torch.empty_like(v) for k, v in res.dev.items()}
        state = ({"O": res.O, "L": res.L, "D": res.D} if b == 0 else
                 {"O": torch.empty_like(res.O), "L": torch.empty_like(res.L),
                  "D": torch.empty_like(res.D)})
        out = res.out if b == 0 else {k: torch.empty_like(v) for k, v in res.out.items()}
        sets.append((dev, state, out))
    h2d = sum(t_.numel() * t_.element_size() for t_ in list(host_in.values())
              + list(host_state.values()))
    d2h = sum(t_.numel() * t_.element_size() for t_ in host_out[0].values())
    uploaded = [torch.cuda.Event() for _ in range(2)]    # set b's inputs are on the device
    computed = [torch.cuda.Event() for _ in range(2)]    # set b's outputs are written
    downloaded = [torch.cuda.Event() for _ in range(2)]  # set b's outputs are on the host
    for b in range(2):
        downloaded[b].record(copy_out)

    def upload(b):
        dev, state, _ = sets[b]
        with torch.cuda.stream(copy):
            copy.wait_event(computed[b])  # the kernels that read this set last are done
            for k in host_in:
                dev[k].copy_(host_in[k], non_blocking=True)
            for k in host_state:
                state[k].copy_(host_state[k], non_blocking=True)
            uploaded[b].record(copy)

    def compute(b):
        dev, state, out = sets[b]
        comp.wait_event(uploaded[b])
        comp.wait_event(downloaded[b])  # the previous use of these outputs is on the host
        fb.flashbob_bob(dev["Q"], dev["K"], dev["V"], state["O"], dev["dO"], state["L"],
                        state["D"], dev["UQ"], dev["UK"], dev["UV"], w.tau, out["dQt"],
                        out["dKt"], out["dVt"], out["ddOt"], out["alpha"], out["E"],
                        causal=w.causal, stream=comp)
        computed[b].record(comp)

    def download(b):
        _, _, out = sets[b]
        with torch.cuda.stream(copy_out):
            copy_out.wait_event(computed[b])
            for k in host_out[b]:
                host_out[b][k].copy_(out[k], non_blocking=True)
            downloaded[b].record(copy_out)

    def run(n):
        upload(0)
        for k in range(n):
            b = k & 1
            compute(b)
            if k + 1 < n:
                upload(1 - b)
            download(b)

    run(2)
    barrier()
    # The same K steps as the device-resident leg: the first upload and the
    # last download (the only copies not overlapped) spread over as many steps.
    n_e2e = max(3, args.steps)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(comp)
    copy.wait_event(t0)
    copy_out.wait_event(t0)
    run(n_e2e)
    comp.wait_stream(copy)
    comp.wait_stream(copy_out)
    t1.record(comp)
    barrier()
    e_ms = reduce_max(t0.elapsed_time(t1), world, "cuda")
    return {"value": job_tflops(w.flops, n_e2e, world, e_ms), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": e_ms / n_e2e, "steps": n_e2e,
            "overlap": "uploads and downloads on two copy streams, two buffer sets"}


def main():
    args = parse_args()
    rank, world, local = dist_env()
    from exact_second_order_gb300.inputs import WORKLOADS, make_inputs
    w = WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, w, rank, world)

    import torch
    import torch.distributed as dist

    from exact_second_order_gb300 import flashbob as fb

    torch.cuda.set_device(local)
    if args.mma_costs:
        return run_mma_costs(fb, torch)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    x = make_inputs(rank_workload(w, rank))
    if args.entry == "jvp":
        dev = {k: v.cuda() for k, v in x.items()}
        return run_jvp(args, w, dev, rank, world, local, barrier, fb, torch)
    res = Resident(w, x, fb, torch)
    uuid = gpu_uuid(torch, local)
    flush, l2_note = l2_flusher(torch, res.input_bytes())
    t = timed_steps(res, args.steps, args.warmup, torch, barrier, uuid, flush)
    del flush
    res_launches = res.launches_per_step()
    res_streams = res.streams_per_step()
    prep_ms = res.prep_ms(torch)
    total_ms = reduce_max(t["total_ms"], world, "cuda")
    ms_per_step = total_ms / args.steps
    flops = w.flops
    value = job_tflops(flops, args.steps, world, total_ms)

    # end to end: pinned host inputs -> device, the C-ABI call, outputs -> host,
    # every step.  Two device copies of the inputs, row state and outputs
    # alternate between steps, and the copies run on a second stream, so a
    # step's uploads and the previous step's downloads overlap the kernels
    # (events order every buffer's reuse).
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, w, x, res, fb, torch, barrier, world)
        del res
        torch.cuda.empty_cache()
    peak, sustained, peak_note = tensor_peak()
    rl = roofline(w, t, peak, peak_note)
    # The committed counters are of the benchmark workload's bytes only.
    rl["traffic"] = read_traffic().get(rl["kernel"]) if w.name == DEFAULT_WORKLOAD else None
    rl["frac_of_sustained"] = rl["achieved"] / sustained
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": dict(config_dict(w), flops_per_step_per_gpu=flops,
                       l2=l2_note,
                       ms_per_call_median=t["median_ms"],
                       pass1_ms=t["p1_ms"], pass2_ms=t["p2_ms"],
                       passes_as_separate_calls_ms=t["passes_ms"],
                       head_group_streams=res_streams, prep_ms_outside_step=prep_ms,
                       pct_of_peak=100.0 * (value / world) / peak,
                       paths="tcgen05" if fb.flashbob_bob_tile_sizes(w.d, fb.FLASHBOB_BF16)[
                           "Br1"] == 128 else "simt"),
        "roofline": rl,
        "gpu_launches": res_launches * args.steps,
        "clocks": t["clocks"],
        "e2e": e2e,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = oracle_baseline(w, oracle_sample(w, x, args.cpu_seconds))
    if rank == 0:
        print(json.dumps(line), flush=True)
    if args.sweep and world == 1:
        res = None
        torch.cuda.empty_cache()
        run_sweep(args, fb, torch, barrier, uuid, peak, peak_note)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
