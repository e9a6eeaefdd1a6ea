#!/usr/bin/env python
"""Throughput of the exact attention backward-over-backward on GB300.

One step = one flashbob_bob call (pass 1 + pass 2) over the long-context
workload (B=1, H=4, N=65536, d=64, bf16 inputs, non-causal) with every input
already resident in device memory.  FLOPs per step follow the fixed GEMM
list of both passes: 38 N^2 d per (batch, head).

Prints one JSON line (rank 0).  ``--impl reference`` times the fp64 CPU
oracle on the host cores instead (rows of the same workload).  ``--entry
jvp`` times flashbob_attention_jvp instead (5 GEMMs, 10 N^2 d per head).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
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
    return ap.parse_args()


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
        self.path = os.path.join(ROOT, "gpurun_out", f"clocks_{os.getpid()}.csv")
        cmd = ["nvidia-smi", f"--query-gpu={SMI_FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "200"]
        if uuid:
            cmd += ["-i", uuid]
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(cmd, stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons, power = [], [], set(), []
        with open(self.path) as fh:
            for line in fh:
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


def oracle_rows_sample(w, x, seconds: float, rows_per_chunk: int = 16, seed: int = 7):
    """Time oracle.bob_rows on seeded rows of head (0, 0) for about
    ``seconds``; returns (rows done, elapsed)."""
    import numpy as np

    from exact_second_order_gb300.inputs import NAMES, as_float64_numpy
    from oracle import bob as orc
    args = [as_float64_numpy(x[k][0, 0]) for k in NAMES]  # query head 0 uses key head 0
    rng = np.random.default_rng(seed)
    done, t0 = 0, time.perf_counter()
    while True:
        rows = rng.choice(w.N, size=rows_per_chunk, replace=False)
        orc.bob_rows(*args, w.tau, rows, causal=w.causal)
        done += rows_per_chunk
        el = time.perf_counter() - t0
        if el >= seconds:
            return done, el


def row_flops(w) -> float:
    """FLOPs credited per oracle row: the row-side GEMMs (pass 1 list) over
    the keys an average query row sees."""
    return 2.0 * PASS1_GEMMS * (w.pairs / w.N) * w.d


def run_reference(args, w, rank, world):
    if rank != 0:
        return
    from exact_second_order_gb300.inputs import make_inputs
    x = make_inputs(w)
    per_step = max(2.0, 60.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_rows_sample(w, x, min(per_step, 2.0))
    t_rows, t_el = 0, 0.0
    for _ in range(args.steps):
        r, el = oracle_rows_sample(w, x, per_step)
        t_rows += r
        t_el += el
    value = t_rows * row_flops(w) / t_el / 1e12
    cores = os.cpu_count()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t_el / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N,
                                        "Nk": w.kv_len, "d": w.d, "Hkv": w.kv_heads,
                                        "causal": w.causal},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{t_rows} seeded rows of head (0,0) through oracle.bob_rows "
                                   f"(fp64 numpy), {row_flops(w):.3e} flops credited per row"},
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

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    assert fb.flashbob_last_device_error() == fb.FLASHBOB_OK
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(None)
    time.sleep(0.3)
    barrier()
    t0.record(stream)
    for _ in range(args.steps):
        step()
    t1.record(stream)
    barrier()
    clocks = sampler.stop()
    assert fb.flashbob_last_device_error() == fb.FLASHBOB_OK
    ms = t0.elapsed_time(t1) / args.steps
    total_ms = reduce_max(t0.elapsed_time(t1), world, "cuda")
    flops = JVP_GEMMS * 2.0 * w.pairs * w.d * w.B * w.H
    value = job_tflops(flops, args.steps, world, total_ms)
    peaks, peak_src = measured_peaks()
    peak = float(peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops")))
    achieved = flops / (ms * 1e-3) / 1e12
    line = {
        "metric": JVP_METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": total_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": w.name, "entry": "flashbob_attention_jvp", "B": w.B, "H": w.H,
                   "Hkv": w.kv_heads, "N": w.N, "Nk": w.kv_len, "d": w.d, "causal": w.causal,
                   "flops_per_step_per_gpu": flops},
        "roofline": {"kernel": "jvp", "bound": "tensor", "achieved": achieved, "peak": peak,
                     "unit": "TFLOP/s", "frac": achieved / peak, "traffic": None,
                     "peak_source": f"bf16_tflops_sustained of {peak_src} peaks"},
        "gpu_launches": args.steps,
        "clocks": clocks,
        "e2e": None,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


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
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    x = make_inputs(rank_workload(w, rank))
    dev = {k: v.cuda() for k, v in x.items()}
    if args.entry == "jvp":
        return run_jvp(args, w, dev, rank, world, local, barrier, fb, torch)
    O, L, D = fb.prep(dev["Q"], dev["K"], dev["V"], dev["dO"], w.tau, causal=w.causal)
    out = fb.alloc_bob_outputs(dev["Q"], K=dev["K"])
    stream = torch.cuda.current_stream()

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        fb.flashbob_bob_pass1(dev["Q"], dev["K"], dev["V"], O, dev["dO"], L, D, dev["UQ"],
                              dev["UK"], dev["UV"], w.tau, out["dQt"], out["ddOt"],
                              out["alpha"], out["E"], causal=w.causal, stream=stream)
        if ev is not None:
            ev[1].record(stream)
        fb.flashbob_bob_pass2(dev["Q"], dev["K"], dev["V"], dev["dO"], L, D, out["alpha"],
                              out["E"], dev["UQ"], dev["UK"], dev["UV"], w.tau, out["dKt"],
                              out["dVt"], causal=w.causal, stream=stream)
        if ev is not None:
            ev[2].record(stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    assert fb.flashbob_last_device_error() == fb.FLASHBOB_OK

    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(local).uuid)
        uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        uuid = None
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    sampler = ClockSampler(uuid)
    time.sleep(0.3)
    barrier()
    for i in range(args.steps):
        step(evs[i])
    barrier()
    clocks = sampler.stop()
    assert fb.flashbob_last_device_error() == fb.FLASHBOB_OK
    # prep (O, L, D) is not part of the step: timed on its own, after it
    pev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    pev[0].record(stream)
    for _ in range(3):
        fb.prep(dev["Q"], dev["K"], dev["V"], dev["dO"], w.tau, causal=w.causal, stream=stream)
    pev[1].record(stream)
    torch.cuda.synchronize()
    prep_ms = pev[0].elapsed_time(pev[1]) / 3
    total_ms = evs[0][0].elapsed_time(evs[-1][2])
    p1_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    p2_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
    total_ms = reduce_max(total_ms, world, "cuda")
    ms_per_step = total_ms / args.steps
    heads = w.B * w.H
    # one Nq x Nk x d GEMM per (batch, head), over the visible pairs only
    unit_flops = 2.0 * w.pairs * w.d * heads
    flops = (PASS1_GEMMS + PASS2_GEMMS) * unit_flops
    value = job_tflops(flops, args.steps, world, total_ms)

    # end to end: pinned host inputs -> device, the C-ABI call, outputs -> host
    e2e = None
    if not args.no_e2e:
        host_in = {k: v.pin_memory() for k, v in x.items()}
        host_state = {"O": O.cpu().pin_memory(), "L": L.cpu().pin_memory(),
                      "D": D.cpu().pin_memory()}
        host_out = {k: torch.empty_like(v, device="cpu").pin_memory() for k, v in out.items()}
        dev_state = {"O": O, "L": L, "D": D}
        h2d = sum(t.numel() * t.element_size() for t in list(host_in.values())
                  + list(host_state.values()))
        d2h = sum(t.numel() * t.element_size() for t in host_out.values())
        n_e2e = max(3, args.steps // 2)

        def e2e_step():
            for k in host_in:
                dev[k].copy_(host_in[k], non_blocking=True)
            for k in host_state:
                dev_state[k].copy_(host_state[k], non_blocking=True)
            fb.flashbob_bob(dev["Q"], dev["K"], dev["V"], O, dev["dO"], L, D, dev["UQ"],
                            dev["UK"], dev["UV"], w.tau, out["dQt"], out["dKt"], out["dVt"],
                            out["ddOt"], out["alpha"], out["E"], causal=w.causal,
                            stream=stream)
            for k in host_out:
                host_out[k].copy_(out[k], non_blocking=True)

        e2e_step()
        barrier()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(n_e2e):
            e2e_step()
        t1.record(stream)
        barrier()
        e_ms = reduce_max(t0.elapsed_time(t1), world, "cuda")
        e2e = {"value": job_tflops(flops, n_e2e, world, e_ms), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e_ms / n_e2e, "steps": n_e2e}

    peaks, peak_src = measured_peaks()
    dominant = "pass1" if p1_ms >= p2_ms else "pass2"
    dom_ms = p1_ms if dominant == "pass1" else p2_ms
    dom_flops = (PASS1_GEMMS if dominant == "pass1" else PASS2_GEMMS) * unit_flops
    achieved = dom_flops / (dom_ms * 1e-3) / 1e12
    peak = float(peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops")))
    traffic = read_traffic().get(dominant)
    in_bytes = sum(t.numel() * t.element_size() for t in dev.values()) + sum(
        t.numel() * t.element_size() for t in (O, L, D))

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "Hkv": w.kv_heads, "N": w.N,
                   "Nk": w.kv_len, "d": w.d, "causal": w.causal,
                   "tau": w.tau, "flops_per_step_per_gpu": flops,
                   "flop_convention": "38*N^2*d*B*H (19 GEMMs of 2*N^2*d); rectangular "
                                      "N*Nk for N^2, causal the pairs j <= i",
                   "l2": f"no flush: inputs {in_bytes / 2**20:.0f} MiB > L2 "
                         f"{L2_BYTES / 2**20:.0f} MiB",
                   "pass1_ms": p1_ms, "pass2_ms": p2_ms,
                   "prep_ms_outside_step": prep_ms,
                   "pct_of_peak": 100.0 * (value / world) / peak,
                   "paths": "tcgen05" if fb.flashbob_bob_tile_sizes(w.d, fb.FLASHBOB_BF16)[
                       "Br1"] == 128 else "simt"},
        "roofline": {"kernel": dominant, "bound": "tensor", "achieved": achieved, "peak": peak,
                     "unit": "TFLOP/s", "frac": achieved / peak, "traffic": traffic,
                     "peak_source": f"bf16_tflops_sustained of {peak_src} peaks"},
        "gpu_launches": 2 * args.steps,
        "clocks": clocks,
        "e2e": e2e,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rows, el = oracle_rows_sample(w, x, args.cpu_seconds)
        line["cpu_baseline"] = {
            "value": rows * row_flops(w) / el / 1e12, "unit": UNIT, "cores": os.cpu_count(),
            "kind": "oracle",
            "sample": f"{rows} seeded rows of head (0,0) through oracle.bob_rows (fp64 numpy, "
                      f"{el:.1f} s); {row_flops(w):.3e} flops credited per row"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
