#!/usr/bin/env python3
"""Benchmark of the W4A16 weight-only GEMM on GB300: µs per call and
effective HBM GB/s at M = 16, as a fraction of the HBM roofline.

Workload (one "step"): the MLP-shaped pair of the 4B-class verifier at one
16-token speculative block -- up-projection K=2560 -> N=9728 and
down-projection K=9728 -> N=2560, INT4 codes uniform in [-8, 7], group 128,
bf16 scales 0.02|N(0,1)| + 1e-3, bf16 X ~ N(0, 1), seed 1.  The packing step
is offline (once per weight) and is timed separately ("pack" in the line).

  value   device-timed throughput (algorithmic bytes / time, GB/s) with all
          inputs resident in HBM; CUDA graph replay of the K steps, the
          buffers rotated over enough copies that every call misses L2.
  e2e     the same metric through the public API with host buffers: each
          step copies both GEMMs' X from pinned host memory (one copy), runs
          both GEMMs, reads both outputs back (one copy), then synchronises.
  roofline  the small-M GEMM kernel: algorithmic bytes per launch over its
          average launch duration, against the measured HBM copy bandwidth.
  cpu_baseline  the CPU oracle (plain C, fp64) timed on a bounded sample.

--impl reference times the CPU oracle as the reference arm (there is no
other implementation of this path to run).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("W4A16 GEMM µs/call and effective HBM GB/s at M=16 "
          "(fraction of roofline)")
WORKLOAD = "w4a16_mlp_pair_m16_up2560x9728_down9728x2560_g128"
M, K_UP, N_UP = 16, 2560, 9728
K_DN, N_DN = 9728, 2560
GROUP = 128
SEED = 1


def algorithmic_bytes(m, k, n, bits=4):
    """Packed W + scales + X read + Y written, each once."""
    return k * n * bits // 8 + (k // GROUP) * n * 2 + m * k * 2 + m * n * 2


# A spin of this many SM cycles (~0.1 ms) is queued on the stream before
# each start event, so that the CPU-side submission of the timed graph is
# over before the GPU reaches it: the region then holds the device time of
# the timed steps and nothing before them.
SPIN_CYCLES = 200_000

BYTES_UP = algorithmic_bytes(M, K_UP, N_UP)
BYTES_DN = algorithmic_bytes(M, K_DN, N_DN)
BYTES_STEP = BYTES_UP + BYTES_DN


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["wq", "reference"], default="wq")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-configuration timings (C1, C3, C4, C5)")
    ap.add_argument("--pdl", type=int, default=1,
                    help="programmatic dependent launch between the GEMMs")
    ap.add_argument("--sweep", action="store_true",
                    help="time every benchmark GEMM shape and print a table "
                         "(one JSON object per shape) instead of the bench line")
    ap.add_argument("--regime", type=int, default=-1,
                    help="run every GEMM on one kernel family (0 warp-MMA small-M, "
                         "1 tiled tensor-core, 2 tensor-memory small-M, 3 tensor-memory "
                         "tiled, 4 tensor-memory small-M with overlapping launches); "
                         "-1 automatic")
    ap.add_argument("--only", default="",
                    help="sweep: only cases whose name contains this text")
    ap.add_argument("--shape", default="",
                    help="sweep: one extra shape M,K,N,bits (e.g. 1024,2560,9728,4)")
    return ap.parse_args()


# ------------------------------------------------------------ helpers ---
def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(ms, dev, pg):
    """The slowest rank's time: every rank's timed region ends only when all
    ranks have finished their share (replicas, weak scaling)."""
    if pg is None:
        return ms
    import torch
    t = torch.tensor([float(ms)], device=dev)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(bytes_per_step, steps, world, ms):
    """Whole-job throughput: the bytes every rank moved over the slowest
    rank's time."""
    return bytes_per_step * steps * world / (ms * 1e-3) / 1e9


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:  # noqa: BLE001
        return 6800.0, "fallback"


# The kernel family the headline step runs, its source files (the ncu
# traffic figure is keyed by their hash) and its name in the launch list.
FAMILY_SOURCES = {0: ("wq_gemm_small.cu", "wq_device.cuh"),
                  4: ("wq_gemm_stream.cu", "wq_device.cuh", "wq_tmem_dequant.cuh",
                      "wq_tcgen05.cuh")}
FAMILY_KERNELS = {0: "gemm_small_kernel<4, CH> (CH = 4 up, 2 down)",
                  4: "gemm_stream_kernel<4>"}


def kernel_source_hash(family):
    h = hashlib.sha256()
    for f in FAMILY_SOURCES.get(family, ()):
        with open(os.path.join(ROOT, "w4a16_weight_only_wq_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload_key, family):
    """DRAM bytes per launch from a committed ncu summary, if it was taken
    on the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "small_gemm_dram_traffic.txt")
    if not os.path.exists(path):
        return None
    src = kernel_source_hash(family)
    for line in open(path):
        parts = line.split()
        if len(parts) == 3 and not line.startswith("#") and parts[0] == src \
                and parts[1] == workload_key:
            return float(parts[2])
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons during a region."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except FileNotFoundError:
            self.proc = None
        time.sleep(0.15)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                smax = float(f[1])
            except ValueError:
                continue
            for nm, v in zip(names, f[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------- workload ---
def make_inputs():
    from tests import synth
    up = synth.GemmCase("up", M, K_UP, N_UP, 4, SEED).draw()
    dn = synth.GemmCase("down", M, K_DN, N_DN, 4, SEED).draw()
    return up, dn


def cpu_oracle_rate(up, dn, budget_s=12.0, max_steps=500):
    """Time the CPU oracle on whole steps (both GEMMs) until the budget is
    spent; returns (GB/s, steps, seconds, threads)."""
    import oracle
    threads = min(os.cpu_count() or 1, M)
    p_up = oracle.pack(up["q"], 4)
    p_dn = oracle.pack(dn["q"], 4)
    steps, t0 = 0, time.perf_counter()
    while True:
        oracle.gemm(up["X"], p_up, up["s"], K_UP, N_UP, 4, nthreads=threads)
        oracle.gemm(dn["X"], p_dn, dn["s"], K_DN, N_DN, 4, nthreads=threads)
        steps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or steps >= max_steps:
            break
    return BYTES_STEP * steps / el / 1e9, steps, el, threads


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    up, dn = make_inputs()
    budget = 60.0
    rate, steps, el, threads = cpu_oracle_rate(up, dn, budget_s=budget,
                                               max_steps=max(1, args.steps))
    sample = (f"{steps} whole steps (up + down GEMM at M=16 on the same seeded "
              f"inputs) in {el:.1f} s; unpack and dequant single-threaded, "
              f"the fp64 GEMM over {threads} row threads")
    line = {
        "metric": METRIC, "value": rate, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": steps, "warmup": 0, "ms_per_step": el / steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic", "impl": "reference",
        "config": {"workload": WORKLOAD, "M": M, "group": GROUP, "bits": 4},
        "cpu_baseline": {"value": rate, "unit": "GB/s", "cores": threads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": rate, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "note": "the reference arm is the CPU oracle: the pages ship no "
                "implementation of this kernel to install or run",
    }
    print(json.dumps(line), flush=True)
    return 0


def run_wq(args):
    import torch

    rank, world, local_rank = dist_env()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist

    import w4a16_weight_only_wq_gb300 as wq

    up, dn = make_inputs()

    def to_bf16(a):
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)

    # Pack on the GPU (offline step), timed separately.
    q_up = torch.from_numpy(up["q"]).to(dev)
    q_dn = torch.from_numpy(dn["q"]).to(dev)
    wp_up = wq.pack_codes(q_up, 4)
    wp_dn = wq.pack_codes(q_dn, 4)
    s_up, s_dn = to_bf16(up["s"]), to_bf16(dn["s"])
    x_up, x_dn = to_bf16(up["X"]), to_bf16(dn["X"])
    torch.cuda.synchronize()

    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 0) or 132 * 2**20)
    reps = max(4, math.ceil(2.0 * l2 / BYTES_STEP) + 1)
    sets = []
    for _ in range(reps):
        sets.append(dict(
            wu=wp_up.clone(), su=s_up.clone(), xu=x_up.clone(),
            yu=torch.empty((M, N_UP), dtype=torch.bfloat16, device=dev),
            wd=wp_dn.clone(), sd=s_dn.clone(), xd=x_dn.clone(),
            yd=torch.empty((M, N_DN), dtype=torch.bfloat16, device=dev)))
    torch.cuda.synchronize()
    wq.wq_set_programmatic_launch(bool(args.pdl))
    wq.wq_debug_force_regime(args.regime)

    stream = torch.cuda.Stream(device=dev)
    sh = int(stream.cuda_stream)

    def step(i):
        b = sets[i % reps]
        st = wq.wq_gemm_w4a16(b["xu"].data_ptr(), b["wu"].data_ptr(),
                              b["su"].data_ptr(), b["yu"].data_ptr(),
                              M, N_UP, K_UP, GROUP, sh)
        st |= wq.wq_gemm_w4a16(b["xd"].data_ptr(), b["wd"].data_ptr(),
                               b["sd"].data_ptr(), b["yd"].data_ptr(),
                               M, N_DN, K_DN, GROUP, sh)
        if st != 0:
            raise RuntimeError(f"wq_gemm_w4a16 failed: {wq.status_string(st)}")

    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):
            step(i)
    stream.synchronize()

    # Graph of S steps (a multiple of the rotation), replayed to cover K.
    S = min(args.steps, reps * max(1, 600 // reps))
    S = max(1, S)
    full, tail = divmod(args.steps, S)

    def capture(nsteps, base):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(nsteps):
                step(base + i)
        return g

    g_full = capture(S, 0) if full else None
    g_tail = capture(tail, full * S) if tail else None

    def replay(g):
        # CUDAGraph.replay() launches on the current stream: make it `stream`
        with torch.cuda.stream(stream):
            g.replay()

    for g in (g_full, g_tail):  # untimed replay (warm-up of the graphs)
        if g is not None:
            replay(g)
    torch.cuda.synchronize()

    def barrier():
        if pg is not None:
            pg.barrier()
        torch.cuda.synchronize()

    clocks = ClockSampler(local_rank)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    clocks.start()
    barrier()
    with torch.cuda.stream(stream):
        torch.cuda._sleep(SPIN_CYCLES)  # covers the CPU-side graph submission
    ev0.record(stream)
    for _ in range(full):
        replay(g_full)
    if g_tail is not None:
        replay(g_tail)
    ev1.record(stream)
    barrier()
    clocks.stop()
    ms = ev0.elapsed_time(ev1)
    clock_note = "sampled during the timed region"
    csum = clocks.summary()
    if csum is None or csum.get("samples", 0) < 3:
        # timed region too short for the sampler: soak the same graph
        soak = ClockSampler(local_rank)
        soak.start()
        t_end = time.time() + 1.0
        while time.time() < t_end:
            replay(g_full or g_tail)
            torch.cuda.synchronize()
        soak.stop()
        csum = soak.summary()
        clock_note = "timed region too short; sampled during a 1 s soak of the same graph"
    ms = max_over_ranks(ms, dev, pg)

    ms_step = ms / args.steps
    value = whole_job_gbs(BYTES_STEP, args.steps, world, ms)

    # Per-GEMM averages: separate graphs of one projection only.
    def time_single(which, n=400):
        def one(i):
            b = sets[i % reps]
            if which == "up":
                wq.wq_gemm_w4a16(b["xu"].data_ptr(), b["wu"].data_ptr(),
                                 b["su"].data_ptr(), b["yu"].data_ptr(),
                                 M, N_UP, K_UP, GROUP, sh)
            else:
                wq.wq_gemm_w4a16(b["xd"].data_ptr(), b["wd"].data_ptr(),
                                 b["sd"].data_ptr(), b["yd"].data_ptr(),
                                 M, N_DN, K_DN, GROUP, sh)
        n = reps * max(1, n // reps)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                one(i)
        replay(g)
        torch.cuda.synchronize()
        a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            torch.cuda._sleep(SPIN_CYCLES)
        a.record(stream)
        for _ in range(5):
            replay(g)
        b_.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b_) * 1e3 / (5 * n)

    us_up = time_single("up")
    us_dn = time_single("down")

    # Every other benchmark configuration, each timed on its own (rank 0).
    configs = {}
    if rank == 0 and not args.no_configs:
        from tests import synth
        for case in synth.C1 + synth.C3 + [c for c in synth.C4 if c.kind == "codes"] + synth.C5:
            r = time_gemm_case(wq, case, stream, sh, l2)
            configs[case.name] = {k_: r[k_] for k_ in ("us", "GB/s", "TFLOP/s", "bound", "frac",
                                                       "regime", "bytes")}

    # End to end through the API with host buffers.  Both GEMMs' inputs sit
    # in one pinned buffer (and one device buffer), and so do both results,
    # so that a step makes one copy each way.
    nx_up, nx_dn, ny_up, ny_dn = M * K_UP, M * K_DN, M * N_UP, M * N_DN
    hx = torch.empty(nx_up + nx_dn, dtype=torch.bfloat16).pin_memory()
    hx[:nx_up].copy_(x_up.cpu().reshape(-1))
    hx[nx_up:].copy_(x_dn.cpu().reshape(-1))
    hy = torch.empty(ny_up + ny_dn, dtype=torch.bfloat16).pin_memory()
    dx = torch.empty(nx_up + nx_dn, dtype=torch.bfloat16, device=dev)
    dy = torch.empty(ny_up + ny_dn, dtype=torch.bfloat16, device=dev)
    ex_up, ex_dn = dx[:nx_up].view(M, K_UP), dx[nx_up:].view(M, K_DN)
    ey_up, ey_dn = dy[:ny_up].view(M, N_UP), dy[ny_up:].view(M, N_DN)
    b0 = sets[0]

    def e2e_step():
        with torch.cuda.stream(stream):
            dx.copy_(hx, non_blocking=True)
            wq.gemm_w4a16(ex_up, b0["wu"], b0["su"], Y=ey_up, stream=stream)
            wq.gemm_w4a16(ex_dn, b0["wd"], b0["sd"], Y=ey_dn, stream=stream)
            hy.copy_(dy, non_blocking=True)
        stream.synchronize()

    for _ in range(20):
        e2e_step()
    n_e2e = min(args.steps, 2000)
    barrier()
    t0 = time.perf_counter()
    for _ in range(n_e2e):
        e2e_step()
    barrier()
    t_e2e = time.perf_counter() - t0
    e2e_val = BYTES_STEP * n_e2e * world / t_e2e / 1e9
    h2d = hx.numel() * 2
    d2h = hy.numel() * 2

    # Offline pack, timed on its own.
    wf = torch.randn(K_UP, N_UP, device=dev) * 0.02
    wq.pack_symmetric(wf, 4)
    torch.cuda.synchronize()
    a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(10):
        wq.pack_symmetric(wf, 4)
    b_.record()
    torch.cuda.synchronize()
    pack_us = a.elapsed_time(b_) * 100.0

    if wq.wq_last_device_error() != wq.WQ_OK:
        raise RuntimeError("a bounded in-kernel wait ran out during the bench")

    peak, peak_kind = measured_peaks()
    us_per_launch = ms_step * 1e3 / 2.0      # both launches move the same bytes
    achieved = (BYTES_STEP / 2) / (us_per_launch * 1e-6) / 1e9
    family = wq.wq_gemm_regime(4, M, N_UP, K_UP)
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak,
                "unit": "GB/s", "frac": achieved / peak,
                "traffic": recorded_traffic(WORKLOAD, family),
                "kernel": FAMILY_KERNELS.get(family, f"kernel family {family}"),
                "peak_source": f"{peak_kind} hbm_gbs (copy bandwidth)",
                "bytes_per_launch": BYTES_STEP // 2}

    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": M, "up_KxN": [K_UP, N_UP],
                   "down_KxN": [K_DN, N_DN], "group": GROUP, "bits": 4,
                   "l2": f"inputs rotated over {reps} buffer sets "
                         f"({reps * BYTES_STEP / 2**20:.0f} MiB > 2 x L2)",
                   "timing": f"CUDA graph of {S} steps replayed, events on the "
                             "launching stream; a 0.1 ms spin queued before the start "
                             "event covers the CPU-side graph submission",
                   "pdl": bool(args.pdl), "parallelism": f"replicas x{world}"},
        "us_per_call": us_per_launch,
        "us_per_call_isolated": {"up": us_up, "down": us_dn},
        "gbs_isolated": {"up": BYTES_UP / us_up / 1e3, "down": BYTES_DN / us_dn / 1e3},
        "pack_us": {"w4_rtn_2560x9728_fp32": pack_us},
        "roofline": roofline,
        "e2e": {"value": e2e_val, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": n_e2e,
                "ms_per_step": t_e2e / n_e2e * 1e3},
        "configs": configs,
        "gpu_launches": 2 * args.steps,
        "clocks": dict(csum or {}, note=clock_note),
    }
    if rank == 0 and not args.no_cpu_baseline:
        rate, steps, el, threads = cpu_oracle_rate(up, dn)
        line["cpu_baseline"] = {
            "value": rate, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{steps} whole steps (up + down at M=16, same inputs) in "
                      f"{el:.1f} s; unpack/dequant single-threaded, fp64 GEMM "
                      f"over {threads} row threads"}
    if pg is not None:
        pg.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def measured_tflops():
    """Dense bf16 tensor peak (burst) of this machine's GPUs, TFLOP/s."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:  # noqa: BLE001
        return 1900.0, "fallback"


def time_gemm_case(wq, case, stream, sh, l2, max_calls=200):
    """Device time of one GEMM shape: a CUDA graph of calls replayed with
    events on the launching stream, the inputs rotated over enough copies
    (> 2 x L2) that every call reads its weights from HBM.  Returns a dict
    with µs per call, GB/s, TFLOP/s, the kernel family and the fraction of
    the roofline that binds (HBM for memory-bound shapes, dense bf16 for
    the rest)."""
    import torch

    dev = torch.device("cuda", torch.cuda.current_device())
    d = case.draw()
    bits, m, k, n = case.bits, case.M, case.K, case.N
    q = torch.from_numpy(d["q"]).to(dev)
    wp = wq.pack_codes(q, bits)
    sc = torch.from_numpy(d["s"].view(np.int16)).view(torch.bfloat16).to(dev)
    x = torch.from_numpy(d["X"].view(np.int16)).view(torch.bfloat16).to(dev)
    nbytes = algorithmic_bytes(m, k, n, bits)
    reps = max(2, math.ceil(2.0 * l2 / nbytes) + 1)
    if reps * nbytes > 8 * 2**30:
        reps = 2
    bufs = [(x.clone(), wp.clone(), sc.clone(),
             torch.empty((m, n), dtype=torch.bfloat16, device=dev))
            for _ in range(reps)]
    fn = wq.wq_gemm_w4a16 if bits == 4 else wq.wq_gemm_w8a16

    def call(i):
        xb, wb, sb, yb = bufs[i % reps]
        st = fn(xb.data_ptr(), wb.data_ptr(), sb.data_ptr(), yb.data_ptr(), m, n, k, GROUP, sh)
        if st != 0:
            raise RuntimeError(wq.status_string(st))

    with torch.cuda.stream(stream):
        for i in range(3):
            call(i)
    stream.synchronize()
    per_graph = reps * max(1, min(max_calls, int(2e9 / max(nbytes, 1))) // reps)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(per_graph):
            call(i)
    with torch.cuda.stream(stream):
        g.replay()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    nrep = 5
    with torch.cuda.stream(stream):
        torch.cuda._sleep(SPIN_CYCLES)  # the graph is submitted while this runs
        a.record(stream)
        for _ in range(nrep):
            g.replay()
        b.record(stream)
    torch.cuda.synchronize()
    us = a.elapsed_time(b) * 1e3 / (nrep * per_graph)
    flops = 2.0 * m * n * k
    peak, peak_kind = measured_peaks()
    tpeak, tpeak_kind = measured_tflops()
    gbs = nbytes / us / 1e3
    tfs = flops / us / 1e6
    # the bound that the shape's arithmetic intensity selects
    tensor_bound = flops / (tpeak * 1e12) > nbytes / (peak * 1e9)
    res = {"case": case.name, "bits": bits, "M": m, "K": k, "N": n,
           "regime": wq.wq_gemm_regime(bits, m, n, k), "us": us, "GB/s": gbs,
           "TFLOP/s": tfs, "hbm_frac": gbs / peak, "peak_source": peak_kind,
           "bound": "tensor" if tensor_bound else "hbm",
           "frac": (tfs / tpeak) if tensor_bound else (gbs / peak),
           "bytes": nbytes, "rotation": reps}
    del bufs, g
    torch.cuda.empty_cache()
    return res


def run_sweep(args):
    """Per-shape timing of every benchmark GEMM (graph replay, L2 defeated by
    rotating buffer copies); one JSON object per line."""
    import torch

    import w4a16_weight_only_wq_gb300 as wq
    from tests import synth

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peak, peak_kind = measured_peaks()
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 0) or 132 * 2**20)
    wq.wq_set_programmatic_launch(bool(args.pdl))
    wq.wq_debug_force_regime(args.regime)
    stream = torch.cuda.Stream(device=dev)
    sh = int(stream.cuda_stream)
    cases = synth.C1 + synth.C2 + synth.C3 + \
        [c for c in synth.C4 if c.kind == "codes"] + synth.C5
    if args.shape:
        m_, k_, n_, b_ = (int(v) for v in args.shape.split(","))
        cases = [synth.GemmCase(f"shape_w{b_}_m{m_}_{k_}x{n_}", m_, k_, n_, b_, 9)]
    cases = [c for c in cases if args.only in c.name]
    for case in cases:
        print(json.dumps(time_gemm_case(wq, case, stream, sh, l2)), flush=True)
    if not args.shape and args.only in "c2_mlp_fused":
        sweep_mlp_pair(wq, synth, stream, sh, l2, peak, peak_kind)
    if not args.shape:
        for T, W in ((8192, 2048), (8192, 1024), (2048, 4096)):
            if args.only in f"swa_drafter_attention_b16_hq32_hkv8_d128_t{T}_w{W}":
                sweep_swa(wq, stream, sh, l2, peak, peak_kind, T, W)
    if wq.wq_last_device_error() != wq.WQ_OK:
        raise RuntimeError("a bounded in-kernel wait ran out during the sweep")
    return 0


def sweep_swa(wq, stream, sh, l2, peak, peak_kind, T, W, B=16, Hq=32, Hkv=8, D=128):
    """The drafter's sliding-window attention: a 16-token block at the end of
    a T-token cached sequence, 32 query heads over 8 key/value heads of 128;
    bytes are Q, the visible keys and values of every head, and O."""
    import torch

    dev = torch.device("cuda", 0)
    full = W == 0 or T <= W
    klo = 0 if full else max(0, T - B - W // 2)
    nk = T - klo
    nbytes = 2 * B * Hq * D * 2 + 2 * Hkv * nk * D * 2
    reps = max(2, math.ceil(2.0 * l2 / (2 * Hkv * nk * D * 2)) + 1)
    g = torch.Generator(device="cpu").manual_seed(T + W)
    q = torch.randn((B, Hq, D), generator=g).to(torch.bfloat16).to(dev)
    k = torch.randn((Hkv, T, D), generator=g).to(torch.bfloat16).to(dev)
    v = torch.randn((Hkv, T, D), generator=g).to(torch.bfloat16).to(dev)
    bufs = [(q.clone(), k.clone(), v.clone(), torch.empty_like(q)) for _ in range(reps)]

    def call(i):
        qb, kb, vb, ob = bufs[i % reps]
        st = wq.wq_swa_attention(qb.data_ptr(), kb.data_ptr(), vb.data_ptr(), ob.data_ptr(), B, Hq,
                                 Hkv, D, T, W, sh)
        if st != 0:
            raise RuntimeError(wq.status_string(st))

    with torch.cuda.stream(stream):
        for i in range(3):
            call(i)
    stream.synchronize()
    per_graph = reps * max(1, 200 // reps)
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr, stream=stream):
        for i in range(per_graph):
            call(i)
    with torch.cuda.stream(stream):
        gr.replay()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        a.record(stream)
        for _ in range(5):
            gr.replay()
        b.record(stream)
    torch.cuda.synchronize()
    us = a.elapsed_time(b) * 1e3 / (5 * per_graph)
    gbs = nbytes / us / 1e3
    print(json.dumps({
        "case": f"swa_drafter_attention_b{B}_hq{Hq}_hkv{Hkv}_d{D}_t{T}_w{W}", "B": B, "Hq": Hq,
        "Hkv": Hkv, "D": D, "T": T, "window": W, "visible_keys": nk, "us": us, "GB/s": gbs,
        "hbm_frac": gbs / peak, "peak_source": peak_kind, "bytes": nbytes,
        "rotation": reps}), flush=True)
    del gr, bufs
    torch.cuda.empty_cache()


def sweep_mlp_pair(wq, synth, stream, sh, l2, peak, peak_kind):
    """The MLP-shaped pair at M=16 through the fused call (one API call for
    both projections, the activation in the up-projection's store), for each
    activation; bytes are both projections' algorithmic bytes."""
    import torch

    dev = torch.device("cuda", 0)
    up_case, dn_case = synth.C2[0], synth.C2[1]
    du, dd = up_case.draw(), dn_case.draw()
    m, k, n1, n2 = up_case.M, up_case.K, up_case.N, dn_case.N
    nbytes = algorithmic_bytes(m, k, n1) + algorithmic_bytes(m, n1, n2)
    reps = max(2, math.ceil(2.0 * l2 / nbytes) + 1)

    def dev_bf16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

    wu = wq.pack_codes(torch.from_numpy(du["q"]).to(dev), 4)
    wd = wq.pack_codes(torch.from_numpy(dd["q"]).to(dev), 4)
    su, sd, x = dev_bf16(du["s"]), dev_bf16(dd["s"]), dev_bf16(du["X"])
    bufs = [(x.clone(), wu.clone(), su.clone(), wd.clone(), sd.clone(),
             torch.empty((m, n1), dtype=torch.bfloat16, device=dev),
             torch.empty((m, n2), dtype=torch.bfloat16, device=dev)) for _ in range(reps)]
    for act_name, act in (("none", wq.WQ_ACT_NONE), ("silu", wq.WQ_ACT_SILU)):
        def call(i):
            xb, wub, sub, wdb, sdb, hb, yb = bufs[i % reps]
            st = wq.wq_mlp_w4a16(xb.data_ptr(), wub.data_ptr(), sub.data_ptr(), wdb.data_ptr(),
                                 sdb.data_ptr(), hb.data_ptr(), yb.data_ptr(), m, k, n1, n2,
                                 GROUP, act, sh)
            if st != 0:
                raise RuntimeError(wq.status_string(st))

        with torch.cuda.stream(stream):
            for i in range(3):
                call(i)
        stream.synchronize()
        per_graph = reps * max(1, 100 // reps)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(per_graph):
                call(i)
        with torch.cuda.stream(stream):
            g.replay()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a.record(stream)
            for _ in range(5):
                g.replay()
            b.record(stream)
        torch.cuda.synchronize()
        us = a.elapsed_time(b) * 1e3 / (5 * per_graph)
        gbs = nbytes / us / 1e3
        print(json.dumps({
            "case": f"c2_mlp_fused_{act_name}_w4_m16_{k}x{n1}x{n2}", "bits": 4, "M": m,
            "K": k, "N1": n1, "N2": n2, "act": act_name, "us_per_pair": us, "GB/s": gbs,
            "hbm_frac": gbs / peak, "peak_source": peak_kind, "bytes": nbytes,
            "rotation": reps}), flush=True)
        del g
    del bufs
    torch.cuda.empty_cache()


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.sweep:
        return run_sweep(args)
    return run_wq(args)


if __name__ == "__main__":
    sys.exit(main())
