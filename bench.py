#!/usr/bin/env python3
"""Benchmark of the DiT blockwise-attention hot path on B300.

One step = one pass of the whole path over one batch of synthetic input that
is already resident in HBM:
  1. dit_attn_fwd        blockwise attention over n_kv_chunks K/V chunks with
                         on-chip log-sum-exp merging (bf16 O, fp32 LSE);
  2. dit_attn_merge      standalone log-sum-exp merge of n fp32 partials (the
                         partials a sequence-parallel split would hand over;
                         produced once, before timing, by dit_attn_fwd_partials);
  3. cfg_combine         classifier-free guidance combine on the latent pair.
Default workload: video DiT, B=1 H=48 S=17550 D=64, n_kv_chunks=16, merge over
16 fp32 partials (the workload whose configuration names the merge).

Prints ONE JSON line (rank 0).  ``value`` is attention TFLOP/s of the whole
step (4 B H S^2 D flops per step / step time, summed over ranks);
per-kernel numbers, the roofline of the dominant kernel, the fp64 CPU oracle
baseline, the end-to-end figure through host buffers and SM clocks sampled
during the timed region are added as objects.

``--impl reference`` times the fp64 CPU oracle as it stands on this host's
cores, on bounded samples of the same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "DiT attention TFLOP/s (fwd, bf16) on 1 B300 and % of dense-BF16 peak; merge GB/s"
NOMINAL_BF16_TFLOPS = 2250.0
NOMINAL_HBM_GBS = 8000.0
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
# Latent channels of the video workload's noise prediction (13 x 60 x 90 latent
# frames; 16 channels is this benchmark's choice).
VIDEO_LATENT = (16, 13, 60, 90)
L2_BYTES = 126e6


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="video")
    ap.add_argument("--heads", type=int, default=None,
                    help="override the head count (a smaller case of the same workload, for profiling)")
    ap.add_argument("--chunks", type=int, default=None, help="n_kv_chunks (default: the workload's largest)")
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--torus-chunks", type=int, default=8,
                    help="K/V chunks of the Torus-style copy/compute overlap measurement")
    ap.add_argument("--no-torus", action="store_true", help="skip the Torus-style overlap measurement")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="CPU-baseline sample budget")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the per-workload attention table")
    ap.add_argument("--config-reps", type=int, default=10,
                    help="timed calls per (workload, chunk count) in the per-workload table")
    return ap.parse_args(argv)


# ------------------------------------------------------------ helpers
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# The sources the attention kernel is compiled from: its device code and the
# launch (tensor maps, grid) in the C ABI file.
ATTN_SOURCES = ("attn_fwd.cuh", "ptx.cuh", "dit_attn.cu")


def kernel_source_hash(names=ATTN_SOURCES):
    """Short hash of the attention kernel's sources; a recorded ncu traffic
    figure is used only while this hash matches the one it was taken on."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "sequence_attention_attn_b300", "csrc")
    for name in sorted(names):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel sources (profiles/traffic.txt: kernel workload hash bytes)."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    try:
        lines = open(path).read().splitlines()
    except OSError:
        return None
    src = kernel_source_hash()
    for line in lines:
        parts = line.split()
        if len(parts) >= 4 and not line.startswith("#") and parts[0] == kernel and parts[1] == workload \
                and parts[2] == src:
            return float(parts[3])
    return None


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def reduce_time_and_units(seconds: float, units: float, world: int, device=None):
    """Max of the timed seconds and sum of the work units over ranks (no-op at
    world size 1).  Uses the default process group (NCCL on GPUs, gloo on CPU)."""
    if world == 1:
        return seconds, units
    import torch
    import torch.distributed as dist
    t = torch.tensor([seconds], dtype=torch.float64, device=device)
    u = torch.tensor([units], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


class ClockSampler:
    """nvidia-smi clock and throttle-reason sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"dit_bench_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path).read().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i, flag in enumerate(r[3]) if flag == "Active"})
        loaded = [r for r in rows if r[2] > 200.0] or rows
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": max(r[1] for r in rows),
                "power_w_max": max(r[2] for r in rows), "samples": len(rows), "reasons": reasons}


# ------------------------------------------------------- CPU baseline
def cpu_oracle_sample(cfg, budget_s: float, seed: int = 7):
    """Time the fp64 oracle, as it stands, on a bounded sample of the workload:
    R query rows (spread over all heads) against all S keys, the merge of those
    rows' n partials, and the CFG combine of a matching slice of the latent.
    Returns (attention flops covered, seconds, description, threads)."""
    import numpy as np
    import torch

    os.environ.setdefault("OMP_NUM_THREADS", str(len(os.sched_getaffinity(0))))
    import oracle
    from sequence_attention_attn_b300 import workloads

    impl = oracle.default()
    g = torch.Generator().manual_seed(seed)
    S, D, BH = cfg.S, cfg.D, cfg.B * cfg.H
    # one head's worth of K/V drawn on the CPU; every sampled row uses it
    k = torch.randn((1, S, D), generator=g).to(torch.bfloat16).double().numpy()
    v = torch.randn((1, S, D), generator=g).to(torch.bfloat16).double().numpy()
    q = torch.randn((1, S, D), generator=g).to(torch.bfloat16).double().numpy()
    n = cfg.merge_n or max(cfg.chunk_counts)

    def run(rows_count):
        rows = np.linspace(0, S - 1, rows_count).astype(np.int64)
        parts, lses = workloads.make_merge(n, rows_count, D, seed=seed)
        ec, eu = workloads.make_cfg((rows_count * D,), seed)
        t0 = time.perf_counter()
        impl.attention_rows(q, k, v, rows)
        impl.lse_merge(parts.numpy(), lses.numpy())
        impl.cfg_combine(ec.numpy(), eu.numpy(), cfg.cfg_w)
        return time.perf_counter() - t0

    rows = 64
    dt = run(rows)
    while dt < budget_s / 4 and rows < cfg.rows:
        rows = min(cfg.rows, int(rows * min(8.0, max(2.0, budget_s / max(dt, 1e-3)))))
        dt = run(rows)
    flops = 4.0 * rows * S * D
    desc = (f"{rows} of {cfg.rows} query rows (all {S} keys each, D={D}), merge of those rows' "
            f"{n} fp32 partials, CFG combine of {rows * D} latent values")
    return flops, dt, desc, impl.num_threads()


def run_reference(args):
    """The oracle, timed as it stands on the host cores (rank 0 only)."""
    rank, world, _local = dist_env()
    if rank != 0:
        return 0
    cfg = select_workload(args)
    n = args.chunks or cfg.merge_n or max(cfg.chunk_counts)
    per_step = max(0.5, min(10.0, 150.0 / max(1, args.steps + args.warmup)))
    flops, dt, desc, threads = cpu_oracle_sample(cfg, per_step)
    rows_per_step = desc.split(" ")[0]
    for _ in range(args.warmup):
        cpu_oracle_sample(cfg, per_step)
    times = []
    t_all = time.perf_counter()
    for _ in range(args.steps):
        f, d, _, _ = cpu_oracle_sample(cfg, per_step)
        times.append((f, d))
    total_f = sum(f for f, _ in times)
    total_t = sum(d for _, d in times)
    value = total_f / total_t / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_t / max(1, args.steps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": workload_config(cfg, n),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": f"per step: {desc}"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "wall_s": time.perf_counter() - t_all,
    }
    del rows_per_step
    print(json.dumps(line), flush=True)
    return 0


def l2_note(cfg, n):
    qkv = 3 * cfg.B * cfg.H * cfg.S * cfg.D * 2
    parts = n * cfg.rows * cfg.D * 4
    big = qkv > L2_BYTES and parts > L2_BYTES
    return (f"{'inputs larger than L2' if big else 'inputs NOT larger than L2'} "
            f"(q+k+v {qkv / 1e6:.0f} MB, merge partials {parts / 1e6:.0f} MB, L2 {L2_BYTES / 1e6:.0f} MB); "
            "no flush")


def workload_config(cfg, n):
    return {"workload": f"{cfg.name}: B={cfg.B} H={cfg.H} S={cfg.S} D={cfg.D}, n_kv_chunks={n}; "
                        f"step = attention + LSE merge of {n} fp32 partials + CFG combine",
            "B": cfg.B, "H": cfg.H, "S": cfg.S, "D": cfg.D, "n_kv_chunks": n,
            "merge_partials": n, "cfg_latent": list(VIDEO_LATENT if cfg.cfg_shape is None else cfg.cfg_shape),
            "l2": l2_note(cfg, n),
            "parallelism": "replicas"}


# ------------------------------------------------------------ our arm
def select_workload(args):
    """The named workload, with the head count overridden if --heads is given."""
    import dataclasses
    from sequence_attention_attn_b300 import workloads
    cfg = workloads.BY_NAME[args.workload]
    if args.heads is not None:
        if args.heads < 1:
            raise SystemExit("--heads must be >= 1")
        cfg = dataclasses.replace(cfg, H=args.heads)
    return cfg


def run_ours(args):
    import torch
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from sequence_attention_attn_b300 import dit_attn, workloads
    cfg = select_workload(args)
    n = args.chunks or cfg.merge_n or max(cfg.chunk_counts)
    peaks, peak_src = load_peaks()

    q, k, v = workloads.make_qkv(cfg, seed=workloads.seed_for(cfg, rank), generator_device="cuda")
    B, H, S, D = q.shape
    rows = B * H * S
    out = torch.empty_like(q)
    lse = torch.empty((B, H, S), dtype=torch.float32, device=dev)
    parts, part_lse = dit_attn.attention_partials(q, k, v, n)
    m_out = torch.empty((rows, D), dtype=torch.float32, device=dev)
    m_lse = torch.empty((rows,), dtype=torch.float32, device=dev)
    latent = VIDEO_LATENT if cfg.cfg_shape is None else cfg.cfg_shape
    eps_c, eps_u = workloads.make_cfg(latent, seed=workloads.seed_for(cfg, 300 + rank), device="cuda")
    c_out = torch.empty_like(eps_c)
    torch.cuda.synchronize()
    if dit_attn.dit_last_device_status() != 0:
        raise RuntimeError("device-side timeout while preparing inputs")

    stream = torch.cuda.current_stream()
    sptr = stream.cuda_stream

    def step():
        dit_attn.dit_attn_fwd(q, k, v, out, lse, n, sptr)
        dit_attn.dit_attn_merge(parts, part_lse, m_out, m_lse, sptr)
        dit_attn.cfg_combine(eps_c, eps_u, cfg.cfg_w, c_out, sptr)

    launches_per_step = 2 + (1 if eps_c.numel() % 4 == 0 else 2)  # attention, merge, CFG (+ its tail)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    t_start.record(stream)
    for i in range(K):
        evs[i][0].record(stream)
        dit_attn.dit_attn_fwd(q, k, v, out, lse, n, sptr)
        evs[i][1].record(stream)
        dit_attn.dit_attn_merge(parts, part_lse, m_out, m_lse, sptr)
        evs[i][2].record(stream)
        dit_attn.cfg_combine(eps_c, eps_u, cfg.cfg_w, c_out, sptr)
        evs[i][3].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if world > 1:
        torch.distributed.barrier()
    status = dit_attn.dit_last_device_status()
    if status != 0:
        raise RuntimeError(f"device status {status} after the timed region")

    total_s = t_start.elapsed_time(t_end) / 1e3
    attn_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    merge_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
    cfg_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in evs)
    flops = cfg.flops
    max_s, units = reduce_time_and_units(total_s, flops * K, world, dev)
    value = units / max_s / 1e12

    merge_bytes = 4.0 * rows * (n * (D + 1) + D + 1)
    cfg_bytes = 12.0 * eps_c.numel()
    attn_tflops = flops / (attn_ms / 1e3) / 1e12
    # One fixed denominator: the measured bf16 burst peak (the kernel runs for
    # a few ms at a time); sustained and nominal fractions are reported beside it.
    peak = peaks["bf16_tflops"]
    traffic = recorded_traffic("attn_fwd", cfg.name)

    # ---- end to end through host buffers (pinned), copies inside the timed region
    e2e = run_e2e(args, q, k, v, parts, part_lse, eps_c, eps_u, out, lse, m_out, m_lse, c_out, n, cfg,
                  world, dev)

    hbm_cfg = cfg_hbm_sweep(peaks, dev)
    per_config = None if args.no_configs else measure_configs(peaks, dev, rank, args.config_reps)
    if per_config is not None and cfg.name in per_config:
        per_config[cfg.name]["lse_merge_in_step"] = {
            "n_partials": n, "ms": merge_ms, "gbs": merge_bytes / (merge_ms / 1e3) / 1e9,
            "frac_of_measured_hbm": merge_bytes / (merge_ms / 1e3) / 1e9 / peaks["hbm_gbs"]}
    torus = None if args.no_torus else torus_overlap(q, k, v, cfg, dev, args.torus_chunks)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        f, dt, desc, threads = cpu_oracle_sample(cfg, args.cpu_seconds)
        cpu = {"value": f / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
               "sample": desc, "seconds": dt}

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": 1e3 * max_s / K, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(cfg, n),
        "roofline": {"bound": "tensor", "kernel": "attn_fwd", "achieved": attn_tflops, "peak": peak,
                     "unit": "TFLOP/s", "frac": attn_tflops / peak, "traffic": traffic,
                     "peak_source": f"{peak_src} burst bf16",
                     "frac_of_measured_sustained": attn_tflops / peaks["bf16_tflops_sustained"],
                     "frac_of_nominal_2250": attn_tflops / NOMINAL_BF16_TFLOPS,
                     "algorithmic_flops_per_launch": flops},
        "kernels": {
            "attn_fwd": {"ms": attn_ms, "tflops": attn_tflops,
                         "frac_of_measured_burst": attn_tflops / peaks["bf16_tflops"],
                         "frac_of_measured_sustained": attn_tflops / peaks["bf16_tflops_sustained"]},
            "lse_merge": {"ms": merge_ms, "bytes": merge_bytes, "gbs": merge_bytes / (merge_ms / 1e3) / 1e9,
                          "frac_of_measured_hbm": merge_bytes / (merge_ms / 1e3) / 1e9 / peaks["hbm_gbs"],
                          "frac_of_nominal_8000": merge_bytes / (merge_ms / 1e3) / 1e9 / NOMINAL_HBM_GBS},
            "cfg_combine": {"ms": cfg_ms, "bytes": cfg_bytes, "gbs": cfg_bytes / (cfg_ms / 1e3) / 1e9,
                            "note": "latent pair fits in L2; launch-bound"},
        },
        "configs": per_config,
        "cfg_hbm": hbm_cfg,
        "torus_overlap": torus,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches_per_step * K,
        "clocks": clk,
        "peaks": {**peaks, "source": peak_src},
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


class L2Flush:
    """Writes a buffer twice the size of L2 so that the next call reads its
    inputs from HBM."""

    def __init__(self, dev):
        import torch
        self.buf = torch.empty(int(2 * L2_BYTES) // 4, dtype=torch.float32, device=dev)

    def __call__(self):
        self.buf.zero_()


# A spin kernel of about 1 ms queued before a timed region, so that the calls
# after it are all enqueued before the GPU reaches the first event: the time
# measured is the device's, not the host's launch rate.
HOLD_CYCLES = 2_000_000


def time_calls(fn, flush, reps, warmup=3):
    """Per-call device time of fn() (CUDA events on the current stream) with L2
    flushed before every call (outside the events); returns (median ms of the
    flushed calls, mean ms of `reps` back-to-back calls without flushing).
    Each timed region starts behind a spin kernel (see HOLD_CYCLES)."""
    import torch
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        fn()
    cold = []
    for _ in range(reps):
        flush()
        torch.cuda._sleep(HOLD_CYCLES // 8)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        e1.synchronize()
        cold.append(e0.elapsed_time(e1))
    torch.cuda._sleep(HOLD_CYCLES)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        fn()
    e1.record(stream)
    e1.synchronize()
    return statistics.median(cold), e0.elapsed_time(e1) / reps


# One device's share of the heads under an 8-way head-parallel split (the
# heads a device computes after an all-to-all), per workload.
HEAD_SHARE = {"dit_xl2_512": 2, "pixart_1024": 2, "flux_mmdit": 3, "video": 6}
SPLIT_COUNTS = (2, 4)


def measure_head_share(cfg, q, k, v, heads, peaks, flush, reps):
    """The merged launch against the chunk-parallel one (dit_attn_fwd_split at
    SPLIT_COUNTS chunks) on the first `heads` heads of the workload: the few
    (batch, head, query-tile pair) units of such a launch leave SMs idle,
    which the chunks fill."""
    import torch
    from sequence_attention_attn_b300 import dit_attn
    qs, ks, vs = (t[:, :heads].contiguous() for t in (q, k, v))
    B, H, S, D = qs.shape
    flops = 4.0 * B * H * S * S * D
    out = torch.empty_like(qs)
    lse = torch.empty((B, H, S), dtype=torch.float32, device=qs.device)

    def rec(ms, ms_warm):
        tf = flops / (ms / 1e3) / 1e12
        return {"ms": ms, "tflops": tf, "frac_of_measured_burst": tf / peaks["bf16_tflops"],
                "ms_warm": ms_warm, "tflops_warm": flops / (ms_warm / 1e3) / 1e12}

    res = {"heads": heads, "B": B, "S": S, "D": D, "gflop": flops / 1e9,
           "merged": rec(*time_calls(lambda: dit_attn.dit_attn_fwd(qs, ks, vs, out, lse, 1), flush, reps)),
           "split": {}}
    for n in SPLIT_COUNTS:
        ws = torch.empty(dit_attn.dit_attn_split_workspace_bytes(B, H, S, D, n), dtype=torch.uint8,
                         device=qs.device)
        res["split"][str(n)] = rec(*time_calls(lambda: dit_attn.dit_attn_fwd_split(qs, ks, vs, out, lse, n, ws),
                                               flush, reps))
        del ws
    return res


def measure_configs(peaks, dev, rank, reps=10):
    """Attention TFLOP/s of every workload at each chunk count it lists, plus
    the CFG combine on the latent pairs the workloads name (latency: they sit
    in L2 sizes).  Inputs are drawn on the device with the workloads'
    generators.  Each launch is timed alone with L2 flushed before it
    ("ms"); "ms_warm" is the mean of back-to-back calls with L2 warm (inputs
    that a previous layer just wrote sit in L2 too), where consecutive
    launches overlap their launch gap (programmatic dependent launch)."""
    import torch
    from sequence_attention_attn_b300 import dit_attn, workloads
    flush = L2Flush(dev)
    table = {}
    for cfg in workloads.CONFIGS:
        q, k, v = workloads.make_qkv(cfg, seed=workloads.seed_for(cfg, rank), generator_device="cuda")
        out = torch.empty_like(q)
        lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
        entry = {"B": cfg.B, "H": cfg.H, "S": cfg.S, "D": cfg.D, "gflop": cfg.flops / 1e9, "attn": {}}
        for n in cfg.chunk_counts:
            ms, ms_warm = time_calls(lambda: dit_attn.dit_attn_fwd(q, k, v, out, lse, n), flush, reps)
            tf = cfg.flops / (ms / 1e3) / 1e12
            entry["attn"][str(n)] = {
                "ms": ms, "tflops": tf, "frac_of_measured_burst": tf / peaks["bf16_tflops"],
                "frac_of_nominal_2250": tf / NOMINAL_BF16_TFLOPS,
                "ms_warm": ms_warm, "tflops_warm": cfg.flops / (ms_warm / 1e3) / 1e12}
        share = HEAD_SHARE.get(cfg.name)
        if share is not None:
            entry["head_share"] = measure_head_share(cfg, q, k, v, share, peaks, flush, reps)
        if cfg.cfg_shape is not None:
            eps_c, eps_u = workloads.make_cfg(cfg.cfg_shape, seed=workloads.seed_for(cfg, 100), device=dev)
            c_out = torch.empty_like(eps_c)
            ms, ms_warm = time_calls(lambda: dit_attn.cfg_combine(eps_c, eps_u, cfg.cfg_w, c_out), flush, reps)
            nbytes = 12.0 * eps_c.numel()
            entry["cfg_combine"] = {"numel_per_operand": eps_c.numel(), "bytes": nbytes, "ms": ms,
                                    "gbs": nbytes / (ms / 1e3) / 1e9, "ms_warm": ms_warm,
                                    "note": "operands fit in L2: launch latency, not bandwidth"}
        table[cfg.name] = entry
        del q, k, v, out, lse
    if dit_attn.dit_last_device_status() != 0:
        raise RuntimeError("device-side timeout in the per-workload table")
    del flush
    torch.cuda.empty_cache()
    return table


def cfg_hbm_sweep(peaks, dev, sizes=(1 << 24, 1 << 26, 1 << 28), reps=10):
    """The CFG combine and its rel-MAE-fused forms (device atomics, and the
    no-workspace form with a fixed summation order) on operands larger than L2
    (2^24, 2^26 and 2^28 fp32 elements each: 0.2, 0.8 and 3.2 GB of
    algorithmic traffic per call), outside the timed step: the bandwidth
    figure the workload latents (L2-resident) cannot show.  The top-level
    figures are those of 2^26 elements; "sweep" holds every size."""
    import torch
    from sequence_attention_attn_b300 import dit_attn
    stream = torch.cuda.current_stream()
    sweep = []
    for numel in sizes:
        g = torch.Generator(device=dev).manual_seed(5)
        c = torch.randn(numel, generator=g, device=dev)
        u = torch.randn(numel, generator=g, device=dev)
        o = torch.empty_like(c)
        sums = torch.empty(3, dtype=torch.float64, device=dev)
        res = {"numel_per_operand": numel, "bytes_per_call": 12.0 * numel, "l2": "operands larger than L2; no flush"}
        for name, fn in (("cfg_combine", lambda: dit_attn.cfg_combine(c, u, 4.5, o, stream.cuda_stream)),
                         ("cfg_combine_relmae", lambda: dit_attn.cfg_combine_relmae(c, u, 4.5, o, sums,
                                                                                    stream.cuda_stream)),
                         ("cfg_combine_relmae_static",
                          lambda: dit_attn.cfg_combine_relmae_static(c, u, 4.5, o, sums, stream.cuda_stream))):
            for _ in range(3):
                fn()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                fn()
            e1.record(stream)
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / reps
            gbs = 12.0 * numel / (ms / 1e3) / 1e9
            res[name] = {"ms": ms, "gbs": gbs, "frac_of_measured_hbm": gbs / peaks["hbm_gbs"],
                         "frac_of_nominal_8000": gbs / NOMINAL_HBM_GBS}
        res["rel_mae"] = float(sums[2])
        sweep.append(res)
        del c, u, o
    torch.cuda.empty_cache()
    main = next(r for r in sweep if r["numel_per_operand"] == 1 << 26) if (1 << 26) in sizes else sweep[-1]
    return {**main, "sweep": [{"numel_per_operand": r["numel_per_operand"],
                               "cfg_combine_gbs": r["cfg_combine"]["gbs"],
                               "cfg_combine_relmae_gbs": r["cfg_combine_relmae"]["gbs"],
                               "cfg_combine_relmae_static_gbs": r["cfg_combine_relmae_static"]["gbs"]}
                              for r in sweep]}


def torus_overlap(q, k, v, cfg, dev, n, reps=5):
    """Host-to-result time of the chunked attention when K/V arrive from pinned
    host memory: (a) serial -- copy q, k, v, then the partials kernel and the
    LSE merge; (b) Torus-style -- copy q, then dit_attn_fwd_torus copies K/V
    chunk by chunk on a side stream while the chunks already landed are
    computed.  Both end with the fp32 output read back to the host.  Also
    timed: the copies alone and the computation alone (their maximum is
    what perfect overlap would reach)."""
    import torch
    from sequence_attention_attn_b300 import dit_attn
    B, H, S, D = q.shape
    rows = B * H * S
    hq, hk, hv = (torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (q, k, v))
    for h, t in zip((hq, hk, hv), (q, k, v)):
        h.copy_(t)
    qd, kd, vd = (torch.empty_like(t) for t in (q, k, v))
    parts = torch.empty((n, rows, D), dtype=torch.float32, device=dev)
    lses = torch.empty((n, rows), dtype=torch.float32, device=dev)
    out = torch.empty((rows, D), dtype=torch.float32, device=dev)
    lse = torch.empty((rows,), dtype=torch.float32, device=dev)
    h_out = torch.empty((rows, D), dtype=torch.float32, pin_memory=True)
    stream = torch.cuda.current_stream()
    side = torch.cuda.Stream(device=dev)
    sptr = stream.cuda_stream

    def copies():
        for d, h in ((qd, hq), (kd, hk), (vd, hv)):
            d.copy_(h, non_blocking=True)

    def compute():
        dit_attn.dit_attn_fwd_partials(qd, kd, vd, parts, lses, n, sptr)
        dit_attn.dit_attn_merge(parts, lses, out, lse, sptr)

    def serial():
        copies()
        compute()
        h_out.copy_(out, non_blocking=True)

    def torus():
        qd.copy_(hq, non_blocking=True)
        dit_attn.dit_attn_fwd_torus(qd, hk, hv, kd, vd, parts, lses, out, lse, n, sptr, side)
        h_out.copy_(out, non_blocking=True)

    def copy_only():
        copies()
        h_out.copy_(out, non_blocking=True)

    res = {"n_kv_chunks": n, "h2d_bytes": 3 * q.numel() * 2, "d2h_bytes": rows * D * 4,
           "source": "K/V from pinned host memory, copies on a side stream; serial arm: one stream"}
    for name, fn in (("serial_ms", serial), ("torus_ms", torus), ("copy_only_ms", copy_only),
                     ("compute_only_ms", compute)):
        for _ in range(2):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        res[name] = e0.elapsed_time(e1) / reps
        if name == "torus_ms":
            # the overlapped result is the serial one, bit for bit
            torus_out = out.clone()
            serial()
            torch.cuda.synchronize()
            res["torus_equals_serial"] = bool(torch.equal(torus_out, out))
            del torus_out
    if dit_attn.dit_last_device_status() != 0:
        raise RuntimeError("device-side timeout in the Torus-style measurement")
    res["overlap_gain"] = res["serial_ms"] / res["torus_ms"]
    res["perfect_overlap_ms"] = max(res["copy_only_ms"], res["compute_only_ms"])
    res["torus_tflops"] = cfg.flops / (res["torus_ms"] / 1e3) / 1e12
    del parts, lses, qd, kd, vd
    return res


def run_e2e(args, q, k, v, parts, part_lse, eps_c, eps_u, out, lse, m_out, m_lse, c_out, n, cfg, world, dev):
    import torch
    from sequence_attention_attn_b300 import dit_attn
    ins = [q, k, v, parts, part_lse, eps_c, eps_u]
    outs = [out, lse, m_out, m_lse, c_out]
    h_in = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in ins]
    for h, t in zip(h_in, ins):
        h.copy_(t)
    h_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs]
    stream = torch.cuda.current_stream()
    sptr = stream.cuda_stream
    h2d = sum(t.numel() * t.element_size() for t in ins)
    d2h = sum(t.numel() * t.element_size() for t in outs)

    side = torch.cuda.Stream(device=dev)
    landed = torch.cuda.Event()

    def one():
        # q, k, v on the compute stream; the merge and CFG inputs on a side
        # stream, so that their copy overlaps the attention, and the attention
        # output is read back while they are still coming in.
        side.wait_stream(stream)
        for d, h in zip(ins[:3], h_in[:3]):
            d.copy_(h, non_blocking=True)
        with torch.cuda.stream(side):
            for d, h in zip(ins[3:], h_in[3:]):
                d.copy_(h, non_blocking=True)
            landed.record(side)
        dit_attn.dit_attn_fwd(q, k, v, out, lse, n, sptr)
        for h, d in zip(h_out[:2], outs[:2]):
            h.copy_(d, non_blocking=True)
        stream.wait_event(landed)
        dit_attn.dit_attn_merge(parts, part_lse, m_out, m_lse, sptr)
        dit_attn.cfg_combine(eps_c, eps_u, cfg.cfg_w, c_out, sptr)
        for h, d in zip(h_out[2:], outs[2:]):
            h.copy_(d, non_blocking=True)

    one()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.e2e_steps):
        one()
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    max_s, units = reduce_time_and_units(dt, cfg.flops * args.e2e_steps, world, dev)
    # The host link alone, after the timed steps: the largest input (the merge
    # partials) copied once from pinned memory, CUDA events on the copy's
    # stream.  The step cannot be faster than its H2D bytes at this rate.
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    parts.copy_(h_in[3], non_blocking=True)
    e1.record(stream)
    e1.synchronize()
    link_gbs = parts.numel() * parts.element_size() / (e0.elapsed_time(e1) / 1e3) / 1e9
    ms_step = 1e3 * max_s / args.e2e_steps
    bound_ms = h2d / (link_gbs * 1e9) * 1e3
    return {"value": units / max_s / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": args.e2e_steps, "ms_per_step": ms_step,
            "host_h2d_gbs": link_gbs, "h2d_bound_ms": bound_ms, "frac_of_h2d_bound": bound_ms / ms_step}


def main(argv=None):
    args = parse_args(argv)
    if args.steps < 1 or args.warmup < 0:
        raise SystemExit("--steps must be >= 1 and --warmup >= 0")
    rank, world, _ = dist_env()
    if args.gpus > 1 and world == 1:
        # not launched by torchrun: relaunch one rank per GPU on this node
        cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={args.gpus}",
               "--master-addr", "127.0.0.1", "--master-port", "29531", os.path.abspath(__file__),
               *(argv if argv is not None else sys.argv[1:])]
        return subprocess.call(cmd)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
