"""Benchmark of the selective-scan hot path on GB300.

Workload (one "step"): one ssm_scan_fwd over the long-sequence bf16
selective-scan workload batch 4, L 16384, 5120 channels, N 16, one B/C group
(z gate and softplus on, final_state returned, y in fp32), inputs resident in
HBM.  Metric: scan elements per second, B*L*D*N / time, whole job.
`other_paths` adds the other workloads' device times against their rooflines:
the scan at batch 8, L 2048, 1536 channels and at batch 1, L 128, 1536
channels (fp32; launch-latency bound, timed as CUDA-graph replays), the
chunked SSD, the decode steps, the Mamba-3 forms and the gradients.

Usage:  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
        python bench.py --profile NAME [--reps R]   (one workload, for ncu)
        python bench.py --peaks                     (arithmetic-unit probes)
Under torchrun each rank runs its own copy of the workload on its GPU
(independent problems, no collective on the data path: weak scaling); the
timed region is bracketed by barriers and the slowest rank's time is used.

--impl reference times the fp64 CPU oracle (the only reference this method
has) on a bounded sample of the same workload, on the host's cores.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

BATCH, DIM, SEQLEN, DSTATE, NGROUPS = 4, 5120, 16384, 16, 1
METRIC = "scan elements/s (B*L*D*N per s)"
UNIT = "elements/s"
WORKLOAD = ("selective scan, bf16 inputs / fp32 state / fp32 y, batch 4, L 16384, "
            "D 5120, N 16, 1 B/C group, z gate + softplus(delta + bias), final_state")

# Roofline of the scan kernel: multi-function-unit (MUFU) bound.  Per
# element (b, l, d, n) one exp2; per (b, l, d) two MUFU ops for softplus
# (ex2, rcp) and two for the silu gate (ex2, rcp).  Peak = 152 SMs x 32 MUFU
# results per clock (the ex2 rate measured on GB300 by `bench.py --peaks`:
# 31.7 per SM per clock) x 2070 MHz (maximum SM clock).
SMS, MUFU_PER_CLK, SM_MAX_MHZ = 152, 32, 2070.0
HBM_PEAK_GBS = 6778.0  # measured copy bandwidth of the GB300s
BF16_PEAK_TFLOPS = 1908.5  # measured cuBLAS bf16 GEMM burst rate of the GB300s
MUFU_PEAK_GOPS = SMS * MUFU_PER_CLK * SM_MAX_MHZ * 1e6 / 1e9
# FP32 pipe: 128 lane-operations per SM per clock (FFMA rate measured by
# `bench.py --peaks`: 121 per SM per clock).
FP32_PER_CLK = 128
FP32_PEAK_GOPS = SMS * FP32_PER_CLK * SM_MAX_MHZ * 1e6 / 1e9
# The scan gradient's arithmetic per element (b, l, d, n), counted on the FP32
# pipe with no recomputation: the state h_t (dl*u*B, one FMA), the adjoint
# (lambda += dy0 C, lambda *= a, and dl*A for a), dC (dy0 h), dB (lambda dl u),
# dA (lambda h_{t-1} a, times dl), d dl (two FMAs), du (one FMA): 12 ops.
SCAN_BWD_FP32_PER_ELEMENT = 12
# DRAM bytes per launch of the scan kernel on this workload, from one ncu
# capture (dram__bytes_read.sum + dram__bytes_write.sum) of the same kernel
# build on batch 4, L 4096, 5120 channels (a quarter of the sequence, the same
# channel blocks), scaled by 4; None whenever the kernel has changed since.
SCAN_TRAFFIC_BYTES = 3279446016  # (506.05 MB + 313.81 MB) x 4


def algorithmic_counts():
    bld = BATCH * SEQLEN * DIM
    elements = bld * DSTATE
    mufu = elements + 4 * bld
    # bytes: u, delta, z (bf16) in; y (fp32) out; B, C (bf16) in; A, D, bias;
    # final_state out
    hbm = bld * (3 * 2 + 4) + 2 * BATCH * NGROUPS * DSTATE * SEQLEN * 2 \
        + DIM * DSTATE * 4 + 2 * DIM * 4 + BATCH * DIM * DSTATE * 4
    return elements, mufu, hbm


# ------------------------------------------------------------------ ranks

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend):
    if world <= 1:
        return None
    import torch.distributed as dist
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    dist.init_process_group(backend=backend)
    return dist


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(dist, value: float, device=None) -> float:
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(dist, value: float, device=None) -> float:
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 50):
        self.gpu = gpu_index
        self.period = period_ms
        self.proc = None
        self.lines = []
        self._t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", f"-lms", str(self.period)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()
        time.sleep(0.3)  # let the first sample arrive

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is None:
            return
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()

    def summary(self, t0: float, t1: float):
        rows = [l for (t, l) in self.lines if t0 - 0.05 <= t <= t1 + 0.15] or \
               [l for (_, l) in self.lines[-3:]]
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            parts = [p.strip() for p in r.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ ours

def make_inputs(rank):
    from state_space_model_selective_gb300 import inputs
    return inputs.scan_inputs(BATCH, DIM, SEQLEN, DSTATE, NGROUPS, "bf16", seed=1002 + rank,
                              gate=True, dskip="ones", device="cpu")


def cpu_baseline(inp, max_seconds=20.0):
    """Time the fp64 oracle (as it stands) on a bounded sample of the workload:
    the first `nb` batch rows of the same inputs, nb grown until one run takes
    at least ~2 s (capped so the total stays within max_seconds); when the
    whole workload takes less, it is run repeatedly for ~2 s and the mean
    taken."""
    import oracle
    nb, elapsed, el = 1, 0.0, 0
    dims = None
    while True:
        sl = slice(0, nb)
        args = (inp["u"][sl], inp["delta"][sl], inp["A"], inp["B"][sl], inp["C"][sl],
                inp["D"], inp["z"][sl], inp["delta_bias"], True)
        t0 = time.perf_counter()
        oracle.scan(*args)
        elapsed = time.perf_counter() - t0
        el = nb * SEQLEN * DIM * DSTATE
        dims = nb
        if elapsed >= 2.0 or nb >= BATCH or elapsed * 2 * 2 > max_seconds:
            break
        nb = min(BATCH, nb * 2)
    runs = 1
    if elapsed < 2.0:
        runs = max(1, min(int(2.0 / max(elapsed, 1e-3)), int(max_seconds / max(elapsed, 1e-3))))
        t0 = time.perf_counter()
        for _ in range(runs):
            oracle.scan(*args)
        elapsed = (time.perf_counter() - t0) / runs
    return {"value": el / elapsed, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"batch rows 0..{dims - 1} of the workload ({dims}x{DIM}x{SEQLEN}x{DSTATE} "
                      f"= {el} elements), fp64, mean of {runs} run(s), {elapsed:.2f} s each"}


def run_ours(args):
    import torch
    from state_space_model_selective_gb300 import binding

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = init_dist(world, "nccl")

    host = make_inputs(rank)
    # pinned host copies (the e2e leg copies them in every step)
    pinned = {k: (v.pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in host.items()}
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in host.items()}
    y = torch.empty((BATCH, DIM, SEQLEN), dtype=torch.float32, device=dev)
    fs = torch.empty((BATCH, DIM, DSTATE), dtype=torch.float32, device=dev)
    ws = torch.empty(binding.ssm_scan_workspace_bytes(BATCH, DIM, SEQLEN, DSTATE, NGROUPS),
                     dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        binding.ssm_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"],
                             d["delta_bias"], True, out_dtype=torch.float32, y=y,
                             final_state=fs, workspace=ws, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    assert binding.ssm_last_device_status(ws) == 0

    sampler = ClockSampler(local)
    sampler.start()
    barrier(dist)
    torch.cuda.synchronize(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_wall0 = time.time()
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    t_wall1 = time.time()
    barrier(dist)
    sampler.stop()
    ms_local = ev0.elapsed_time(ev1)
    ms = max_over_ranks(dist, ms_local, dev)
    clocks = sampler.summary(t_wall0, t_wall1)
    assert binding.ssm_last_device_status(ws) == 0

    elements, mufu, hbm = algorithmic_counts()
    total_elements = sum_over_ranks(dist, float(elements * args.steps), dev)
    value = total_elements / (ms / 1e3)
    per_launch_s = ms_local / 1e3 / args.steps
    achieved = mufu / per_launch_s / 1e9

    # ---- e2e: the scan through ssm_scan_fwd_host, the entry point for host-
    # resident activations: every step copies u, delta, z, B, C in from pinned host
    # memory and y and the final state out (the library pipelines the copies with
    # the scan over segments of the sequence); A, D and delta_bias are parameters
    # resident on the device
    e2e_steps = max(3, min(args.steps, 20))
    names = ["u", "delta", "z", "B", "C"]
    h2d = sum(pinned[k].numel() * pinned[k].element_size() for k in names)
    y_host = torch.empty(y.shape, dtype=y.dtype, pin_memory=True)
    fs_host = torch.empty(fs.shape, dtype=fs.dtype, pin_memory=True)
    d2h = y_host.numel() * 4 + fs_host.numel() * 4
    ws_host = torch.empty(binding.ssm_scan_fwd_host_workspace_bytes(
        BATCH, DIM, SEQLEN, DSTATE, NGROUPS, torch.bfloat16, torch.float32),
        dtype=torch.uint8, device=dev)

    def e2e_step():
        binding.ssm_scan_fwd_host(pinned["u"], pinned["delta"], d["A"], pinned["B"], pinned["C"],
                                  y_host, fs_host, d["D"], pinned["z"], d["delta_bias"], True,
                                  workspace=ws_host, stream=stream)

    e2e_step()
    torch.cuda.synchronize(dev)
    # five windows of steps, each timed whole (copies in and out of every step
    # inside it); the median window is reported and all five are listed, so a
    # stall of the shared host link in one or two windows does not decide the
    # number
    n_windows = 5
    win_steps = max(1, e2e_steps // n_windows)
    e2e_windows = []
    for _ in range(n_windows):
        barrier(dist)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(win_steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        w_ms = max_over_ranks(dist, e0.elapsed_time(e1), dev)
        w_total = sum_over_ranks(dist, float(elements * win_steps), dev)
        e2e_windows.append(w_total / (w_ms / 1e3))
    e2e_value = statistics.median(e2e_windows)

    paths = measure_other_paths(dev) if rank == 0 else None

    out = None
    if rank == 0:
        cpu = cpu_baseline(host) if world == 1 else None  # rank 0 at N=1 only
        out = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic",
            "config": {"workload": WORKLOAD, "batch": BATCH, "seqlen": SEQLEN, "dim": DIM,
                       "dstate": DSTATE, "ngroups": NGROUPS, "in_dtype": "bf16",
                       "state_dtype": "f32", "out_dtype": "f32",
                       "l2": "inputs 2.0 GB > 129 MB L2 (no flush)",
                       "parallelism": f"independent workload per GPU x{world}"},
            "e2e": {"value": e2e_value, "unit": UNIT,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "timing": f"median of {n_windows} windows of {win_steps} steps",
                    "windows": e2e_windows},
            "gpu_launches": args.steps,
            "roofline": {"bound": "alu", "achieved": achieved, "peak": MUFU_PEAK_GOPS,
                         "unit": "Gop/s (MUFU)", "frac": achieved / MUFU_PEAK_GOPS,
                         "traffic": SCAN_TRAFFIC_BYTES,
                         "algorithmic_mufu_ops_per_launch": mufu,
                         "algorithmic_hbm_bytes_per_launch": hbm,
                         "hbm_gbs_at_this_time": hbm / per_launch_s / 1e9},
            "clocks": clocks,
            "cpu_baseline": cpu,
            "other_paths": paths,
        }
        print(json.dumps(out), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return out


def measure_other_paths(dev, reps=20):
    """Device time of the chunked SSD (batch 32, L 256, 32 heads, headdim 64,
    d_state 128, bf16 in, fp32 y) and of one decode step (batch 256, 32 heads,
    headdim 64, d_state 128, fp32), Mamba-2 and Mamba-3 SISO forms, against
    the HBM roofline of their algorithmic bytes."""
    import torch
    from state_space_model_selective_gb300 import binding, inputs
    res = {}
    inp = inputs.ssd_inputs(32, 256, 32, 64, 128, 1, "bf16", seed=1004, device="cuda")
    y = torch.empty(inp["x"].shape, device=dev)
    fs = torch.empty(32, 32, 64, 128, device=dev)

    def ssd():
        binding.ssd_chunked_fwd(inp["x"], inp["dt"], inp["A_head"], inp["B"], inp["C"], 64,
                                out_dtype=torch.float32, y=y, final_state=fs)
    ms = _time(ssd, reps)
    nbytes = inp["x"].numel() * 2 + y.numel() * 4 + 2 * inp["B"].numel() * 2 + \
        inp["dt"].numel() * 4 + fs.numel() * 4
    el = 32 * 256 * 32 * 64 * 128
    res["ssd_chunked_fwd"] = {
        "workload": "chunked SSD bf16 in / fp32 y, batch 32, L 256, 32 heads, headdim 64, "
                    "d_state 128, chunk 64", "ms": ms, "elements_per_s": el / (ms / 1e3),
        "roofline": {"bound": "hbm", "achieved": nbytes / (ms / 1e3) / 1e9,
                     "peak": HBM_PEAK_GBS, "unit": "GB/s",
                     "frac": nbytes / (ms / 1e3) / 1e9 / HBM_PEAK_GBS,
                     "algorithmic_bytes": nbytes}}
    del inp
    res["ssm_scan_fwd_b8_l2048"] = _measure_scan(dev, 8, 1536, 2048, "bf16", reps)
    res["ssm_scan_fwd_b1_l128_f32"] = _measure_scan(dev, 1, 1536, 128, "f32", reps, graph=True)
    res["ssm_scan_bwd"] = _measure_scan_bwd(dev, reps)
    res["ssd_chunked_bwd"] = _measure_ssd_bwd(dev, reps)
    res["ssd_mamba3_bwd"] = _measure_mamba3_bwd(dev, reps)
    res["ssd_mamba3_mimo_bwd"] = _measure_mimo_bwd(dev, reps)
    m3 = inputs.mamba3_inputs(32, 256, 32, 64, 128, 1, "bf16", seed=1006, device="cuda")

    def ssd_m3():
        binding.ssd_mamba3_fwd(m3["x"], m3["dt"], m3["lam"], m3["A_head"], m3["B"], m3["C"], 64,
                               out_dtype=torch.float32, y=y, final_state=fs,
                               prev_B=m3["prev_B"], prev_x=m3["prev_x"])
    ms = _time(ssd_m3, reps)
    nbytes3 = nbytes + m3["lam"].numel() * 4 + m3["prev_B"].numel() * 2 + m3["prev_x"].numel() * 2
    res["ssd_mamba3_fwd"] = {
        "workload": "Mamba-3 SISO chunked prefill bf16 in / fp32 y, batch 32, L 256, 32 heads, "
                    "headdim 64, d_state 128, chunk 64", "ms": ms,
        "elements_per_s": el / (ms / 1e3),
        "roofline": {"bound": "hbm", "achieved": nbytes3 / (ms / 1e3) / 1e9,
                     "peak": HBM_PEAK_GBS, "unit": "GB/s",
                     "frac": nbytes3 / (ms / 1e3) / 1e9 / HBM_PEAK_GBS,
                     "algorithmic_bytes": nbytes3}}
    del m3, y, fs
    mi = inputs.mamba3_mimo_inputs(32, 256, 4, 32, 64, 128, 1, "bf16", seed=1007, device="cuda")
    ym = torch.empty(mi["x"].shape, device=dev)
    fsm = torch.empty(32, 32, 64, 128, device=dev)

    def ssd_mimo():
        binding.ssd_mamba3_mimo_fwd(mi["x"], mi["dt"], mi["lam"], mi["A_head"], mi["B"], mi["C"],
                                    16, out_dtype=torch.float32, y=ym, final_state=fsm,
                                    prev_B=mi["prev_B"], prev_x=mi["prev_x"])
    ms = _time(ssd_mimo, reps)
    nbm = (mi["x"].numel() * 2 + ym.numel() * 4 + 2 * mi["B"].numel() * 2 +
           2 * mi["dt"].numel() * 4 + fsm.numel() * 4 + mi["prev_B"].numel() * 2 +
           mi["prev_x"].numel() * 2)
    res["ssd_mamba3_mimo_fwd"] = {
        "workload": "Mamba-3 MIMO rank 4 chunked prefill bf16 in / fp32 y, batch 32, L 256, "
                    "32 heads, headdim 64, d_state 128, chunk 16", "ms": ms,
        "elements_per_s": el * 4 / (ms / 1e3),
        "roofline": {"bound": "hbm", "achieved": nbm / (ms / 1e3) / 1e9,
                     "peak": HBM_PEAK_GBS, "unit": "GB/s",
                     "frac": nbm / (ms / 1e3) / 1e9 / HBM_PEAK_GBS, "algorithmic_bytes": nbm}}
    del mi, ym, fsm
    res["ssm_mamba3_rope"] = _measure_rope(dev, reps)
    g = torch.Generator(device="cuda")
    g.manual_seed(1005)
    B_, H, P, N = 256, 32, 64, 128
    state = 0.1 * torch.randn(B_, H, P, N, device=dev, generator=g)
    x = torch.randn(B_, H, P, device=dev, generator=g)
    Bm = torch.randn(B_, 1, N, device=dev, generator=g)
    Cm = torch.randn(B_, 1, N, device=dev, generator=g)
    dt = torch.nn.functional.softplus(torch.randn(B_, H, device=dev, generator=g) - 4)
    A = -(1 + 15 * torch.rand(H, device=dev, generator=g))
    D = torch.ones(H, device=dev)
    yd = torch.empty_like(x)

    def dec():
        binding.ssm_decode_step(state, x, dt, A, Bm, Cm, D, y=yd)
    ms = _time(dec, reps)
    nbytes = 2 * state.numel() * 4 + 2 * x.numel() * 4 + 2 * Bm.numel() * 4 + dt.numel() * 4
    res["ssm_decode_step"] = {
        "workload": "decode step fp32, batch 256, 32 heads, headdim 64, d_state 128",
        "ms": ms, "elements_per_s": state.numel() / (ms / 1e3),
        "roofline": {"bound": "hbm", "achieved": nbytes / (ms / 1e3) / 1e9,
                     "peak": HBM_PEAK_GBS, "unit": "GB/s",
                     "frac": nbytes / (ms / 1e3) / 1e9 / HBM_PEAK_GBS,
                     "algorithmic_bytes": nbytes}}
    lam = torch.sigmoid(torch.randn(B_, H, device=dev, generator=g))
    xp = torch.randn(B_, H, P, device=dev, generator=g)
    Bp = torch.randn(B_, 1, N, device=dev, generator=g)

    def dec_m3():
        binding.ssm_decode_step_mamba3(state, Bp, xp, x, dt, lam, A, Bm, Cm, D, y=yd)
    ms = _time(dec_m3, reps)
    nbytes3 = nbytes + lam.numel() * 4 + xp.numel() * 4 + Bp.numel() * 4
    xr = torch.randn(B_, 4, H, P, device=dev, generator=g)
    xpr = torch.randn(B_, 4, H, P, device=dev, generator=g)
    Br = torch.randn(B_, 4, 1, N, device=dev, generator=g)
    Cr = torch.randn(B_, 4, 1, N, device=dev, generator=g)
    Bpr = torch.randn(B_, 4, 1, N, device=dev, generator=g)
    yr = torch.empty_like(xr)

    def dec_mimo():
        binding.ssm_decode_step_mamba3_mimo(state, Bpr, xpr, xr, dt, lam, A, Br, Cr, D, y=yr)
    ms_m = _time(dec_mimo, reps)
    nbytes_m = (2 * state.numel() * 4 + (xr.numel() + xpr.numel() + yr.numel()) * 4 +
                (Br.numel() + Cr.numel() + Bpr.numel()) * 4 + 2 * dt.numel() * 4)
    res["ssm_decode_step_mamba3_mimo"] = {
        "workload": "Mamba-3 MIMO rank 4 decode step fp32, batch 256, 32 heads, headdim 64, "
                    "d_state 128", "ms": ms_m, "elements_per_s": state.numel() / (ms_m / 1e3),
        "roofline": {"bound": "hbm", "achieved": nbytes_m / (ms_m / 1e3) / 1e9,
                     "peak": HBM_PEAK_GBS, "unit": "GB/s",
                     "frac": nbytes_m / (ms_m / 1e3) / 1e9 / HBM_PEAK_GBS,
                     "algorithmic_bytes": nbytes_m}}
    res["ssm_decode_step_mamba3"] = {
        "workload": "Mamba-3 SISO decode step fp32, batch 256, 32 heads, headdim 64, d_state 128",
        "ms": ms, "elements_per_s": state.numel() / (ms / 1e3),
        "roofline": {"bound": "hbm", "achieved": nbytes3 / (ms / 1e3) / 1e9,
                     "peak": HBM_PEAK_GBS, "unit": "GB/s",
                     "frac": nbytes3 / (ms / 1e3) / 1e9 / HBM_PEAK_GBS,
                     "algorithmic_bytes": nbytes3}}
    return res


def _measure_scan(dev, batch, dim, seqlen, dt, reps, graph=False):
    """The forward scan (gate, softplus, final_state, y in fp32) on one of the
    other scan workloads, against the MUFU roofline like the benchmark step.
    With graph=True (the 3.1e6-element fp32 workload, whose launch overhead is
    larger than its work) the calls are captured in a CUDA graph and timed as
    replays, and the plain back-to-back launch time is reported beside it."""
    import torch
    from state_space_model_selective_gb300 import binding, inputs
    seed = {2048: 1002, 128: 1001}.get(seqlen, 1000)
    x = inputs.scan_inputs(batch, dim, seqlen, DSTATE, 1, dt, seed=seed, device="cuda")
    y = torch.empty((batch, dim, seqlen), dtype=torch.float32, device=dev)
    fs = torch.empty((batch, dim, DSTATE), dtype=torch.float32, device=dev)
    ws = torch.empty(binding.ssm_scan_workspace_bytes(batch, dim, seqlen, DSTATE, 1),
                     dtype=torch.uint8, device=dev)

    def fwd():
        binding.ssm_scan_fwd(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"],
                             x["delta_bias"], True, out_dtype=torch.float32, y=y,
                             final_state=fs, workspace=ws)
    ms = _time(fwd, reps)
    out = {}
    if graph:
        out["ms_plain_launches"] = ms
        ms = _time_graph(fwd, 200)
    assert binding.ssm_last_device_status(ws) == 0
    bld = batch * seqlen * dim
    el = bld * DSTATE
    mufu = el + 4 * bld
    achieved = mufu / (ms / 1e3) / 1e9
    path = "sequence-parallel scan" if batch * dim <= 3072 else "chained scan"
    out.update({
        "workload": f"selective scan {dt} in / fp32 y, batch {batch}, L {seqlen}, {dim} "
                    f"channels, d_state 16, 1 group, gate, softplus ({path})",
        "ms": ms, "elements_per_s": el / (ms / 1e3),
        "timing": "CUDA-graph replay of 200 calls" if graph else f"mean of {reps} launches",
        "roofline": {"bound": "alu", "achieved": achieved, "peak": MUFU_PEAK_GOPS,
                     "unit": "Gop/s (MUFU)", "frac": achieved / MUFU_PEAK_GOPS,
                     "algorithmic_mufu_ops": mufu}})
    return out


def _measure_rope(dev, reps):
    """Mamba-3's data-dependent rotation of B and C (ssm_mamba3_rope) on the SSD
    workload (batch 32, L 256, 32 heads, one group, d_state 128, bf16 B, C), against
    the HBM roofline of its algorithmic bytes: dt, theta, B, C in; the per-head
    rotated B, C out."""
    import torch
    from state_space_model_selective_gb300 import binding, inputs
    Bn, L, H, P, N = 32, 256, 32, 64, 128
    inp = inputs.ssd_inputs(Bn, L, H, P, N, 1, "bf16", seed=1004, device=dev)
    r = inputs.rope_inputs(Bn, L, H, N, seed=1008, device=dev)
    Br = torch.empty(Bn, L, H, N, dtype=torch.bfloat16, device=dev)
    Cr = torch.empty_like(Br)
    ang = torch.empty(Bn, H, N // 2, device=dev)

    def rope():
        binding.ssm_mamba3_rope(inp["B"], inp["C"], inp["dt"], r["theta"], r["angle0"],
                                B_rot=Br, C_rot=Cr, angle_out=ang)
    ms = _time(rope, reps)
    nbytes = (inp["dt"].numel() * 4 + r["theta"].numel() * 4 + 2 * inp["B"].numel() * 2 +
              2 * Br.numel() * 2 + 2 * ang.numel() * 4)
    return {"workload": "Mamba-3 RoPE on B, C: bf16, batch 32, L 256, 32 heads, 1 group, "
                        "d_state 128 (per-head rotated B, C out)", "ms": ms,
            "roofline": {"bound": "hbm", "achieved": nbytes / (ms / 1e3) / 1e9,
                         "peak": HBM_PEAK_GBS, "unit": "GB/s",
                         "frac": nbytes / (ms / 1e3) / 1e9 / HBM_PEAK_GBS,
                         "algorithmic_bytes": nbytes}}


def _measure_scan_bwd(dev, reps):
    """The scan gradient (ssm_scan_bwd: checkpointing forward, reverse sweep,
    reductions) on the batch 8, L 2048, 1536-channel scan workload (bf16,
    d_state 16, D, gate, bias, softplus), against the FP32 pipe."""
    import torch
    from state_space_model_selective_gb300 import binding, inputs
    BATCH, DIM, SEQLEN = 8, 1536, 2048
    inp = inputs.scan_inputs(BATCH, DIM, SEQLEN, DSTATE, 1, "bf16", seed=1002, device=dev)
    g = torch.Generator(device=dev)
    g.manual_seed(1008)
    dy = torch.randn(BATCH, DIM, SEQLEN, device=dev, generator=g).to(torch.bfloat16)
    f = dict(dtype=torch.float32, device=dev)
    act = (BATCH, DIM, SEQLEN)
    out = {"du": torch.empty(act, **f), "ddelta": torch.empty(act, **f),
           "dz": torch.empty(act, **f), "dA": torch.empty(DIM, DSTATE, **f),
           "dB": torch.empty(BATCH, 1, DSTATE, SEQLEN, **f),
           "dC": torch.empty(BATCH, 1, DSTATE, SEQLEN, **f), "dD": torch.empty(DIM, **f),
           "ddelta_bias": torch.empty(DIM, **f),
           "dinitial_state": torch.empty(BATCH, DIM, DSTATE, **f)}
    ws = torch.empty(binding.ssm_scan_bwd_workspace_bytes(BATCH, DIM, SEQLEN, DSTATE, 1),
                     dtype=torch.uint8, device=dev)

    def bwd():
        binding.ssm_scan_bwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], dy, inp["D"],
                             inp["z"], inp["delta_bias"], True, workspace=ws, out=out)
    ms = _time(bwd, reps)
    el = BATCH * SEQLEN * DIM * DSTATE
    ops = SCAN_BWD_FP32_PER_ELEMENT * el
    achieved = ops / (ms / 1e3) / 1e9
    # a training step's scan: the forward keeping checkpoints, then the gradient
    # from them (no second forward recurrence)
    y = torch.empty(BATCH, DIM, SEQLEN, **f)
    fs = torch.empty(BATCH, DIM, DSTATE, **f)
    ck = torch.empty(binding.ssm_scan_checkpoint_bytes(BATCH, DIM, SEQLEN) // 4, **f)
    wsf = torch.empty(binding.ssm_scan_workspace_bytes(BATCH, DIM, SEQLEN), dtype=torch.uint8,
                      device=dev)

    def train():
        binding.ssm_scan_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"],
                             inp["z"], inp["delta_bias"], True, out_dtype=torch.float32, y=y,
                             final_state=fs, workspace=wsf, checkpoints=ck)
        binding.ssm_scan_bwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], dy, inp["D"],
                             inp["z"], inp["delta_bias"], True, workspace=ws, out=out,
                             checkpoints=ck)
    ms_train = _time(train, reps)
    return {"workload": "selective-scan gradient bf16 in / fp32 gradients, batch 8, L 2048, "
                        "1536 channels, d_state 16, D, gate, bias, softplus",
            "ms": ms, "elements_per_s": el / (ms / 1e3),
            "train_step_ms": ms_train,
            "train_step": "forward keeping checkpoints + gradient from them",
            "roofline": {"bound": "alu", "achieved": achieved, "peak": FP32_PEAK_GOPS,
                         "unit": "Gop/s (FP32 pipe)", "frac": achieved / FP32_PEAK_GOPS,
                         "algorithmic_fp32_ops": ops}}


def _measure_ssd_bwd(dev, reps):
    """The chunked SSD's gradient (ssd_chunked_bwd: block-state forward, reverse
    block walk on the tensor cores, head and batch sums) on the SSD workload
    (bf16, batch 32, L 256, 32 heads, headdim 64, d_state 128), against the bf16
    tensor peak.  Algorithmic FLOPs per 128-step block and head: the nine
    distinct products of the chunked gradient at full precision, 2 (3 Q^2 N +
    2 Q^2 P + 4 Q P N); the kernel's hi/lo splits and its second (transposed)
    Q x Q product are not counted."""
    import torch
    from state_space_model_selective_gb300 import binding, inputs
    Bn, L, H, P, N = 32, 256, 32, 64, 128
    inp = inputs.ssd_inputs(Bn, L, H, P, N, 1, "bf16", seed=1004, device=dev)
    g = torch.Generator(device=dev)
    g.manual_seed(1009)
    dy = torch.randn(Bn, L, H, P, device=dev, generator=g).to(torch.bfloat16)
    f = dict(dtype=torch.float32, device=dev)
    out = {"dx": torch.empty(Bn, L, H, P, **f), "ddt": torch.empty(Bn, L, H, **f),
           "dA_head": torch.empty(H, **f), "dB": torch.empty(Bn, L, 1, N, **f),
           "dC": torch.empty(Bn, L, 1, N, **f), "dinitial_state": torch.empty(Bn, H, P, N, **f)}
    ws = torch.empty(binding.ssd_chunked_bwd_workspace_bytes(Bn, L, H, P, N, 1),
                     dtype=torch.uint8, device=dev)

    def bwd():
        binding.ssd_chunked_bwd(inp["x"], inp["dt"], inp["A_head"], inp["B"], inp["C"], dy, 64,
                                workspace=ws, out=out)
    ms = _time(bwd, reps)
    # a training step's SSD: the forward keeping block states, then the gradient
    # from them (no second forward)
    y = torch.empty(Bn, L, H, P, **f)
    fs = torch.empty(Bn, H, P, N, **f)
    bs = torch.empty(binding.ssd_chunked_checkpoint_bytes(Bn, L, H, P, N) // 4, **f)

    def train():
        binding.ssd_chunked_fwd(inp["x"], inp["dt"], inp["A_head"], inp["B"], inp["C"], 64,
                                out_dtype=torch.float32, y=y, final_state=fs, block_states=bs)
        binding.ssd_chunked_bwd(inp["x"], inp["dt"], inp["A_head"], inp["B"], inp["C"], dy, 64,
                                workspace=ws, out=out, block_states=bs)
    ms_train = _time(train, reps)
    Q = 128
    flops = 2 * (3 * Q * Q * N + 2 * Q * Q * P + 4 * Q * P * N) * Bn * H * (L // Q)
    achieved = flops / (ms / 1e3) / 1e12
    return {"workload": "chunked-SSD gradient bf16 in / fp32 gradients, batch 32, L 256, 32 "
                        "heads, headdim 64, d_state 128, chunk 64",
            "ms": ms, "elements_per_s": Bn * L * H * P * N / (ms / 1e3),
            "train_step_ms": ms_train,
            "train_step": "forward keeping block states + gradient from them",
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": BF16_PEAK_TFLOPS,
                         "unit": "TFLOP/s", "frac": achieved / BF16_PEAK_TFLOPS,
                         "algorithmic_flops": flops}}


def _measure_mamba3_bwd(dev, reps):
    """The Mamba-3 SISO gradient (ssd_mamba3_bwd: the Mamba-3 forward for the block
    states, the SSD gradient with the Mamba-3 input weights, elementwise kernels for
    lambda, the diagonal correction and the previous token) on the SSD workload
    with lambda, an initial state and a previous token, against the bf16 tensor
    peak with the SSD gradient's algorithmic FLOPs (the Mamba-3 extras are
    elementwise)."""
    import torch
    from state_space_model_selective_gb300 import binding, inputs
    Bn, L, H, P, N = 32, 256, 32, 64, 128
    m3 = inputs.mamba3_inputs(Bn, L, H, P, N, 1, "bf16", seed=1006, device=dev)
    g = torch.Generator(device=dev)
    g.manual_seed(1010)
    dy = torch.randn(Bn, L, H, P, device=dev, generator=g).to(torch.bfloat16)
    ws = torch.empty(binding.ssd_mamba3_bwd_workspace_bytes(Bn, L, H, P, N, 1),
                     dtype=torch.uint8, device=dev)

    def bwd():
        binding.ssd_mamba3_bwd(m3["x"], m3["dt"], m3["lam"], m3["A_head"], m3["B"], m3["C"], dy,
                               64, m3["h0"], m3["prev_B"], m3["prev_x"], workspace=ws)
    ms = _time(bwd, reps)
    # a training step: the forward keeping block states, then the gradient from them
    f = dict(dtype=torch.float32, device=dev)
    y = torch.empty(Bn, L, H, P, **f)
    fs = torch.empty(Bn, H, P, N, **f)
    bs = torch.empty(binding.ssd_chunked_checkpoint_bytes(Bn, L, H, P, N) // 4, **f)

    def train():
        binding.ssd_mamba3_fwd(m3["x"], m3["dt"], m3["lam"], m3["A_head"], m3["B"], m3["C"], 64,
                               out_dtype=torch.float32, y=y, final_state=fs,
                               initial_state=m3["h0"], prev_B=m3["prev_B"],
                               prev_x=m3["prev_x"], block_states=bs)
        binding.ssd_mamba3_bwd(m3["x"], m3["dt"], m3["lam"], m3["A_head"], m3["B"], m3["C"], dy,
                               64, m3["h0"], m3["prev_B"], m3["prev_x"], workspace=ws,
                               block_states=bs)
    ms_train = _time(train, reps)
    Q = 128
    flops = 2 * (3 * Q * Q * N + 2 * Q * Q * P + 4 * Q * P * N) * Bn * H * (L // Q)
    achieved = flops / (ms / 1e3) / 1e12
    return {"workload": "Mamba-3 SISO gradient bf16 in / fp32 gradients, batch 32, L 256, "
                        "32 heads, headdim 64, d_state 128, chunk 64, initial state and "
                        "previous token", "ms": ms,
            "elements_per_s": Bn * L * H * P * N / (ms / 1e3),
            "train_step_ms": ms_train,
            "train_step": "forward keeping block states + gradient from them",
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": BF16_PEAK_TFLOPS,
                         "unit": "TFLOP/s", "frac": achieved / BF16_PEAK_TFLOPS,
                         "algorithmic_flops": flops}}


def _measure_mimo_bwd(dev, reps):
    """The Mamba-3 MIMO gradient (ssd_mamba3_mimo_bwd) on the pages' MIMO shape (batch
    32, L 256, rank 4, 32 heads, headdim 64, d_state 128, chunk 16) with an initial
    state and a previous token, against the bf16 tensor peak with the SSD gradient's
    algorithmic FLOPs over the L R sub-tokens."""
    import torch
    from state_space_model_selective_gb300 import binding, inputs
    Bn, L, R, H, P, N = 32, 256, 4, 32, 64, 128
    m = inputs.mamba3_mimo_inputs(Bn, L, R, H, P, N, 1, "bf16", seed=1007, device=dev)
    g = torch.Generator(device=dev)
    g.manual_seed(1011)
    dy = torch.randn(Bn, L, R, H, P, device=dev, generator=g).to(torch.bfloat16)
    ws = torch.empty(binding.ssd_mamba3_mimo_bwd_workspace_bytes(Bn, L, R, H, P, N, 1),
                     dtype=torch.uint8, device=dev)

    def bwd():
        binding.ssd_mamba3_mimo_bwd(m["x"], m["dt"], m["lam"], m["A_head"], m["B"], m["C"], dy,
                                    16, m["h0"], m["prev_B"], m["prev_x"], workspace=ws)
    ms = _time(bwd, reps)
    f = dict(dtype=torch.float32, device=dev)
    y = torch.empty(Bn, L, R, H, P, **f)
    fs = torch.empty(Bn, H, P, N, **f)
    bs = torch.empty(binding.ssd_chunked_checkpoint_bytes(Bn, L * R, H, P, N) // 4, **f)

    def train():
        binding.ssd_mamba3_mimo_fwd(m["x"], m["dt"], m["lam"], m["A_head"], m["B"], m["C"], 16,
                                    out_dtype=torch.float32, y=y, final_state=fs,
                                    initial_state=m["h0"], prev_B=m["prev_B"],
                                    prev_x=m["prev_x"], block_states=bs)
        binding.ssd_mamba3_mimo_bwd(m["x"], m["dt"], m["lam"], m["A_head"], m["B"], m["C"], dy,
                                    16, m["h0"], m["prev_B"], m["prev_x"], workspace=ws,
                                    block_states=bs)
    ms_train = _time(train, reps)
    Q = 128
    flops = 2 * (3 * Q * Q * N + 2 * Q * Q * P + 4 * Q * P * N) * Bn * H * (L * R // Q)
    achieved = flops / (ms / 1e3) / 1e12
    return {"workload": "Mamba-3 MIMO gradient bf16 in / fp32 gradients, batch 32, L 256, "
                        "rank 4, 32 heads, headdim 64, d_state 128, chunk 16, initial state "
                        "and previous token", "ms": ms,
            "elements_per_s": Bn * L * R * H * P * N / (ms / 1e3),
            "train_step_ms": ms_train,
            "train_step": "forward keeping block states + gradient from them",
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": BF16_PEAK_TFLOPS,
                         "unit": "TFLOP/s", "frac": achieved / BF16_PEAK_TFLOPS,
                         "algorithmic_flops": flops}}


def _time_graph(fn, n):
    """Mean device time per call of fn, captured n times in a CUDA graph and
    replayed (the launch overhead of single calls removed)."""
    import torch
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for _ in range(3):
            fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(n):
            fn()
    g.replay()
    torch.cuda.synchronize()
    times = []
    with torch.cuda.stream(s):  # the replay runs on the current stream
        for _ in range(5):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            g.replay()
            e1.record(s)
            e1.synchronize()
            times.append(e0.elapsed_time(e1) / n)
    return statistics.median(times)


def _time(fn, reps):
    import torch
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    s = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for _ in range(reps):
        fn()
    e1.record(s)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


# ------------------------------------------------------------------ reference

def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return None
    from state_space_model_selective_gb300 import inputs
    inp = inputs.scan_inputs(BATCH, DIM, SEQLEN, DSTATE, NGROUPS, "bf16", seed=1002, gate=True,
                             dskip="ones", device="cpu")
    import oracle
    # each step: the oracle over one batch row of the workload (bounded sample)
    sl = slice(0, 1)
    a = (inp["u"][sl], inp["delta"][sl], inp["A"], inp["B"][sl], inp["C"][sl], inp["D"],
         inp["z"][sl], inp["delta_bias"], True)
    oracle.scan(*a)  # one untimed warm-up run (the oracle has no state to warm)
    steps = max(1, min(args.steps, 5))
    t0 = time.perf_counter()
    for _ in range(steps):
        oracle.scan(*a)
    el = time.perf_counter() - t0
    elements = steps * SEQLEN * DIM * DSTATE
    value = elements / el
    sample = (f"{steps} step(s), each the fp64 oracle over batch row 0 of the workload "
              f"(1x{DIM}x{SEQLEN}x{DSTATE} elements)")
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
           "n_gpus": world, "steps": steps, "warmup": args.warmup,
           "ms_per_step": el / steps * 1e3, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": WORKLOAD, "batch": BATCH, "seqlen": SEQLEN, "dim": DIM,
                      "dstate": DSTATE},
           "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0},
           "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(),
                            "kind": "oracle", "sample": sample}}
    print(json.dumps(out), flush=True)
    return out


# ------------------------------------------------------------------ profiling

def _profile_setup(name):
    """One workload as a callable (inputs drawn on the GPU, seeded), the target
    of ncu captures: `python bench.py --profile NAME --reps R`."""
    import torch
    from state_space_model_selective_gb300 import binding, inputs
    dev = torch.device("cuda")
    scans = {"scan": (4, 5120, 16384, "bf16", 1003), "scan_l4096": (4, 5120, 4096, "bf16", 1003),
             "scan_b8": (8, 1536, 2048, "bf16", 1002), "scan_b1_f32": (1, 1536, 128, "f32", 1001),
             # one middle segment of the end-to-end leg: 2560 channels of one batch row,
             # which the sequence-parallel kernel scans
             "scan_segment": (1, 2560, 16384, "bf16", 1003)}
    if name in scans:
        B, D, L, dt, seed = scans[name]
        inp = inputs.scan_inputs(B, D, L, 16, 1, dt, seed=seed, device="cuda")
        y = torch.empty(B, D, L, device=dev)
        fs = torch.empty(B, D, 16, device=dev)
        ws = torch.empty(binding.ssm_scan_workspace_bytes(B, D, L), dtype=torch.uint8, device=dev)

        def fn():
            binding.ssm_scan_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"],
                                 inp["z"], inp["delta_bias"], True, out_dtype=torch.float32,
                                 y=y, final_state=fs, workspace=ws)
        return fn, lambda: binding.ssm_last_device_status(ws) == 0
    if name == "ssd":
        inp = inputs.ssd_inputs(32, 256, 32, 64, 128, 1, "bf16", seed=1004, device="cuda")
        y = torch.empty(inp["x"].shape, device=dev)
        fs = torch.empty(32, 32, 64, 128, device=dev)

        def fn():
            binding.ssd_chunked_fwd(inp["x"], inp["dt"], inp["A_head"], inp["B"], inp["C"], 64,
                                    out_dtype=torch.float32, y=y, final_state=fs)
        return fn, None
    if name == "scan_bwd":
        B, D, L = 8, 1536, 2048
        inp = inputs.scan_inputs(B, D, L, 16, 1, "bf16", seed=1002, device="cuda")
        g = torch.Generator(device=dev)
        g.manual_seed(1008)
        dy = torch.randn(B, D, L, device=dev, generator=g).to(torch.bfloat16)
        ws = torch.empty(binding.ssm_scan_bwd_workspace_bytes(B, D, L), dtype=torch.uint8,
                         device=dev)

        def fn():
            binding.ssm_scan_bwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], dy,
                                 inp["D"], inp["z"], inp["delta_bias"], True, workspace=ws)
        return fn, lambda: binding.ssm_last_device_status(ws) == 0
    if name in ("ssd_bwd", "m3_bwd", "mimo_bwd"):
        g = torch.Generator(device=dev)
        if name == "ssd_bwd":
            inp = inputs.ssd_inputs(32, 256, 32, 64, 128, 1, "bf16", seed=1004, device="cuda")
            g.manual_seed(1009)
            dy = torch.randn(32, 256, 32, 64, device=dev, generator=g).to(torch.bfloat16)
            ws = torch.empty(binding.ssd_chunked_bwd_workspace_bytes(32, 256, 32),
                             dtype=torch.uint8, device=dev)

            def fn():
                binding.ssd_chunked_bwd(inp["x"], inp["dt"], inp["A_head"], inp["B"], inp["C"],
                                        dy, 64, workspace=ws)
        elif name == "m3_bwd":
            m3 = inputs.mamba3_inputs(32, 256, 32, 64, 128, 1, "bf16", seed=1006, device="cuda")
            g.manual_seed(1010)
            dy = torch.randn(32, 256, 32, 64, device=dev, generator=g).to(torch.bfloat16)
            ws = torch.empty(binding.ssd_mamba3_bwd_workspace_bytes(32, 256, 32),
                             dtype=torch.uint8, device=dev)

            def fn():
                binding.ssd_mamba3_bwd(m3["x"], m3["dt"], m3["lam"], m3["A_head"], m3["B"],
                                       m3["C"], dy, 64, m3["h0"], m3["prev_B"], m3["prev_x"],
                                       workspace=ws)
        else:
            m = inputs.mamba3_mimo_inputs(32, 256, 4, 32, 64, 128, 1, "bf16", seed=1007,
                                          device="cuda")
            g.manual_seed(1011)
            dy = torch.randn(32, 256, 4, 32, 64, device=dev, generator=g).to(torch.bfloat16)
            ws = torch.empty(binding.ssd_mamba3_mimo_bwd_workspace_bytes(32, 256, 4, 32),
                             dtype=torch.uint8, device=dev)

            def fn():
                binding.ssd_mamba3_mimo_bwd(m["x"], m["dt"], m["lam"], m["A_head"], m["B"],
                                            m["C"], dy, 16, m["h0"], m["prev_B"], m["prev_x"],
                                            workspace=ws)
        return fn, lambda: binding.ssm_last_device_status(ws) == 0
    if name == "decode_mimo":
        g = torch.Generator(device=dev)
        g.manual_seed(1005)
        B_, H, P, N, R = 256, 32, 64, 128, 4
        state = 0.1 * torch.randn(B_, H, P, N, device=dev, generator=g)
        dt = torch.nn.functional.softplus(torch.randn(B_, H, device=dev, generator=g) - 4)
        lam = torch.sigmoid(torch.randn(B_, H, device=dev, generator=g))
        A = -(1 + 15 * torch.rand(H, device=dev, generator=g))
        D = torch.ones(H, device=dev)
        xr, xpr = (torch.randn(B_, R, H, P, device=dev, generator=g) for _ in range(2))
        Br, Cr, Bpr = (torch.randn(B_, R, 1, N, device=dev, generator=g) for _ in range(3))
        yr = torch.empty_like(xr)

        def fn():
            binding.ssm_decode_step_mamba3_mimo(state, Bpr, xpr, xr, dt, lam, A, Br, Cr, D, y=yr)
        return fn, None
    if name == "decode":
        inp = inputs.decode_inputs(256, 32, 64, 128, 1, 1, "f32", seed=1005, device="cuda")
        state = inp["state"]

        def fn():
            binding.ssm_decode_step(state, inp["x"][0], inp["dt"][0], inp["A"], inp["B"][0],
                                    inp["C"][0], inp["D"])
        return fn, None
    if name == "rope":
        Bn, L, H, P, N = 32, 256, 32, 64, 128
        inp = inputs.ssd_inputs(Bn, L, H, P, N, 1, "bf16", seed=1004, device=dev)
        r = inputs.rope_inputs(Bn, L, H, N, seed=1008, device=dev)
        Br = torch.empty(Bn, L, H, N, dtype=torch.bfloat16, device=dev)
        Cr = torch.empty_like(Br)
        ang = torch.empty(Bn, H, N // 2, device=dev)

        def fn():
            binding.ssm_mamba3_rope(inp["B"], inp["C"], inp["dt"], r["theta"], r["angle0"],
                                    B_rot=Br, C_rot=Cr, angle_out=ang)
        return fn, None
    raise SystemExit(f"unknown workload {name!r}")


PROFILE_WORKLOADS = ["scan", "scan_l4096", "scan_b8", "scan_b1_f32", "scan_segment", "ssd",
                     "decode", "decode_mimo", "scan_bwd", "ssd_bwd", "m3_bwd", "mimo_bwd", "rope"]


def run_profile(name, reps):
    """Runs one workload `reps` times (the process exits non-zero on any error):
    scan: the benchmark step's scan; scan_l4096: the same channels over L 4096;
    scan_b8: batch 8, L 2048, 1536 channels; scan_b1_f32: batch 1, L 128, 1536
    channels, fp32; scan_segment: 2560 channels of one batch row over L 16384 (a
    segment of the end-to-end leg); ssd: chunked SSD batch 32, L 256, 32 heads; decode,
    decode_mimo: decode steps batch 256, 32 heads; scan_bwd, ssd_bwd, m3_bwd,
    mimo_bwd: the gradients on those workloads; rope: Mamba-3's rotation of B
    and C on the SSD workload."""
    import torch
    fn, check = _profile_setup(name)
    for _ in range(reps):
        fn()
    torch.cuda.synchronize()
    if check is not None:
        assert check(), "device-side status not OK"
    print(f"{name}: {reps} runs ok", flush=True)


# ------------------------------------------------------------------ peaks

PEAKS_SRC = os.path.join(ROOT, "bench_peaks.cu")
PEAKS_LIB = os.path.join(ROOT, "_build", "libbench_peaks.so")


def build_peaks(force=False):
    """Compiles bench_peaks.cu (sm_103a) into _build/libbench_peaks.so."""
    if not force and os.path.exists(PEAKS_LIB) and \
            os.path.getmtime(PEAKS_LIB) >= os.path.getmtime(PEAKS_SRC):
        return PEAKS_LIB
    import shutil
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    os.makedirs(os.path.dirname(PEAKS_LIB), exist_ok=True)
    r = subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                        "-lineinfo", "-Xcompiler", "-fPIC", "-shared", "-o", PEAKS_LIB, PEAKS_SRC,
                        "-cudart", "static"], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on bench_peaks.cu:\n{r.stderr}")
    return PEAKS_LIB


def _sm_clock_mhz():
    import torch
    try:
        r = subprocess.run(["nvidia-smi", "--query-gpu=clocks.sm", "--format=csv,noheader,nounits",
                            f"--id={torch.cuda.current_device()}"],
                           capture_output=True, text=True, timeout=10)
        return float(r.stdout.strip().splitlines()[0])
    except Exception:
        return None


def run_peaks(iters=20000, reps=3):
    """Per-clock throughput of the units the scan uses, on this GPU: MUFU ex2,
    fp32 FMA, packed fp32x2 FMA (per SM per clock, the SM clock sampled with
    nvidia-smi after each probe), the scan's per-step arithmetic mixes
    (sub-partition cycles per element), shared-load costs, latencies, and the
    issue-slot sharing of MUFU, FP32 and broadcast loads (cycles per warp-step
    from clock64)."""
    import ctypes
    import torch
    lib = ctypes.CDLL(build_peaks())
    vp, i = ctypes.c_void_p, ctypes.c_int
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    sms = props.multi_processor_count
    out = torch.empty(sms * 8 * 256, device="cuda")
    cyc = torch.empty(sms * 8, dtype=torch.int64, device="cuda")
    st = torch.cuda.current_stream()
    sp, op = vp(st.cuda_stream), vp(out.data_ptr())
    res = {"sms": sms, "gpu": props.name}

    def timed(launch):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        n = launch()
        e1.record(st)
        torch.cuda.synchronize()
        return n, e0.elapsed_time(e1) / 1e3, _sm_clock_mhz()

    lib.ssm_peak_probe.restype = ctypes.c_double
    lib.ssm_peak_probe.argtypes = [i] * 4 + [vp, vp]
    for kind, name, blocks, threads in ((0, "mufu_ex2", sms * 8, 256), (1, "ffma", sms * 8, 256),
                                        (2, "ffma2_lanes", sms * 8, 256),
                                        (0, "mufu_ex2_1warp_per_smsp", sms * 4, 32),
                                        (2, "ffma2_lanes_1warp_per_smsp", sms * 4, 32)):
        best = None
        for _ in range(reps):
            n, sec, mhz = timed(lambda: lib.ssm_peak_probe(kind, blocks, threads, iters, op, sp))
            if n <= 0:
                raise RuntimeError("probe launch failed")
            if best is None or n / sec > best[0]:
                best = (n / sec, mhz)
        rate, mhz = best
        res[name] = {"per_s": rate, "sm_mhz": mhz,
                     "per_sm_per_clk": rate / sms / (mhz * 1e6) if mhz else None}
    # the issue-slot sharing of MUFU, FP32 and broadcast shared loads
    lib.ssm_overlap_probe.restype = i
    lib.ssm_overlap_probe.argtypes = [i, i, i, vp, vp, vp]
    names = ["8x(FMUL+MUFU ex2)", "32 FFMA", "16 FFMA2", "8 broadcast LDS.128",
             "8x(FMUL+MUFU) + 24 FFMA", "8x(FMUL+MUFU) + 12 FFMA2",
             "8x(FMUL+MUFU) + 24 FFMA + 4 LDS.128", "8x(FMUL+MUFU) + 12 FFMA2 + 8 LDS.128"]
    ov = {}
    for wps in (2, 4):
        for which, nm in enumerate(names):
            it = 2000
            lib.ssm_overlap_probe(which, sms * wps, 10, op, vp(cyc.data_ptr()), sp)
            if not lib.ssm_overlap_probe(which, sms * wps, it, op, vp(cyc.data_ptr()), sp):
                raise RuntimeError("overlap probe launch failed")
            torch.cuda.synchronize()
            mx = int(cyc[:sms * wps].max().item())
            ov[f"{nm} @ {wps} warps/SMSP"] = mx / (it * 8 * wps)  # cycles per warp-step
    res["issue_sharing_cycles_per_warp_step"] = ov
    # the scan's per-step arithmetic from registers (ns states per thread;
    # scalar, and scalar vs packed fp32x2): sub-partition cycles per element
    lib.ssm_scan_mix_probe.restype = ctypes.c_double
    lib.ssm_scan_mix_probe.argtypes = [i] * 4 + [vp, vp]
    lib.ssm_scan_mix2_probe.restype = ctypes.c_double
    lib.ssm_scan_mix2_probe.argtypes = [i] * 5 + [vp, vp]
    mix, mix2 = {}, {}
    for ns in (4, 8, 16):
        for wps in (1, 2, 3, 4):
            steps = 4000
            lib.ssm_scan_mix_probe(ns, sms * 4 * wps, 32, 100, op, sp)
            _, sec, mhz = timed(lambda: lib.ssm_scan_mix_probe(ns, sms * 4 * wps, 32, steps, op, sp))
            mix[f"ns{ns}_{wps}warp_per_smsp"] = sec * (mhz or SM_MAX_MHZ) * 1e6 / steps / (wps * 32 * ns)
        for packed in (0, 1):
            for wps in (1, 2, 4):
                steps = 4000
                lib.ssm_scan_mix2_probe(ns, packed, sms * 4 * wps, 32, 100, op, sp)
                _, sec, mhz = timed(lambda: lib.ssm_scan_mix2_probe(ns, packed, sms * 4 * wps, 32,
                                                                    steps, op, sp))
                mix2[f"{'x2' if packed else 'f32'}_ns{ns}_{wps}warp_per_smsp"] = \
                    sec * (mhz or SM_MAX_MHZ) * 1e6 / steps / (wps * 32 * ns)
    res["scan_step_mix_cycles_per_element"] = mix
    res["scan_full_mix_cycles_per_element"] = mix2
    # shared-memory load cost by width and address pattern: SM clocks per
    # warp-wide load instruction (1 = one 128-byte wavefront per clock)
    lib.ssm_lds_probe.restype = ctypes.c_double
    lib.ssm_lds_probe.argtypes = [i] * 5 + [vp, vp]
    lds = {}
    pat = {0: "same_addr", 1: "4addr_lane_mod4", 2: "4addr_per_quarter", 3: "32addr"}
    for width in (4, 8, 16):
        for pattern in (0, 1, 2, 3):
            its = 4000
            lib.ssm_lds_probe(width, pattern, sms * 4, 512, 50, op, sp)
            n, sec, mhz = timed(lambda: lib.ssm_lds_probe(width, pattern, sms * 4, 512, its, op, sp))
            lds[f"lds{width * 8}_{pat[pattern]}"] = sec * (mhz or SM_MAX_MHZ) * 1e6 * sms / n
    res["lds_clocks_per_warp_load"] = lds
    lib.ssm_latency_probe.restype = ctypes.c_float
    lib.ssm_latency_probe.argtypes = [i, i, vp, vp]
    lat = {}
    for kind, name in ((0, "ex2"), (1, "rcp"), (2, "ffma"), (3, "ffma2"), (4, "lds")):
        lib.ssm_latency_probe(kind, 64, op, sp)
        lat[name] = lib.ssm_latency_probe(kind, 2000, op, sp)
    res["latency_cycles"] = lat
    return res


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--profile", choices=PROFILE_WORKLOADS, default=None)
    p.add_argument("--reps", type=int, default=3)
    p.add_argument("--peaks", action="store_true")
    args = p.parse_args(argv)
    if args.profile:
        return run_profile(args.profile, args.reps)
    if args.peaks:
        import torch
        torch.cuda.init()
        print(json.dumps(run_peaks()), flush=True)
        return None
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    main()
