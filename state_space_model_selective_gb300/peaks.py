"""Measure the per-clock throughput of the units the selective scan uses:
MUFU ex2, fp32 FMA and packed fp32x2 FMA, on the current GPU.

Prints one JSON line with results per second and per SM per clock (the SM
clock is sampled with nvidia-smi during each probe).  These rates, times the
SM count and the maximum SM clock, are the scan's arithmetic roofline.
"""
from __future__ import annotations

import ctypes
import json
import os
import subprocess

import torch

_LIB = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libssm_peaks.so")


def _sm_clock_mhz():
    try:
        r = subprocess.run(["nvidia-smi", "--query-gpu=clocks.sm", "--format=csv,noheader,nounits",
                            f"--id={torch.cuda.current_device()}"],
                           capture_output=True, text=True, timeout=10)
        return float(r.stdout.strip().splitlines()[0])
    except Exception:
        return None


def measure(iters: int = 20000, reps: int = 3) -> dict:
    lib = ctypes.CDLL(_LIB)
    lib.ssm_peak_probe.restype = ctypes.c_double
    lib.ssm_peak_probe.argtypes = [ctypes.c_int] * 4 + [ctypes.c_void_p, ctypes.c_void_p]
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    sms = props.multi_processor_count
    blocks, threads = sms * 8, 256
    out = torch.empty(blocks * threads, device="cuda")
    stream = torch.cuda.current_stream()
    res = {"sms": sms, "gpu": props.name}
    for kind, name in ((0, "mufu_ex2"), (1, "ffma"), (2, "ffma2_lanes")):
        best = None
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            n = lib.ssm_peak_probe(kind, blocks, threads, iters, ctypes.c_void_p(out.data_ptr()),
                                   ctypes.c_void_p(stream.cuda_stream))
            e1.record(stream)
            torch.cuda.synchronize()
            mhz = _sm_clock_mhz()
            ms = e0.elapsed_time(e1)
            if n <= 0:
                raise RuntimeError("probe launch failed")
            rate = n / (ms / 1e3)
            if best is None or rate > best[0]:
                best = (rate, mhz)
        rate, mhz = best
        res[name] = {"per_s": rate, "sm_mhz": mhz,
                     "per_sm_per_clk": rate / sms / (mhz * 1e6) if mhz else None}
    # the same probes with one warp per SM sub-partition (4 per SM)
    for kind, name in ((0, "mufu_ex2_1warp_per_smsp"), (2, "ffma2_lanes_1warp_per_smsp")):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        n = lib.ssm_peak_probe(kind, sms * 4, 32, iters, ctypes.c_void_p(out.data_ptr()),
                               ctypes.c_void_p(stream.cuda_stream))
        e1.record(stream)
        torch.cuda.synchronize()
        mhz = _sm_clock_mhz()
        rate = n / (e0.elapsed_time(e1) / 1e3)
        res[name] = {"per_s": rate, "sm_mhz": mhz,
                     "per_sm_per_clk": rate / sms / (mhz * 1e6) if mhz else None}
    # the scan's per-step arithmetic (ns states per thread, scalar fp32):
    # SM-sub-partition cycles per element with 1..4 warps per sub-partition
    lib.ssm_scan_mix_probe.restype = ctypes.c_double
    lib.ssm_scan_mix_probe.argtypes = [ctypes.c_int] * 4 + [ctypes.c_void_p, ctypes.c_void_p]
    mix = {}
    for ns in (4, 8, 16):
        for wps in (1, 2, 3, 4):
            steps = 4000
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            lib.ssm_scan_mix_probe(ns, sms * 4 * wps, 32, 100, ctypes.c_void_p(out.data_ptr()),
                                   ctypes.c_void_p(stream.cuda_stream))
            e0.record(stream)
            lib.ssm_scan_mix_probe(ns, sms * 4 * wps, 32, steps,
                                   ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(stream.cuda_stream))
            e1.record(stream)
            torch.cuda.synchronize()
            mhz = _sm_clock_mhz() or 2070.0
            cyc = e0.elapsed_time(e1) / 1e3 * mhz * 1e6 / steps
            mix[f"ns{ns}_{wps}warp_per_smsp"] = cyc / (wps * 32 * ns)  # cycles per element
    res["scan_step_mix"] = mix
    # full per-element arithmetic, scalar vs packed fp32x2 (cycles per element
    # per sub-partition; 4 MUFU cycles per 32 elements = 0.125)
    lib.ssm_scan_mix2_probe.restype = ctypes.c_double
    lib.ssm_scan_mix2_probe.argtypes = [ctypes.c_int] * 5 + [ctypes.c_void_p, ctypes.c_void_p]
    mix2 = {}
    for packed in (0, 1):
        for ns in (4, 8, 16):
            for wps in (1, 2, 4):
                steps = 4000
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                lib.ssm_scan_mix2_probe(ns, packed, sms * 4 * wps, 32, 100,
                                        ctypes.c_void_p(out.data_ptr()),
                                        ctypes.c_void_p(stream.cuda_stream))
                e0.record(stream)
                lib.ssm_scan_mix2_probe(ns, packed, sms * 4 * wps, 32, steps,
                                        ctypes.c_void_p(out.data_ptr()),
                                        ctypes.c_void_p(stream.cuda_stream))
                e1.record(stream)
                torch.cuda.synchronize()
                mhz = _sm_clock_mhz() or 2070.0
                cyc = e0.elapsed_time(e1) / 1e3 * mhz * 1e6 / steps
                mix2[f"{'x2' if packed else 'f32'}_ns{ns}_{wps}warp_per_smsp"] = cyc / (wps * 32 * ns)
    res["scan_full_mix"] = mix2
    # shared-memory load cost by width and address pattern: SM clocks per
    # warp-wide load instruction (1 = one 128-byte wavefront per clock)
    lib.ssm_lds_probe.restype = ctypes.c_double
    lib.ssm_lds_probe.argtypes = [ctypes.c_int] * 5 + [ctypes.c_void_p, ctypes.c_void_p]
    lds = {}
    names = {0: "same_addr", 1: "4addr_lane_mod4", 2: "4addr_per_quarter", 3: "32addr"}
    for width in (4, 8, 16):
        for pattern in (0, 1, 2, 3):
            its = 4000
            lib.ssm_lds_probe(width, pattern, sms * 4, 512, 50, ctypes.c_void_p(out.data_ptr()),
                              ctypes.c_void_p(stream.cuda_stream))
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            n = lib.ssm_lds_probe(width, pattern, sms * 4, 512, its,
                                  ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(stream.cuda_stream))
            e1.record(stream)
            torch.cuda.synchronize()
            mhz = _sm_clock_mhz() or 2070.0
            clocks = e0.elapsed_time(e1) / 1e3 * mhz * 1e6
            lds[f"lds{width * 8}_{names[pattern]}"] = clocks * sms / n
    res["lds_clocks_per_warp_load"] = lds
    lib.ssm_latency_probe.restype = ctypes.c_float
    lib.ssm_latency_probe.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    lat = {}
    for kind, name in ((0, "ex2"), (1, "rcp"), (2, "ffma"), (3, "ffma2"), (4, "lds")):
        lib.ssm_latency_probe(kind, 64, ctypes.c_void_p(out.data_ptr()),
                              ctypes.c_void_p(stream.cuda_stream))
        lat[name] = lib.ssm_latency_probe(kind, 2000, ctypes.c_void_p(out.data_ptr()),
                                          ctypes.c_void_p(stream.cuda_stream))
    res["latency_cycles"] = lat
    return res


if __name__ == "__main__":
    torch.cuda.init()
    print(json.dumps(measure()))
