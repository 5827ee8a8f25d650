"""Run one workload a few times on the GPU (the target of ncu captures).

    python -m state_space_model_selective_gb300.profile_run scan   [--reps 5]
    python -m state_space_model_selective_gb300.profile_run ssd    [--reps 5]
    python -m state_space_model_selective_gb300.profile_run decode [--reps 5]
    python -m state_space_model_selective_gb300.profile_run scan_bwd [--reps 5]
    python -m state_space_model_selective_gb300.profile_run ssd_bwd [--reps 5]
    python -m state_space_model_selective_gb300.profile_run decode_mimo [--reps 5]
    python -m state_space_model_selective_gb300.profile_run m3_bwd [--reps 5]
    python -m state_space_model_selective_gb300.profile_run mimo_bwd [--reps 5]

scan:     selective scan, bf16 in / fp32 y, batch 8, L 2048, D 1536, N 16
ssd:      chunked SSD, bf16 in / fp32 y, batch 32, L 256, 32 heads, headdim 64, N 128
decode:   decode step, fp32, batch 256, 32 heads, headdim 64, N 128
scan_bwd: the scan's gradient on the scan workload (D, gate, bias, softplus)
ssd_bwd:  the chunked SSD's gradient on the SSD workload
decode_mimo: Mamba-3 MIMO rank-4 decode step, fp32, batch 256, 32 heads, headdim 64, N 128
m3_bwd:   Mamba-3 SISO gradient on the SSD workload (initial state, previous token)
mimo_bwd: Mamba-3 MIMO rank-4 gradient, batch 32, L 256, 32 heads, headdim 64, N 128, chunk 16
Inputs are drawn on the GPU (seeded); the process exits non-zero on any error.
"""
from __future__ import annotations

import argparse

import torch

from . import binding, inputs


def main(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("workload",
                   choices=["scan", "ssd", "decode", "scan_bwd", "ssd_bwd", "decode_mimo",
                            "m3_bwd", "mimo_bwd"])
    p.add_argument("--reps", type=int, default=5)
    a = p.parse_args(argv)
    dev = torch.device("cuda")
    if a.workload == "scan":
        B, D, L = 8, 1536, 2048
        inp = inputs.scan_inputs(B, D, L, 16, 1, "bf16", seed=1002, device="cuda")
        y = torch.empty(B, D, L, device=dev)
        fs = torch.empty(B, D, 16, device=dev)
        ws = torch.empty(binding.ssm_scan_workspace_bytes(B, D, L), dtype=torch.uint8, device=dev)
        for _ in range(a.reps):
            binding.ssm_scan_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"],
                                 inp["z"], inp["delta_bias"], True, out_dtype=torch.float32,
                                 y=y, final_state=fs, workspace=ws)
        torch.cuda.synchronize()
        assert binding.ssm_last_device_status(ws) == 0
    elif a.workload == "ssd":
        inp = inputs.ssd_inputs(32, 256, 32, 64, 128, 1, "bf16", seed=1004, device="cuda")
        y = torch.empty(inp["x"].shape, device=dev)
        fs = torch.empty(32, 32, 64, 128, device=dev)
        for _ in range(a.reps):
            binding.ssd_chunked_fwd(inp["x"], inp["dt"], inp["A_head"], inp["B"], inp["C"], 64,
                                    out_dtype=torch.float32, y=y, final_state=fs)
        torch.cuda.synchronize()
    elif a.workload == "scan_bwd":
        B, D, L = 8, 1536, 2048
        inp = inputs.scan_inputs(B, D, L, 16, 1, "bf16", seed=1002, device="cuda")
        g = torch.Generator(device=dev)
        g.manual_seed(1008)
        dy = torch.randn(B, D, L, device=dev, generator=g).to(torch.bfloat16)
        ws = torch.empty(binding.ssm_scan_bwd_workspace_bytes(B, D, L), dtype=torch.uint8,
                         device=dev)
        for _ in range(a.reps):
            binding.ssm_scan_bwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], dy,
                                 inp["D"], inp["z"], inp["delta_bias"], True, workspace=ws)
        torch.cuda.synchronize()
        assert binding.ssm_last_device_status(ws) == 0
    elif a.workload == "ssd_bwd":
        inp = inputs.ssd_inputs(32, 256, 32, 64, 128, 1, "bf16", seed=1004, device="cuda")
        g = torch.Generator(device=dev)
        g.manual_seed(1009)
        dy = torch.randn(32, 256, 32, 64, device=dev, generator=g).to(torch.bfloat16)
        ws = torch.empty(binding.ssd_chunked_bwd_workspace_bytes(32, 256, 32), dtype=torch.uint8,
                         device=dev)
        for _ in range(a.reps):
            binding.ssd_chunked_bwd(inp["x"], inp["dt"], inp["A_head"], inp["B"], inp["C"], dy,
                                    64, workspace=ws)
        torch.cuda.synchronize()
        assert binding.ssm_last_device_status(ws) == 0
    elif a.workload == "m3_bwd":
        m3 = inputs.mamba3_inputs(32, 256, 32, 64, 128, 1, "bf16", seed=1006, device="cuda")
        g = torch.Generator(device=dev)
        g.manual_seed(1010)
        dy = torch.randn(32, 256, 32, 64, device=dev, generator=g).to(torch.bfloat16)
        ws = torch.empty(binding.ssd_mamba3_bwd_workspace_bytes(32, 256, 32), dtype=torch.uint8,
                         device=dev)
        for _ in range(a.reps):
            binding.ssd_mamba3_bwd(m3["x"], m3["dt"], m3["lam"], m3["A_head"], m3["B"], m3["C"],
                                   dy, 64, m3["h0"], m3["prev_B"], m3["prev_x"], workspace=ws)
        torch.cuda.synchronize()
        assert binding.ssm_last_device_status(ws) == 0
    elif a.workload == "mimo_bwd":
        m = inputs.mamba3_mimo_inputs(32, 256, 4, 32, 64, 128, 1, "bf16", seed=1007,
                                      device="cuda")
        g = torch.Generator(device=dev)
        g.manual_seed(1011)
        dy = torch.randn(32, 256, 4, 32, 64, device=dev, generator=g).to(torch.bfloat16)
        ws = torch.empty(binding.ssd_mamba3_mimo_bwd_workspace_bytes(32, 256, 4, 32),
                         dtype=torch.uint8, device=dev)
        for _ in range(a.reps):
            binding.ssd_mamba3_mimo_bwd(m["x"], m["dt"], m["lam"], m["A_head"], m["B"], m["C"],
                                        dy, 16, m["h0"], m["prev_B"], m["prev_x"], workspace=ws)
        torch.cuda.synchronize()
        assert binding.ssm_last_device_status(ws) == 0
    elif a.workload == "decode_mimo":
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
        for _ in range(a.reps):
            binding.ssm_decode_step_mamba3_mimo(state, Bpr, xpr, xr, dt, lam, A, Br, Cr, D, y=yr)
        torch.cuda.synchronize()
    else:
        inp = inputs.decode_inputs(256, 32, 64, 128, 1, 1, "f32", seed=1005, device="cuda")
        state = inp["state"]
        for _ in range(a.reps):
            binding.ssm_decode_step(state, inp["x"][0], inp["dt"][0], inp["A"], inp["B"][0],
                                    inp["C"][0], inp["D"])
        torch.cuda.synchronize()
    print(f"{a.workload}: {a.reps} runs ok")


if __name__ == "__main__":
    main()
