"""Seeded synthetic inputs shaped like the pages' workloads.

This module holds no arithmetic of the method itself: it only draws random
numbers and shapes them into the distributions the workloads name.  Both the
CUDA path and the fp64 oracle consume exactly the tensors returned here
(bf16 values are upcast exactly by the oracle).

Recipes (fixed draw order, one ``torch.Generator`` per call):

* selective scan (``scan_inputs``): u, z ~ N(0, 1); raw delta = 0.5 N(0, 1);
  per-channel dt0 = exp(U[ln 1e-3, ln 1e-1]) and delta_bias = inv_softplus(dt0)
  = log(expm1(dt0)), so the kernel's softplus(delta + bias) has the stated
  distribution; A[d, n] = -(n + 1); B, C ~ N(0, 1) of shape (B, G, N, L)
  shared by the channels of a group; D = 1.
* chunked SSD (``ssd_inputs``): x, B, C ~ N(0, 1); dt = softplus(N(0, 1) - 4);
  A_head = -U[1, 16].
* decode (``decode_inputs``): state ~ N(0, 0.1) (standard deviation 0.1);
  per step x, B, C ~ N(0, 1), dt = softplus(N(0, 1) - 4); A_head = -U[1, 16];
  D = 1, no gate unless asked for.

Tensors are created on the CPU by default so that the same seed gives the
same values on any machine; pass ``device="cuda"`` to draw large workloads
directly on the GPU with a CUDA generator (used by the benchmark, whose
inputs need not match any stored value).
"""
from __future__ import annotations

import math

import torch

_DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


def torch_dtype(name: str) -> torch.dtype:
    return _DTYPES[name]


def _gen(seed: int, device: str) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _randn(shape, g, device):
    return torch.randn(*shape, generator=g, device=device, dtype=torch.float32)


def _rand(shape, g, device):
    return torch.rand(*shape, generator=g, device=device, dtype=torch.float32)


def scan_inputs(batch: int, dim: int, seqlen: int, dstate: int = 16, ngroups: int = 1,
                dtype: str = "bf16", seed: int = 1002, gate: bool = True,
                dskip: str = "ones", device: str = "cpu") -> dict:
    """Inputs of the selective scan in the layouts the C ABI takes.

    u, delta, z: (batch, dim, seqlen); A: (dim, dstate) fp32;
    B, C: (batch, ngroups, dstate, seqlen); D, delta_bias: (dim,) fp32.
    ``dskip`` is "ones" (the workloads' D = 1), "randn" or "none".
    """
    g = _gen(seed, device)
    td = _DTYPES[dtype]
    u = _randn((batch, dim, seqlen), g, device)
    delta = 0.5 * _randn((batch, dim, seqlen), g, device)
    z = _randn((batch, dim, seqlen), g, device)
    Bm = _randn((batch, ngroups, dstate, seqlen), g, device)
    Cm = _randn((batch, ngroups, dstate, seqlen), g, device)
    lo, hi = math.log(1e-3), math.log(1e-1)
    dt0 = torch.exp(lo + (hi - lo) * _rand((dim,), g, device))
    delta_bias = torch.log(torch.expm1(dt0))
    A = -torch.arange(1, dstate + 1, dtype=torch.float32, device=device).repeat(dim, 1)
    if dskip == "ones":
        D = torch.ones(dim, dtype=torch.float32, device=device)
    elif dskip == "randn":
        D = _randn((dim,), g, device)
    else:
        D = None
    return {
        "u": u.to(td).contiguous(),
        "delta": delta.to(td).contiguous(),
        "A": A.contiguous(),
        "B": Bm.to(td).contiguous(),
        "C": Cm.to(td).contiguous(),
        "D": D,
        "z": z.to(td).contiguous() if gate else None,
        "delta_bias": delta_bias.contiguous(),
        "delta_softplus": True,
    }


def ssd_inputs(batch: int, seqlen: int, nheads: int, headdim: int, dstate: int,
               ngroups: int = 1, dtype: str = "bf16", seed: int = 1004,
               device: str = "cpu") -> dict:
    """Inputs of the chunked SSD: x (B, L, H, P); dt (B, L, H) fp32;
    A_head (H,) fp32; B, C (B, L, G, N)."""
    g = _gen(seed, device)
    td = _DTYPES[dtype]
    x = _randn((batch, seqlen, nheads, headdim), g, device)
    Bm = _randn((batch, seqlen, ngroups, dstate), g, device)
    Cm = _randn((batch, seqlen, ngroups, dstate), g, device)
    dt = torch.nn.functional.softplus(_randn((batch, seqlen, nheads), g, device) - 4.0)
    A_head = -(1.0 + 15.0 * _rand((nheads,), g, device))
    return {
        "x": x.to(td).contiguous(),
        "dt": dt.contiguous(),
        "A_head": A_head.contiguous(),
        "B": Bm.to(td).contiguous(),
        "C": Cm.to(td).contiguous(),
    }


def mamba3_inputs(batch: int, seqlen: int, nheads: int, headdim: int, dstate: int,
                  ngroups: int = 1, dtype: str = "bf16", seed: int = 1006,
                  device: str = "cpu") -> dict:
    """Inputs of the Mamba-3 SISO prefill: those of ``ssd_inputs`` (drawn first,
    from the same seed) plus lam (B, L, H) fp32 = sigmoid(N(0, 1)); the token
    before the first, prev_B (B, G, N) and prev_x (B, H, P); and an initial
    state h0 (B, H, P, N) fp32 ~ 0.1 N(0, 1)."""
    out = ssd_inputs(batch, seqlen, nheads, headdim, dstate, ngroups, dtype, seed, device)
    g = _gen(seed + 7919, device)
    td = _DTYPES[dtype]
    out["lam"] = torch.sigmoid(_randn((batch, seqlen, nheads), g, device)).contiguous()
    out["prev_B"] = _randn((batch, ngroups, dstate), g, device).to(td).contiguous()
    out["prev_x"] = _randn((batch, nheads, headdim), g, device).to(td).contiguous()
    out["h0"] = (0.1 * _randn((batch, nheads, headdim, dstate), g, device)).contiguous()
    return out


def mamba3_mimo_inputs(batch: int, seqlen: int, rank: int, nheads: int, headdim: int,
                       dstate: int, ngroups: int = 1, dtype: str = "bf16", seed: int = 1007,
                       device: str = "cpu") -> dict:
    """Inputs of the Mamba-3 MIMO prefill, rank inside the time position:
    x (B, L, R, H, P), B, C (B, L, R, G, N) ~ N(0, 1) in dtype; dt (B, L, H) =
    softplus(N(0, 1) - 4); lam (B, L, H) = sigmoid(N(0, 1)); A_head (H,) =
    -U[1, 16]; the token before the first, prev_B (B, R, G, N) and prev_x
    (B, R, H, P); an initial state h0 (B, H, P, N) ~ 0.1 N(0, 1)."""
    g = _gen(seed, device)
    td = _DTYPES[dtype]
    x = _randn((batch, seqlen, rank, nheads, headdim), g, device)
    Bm = _randn((batch, seqlen, rank, ngroups, dstate), g, device)
    Cm = _randn((batch, seqlen, rank, ngroups, dstate), g, device)
    dt = torch.nn.functional.softplus(_randn((batch, seqlen, nheads), g, device) - 4.0)
    lam = torch.sigmoid(_randn((batch, seqlen, nheads), g, device))
    A_head = -(1.0 + 15.0 * _rand((nheads,), g, device))
    prev_B = _randn((batch, rank, ngroups, dstate), g, device)
    prev_x = _randn((batch, rank, nheads, headdim), g, device)
    h0 = 0.1 * _randn((batch, nheads, headdim, dstate), g, device)
    return {"x": x.to(td).contiguous(), "dt": dt.contiguous(), "lam": lam.contiguous(),
            "A_head": A_head.contiguous(), "B": Bm.to(td).contiguous(),
            "C": Cm.to(td).contiguous(), "prev_B": prev_B.to(td).contiguous(),
            "prev_x": prev_x.to(td).contiguous(), "h0": h0.contiguous()}


def decode_inputs(batch: int, nheads: int, headdim: int, dstate: int, ngroups: int = 1,
                  steps: int = 1, dtype: str = "f32", seed: int = 1005,
                  gate: bool = False, dskip: str = "ones", device: str = "cpu") -> dict:
    """Inputs of ``steps`` chained decode steps.

    state (B, H, P, N) fp32; per step t: x[t], z[t] (B, H, P); dt[t] (B, H) fp32;
    B[t], C[t] (B, G, N); A_head, D (H,) fp32.
    """
    g = _gen(seed, device)
    td = _DTYPES[dtype]
    state = 0.1 * _randn((batch, nheads, headdim, dstate), g, device)
    A_head = -(1.0 + 15.0 * _rand((nheads,), g, device))
    if dskip == "ones":
        D = torch.ones(nheads, dtype=torch.float32, device=device)
    elif dskip == "randn":
        D = _randn((nheads,), g, device)
    else:
        D = None
    xs, dts, Bs, Cs, zs = [], [], [], [], []
    for _ in range(steps):
        xs.append(_randn((batch, nheads, headdim), g, device).to(td))
        Bs.append(_randn((batch, ngroups, dstate), g, device).to(td))
        Cs.append(_randn((batch, ngroups, dstate), g, device).to(td))
        dts.append(torch.nn.functional.softplus(_randn((batch, nheads), g, device) - 4.0))
        zs.append(_randn((batch, nheads, headdim), g, device).to(td) if gate else None)
    return {"state": state.contiguous(), "A": A_head.contiguous(), "D": D,
            "x": xs, "dt": dts, "B": Bs, "C": Cs, "z": zs}


def rope_inputs(batch: int, seqlen: int, nheads: int, dstate: int, seed: int = 1008,
                device: str = "cpu") -> dict:
    """Inputs of Mamba-3's data-dependent rotation (no page gives their
    distribution): theta (B, L, H, N/2) fp32 ~ N(0, 1), one angular rate per
    head and state pair, and a starting angle angle0 (B, H, N/2) fp32 ~
    U[-pi, pi)."""
    g = _gen(seed, device)
    theta = _randn((batch, seqlen, nheads, dstate // 2), g, device).contiguous()
    angle0 = ((_rand((batch, nheads, dstate // 2), g, device) * 2.0 - 1.0) * 3.141592653589793)
    return {"theta": theta, "angle0": angle0.contiguous()}
