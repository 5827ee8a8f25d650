"""Mamba-3's data-dependent rotation of B and C (ssm_mamba3_rope) through the
C ABI, against the fp64 oracle ("Mamba-3 NKI Kernels for AWS Neuron", section
"How it works", Phase 1): alone, then feeding the SISO and MIMO prefills and
128 chained decode steps, each compared with the oracle's rotation followed by
its recurrence."""
import numpy as np
import pytest
import torch

import oracle
from state_space_model_selective_gb300 import binding, inputs
from tests.helpers import TOL_BF16, TOL_F32, assert_close, to64

pytestmark = pytest.mark.gpu

BF16_ULP = 2.0 ** -7  # spacing of bf16 values in [1, 2)


def _bf16_round(a):
    """fp64 values rounded to bf16 and back (torch's round-to-nearest-even)."""
    return torch.from_numpy(np.ascontiguousarray(a)).to(torch.float32).to(torch.bfloat16)


CASES = [  # batch, seqlen, rank, nheads, ngroups, dstate, dtype, with angle0
    (2, 100, 1, 4, 2, 128, "f32", True),
    (1, 256, 1, 8, 1, 128, "bf16", False),
    (2, 33, 4, 4, 4, 128, "bf16", True),
    (3, 17, 2, 6, 3, 16, "f32", False),
    (2, 700, 1, 2, 1, 6, "bf16", True),   # 3 pairs: scalar loads, a 512-step tile + tail
    (1, 75, 1, 2, 1, 160, "f32", True),   # 80 pairs: two CTAs per head, the second partial
    (1, 1, 3, 2, 2, 128, "bf16", True),   # one step (a decode step's rotation), rank 3
]


@pytest.mark.parametrize("case", CASES, ids=[f"B{c[0]}L{c[1]}R{c[2]}H{c[3]}G{c[4]}N{c[5]}{c[6]}"
                                             for c in CASES])
def test_rope_matches_oracle(case):
    batch, seqlen, rank, nheads, ngroups, dstate, dt_name, with_a0 = case
    td = inputs.torch_dtype(dt_name)
    g = torch.Generator().manual_seed(seqlen + rank)
    shape = (batch, seqlen, ngroups, dstate) if rank == 1 else (batch, seqlen, rank, ngroups, dstate)
    B = torch.randn(*shape, generator=g).to(td)
    C = torch.randn(*shape, generator=g).to(td)
    dt = torch.nn.functional.softplus(torch.randn(batch, seqlen, nheads, generator=g) - 4)
    r = inputs.rope_inputs(batch, seqlen, nheads, dstate, seed=50 + seqlen)
    a0 = r["angle0"] if with_a0 else None
    Br, Cr, ang = binding.ssm_mamba3_rope(B.cuda(), C.cuda(), dt.cuda(), r["theta"].cuda(),
                                          None if a0 is None else a0.cuda())
    torch.cuda.synchronize()
    Br_ref, Cr_ref, ang_ref = oracle.mamba3_rope(B, C, dt, r["theta"], a0)
    if dt_name == "f32":
        assert_close(Br, Br_ref, TOL_F32, "B_rot")
        assert_close(Cr, Cr_ref, TOL_F32, "C_rot")
    else:
        # the fp32 rotation rounded to bf16: within one bf16 step, at the
        # scale of the rotated pair's norm, of the correctly rounded fp64
        # value (an output near zero comes from cancellation, so its own ulp
        # is not the scale of the error)
        for got, ref, name in ((Br, Br_ref, "B_rot"), (Cr, Cr_ref, "C_rot")):
            r16 = to64(_bf16_round(ref))
            diff = np.abs(to64(got) - r16)
            norm = np.sqrt(ref[..., 0::2] ** 2 + ref[..., 1::2] ** 2).repeat(2, axis=-1)
            ulp = BF16_ULP * np.exp2(np.floor(np.log2(np.maximum(norm, 1e-30))))
            assert np.all(diff <= ulp * 1.0001), (name, float(np.max(diff / ulp)))
            assert_close(got, ref, 2.0 ** -8, name)
    np.testing.assert_allclose(to64(ang), ang_ref, rtol=2e-6, atol=2e-6)


def test_rope_empty_sequence_hands_the_angle_on():
    """seqlen 0: no rows to rotate; the final angle is the initial one."""
    r = inputs.rope_inputs(2, 1, 3, 16, seed=5, device="cuda")
    B = torch.zeros(2, 0, 1, 16, device="cuda")
    dt = torch.zeros(2, 0, 3, device="cuda")
    th = torch.zeros(2, 0, 3, 8, device="cuda")
    Br, Cr, ang = binding.ssm_mamba3_rope(B, B.clone(), dt, th, r["angle0"])
    torch.cuda.synchronize()
    assert Br.shape == (2, 0, 3, 16) and Cr.shape == (2, 0, 3, 16)
    assert torch.equal(ang, r["angle0"])


def test_rope_resumes_in_place():
    """Three calls over consecutive pieces, the angle updated in place,
    give the bits of one call over the whole sequence."""
    batch, seqlen, nheads, ngroups, dstate = 2, 90, 4, 2, 64
    g = torch.Generator().manual_seed(7)
    B = torch.randn(batch, seqlen, ngroups, dstate, generator=g).cuda()
    C = torch.randn(batch, seqlen, ngroups, dstate, generator=g).cuda()
    dt = torch.nn.functional.softplus(torch.randn(batch, seqlen, nheads, generator=g) - 4).cuda()
    r = inputs.rope_inputs(batch, seqlen, nheads, dstate, seed=77, device="cuda")
    Bw, Cw, aw = binding.ssm_mamba3_rope(B, C, dt, r["theta"], r["angle0"])
    ang = r["angle0"].clone()
    pieces = []
    for a, b in ((0, 30), (30, 31), (31, 90)):
        Bp, Cp, _ = binding.ssm_mamba3_rope(B[:, a:b].contiguous(), C[:, a:b].contiguous(),
                                            dt[:, a:b].contiguous(),
                                            r["theta"][:, a:b].contiguous(), ang, angle_out=ang)
        pieces.append((Bp, Cp))
    torch.cuda.synchronize()
    # the angle carried between calls is rounded once per call; the pieces
    # agree with the whole to that rounding
    assert_close(torch.cat([p[0] for p in pieces], 1), Bw, 1e-6, "B_rot")
    assert_close(torch.cat([p[1] for p in pieces], 1), Cw, 1e-6, "C_rot")
    assert_close(ang, aw, 1e-6, "angle")


@pytest.mark.parametrize("rank", [1, 4])
def test_mamba3_prefill_with_rope_matches_oracle(rank):
    """bf16 prefill: B and C rotated on the GPU (bf16 out, one row per head)
    feeding ssd_mamba3_fwd / ssd_mamba3_mimo_fwd with ngroups = nheads; the
    oracle rotates in fp64, rounds to bf16 as the pipeline does, and runs its
    recurrence."""
    batch, seqlen, nheads, headdim, dstate = 2, 256, 4, 64, 128
    if rank == 1:
        inp = inputs.mamba3_inputs(batch, seqlen, nheads, headdim, dstate, 1, "bf16", seed=260)
    else:
        inp = inputs.mamba3_mimo_inputs(batch, seqlen, rank, nheads, headdim, dstate, 1, "bf16",
                                        seed=261)
    r = inputs.rope_inputs(batch, seqlen, nheads, dstate, seed=262)
    d = {k: v.cuda() for k, v in inp.items()}
    Br, Cr, _ = binding.ssm_mamba3_rope(d["B"], d["C"], d["dt"], r["theta"].cuda(),
                                        r["angle0"].cuda())
    if rank == 1:
        y, fs = binding.ssd_mamba3_fwd(d["x"], d["dt"], d["lam"], d["A_head"], Br, Cr, 64,
                                       out_dtype=torch.float32, initial_state=d["h0"])
    else:
        y, fs = binding.ssd_mamba3_mimo_fwd(d["x"], d["dt"], d["lam"], d["A_head"], Br, Cr, 16,
                                            out_dtype=torch.float32, initial_state=d["h0"])
    torch.cuda.synchronize()
    Br_ref, Cr_ref, _ = oracle.mamba3_rope(inp["B"], inp["C"], inp["dt"], r["theta"],
                                           r["angle0"])
    B16, C16 = _bf16_round(Br_ref), _bf16_round(Cr_ref)
    if rank == 1:
        y_ref, fs_ref = oracle.mamba3_recurrence(inp["x"], inp["dt"], inp["lam"],
                                                 inp["A_head"], B16, C16, inp["h0"])
    else:
        y_ref, fs_ref = oracle.mamba3_mimo_recurrence(inp["x"], inp["dt"], inp["lam"],
                                                      inp["A_head"], B16, C16, inp["h0"])
    assert_close(y, y_ref, TOL_BF16, "y")
    assert_close(fs, fs_ref, TOL_BF16, "final_state")


def test_mamba3_decode_with_rope_128_steps():
    """fp32 decode, 128 chained steps: each step rotates its B and C (seqlen 1,
    the angle updated in place) and runs ssm_decode_step_mamba3; the oracle
    rotates the whole sequence at once and chains its decode steps."""
    batch, nheads, headdim, dstate, steps = 4, 4, 64, 128, 128
    g = torch.Generator().manual_seed(270)
    x = torch.randn(steps, batch, nheads, headdim, generator=g)
    Bm = torch.randn(steps, batch, 1, dstate, generator=g)
    Cm = torch.randn(steps, batch, 1, dstate, generator=g)
    dt = torch.nn.functional.softplus(torch.randn(steps, batch, nheads, generator=g) - 4)
    lam = torch.sigmoid(torch.randn(steps, batch, nheads, generator=g))
    A = -(1.0 + 15.0 * torch.rand(nheads, generator=g))
    D = torch.randn(nheads, generator=g)
    state0 = 0.1 * torch.randn(batch, nheads, headdim, dstate, generator=g)
    r = inputs.rope_inputs(batch, steps, nheads, dstate, seed=271)
    # the oracle: the sequence's rotation at once, then the decode chain
    Bseq = Bm.permute(1, 0, 2, 3).contiguous()  # (batch, steps, 1, N)
    Cseq = Cm.permute(1, 0, 2, 3).contiguous()
    dtseq = dt.permute(1, 0, 2).contiguous()
    Br_ref, Cr_ref, ang_ref = oracle.mamba3_rope(Bseq, Cseq, dtseq, r["theta"], r["angle0"])
    st_ref = state0.double().numpy()
    prevB_ref = np.zeros((batch, nheads, dstate))
    prevx_ref = np.zeros((batch, nheads, headdim))
    # the GPU: one rotation and one decode step per token
    state = state0.cuda()
    ang = r["angle0"].cuda()
    theta = r["theta"].cuda()
    prevB = torch.zeros(batch, nheads, dstate, device="cuda")
    prevx = torch.zeros(batch, nheads, headdim, device="cuda")
    for t in range(steps):
        Bt, Ct, _ = binding.ssm_mamba3_rope(Bm[t].unsqueeze(1).cuda(), Cm[t].unsqueeze(1).cuda(),
                                            dt[t].unsqueeze(1).cuda(),
                                            theta[:, t:t + 1].contiguous(), ang, angle_out=ang)
        Bt, Ct = Bt[:, 0].contiguous(), Ct[:, 0].contiguous()  # (batch, H, N): ngroups = H
        xt = x[t].cuda()
        y = binding.ssm_decode_step_mamba3(state, prevB, prevx, xt, dt[t].cuda(), lam[t].cuda(),
                                           A.cuda(), Bt, Ct, D.cuda())
        prevB, prevx = Bt, xt
        y_ref, st_ref = oracle.mamba3_decode_step(st_ref, prevB_ref, prevx_ref, x[t], dt[t],
                                                  lam[t], A, Br_ref[:, t], Cr_ref[:, t], D)
        prevB_ref, prevx_ref = Br_ref[:, t], x[t].double().numpy()
        assert_close(y, y_ref, TOL_F32, f"y step {t}")
    torch.cuda.synchronize()
    assert_close(state, st_ref, TOL_F32, "final state")
    np.testing.assert_allclose(to64(ang), ang_ref, rtol=2e-6, atol=2e-6)
