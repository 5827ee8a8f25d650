"""Parity of the CUDA decode step (through the C ABI) with the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from state_space_model_selective_gb300 import binding, inputs
from tests.helpers import TOL_BF16, TOL_F32, assert_close, to64, assert_elementwise

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("batch,nheads,headdim,dstate,ngroups,dtype,gate",
                         [(2, 4, 64, 128, 1, "f32", True), (3, 6, 16, 64, 2, "f32", False),
                          (1, 2, 8, 16, 1, "f32", True), (2, 4, 32, 256, 4, "bf16", True),
                          (5, 3, 7, 32, 1, "bf16", False),
                          # dstate 128 runs the bulk-copy kernel: tiles of up to 64 rows
                          (3, 2, 100, 128, 1, "bf16", True),   # a 64-row and a 36-row tile
                          (2, 3, 8, 128, 3, "f32", False),     # one short tile per head
                          (1, 1, 192, 128, 1, "f32", True)])   # three full tiles, one head
def test_decode_chain_matches_oracle(batch, nheads, headdim, dstate, ngroups, dtype, gate):
    steps = 6
    inp = inputs.decode_inputs(batch, nheads, headdim, dstate, ngroups, steps, dtype, seed=31,
                               gate=gate, dskip="randn")
    state = inp["state"].cuda()
    ref_state = inp["state"]
    tol = TOL_F32 if dtype == "f32" else TOL_BF16
    for t in range(steps):
        z = inp["z"][t]
        y = binding.ssm_decode_step(state, inp["x"][t].cuda(), inp["dt"][t].cuda(),
                                    inp["A"].cuda(), inp["B"][t].cuda(), inp["C"][t].cuda(),
                                    inp["D"].cuda(), None if z is None else z.cuda())
        y_ref, ref_state = oracle.decode_step(ref_state, inp["x"][t], inp["dt"][t], inp["A"],
                                              inp["B"][t], inp["C"][t], inp["D"], z)
        if dtype == "f32":
            assert_close(y, y_ref, tol, f"y step {t}")
        else:  # bf16 y: the rounding of the exact result, within one bf16 ulp
            assert_close(y, y_ref, 2 ** -7, f"y step {t}")
        assert_close(state, ref_state, tol, f"state step {t}")


def test_workload_decode_128_steps():
    """batch 256, 32 heads, headdim 64, dstate 128, fp32, 128 chained steps;
    y of every step and the final state checked on every batch row."""
    batch, nheads, headdim, dstate, steps = 256, 32, 64, 128, 128
    g = torch.Generator(device="cuda")
    g.manual_seed(1005)
    state = 0.1 * torch.randn(batch, nheads, headdim, dstate, device="cuda", generator=g)
    A = -(1.0 + 15.0 * torch.rand(nheads, device="cuda", generator=g))
    D = torch.ones(nheads, device="cuda")
    sample = torch.arange(batch)
    ref_state = state[sample].cpu()
    for t in range(steps):
        x = torch.randn(batch, nheads, headdim, device="cuda", generator=g)
        Bm = torch.randn(batch, 1, dstate, device="cuda", generator=g)
        Cm = torch.randn(batch, 1, dstate, device="cuda", generator=g)
        dt = torch.nn.functional.softplus(torch.randn(batch, nheads, device="cuda", generator=g) - 4)
        y = binding.ssm_decode_step(state, x, dt, A, Bm, Cm, D)
        y_ref, ref_state = oracle.decode_step(ref_state, x[sample].cpu(), dt[sample].cpu(), A.cpu(),
                                              Bm[sample].cpu(), Cm[sample].cpu(), D.cpu())
        assert_close(y[sample], y_ref, TOL_F32, f"y step {t}")
    assert_close(state[sample], ref_state, TOL_F32, "final state")
    assert_elementwise(state, ref_state, "final state")
    assert torch.isfinite(state).all()
