"""Parity of the Mamba-3 SISO prefill (tensor-core single-SSD form) and decode
step, through the C ABI, with the fp64 oracle's step-by-step recurrence."""
import numpy as np
import pytest
import torch

import oracle
from state_space_model_selective_gb300 import binding, inputs
from tests.helpers import TOL_BF16, TOL_F32, assert_close

pytestmark = pytest.mark.gpu


def _prefill(inp, h0=None, prev=False, out_dtype=torch.float32):
    d = {k: v.cuda() for k, v in inp.items()}
    batch, seqlen, nheads, headdim = d["x"].shape
    y = torch.full(d["x"].shape, float("nan"), dtype=out_dtype, device="cuda")
    fs = torch.full((batch, nheads, headdim, d["B"].shape[3]), float("nan"), device="cuda")
    binding.ssd_mamba3_fwd(d["x"], d["dt"], d["lam"], d["A_head"], d["B"], d["C"], 64,
                           out_dtype=out_dtype, y=y, final_state=fs,
                           initial_state=None if h0 is None else h0.cuda(),
                           prev_B=d["prev_B"] if prev else None,
                           prev_x=d["prev_x"] if prev else None)
    torch.cuda.synchronize()
    return y, fs


def _ref(inp, h0=None, prev=False):
    return oracle.mamba3_recurrence(inp["x"], inp["dt"], inp["lam"], inp["A_head"], inp["B"],
                                    inp["C"], None if h0 is None else h0.double().numpy(),
                                    inp["prev_B"] if prev else None,
                                    inp["prev_x"] if prev else None)


CASES = [  # batch, seqlen, nheads, ngroups, initial state, previous token
    (1, 64, 2, 1, False, False),    # one partial 128-step block
    (2, 128, 4, 1, False, True),    # one full block, previous token
    (2, 192, 4, 2, True, True),     # a full and a half block, 2 groups, resumed
    (3, 256, 6, 3, True, False),    # two blocks, 3 groups
    (1, 640, 2, 1, False, False),   # five blocks
]


@pytest.mark.parametrize("case", CASES,
                         ids=[f"B{c[0]}L{c[1]}H{c[2]}G{c[3]}h{int(c[4])}p{int(c[5])}" for c in CASES])
def test_mamba3_prefill_matches_recurrence(case):
    batch, seqlen, nheads, ngroups, use_h0, use_prev = case
    inp = inputs.mamba3_inputs(batch, seqlen, nheads, 64, 128, ngroups, "bf16", seed=200 + seqlen)
    h0 = inp["h0"] if use_h0 else None
    y, fs = _prefill(inp, h0, use_prev)
    y_ref, fs_ref = _ref(inp, h0, use_prev)
    assert_close(y, y_ref, TOL_BF16, "y")
    assert_close(fs, fs_ref, TOL_BF16, "final_state")


def test_mamba3_lambda_one_equals_mamba2_ssd():
    """lambda = 1: the Mamba-3 prefill is the Mamba-2 chunked SSD."""
    inp = inputs.mamba3_inputs(2, 256, 4, 64, 128, 1, "bf16", seed=211)
    inp["lam"] = torch.ones_like(inp["lam"])
    y3, f3 = _prefill(inp, inp["h0"], prev=True)
    d = {k: v.cuda() for k, v in inp.items()}
    y2, f2 = binding.ssd_chunked_fwd(d["x"], d["dt"], d["A_head"], d["B"], d["C"], 64,
                                     out_dtype=torch.float32, initial_state=d["h0"])
    torch.cuda.synchronize()
    assert_close(y3, y2.double().cpu().numpy(), 1e-5, "y")
    assert_close(f3, f2.double().cpu().numpy(), 1e-5, "final_state")


def test_mamba3_bf16_output_is_rounded_fp32_output():
    inp = inputs.mamba3_inputs(2, 256, 4, 64, 128, 1, "bf16", seed=213)
    y32, f32 = _prefill(inp, prev=True)
    y16, f16 = _prefill(inp, prev=True, out_dtype=torch.bfloat16)
    assert torch.equal(y16, y32.to(torch.bfloat16)) and torch.equal(f16, f32)


@pytest.mark.parametrize("split", [128, 64])
def test_mamba3_resume_equals_whole_sequence(split):
    """Prefill over L steps equals prefill over the first `split` steps, then
    the rest from its final state with the split's last token as the
    previous token."""
    batch, nheads, L = 2, 4, 384
    inp = inputs.mamba3_inputs(batch, L, nheads, 64, 128, 1, "bf16", seed=217)
    y_all, fs_all = _prefill(inp)
    first = {k: (v[:, :split].contiguous() if k in ("x", "dt", "lam", "B", "C") else v)
             for k, v in inp.items()}
    rest = {k: (v[:, split:].contiguous() if k in ("x", "dt", "lam", "B", "C") else v)
            for k, v in inp.items()}
    rest["prev_B"] = inp["B"][:, split - 1].contiguous()
    rest["prev_x"] = inp["x"][:, split - 1].contiguous()
    y1, fs1 = _prefill(first)
    y2, fs2 = _prefill(rest, h0=fs1.cpu(), prev=True)
    y_cat = torch.cat([y1, y2], dim=1)
    y_ref, fs_ref = _ref(inp)
    assert_close(y_cat, y_ref, TOL_BF16, "y")
    assert_close(fs2, fs_ref, TOL_BF16, "final_state")
    # the two runs cut the sequence into different 128-step blocks; each is
    # within ~1e-5 of the exact result (16-bit split operands), so they agree
    # to a few 1e-5
    assert_close(y_cat, y_all.double().cpu().numpy(), 5e-5, "y (runs)")
    assert_close(fs2, fs_all.double().cpu().numpy(), 5e-5, "final_state (runs)")


@pytest.mark.parametrize("batch,nheads,headdim,dstate,ngroups,dtype,gate",
                         [(2, 4, 64, 128, 1, "f32", True), (3, 2, 100, 128, 1, "bf16", False),
                          (3, 6, 16, 64, 2, "f32", False), (2, 4, 32, 256, 4, "bf16", True)])
def test_mamba3_decode_chain_matches_oracle(batch, nheads, headdim, dstate, ngroups, dtype, gate):
    steps = 6
    inp = inputs.decode_inputs(batch, nheads, headdim, dstate, ngroups, steps + 1, dtype, seed=41,
                               gate=gate, dskip="randn")
    g = torch.Generator().manual_seed(43)
    lams = [torch.sigmoid(torch.randn(batch, nheads, generator=g)) for _ in range(steps)]
    tol = TOL_F32 if dtype == "f32" else TOL_BF16
    state = inp["state"].clone().cuda()
    st_ref = inp["state"].double().numpy()
    D = inp["D"].cuda()
    for t in range(1, steps + 1):  # step 0's x and B serve as the previous token
        c = lambda v: None if v is None else v.cuda()  # noqa: E731
        y = binding.ssm_decode_step_mamba3(state, c(inp["B"][t - 1]), c(inp["x"][t - 1]),
                                           c(inp["x"][t]), c(inp["dt"][t]), c(lams[t - 1]),
                                           inp["A"].cuda(), c(inp["B"][t]), c(inp["C"][t]), D,
                                           c(inp["z"][t]))
        torch.cuda.synchronize()
        y_ref, st_ref = oracle.mamba3_decode_step(st_ref, inp["B"][t - 1], inp["x"][t - 1],
                                                  inp["x"][t], inp["dt"][t], lams[t - 1],
                                                  inp["A"], inp["B"][t], inp["C"][t], inp["D"],
                                                  inp["z"][t])
        if dtype == "f32":
            assert_close(y, y_ref, tol, f"y step {t}")
        else:  # bf16 y: the rounding of the exact result, within one bf16 ulp
            assert_close(y, y_ref, 2 ** -7, f"y step {t}")
        assert_close(state, st_ref, tol, f"state step {t}")


def test_mamba3_prefill_then_decode_handoff():
    """Prefill over 128 steps, then 64 decode steps (previous token = the last
    one seen), equal the prefill over all 192 steps."""
    batch, nheads, L0, L1 = 2, 4, 128, 64
    inp = inputs.mamba3_inputs(batch, L0 + L1, nheads, 64, 128, 1, "bf16", seed=223)
    y_all, fs_all = _prefill(inp)
    first = {k: (v[:, :L0].contiguous() if k in ("x", "dt", "lam", "B", "C") else v)
             for k, v in inp.items()}
    _, state = _prefill(first)
    d = {k: v.cuda() for k, v in inp.items()}
    ys = []
    for t in range(L0, L0 + L1):
        y = binding.ssm_decode_step_mamba3(state, d["B"][:, t - 1].contiguous(),
                                           d["x"][:, t - 1].contiguous(),
                                           d["x"][:, t].contiguous(), d["dt"][:, t].contiguous(),
                                           d["lam"][:, t].contiguous(), d["A_head"],
                                           d["B"][:, t].contiguous(), d["C"][:, t].contiguous(),
                                           y=torch.empty(batch, nheads, 64, dtype=torch.bfloat16,
                                                         device="cuda"))
        ys.append(y.float())
    torch.cuda.synchronize()
    # bf16 decode outputs against the prefill's fp32 outputs: one bf16 ulp
    assert_close(torch.stack(ys, dim=1), y_all[:, L0:].double().cpu().numpy(), 2 ** -7, "y")
    assert_close(state, fs_all.double().cpu().numpy(), 5e-5, "state")
