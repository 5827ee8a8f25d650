"""Parity of the Mamba-3 MIMO (rank R) prefill -- the tensor-core SSD over
rank-flattened sub-tokens -- and decode step, through the C ABI, with the fp64
oracle's rank-R recurrence."""
import pytest
import torch

import oracle
from state_space_model_selective_gb300 import binding, inputs
from tests.helpers import TOL_BF16, TOL_F32, assert_close

pytestmark = pytest.mark.gpu

_STEP_KEYS = ("x", "dt", "lam", "B", "C")


def _prefill(inp, h0=None, prev=False, out_dtype=torch.float32):
    d = {k: v.cuda() for k, v in inp.items()}
    rank = d["x"].shape[2]
    y = torch.full(d["x"].shape, float("nan"), dtype=out_dtype, device="cuda")
    batch, _, _, nheads, headdim = d["x"].shape
    fs = torch.full((batch, nheads, headdim, d["B"].shape[4]), float("nan"), device="cuda")
    binding.ssd_mamba3_mimo_fwd(d["x"], d["dt"], d["lam"], d["A_head"], d["B"], d["C"],
                                64 // rank, out_dtype=out_dtype, y=y, final_state=fs,
                                initial_state=None if h0 is None else h0.cuda(),
                                prev_B=d["prev_B"] if prev else None,
                                prev_x=d["prev_x"] if prev else None)
    torch.cuda.synchronize()
    return y, fs


def _ref(inp, h0=None, prev=False):
    return oracle.mamba3_mimo_recurrence(inp["x"], inp["dt"], inp["lam"], inp["A_head"],
                                         inp["B"], inp["C"],
                                         None if h0 is None else h0.double().numpy(),
                                         inp["prev_B"] if prev else None,
                                         inp["prev_x"] if prev else None)


CASES = [  # batch, seqlen (steps), rank, nheads, ngroups, initial state, previous token
    (1, 16, 4, 2, 1, False, False),   # 64 sub-tokens: one partial 128-row block
    (2, 32, 4, 4, 1, False, True),    # one full block
    (2, 80, 4, 4, 2, True, True),     # 2.5 blocks, 2 groups, resumed
    (1, 160, 4, 2, 1, False, False),  # five blocks
    (2, 96, 2, 4, 2, True, True),     # rank 2: 1.5 blocks
]


@pytest.mark.parametrize("case", CASES,
                         ids=[f"B{c[0]}L{c[1]}R{c[2]}H{c[3]}G{c[4]}h{int(c[5])}p{int(c[6])}"
                              for c in CASES])
def test_mimo_prefill_matches_recurrence(case):
    batch, seqlen, rank, nheads, ngroups, use_h0, use_prev = case
    inp = inputs.mamba3_mimo_inputs(batch, seqlen, rank, nheads, 64, 128, ngroups, "bf16",
                                    seed=300 + seqlen)
    h0 = inp["h0"] if use_h0 else None
    y, fs = _prefill(inp, h0, use_prev)
    y_ref, fs_ref = _ref(inp, h0, use_prev)
    assert_close(y, y_ref, TOL_BF16, "y")
    assert_close(fs, fs_ref, TOL_BF16, "final_state")


def test_mimo_rank_one_is_siso():
    inp = inputs.mamba3_mimo_inputs(2, 128, 1, 4, 64, 128, 1, "bf16", seed=311)
    y1, f1 = _prefill(inp, inp["h0"], prev=True)
    d = {k: v.cuda() for k, v in inp.items()}
    y2, f2 = binding.ssd_mamba3_fwd(d["x"][:, :, 0], d["dt"], d["lam"], d["A_head"],
                                    d["B"][:, :, 0], d["C"][:, :, 0], 64,
                                    out_dtype=torch.float32, initial_state=d["h0"],
                                    prev_B=d["prev_B"][:, 0], prev_x=d["prev_x"][:, 0])
    torch.cuda.synchronize()
    assert torch.equal(y1[:, :, 0], y2) and torch.equal(f1, f2)


@pytest.mark.parametrize("rank,dtype,gate", [(4, "f32", True), (4, "bf16", False),
                                             (2, "f32", False), (2, "bf16", True)])
def test_mimo_decode_chain_matches_oracle(rank, dtype, gate):
    batch, nheads, headdim, dstate, steps = 3, 4, 100, 128, 5
    inp = inputs.mamba3_mimo_inputs(batch, steps + 1, rank, nheads, headdim, dstate, 2, dtype,
                                    seed=321)
    g = torch.Generator().manual_seed(322)
    D = torch.randn(nheads, generator=g)
    zs = [torch.randn(batch, rank, nheads, headdim, generator=g).to(inp["x"].dtype) if gate
          else None for _ in range(steps + 1)]
    tol = TOL_F32 if dtype == "f32" else TOL_BF16
    state = inp["h0"].clone().cuda()
    st_ref = inp["h0"].double().numpy()
    for t in range(1, steps + 1):  # step 0's x and B serve as the previous token
        c = lambda v: None if v is None else v.contiguous().cuda()  # noqa: E731
        y = binding.ssm_decode_step_mamba3_mimo(
            state, c(inp["B"][:, t - 1]), c(inp["x"][:, t - 1]), c(inp["x"][:, t]),
            c(inp["dt"][:, t]), c(inp["lam"][:, t]), inp["A_head"].cuda(), c(inp["B"][:, t]),
            c(inp["C"][:, t]), D.cuda(), c(zs[t]))
        torch.cuda.synchronize()
        y_ref, st_ref = oracle.mamba3_mimo_decode_step(
            st_ref, inp["B"][:, t - 1], inp["x"][:, t - 1], inp["x"][:, t], inp["dt"][:, t],
            inp["lam"][:, t], inp["A_head"], inp["B"][:, t], inp["C"][:, t], D, zs[t])
        if dtype == "f32":
            assert_close(y, y_ref, tol, f"y step {t}")
        else:  # bf16 y: the rounding of the exact result, within one bf16 ulp
            assert_close(y, y_ref, 2 ** -7, f"y step {t}")
        assert_close(state, st_ref, tol, f"state step {t}")


def test_mimo_prefill_then_decode_handoff():
    """Prefill over 32 steps, then 16 decode steps (previous token = the last one
    seen), equal the prefill over all 48 steps."""
    batch, nheads, rank, L0, L1 = 2, 4, 4, 32, 16
    inp = inputs.mamba3_mimo_inputs(batch, L0 + L1, rank, nheads, 64, 128, 1, "bf16", seed=331)
    y_all, fs_all = _prefill(inp)
    first = {k: (v[:, :L0].contiguous() if k in _STEP_KEYS else v) for k, v in inp.items()}
    _, state = _prefill(first)
    d = {k: v.cuda() for k, v in inp.items()}
    ys = []
    for t in range(L0, L0 + L1):
        y = binding.ssm_decode_step_mamba3_mimo(
            state, d["B"][:, t - 1].contiguous(), d["x"][:, t - 1].contiguous(),
            d["x"][:, t].contiguous(), d["dt"][:, t].contiguous(), d["lam"][:, t].contiguous(),
            d["A_head"], d["B"][:, t].contiguous(), d["C"][:, t].contiguous())
        ys.append(y.float())
    torch.cuda.synchronize()
    assert_close(torch.stack(ys, dim=1), y_all[:, L0:].double().cpu().numpy(), 2 ** -7, "y")
    assert_close(state, fs_all.double().cpu().numpy(), 5e-5, "state")
