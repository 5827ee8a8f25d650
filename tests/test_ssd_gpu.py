"""Parity of the tensor-core chunked SSD (through the C ABI) with the fp64 oracle's
step-by-step recurrence."""
import numpy as np
import pytest
import torch

import oracle
from state_space_model_selective_gb300 import binding, inputs
from tests.helpers import TOL_BF16, assert_close, assert_elementwise

pytestmark = pytest.mark.gpu


def _run(inp, out_dtype=torch.float32, poison=True, h0=None):
    d = {k: v.cuda() for k, v in inp.items()}
    x = d["x"]
    batch, seqlen, nheads, headdim = x.shape
    y = torch.empty(x.shape, dtype=out_dtype, device="cuda")
    fs = torch.empty((batch, nheads, headdim, d["B"].shape[3]), device="cuda")
    if poison:
        y.fill_(float("nan"))
        fs.fill_(float("nan"))
    binding.ssd_chunked_fwd(d["x"], d["dt"], d["A_head"], d["B"], d["C"], 64, out_dtype=out_dtype,
                            y=y, final_state=fs,
                            initial_state=None if h0 is None else h0.cuda())
    torch.cuda.synchronize()
    return y, fs


def _slice_steps(inp, t0, t1):
    return {k: (v[:, t0:t1].contiguous() if k in ("x", "dt", "B", "C") else v)
            for k, v in inp.items()}


CASES = [  # batch, seqlen, nheads, ngroups
    (1, 64, 2, 1),     # one partial 128-step block
    (2, 128, 4, 1),    # one full block
    (2, 192, 4, 2),    # a full block and a half block, 2 groups
    (3, 256, 6, 3),    # two blocks, 3 groups
    (1, 640, 2, 1),    # five blocks: long carried state
]


@pytest.mark.parametrize("case", CASES, ids=[f"B{c[0]}L{c[1]}H{c[2]}G{c[3]}" for c in CASES])
def test_ssd_matches_recurrence(case):
    batch, seqlen, nheads, ngroups = case
    inp = inputs.ssd_inputs(batch, seqlen, nheads, 64, 128, ngroups, "bf16", seed=40 + seqlen)
    y, fs = _run(inp)
    y_ref, fs_ref = oracle.ssd_recurrence(inp["x"], inp["dt"], inp["A_head"], inp["B"], inp["C"])
    assert_close(y, y_ref, TOL_BF16, "y")
    assert_close(fs, fs_ref, TOL_BF16, "final_state")


def test_ssd_bf16_output_is_rounded_fp32_output():
    inp = inputs.ssd_inputs(2, 256, 4, 64, 128, 1, "bf16", seed=3)
    y32, f32 = _run(inp, torch.float32)
    y16, f16 = _run(inp, torch.bfloat16)
    assert torch.equal(y16, y32.to(torch.bfloat16))
    assert torch.equal(f16, f32)


def test_ssd_deterministic():
    inp = inputs.ssd_inputs(2, 256, 4, 64, 128, 1, "bf16", seed=4)
    a = _run(inp)
    b = _run(inp)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_ssd_zero_length():
    x = torch.zeros(2, 0, 4, 64, dtype=torch.bfloat16, device="cuda")
    dt = torch.zeros(2, 0, 4, device="cuda")
    A = -torch.ones(4, device="cuda")
    B = torch.zeros(2, 0, 1, 128, dtype=torch.bfloat16, device="cuda")
    fs = torch.full((2, 4, 64, 128), 7.0, device="cuda")
    binding.ssd_chunked_fwd(x, dt, A, B, B, 64, final_state=fs)
    torch.cuda.synchronize()
    assert torch.count_nonzero(fs).item() == 0


def test_prefill_then_decode_handoff():
    """The SSD's final state seeds the decode step: 128 prefill steps by the
    chunked SSD, then 64 chained decode steps, equal the SSD over all 192
    steps (outputs of the decoded steps and the final state)."""
    batch, L0, L1, nheads = 2, 128, 64, 4
    inp = inputs.ssd_inputs(batch, L0 + L1, nheads, 64, 128, 1, "bf16", seed=12)
    y_all, fs_all = _run(inp)
    pre = {k: (v[:, :L0].contiguous() if v.dim() > 1 else v) for k, v in inp.items()}
    _, state = _run(pre)
    d = {k: v.cuda() for k, v in inp.items()}
    for t in range(L0, L0 + L1):
        y = binding.ssm_decode_step(state, d["x"][:, t].contiguous(), d["dt"][:, t].contiguous(),
                                    d["A_head"], d["B"][:, t].contiguous(),
                                    d["C"][:, t].contiguous())
        assert_close(y.float(), y_all[:, t], 2 ** -7, f"decoded step {t}")
    assert_close(state, fs_all, TOL_BF16, "final state after decode")


def test_workload_ssd_B32_L256_H32():
    """Chunked SSD bf16, batch 32, L 256, 32 heads, headdim 64, d_state 128,
    chunk 64; every output element checked against the sequential recurrence
    (eight batch rows per oracle call)."""
    inp = inputs.ssd_inputs(32, 256, 32, 64, 128, 1, "bf16", seed=1004)
    y, fs = _run(inp, poison=False)
    assert torch.isfinite(y).all() and torch.isfinite(fs).all()
    y_ref = np.empty(tuple(y.shape))
    fs_ref = np.empty(tuple(fs.shape))
    for b0 in range(0, 32, 8):
        sl = slice(b0, b0 + 8)
        y_ref[sl], fs_ref[sl] = oracle.ssd_recurrence(inp["x"][sl], inp["dt"][sl],
                                                      inp["A_head"], inp["B"][sl], inp["C"][sl])
    assert_close(y, y_ref, TOL_BF16, "y")
    assert_close(fs, fs_ref, TOL_BF16, "final_state")
    assert_elementwise(y, y_ref, "y")


@pytest.mark.parametrize("seqlen", [64, 192, 256])
def test_ssd_initial_state_matches_recurrence(seqlen):
    """Prefill resumed from a given state: the recurrence starts at h0."""
    batch, nheads = 2, 4
    inp = inputs.ssd_inputs(batch, seqlen, nheads, 64, 128, 2, "bf16", seed=70 + seqlen)
    h0 = torch.randn(batch, nheads, 64, 128, generator=torch.Generator().manual_seed(5))
    y, fs = _run(inp, h0=h0)
    y_ref, fs_ref = oracle.ssd_recurrence(inp["x"], inp["dt"], inp["A_head"], inp["B"], inp["C"],
                                          h0.double().numpy())
    assert_close(y, y_ref, TOL_BF16, "y")
    assert_close(fs, fs_ref, TOL_BF16, "final_state")


@pytest.mark.parametrize("split", [128, 64])
def test_ssd_resume_equals_whole_sequence(split):
    """The SSD over 384 steps equals the SSD over the first `split` steps
    followed by the SSD over the rest from its final state; with the split on a
    128-step block boundary the two runs do the same arithmetic (bit-equal)."""
    batch, nheads, L = 2, 4, 384
    inp = inputs.ssd_inputs(batch, L, nheads, 64, 128, 1, "bf16", seed=81)
    y_all, fs_all = _run(inp)
    y1, fs1 = _run(_slice_steps(inp, 0, split))
    y2, fs2 = _run(_slice_steps(inp, split, L), h0=fs1.cpu())
    y_cat = torch.cat([y1, y2], dim=1)
    if split % 128 == 0:
        assert torch.equal(y_cat, y_all) and torch.equal(fs2, fs_all)
    else:
        assert_close(y_cat, y_all.double().cpu().numpy(), 1e-5, "y")
        assert_close(fs2, fs_all.double().cpu().numpy(), 1e-5, "final_state")


def test_ssd_initial_state_in_place():
    """initial_state may be final_state itself: the state is updated in place."""
    batch, nheads = 2, 4
    inp = inputs.ssd_inputs(batch, 256, nheads, 64, 128, 1, "bf16", seed=90)
    d = {k: v.cuda() for k, v in inp.items()}
    h0 = torch.randn(batch, nheads, 64, 128, generator=torch.Generator().manual_seed(6)).cuda()
    ref_y, ref_fs = _run(inp, h0=h0.cpu())
    state = h0.clone()
    y = torch.empty(d["x"].shape, device="cuda")
    binding.ssd_chunked_fwd(d["x"], d["dt"], d["A_head"], d["B"], d["C"], 64, out_dtype=torch.float32,
                            y=y, final_state=state, initial_state=state)
    torch.cuda.synchronize()
    assert torch.equal(y, ref_y) and torch.equal(state, ref_fs)


def test_ssd_zero_length_passes_state_through():
    x = torch.zeros(2, 0, 4, 64, dtype=torch.bfloat16, device="cuda")
    dt = torch.zeros(2, 0, 4, device="cuda")
    A = -torch.ones(4, device="cuda")
    B = torch.zeros(2, 0, 1, 128, dtype=torch.bfloat16, device="cuda")
    h0 = torch.randn(2, 4, 64, 128, device="cuda")
    fs = torch.full((2, 4, 64, 128), 7.0, device="cuda")
    binding.ssd_chunked_fwd(x, dt, A, B, B, 64, final_state=fs, initial_state=h0)
    torch.cuda.synchronize()
    assert torch.equal(fs, h0)
