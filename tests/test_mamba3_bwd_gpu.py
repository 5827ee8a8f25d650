"""Parity of the Mamba-3 SISO gradient (ssd_mamba3_bwd, through the C ABI) with
the fp64 oracle's reverse-mode derivative of the three-term recurrence (Eq. 9
of "Mamba-3 NKI Kernels for AWS Neuron", section "How it works").

Tolerance.  The call is the tensor-core SSD gradient (with the Mamba-3 input
weights) plus fp32 elementwise kernels, so the per-element gradients carry the
SSD gradient's error class, normwise of order 1e-5: TOL_GRAD = 1e-4 as for
ssd_chunked_bwd; dA_head (a sum over the batch and the sequence in which the
C . dC and B . dB terms largely cancel) TOL_DA = 5e-4 likewise.
"""
import pytest
import torch

import oracle
from state_space_model_selective_gb300 import binding, inputs
from tests.helpers import assert_close

pytestmark = pytest.mark.gpu

TOL_GRAD = 1e-4
TOL_DA = 5e-4
KEYS = [("dx", "dx", TOL_GRAD), ("ddt", "ddt", TOL_GRAD), ("dlam", "dlam", TOL_GRAD),
        ("dA_head", "dA", TOL_DA), ("dB", "dB", TOL_GRAD), ("dC", "dC", TOL_GRAD),
        ("dinitial_state", "dh0", TOL_GRAD), ("dprev_B", "dprev_B", TOL_GRAD),
        ("dprev_x", "dprev_x", TOL_GRAD)]


def _case_inputs(batch, seqlen, nheads, ngroups, seed, h0, prev, dfinal):
    inp = inputs.mamba3_inputs(batch, seqlen, nheads, 64, 128, ngroups, "bf16", seed=seed)
    gen = torch.Generator().manual_seed(seed + 1)
    dy = torch.randn(batch, seqlen, nheads, 64, generator=gen).to(torch.bfloat16)
    df = torch.randn(batch, nheads, 64, 128, generator=gen) if dfinal else None
    if not h0:
        inp["h0"] = None
    if not prev:
        inp["prev_B"] = inp["prev_x"] = None
    return inp, dy, df


def _gpu(inp, dy, dfinal, ws_fill=0xAB):
    c = lambda t: None if t is None else t.cuda()
    batch, seqlen, nheads, _ = inp["x"].shape
    need = binding.ssd_mamba3_bwd_workspace_bytes(batch, seqlen, nheads, 64, 128,
                                                  inp["B"].shape[2])
    ws = torch.full((max(need, 256),), ws_fill, dtype=torch.uint8, device="cuda")
    g = binding.ssd_mamba3_bwd(c(inp["x"]), c(inp["dt"]), c(inp["lam"]), c(inp["A_head"]),
                               c(inp["B"]), c(inp["C"]), c(dy), 64, c(inp["h0"]),
                               c(inp["prev_B"]), c(inp["prev_x"]), c(dfinal), workspace=ws)
    torch.cuda.synchronize()
    if seqlen > 0 and batch * nheads > 0:
        assert binding.ssm_last_device_status(ws) == 0
    return g


def _ref(inp, dy, dfinal):
    return oracle.mamba3_bwd(inp["x"], inp["dt"], inp["lam"], inp["A_head"], inp["B"], inp["C"],
                             dy, inp["h0"], inp["prev_B"], inp["prev_x"], dfinal)


CASES = [  # batch, seqlen, nheads, ngroups, initial state, previous token, final cotangent
    (1, 64, 2, 1, False, False, False),   # one partial block, nothing carried in
    (2, 128, 4, 1, True, True, True),     # one full block, everything given
    (2, 192, 4, 2, True, True, True),     # a block and a half, 2 groups
    (3, 256, 6, 3, False, True, False),   # two blocks, 3 groups, the previous token only
    (1, 640, 2, 1, True, True, True),     # five blocks: the adjoint carried back four times
    (2, 128, 4, 4, True, False, True),    # one head per group
]


@pytest.mark.parametrize("case", CASES, ids=[
    f"B{c[0]}L{c[1]}H{c[2]}G{c[3]}{'s' if c[4] else ''}{'p' if c[5] else ''}{'f' if c[6] else ''}"
    for c in CASES])
def test_mamba3_bwd_matches_oracle(case):
    batch, seqlen, nheads, ngroups, h0, prev, df = case
    inp, dy, dfinal = _case_inputs(batch, seqlen, nheads, ngroups, 300 + seqlen, h0, prev, df)
    g = _gpu(inp, dy, dfinal)
    ref = _ref(inp, dy, dfinal)
    for key, rkey, tol in KEYS:
        if ref[rkey] is None:
            assert g[key] is None, key
            continue
        assert_close(g[key], ref[rkey], tol, key)


def test_mamba3_bwd_lambda_one_is_the_ssd_gradient():
    """At lambda = 1 (no previous-token term, beta = 0) the Mamba-3 recurrence is the
    Mamba-2 SSD's: dx, ddt, dA, dB, dC, dinitial_state equal ssd_chunked_bwd's up to
    rounding (the same kernels with weights w = dt)."""
    inp, dy, dfinal = _case_inputs(2, 256, 4, 2, 410, True, False, True)
    inp["lam"] = torch.ones_like(inp["lam"])
    g = _gpu(inp, dy, dfinal)
    c = lambda t: t.cuda()
    s = binding.ssd_chunked_bwd(c(inp["x"]), c(inp["dt"]), c(inp["A_head"]), c(inp["B"]),
                                c(inp["C"]), c(dy), 64, c(inp["h0"]), c(dfinal))
    torch.cuda.synchronize()
    for key in ("dx", "ddt", "dA_head", "dB", "dC", "dinitial_state"):
        assert_close(g[key], s[key].double().cpu(), 1e-5, key)


def test_mamba3_bwd_deterministic_and_workspace_independent():
    inp, dy, dfinal = _case_inputs(2, 256, 4, 1, 420, True, True, True)
    g1 = _gpu(inp, dy, dfinal, ws_fill=0x00)
    g2 = _gpu(inp, dy, dfinal, ws_fill=0xFF)
    for k, v in g1.items():
        if v is not None:
            assert torch.equal(v, g2[k]), k


def test_mamba3_bwd_empty_sequence():
    inp, dy, dfinal = _case_inputs(2, 0, 4, 1, 430, False, True, True)
    g = _gpu(inp, dy, dfinal)
    assert torch.count_nonzero(g["dA_head"]).item() == 0
    assert torch.equal(g["dinitial_state"].cpu(), dfinal)
    assert torch.count_nonzero(g["dprev_B"]).item() == 0
    assert torch.count_nonzero(g["dprev_x"]).item() == 0


@pytest.mark.parametrize("name,grad", [("dt", "ddt"), ("lam", "dlam")])
def test_mamba3_bwd_directional_derivatives(name, grad):
    """<grad, v> against a central difference of sum(dy y) + sum(dfinal final_state)
    through the CUDA forward (ssd_mamba3_fwd) in the fp32 inputs dt and lambda."""
    inp, dy, dfinal = _case_inputs(1, 256, 4, 1, 440, True, True, True)
    g = _gpu(inp, dy, dfinal)
    base = inp[name]
    v = torch.randn(base.shape, generator=torch.Generator().manual_seed(441)) * base.abs()
    eps = 1e-2

    def loss(t):
        d = {k: (None if u is None else u.cuda()) for k, u in inp.items()}
        d[name] = t.cuda()
        y, fs = binding.ssd_mamba3_fwd(d["x"], d["dt"], d["lam"], d["A_head"], d["B"], d["C"],
                                       64, out_dtype=torch.float32, initial_state=d["h0"],
                                       prev_B=d["prev_B"], prev_x=d["prev_x"])
        return float((y.double().cpu() * dy.double()).sum() +
                     (fs.double().cpu() * dfinal.double()).sum())

    fd = (loss(base + eps * v) - loss(base - eps * v)) / (2 * eps)
    terms = g[grad].double().cpu() * v.double()
    an = float(terms.sum())
    assert abs(fd - an) <= 5e-3 * abs(an) + 1e-3 * float(terms.abs().sum()), (name, fd, an)


def test_mamba3_bwd_full_size_properties():
    """32 x 256 x 32 heads (headdim 64, d_state 128), the bench's Mamba-3 gradient
    workload, in its launch configuration.  With dy zero after step 64, no final
    cotangent and no previous token, the loss depends on the first 64 steps only:
    dx, dB, dC are exactly zero from step 64 on and ddt, dlambda from step 65 on
    (dt_64 and lambda_64 enter the first 64 steps' algebra only through terms that
    cancel), and the first 64 steps, dA and the initial state's gradient match the
    oracle run on those steps alone."""
    batch, seqlen, nheads, T = 32, 256, 32, 64
    inp, dy, _ = _case_inputs(batch, seqlen, nheads, 1, 1006, True, False, False)
    dy[:, T:] = 0
    g = _gpu(inp, dy, None)
    for key in ("dx", "dB", "dC"):
        assert torch.count_nonzero(g[key][:, T:]).item() == 0, key
    for key in ("ddt", "dlam"):
        assert torch.count_nonzero(g[key][:, T + 1:]).item() == 0, key
    head = {k: (v[:, :T].contiguous() if k in ("x", "dt", "lam", "B", "C") else v)
            for k, v in inp.items()}
    ref = _ref(head, dy[:, :T].contiguous(), None)
    for key, rkey, tol in KEYS:
        if ref[rkey] is None:
            continue
        got = g[key][:, :T] if key in ("dx", "ddt", "dlam", "dB", "dC") else g[key]
        assert_close(got, ref[rkey], tol, key)


def test_mamba3_block_states_from_the_forward():
    """ssd_mamba3_fwd keeping block states gives the plain forward's y and final state
    bit for bit, and ssd_mamba3_bwd from those states gives the same bits as
    ssd_mamba3_bwd recomputing them."""
    batch, seqlen, nheads = 2, 320, 4
    inp, dy, dfinal = _case_inputs(batch, seqlen, nheads, 2, 450, True, True, True)
    d = {k: (None if v is None else v.cuda()) for k, v in inp.items()}
    args = (d["x"], d["dt"], d["lam"], d["A_head"], d["B"], d["C"], 64)
    kw = dict(initial_state=d["h0"], prev_B=d["prev_B"], prev_x=d["prev_x"])
    y0, f0 = binding.ssd_mamba3_fwd(*args, out_dtype=torch.float32, **kw)
    bs = torch.full((binding.ssd_chunked_checkpoint_bytes(batch, seqlen, nheads) // 4,),
                    float("nan"), device="cuda")
    y1, f1 = binding.ssd_mamba3_fwd(*args, out_dtype=torch.float32, block_states=bs, **kw)
    torch.cuda.synchronize()
    assert torch.equal(y0, y1) and torch.equal(f0, f1)
    assert not torch.isnan(bs).any()
    g0 = binding.ssd_mamba3_bwd(*args[:6], dy.cuda(), 64, d["h0"], d["prev_B"], d["prev_x"],
                                dfinal.cuda())
    g1 = binding.ssd_mamba3_bwd(*args[:6], dy.cuda(), 64, d["h0"], d["prev_B"], d["prev_x"],
                                dfinal.cuda(), block_states=bs)
    torch.cuda.synchronize()
    for k, v in g0.items():
        assert torch.equal(v, g1[k]), k
