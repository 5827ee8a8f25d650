"""Parity of the tensor-core SSD gradient (ssd_chunked_bwd, through the C ABI)
with the fp64 oracle's reverse-mode derivative of the step recurrence.

Tolerance.  The kernel's products take bf16 operands: x, B, C and dy exactly,
the fp32 intermediates (states, adjoint states, masked decayed Q x Q products)
as bf16 hi + lo pairs (about 16 significant bits, relative error <= 2^-17 per
operand), with fp32 accumulation over K <= 128; the per-element gradients then
carry a normwise error of order 1e-5 (measured 3-5e-6): TOL_SSD_GRAD = 1e-4.
dA_head sums d cs over the batch and the sequence, where the C . dC and B . dB
terms largely cancel, so its error relative to its own size is larger
(measured up to 4.4e-5): TOL_SSD_DA = 5e-4.
"""
import pytest
import torch

import oracle
from state_space_model_selective_gb300 import binding, inputs
from tests.helpers import assert_close

pytestmark = pytest.mark.gpu

TOL_SSD_GRAD = 1e-4
TOL_SSD_DA = 5e-4
KEYS = [("dx", "dx", TOL_SSD_GRAD), ("ddt", "ddt", TOL_SSD_GRAD), ("dA_head", "dA", TOL_SSD_DA),
        ("dB", "dB", TOL_SSD_GRAD), ("dC", "dC", TOL_SSD_GRAD),
        ("dinitial_state", "dh0", TOL_SSD_GRAD)]


def _cotangents(batch, seqlen, nheads, seed, with_dfinal):
    gen = torch.Generator().manual_seed(seed)
    dy = torch.randn(batch, seqlen, nheads, 64, generator=gen).to(torch.bfloat16)
    dfinal = torch.randn(batch, nheads, 64, 128, generator=gen) if with_dfinal else None
    return dy, dfinal


def _gpu(inp, dy, h0=None, dfinal=None, poison=True):
    d = {k: v.cuda() for k, v in inp.items()}
    batch, seqlen, nheads, _ = d["x"].shape
    out = None
    if poison:  # catch elements the kernels never write
        f = dict(dtype=torch.float32, device="cuda")
        out = {"dx": torch.full(tuple(d["x"].shape), float("nan"), **f),
               "ddt": torch.full(tuple(d["dt"].shape), float("nan"), **f),
               "dA_head": torch.full((nheads,), float("nan"), **f),
               "dB": torch.full(tuple(d["B"].shape), float("nan"), **f),
               "dC": torch.full(tuple(d["C"].shape), float("nan"), **f),
               "dinitial_state": torch.full((batch, nheads, 64, 128), float("nan"), **f)}
    need = binding.ssd_chunked_bwd_workspace_bytes(batch, seqlen, nheads, 64, 128,
                                                   d["B"].shape[2])
    ws = torch.full((max(need, 256),), 0xAB, dtype=torch.uint8, device="cuda")
    g = binding.ssd_chunked_bwd(d["x"], d["dt"], d["A_head"], d["B"], d["C"], dy.cuda(), 64,
                                None if h0 is None else h0.cuda(),
                                None if dfinal is None else dfinal.cuda(), workspace=ws, out=out)
    torch.cuda.synchronize()
    if seqlen > 0 and batch * nheads > 0:
        assert binding.ssm_last_device_status(ws) == 0
    return g


def _ref(inp, dy, h0=None, dfinal=None):
    return oracle.ssd_bwd(inp["x"], inp["dt"], inp["A_head"], inp["B"], inp["C"], dy, h0, dfinal)


CASES = [  # batch, seqlen, nheads, ngroups, initial state and final cotangent
    (1, 64, 2, 1, False),    # one partial 128-step block
    (2, 128, 4, 1, True),    # one full block
    (2, 192, 4, 2, True),    # a full block and a half block, 2 groups
    (3, 256, 6, 3, False),   # two blocks, 3 groups
    (1, 640, 2, 1, True),    # five blocks: the adjoint state carried back four times
    (2, 128, 4, 4, True),    # one head per group: no sum over heads
]


@pytest.mark.parametrize("case", CASES,
                         ids=[f"B{c[0]}L{c[1]}H{c[2]}G{c[3]}{'s' if c[4] else ''}" for c in CASES])
def test_ssd_bwd_matches_oracle(case):
    batch, seqlen, nheads, ngroups, state = case
    inp = inputs.ssd_inputs(batch, seqlen, nheads, 64, 128, ngroups, "bf16", seed=60 + seqlen)
    dy, dfinal = _cotangents(batch, seqlen, nheads, 61 + seqlen, state)
    h0 = (0.1 * torch.randn(batch, nheads, 64, 128, generator=torch.Generator().manual_seed(5))
          if state else None)
    g = _gpu(inp, dy, h0, dfinal)
    ref = _ref(inp, dy, h0, dfinal)
    for key, rkey, tol in KEYS:
        assert_close(g[key], ref[rkey], tol, key)


def test_ssd_bwd_deterministic():
    inp = inputs.ssd_inputs(2, 256, 4, 64, 128, 1, "bf16", seed=71)
    dy, dfinal = _cotangents(2, 256, 4, 72, True)
    g1 = _gpu(inp, dy, None, dfinal)
    g2 = _gpu(inp, dy, None, dfinal)
    for k, v in g1.items():
        assert torch.equal(v, g2[k]), k


def test_ssd_bwd_empty_sequence():
    inp = inputs.ssd_inputs(2, 0, 4, 64, 128, 1, "bf16", seed=73)
    dy, dfinal = _cotangents(2, 0, 4, 74, True)
    g = _gpu(inp, dy, None, dfinal, poison=False)
    assert torch.count_nonzero(g["dA_head"]).item() == 0
    assert torch.equal(g["dinitial_state"].cpu(), dfinal)


def test_ssd_bwd_is_vjp_of_forward():
    """<dx, v> against a central difference of sum(dy y) through the CUDA forward:
    y is linear in x, so the difference is exact up to rounding (the forward's
    bf16 x input: v is a bf16-representable direction and eps a power of two)."""
    inp = inputs.ssd_inputs(1, 128, 2, 64, 128, 1, "bf16", seed=75)
    dy, _ = _cotangents(1, 128, 2, 76, False)
    g = _gpu(inp, dy)
    v = torch.randn(inp["x"].shape, generator=torch.Generator().manual_seed(77)).to(torch.bfloat16)
    eps = 0.25

    def loss(x):
        d = {k: t.cuda() for k, t in inp.items()}
        y, _ = binding.ssd_chunked_fwd(x.cuda(), d["dt"], d["A_head"], d["B"], d["C"], 64,
                                       out_dtype=torch.float32)
        return float((y.double().cpu() * dy.double()).sum())

    xp = (inp["x"].float() + eps * v.float()).to(torch.bfloat16)
    xm = (inp["x"].float() - eps * v.float()).to(torch.bfloat16)
    fd = (loss(xp) - loss(xm)) / (2 * eps)
    # the direction actually taken (bf16 rounding of x +- eps v)
    dirv = (xp.double() - xm.double()) / (2 * eps)
    an = float((g["dx"].double().cpu() * dirv).sum())
    assert abs(fd - an) <= 5e-3 * max(1.0, abs(an)), (fd, an)


def test_ssd_bwd_full_size_properties():
    """32 x 256 x 32 heads (headdim 64, d_state 128), the SSD workload, in its
    launch configuration.  With dy zero after step 64 and no final cotangent,
    every gradient at t >= 64 is exactly zero and the rest (including dA, a sum
    over the batch) matches the oracle on the first 64 steps."""
    batch, seqlen, nheads = 32, 256, 32
    inp = inputs.ssd_inputs(batch, seqlen, nheads, 64, 128, 1, "bf16", seed=1004)
    dy, _ = _cotangents(batch, seqlen, nheads, 1009, False)
    T = 64
    dy[:, T:] = 0
    g = _gpu(inp, dy, poison=False)
    for key in ("dx", "ddt", "dB", "dC"):
        assert torch.count_nonzero(g[key][:, T:]).item() == 0, key
    head = {k: (v[:, :T].contiguous() if k in ("x", "dt", "B", "C") else v) for k, v in inp.items()}
    ref = _ref(head, dy[:, :T].contiguous())
    for key, rkey, tol in KEYS:
        got = g[key][:, :T] if key in ("dx", "ddt", "dB", "dC") else g[key]
        assert_close(got, ref[rkey], tol, key)


@pytest.mark.parametrize("name,grad", [("dt", "ddt"), ("A_head", "dA_head")])
def test_ssd_bwd_directional_derivatives(name, grad):
    """<grad, v> against a central difference of sum(dy y) through the CUDA
    forward in the fp32 inputs dt and A_head (the forward is smooth in both)."""
    inp = inputs.ssd_inputs(1, 256, 4, 64, 128, 1, "bf16", seed=93)
    dy, _ = _cotangents(1, 256, 4, 94, False)
    g = _gpu(inp, dy, poison=False)
    gen = torch.Generator().manual_seed(95)
    base = inp[name]
    v = torch.randn(base.shape, generator=gen) * base.abs()  # relative direction
    eps = 1e-2

    def loss(t):
        d = {k: u.cuda() for k, u in inp.items()}
        d[name] = t.cuda()
        y, _ = binding.ssd_chunked_fwd(d["x"], d["dt"], d["A_head"], d["B"], d["C"], 64,
                                       out_dtype=torch.float32)
        return float((y.double().cpu() * dy.double()).sum())

    fd = (loss(base + eps * v) - loss(base - eps * v)) / (2 * eps)
    terms = g[grad].double().cpu() * v.double()
    an = float(terms.sum())
    # O(eps^2) truncation; the bound also scales with sum |g v| (a random
    # direction can make <g, v> cancel far below its terms)
    assert abs(fd - an) <= 5e-3 * abs(an) + 1e-3 * float(terms.abs().sum()), (name, fd, an)


def test_ssd_block_states_from_the_forward():
    """ssd_chunked_fwd with block states gives the plain forward's y and final
    state bit for bit, and ssd_chunked_bwd from those states gives the same bits
    as ssd_chunked_bwd recomputing them."""
    batch, seqlen, nheads = 2, 320, 4
    inp = inputs.ssd_inputs(batch, seqlen, nheads, 64, 128, 2, "bf16", seed=150)
    d = {k: v.cuda() for k, v in inp.items()}
    h0 = 0.1 * torch.randn(batch, nheads, 64, 128, generator=torch.Generator().manual_seed(151))
    h0 = h0.cuda()
    args = (d["x"], d["dt"], d["A_head"], d["B"], d["C"], 64)
    y0, f0 = binding.ssd_chunked_fwd(*args, out_dtype=torch.float32, initial_state=h0)
    bs = torch.full((binding.ssd_chunked_checkpoint_bytes(batch, seqlen, nheads) // 4,),
                    float("nan"), device="cuda")
    y1, f1 = binding.ssd_chunked_fwd(*args, out_dtype=torch.float32, initial_state=h0,
                                     block_states=bs)
    torch.cuda.synchronize()
    assert torch.equal(y0, y1) and torch.equal(f0, f1)
    assert not torch.isnan(bs).any()
    dy, dfinal = _cotangents(batch, seqlen, nheads, 152, True)
    g0 = binding.ssd_chunked_bwd(*args[:5], dy.cuda(), 64, h0, dfinal.cuda())
    g1 = binding.ssd_chunked_bwd(*args[:5], dy.cuda(), 64, h0, dfinal.cuda(), block_states=bs)
    torch.cuda.synchronize()
    for k, v in g0.items():
        assert torch.equal(v, g1[k]), k
