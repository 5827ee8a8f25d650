"""Parity of the CUDA selective-scan gradient (ssm_scan_bwd, through the C ABI)
with the fp64 oracle's reverse-mode derivative.

Tolerance: the kernel differentiates in fp32 from the same (bf16-rounded where
the inputs are bf16) values the oracle reads, so every output is held to a
normwise bound.  Per-element gradients (du, ddelta, dz, dinitial_state) carry
the forward's rounding plus one reverse sweep: TOL_GRAD.  Gradients that are
sums over the batch and the sequence (dA, dD, ddelta_bias) or over a group's
channels (dB, dC) add fp32 rounding that grows with the square root of the
number of terms: TOL_GRAD_SUM.
"""
import pytest
import torch

import oracle
from state_space_model_selective_gb300 import binding, inputs
from tests.helpers import assert_close

pytestmark = pytest.mark.gpu

TOL_GRAD = 2e-5
TOL_GRAD_SUM = 5e-5

KEYS = [("du", "du", TOL_GRAD), ("ddelta", "ddelta", TOL_GRAD), ("dz", "dz", TOL_GRAD),
        ("dinitial_state", "dh0", TOL_GRAD), ("dA", "dA", TOL_GRAD_SUM),
        ("dB", "dB", TOL_GRAD_SUM), ("dC", "dC", TOL_GRAD_SUM), ("dD", "dD", TOL_GRAD_SUM),
        ("ddelta_bias", "dbias", TOL_GRAD_SUM)]


def _dev(t):
    return None if t is None else t.cuda()


def _gpu_grad(inp, dy, h0=None, dfinal=None, poison=True):
    x = {k: (_dev(v) if isinstance(v, torch.Tensor) or v is None else v) for k, v in inp.items()}
    batch, dim, seqlen = x["u"].shape
    need = binding.ssm_scan_bwd_workspace_bytes(batch, dim, seqlen, 16, x["B"].shape[1])
    ws = torch.full((max(need, 256),), 0xAB, dtype=torch.uint8, device="cuda")
    out = None
    if poison:  # catch elements the kernels never write
        f = dict(dtype=torch.float32, device="cuda")
        act = (batch, dim, seqlen)
        out = {"du": torch.full(act, float("nan"), **f),
               "ddelta": torch.full(act, float("nan"), **f),
               "dA": torch.full(tuple(x["A"].shape), float("nan"), **f),
               "dB": torch.full(tuple(x["B"].shape), float("nan"), **f),
               "dC": torch.full(tuple(x["C"].shape), float("nan"), **f),
               "dinitial_state": torch.full((batch, dim, 16), float("nan"), **f)}
        if x["z"] is not None:
            out["dz"] = torch.full(act, float("nan"), **f)
        if x["D"] is not None:
            out["dD"] = torch.full((dim,), float("nan"), **f)
        if x["delta_bias"] is not None:
            out["ddelta_bias"] = torch.full((dim,), float("nan"), **f)
    g = binding.ssm_scan_bwd(x["u"], x["delta"], x["A"], x["B"], x["C"], _dev(dy), x["D"],
                             x["z"], x["delta_bias"], x["delta_softplus"], _dev(h0),
                             _dev(dfinal), workspace=ws, out=out)
    torch.cuda.synchronize()
    if seqlen > 0:  # with no steps nothing runs and the workspace is not touched
        assert binding.ssm_last_device_status(ws) == 0
    return g


def _oracle_grad(inp, dy, h0=None, dfinal=None):
    return oracle.scan_bwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], dy, inp["D"],
                           inp["z"], inp["delta_bias"], inp["delta_softplus"], h0, dfinal)


def _compare(g, ref, skip=()):
    for key, rkey, tol in KEYS:
        if key in skip or ref[rkey] is None:
            continue
        assert g[key] is not None, key
        assert_close(g[key], ref[rkey], tol, key)


def _dy(shape, dtype, seed):
    gen = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=gen).to(inputs.torch_dtype(dtype))


CASES = [
    # batch, dim, seqlen, ngroups, dtype, gate, dskip, softplus, h0/dfinal
    (1, 32, 64, 1, "f32", True, "ones", True, False),      # one tile, one block
    (2, 64, 200, 1, "f32", True, "randn", True, True),     # ragged tail, 4 tiles
    (2, 48, 333, 1, "f32", False, "none", False, False),   # odd L, partial block, no gate
    (3, 96, 256, 2, "bf16", True, "ones", True, True),     # groups
    (2, 40, 130, 4, "bf16", True, "randn", True, False),   # 10 channels per group
    (1, 32, 77, 1, "bf16", True, "ones", False, True),     # odd L with bf16
    (1, 64, 16, 1, "f32", True, "randn", True, True),      # one segment
    (2, 32, 7, 1, "f32", True, "ones", True, True),        # shorter than a segment
]


@pytest.mark.parametrize("case", CASES,
                         ids=[f"B{c[0]}D{c[1]}L{c[2]}G{c[3]}{c[4]}" for c in CASES])
def test_scan_bwd_matches_oracle(case):
    batch, dim, seqlen, ngroups, dt, gate, dskip, softplus, state = case
    inp = inputs.scan_inputs(batch, dim, seqlen, 16, ngroups, dt, seed=300 + seqlen, gate=gate,
                             dskip=dskip)
    inp["delta_softplus"] = softplus
    if not softplus:  # without softplus, delta + bias must stay positive
        inp["delta"] = (inp["delta"].float().abs() * 0.1).to(inp["delta"].dtype)
        inp["delta_bias"] = torch.full_like(inp["delta_bias"], 0.01)
    dy = _dy((batch, dim, seqlen), dt, 7 + seqlen)
    gen = torch.Generator().manual_seed(11)
    h0 = torch.randn(batch, dim, 16, generator=gen) * 0.5 if state else None
    dfinal = torch.randn(batch, dim, 16, generator=gen) if state else None
    g = _gpu_grad(inp, dy, h0, dfinal)
    ref = _oracle_grad(inp, dy, h0, dfinal)
    _compare(g, ref)
    if not gate:
        assert g["dz"] is None


def test_scan_bwd_optional_outputs_without_inputs():
    """dD and ddelta_bias are the derivatives at D = 0 and delta_bias = 0 when
    those inputs are absent; the oracle gives them by passing explicit zeros."""
    inp = inputs.scan_inputs(2, 64, 150, 16, 1, "f32", seed=41, dskip="none")
    inp["delta_bias"] = None
    dy = _dy((2, 64, 150), "f32", 3)
    x = {k: (_dev(v) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    g = binding.ssm_scan_bwd(x["u"], x["delta"], x["A"], x["B"], x["C"], dy.cuda(), None, x["z"],
                             None, True, want_dD=True, want_ddelta_bias=True)
    torch.cuda.synchronize()
    z64 = dict(inp, D=torch.zeros(64), delta_bias=torch.zeros(64))
    ref = _oracle_grad(z64, dy)
    _compare(g, ref)


def test_scan_bwd_deterministic():
    """Two runs give the same bits: every sum is added in a fixed order."""
    inp = inputs.scan_inputs(2, 128, 300, 16, 2, "bf16", seed=8)
    dy = _dy((2, 128, 300), "bf16", 9)
    g1 = _gpu_grad(inp, dy)
    g2 = _gpu_grad(inp, dy)
    for k, v in g1.items():
        if v is not None:
            assert torch.equal(v, g2[k]), k


def test_scan_bwd_empty_sequence():
    """No step: the parameter gradients are zero and dinitial_state = dfinal."""
    inp = inputs.scan_inputs(2, 32, 0, 16, 1, "f32", seed=2)
    dfinal = torch.randn(2, 32, 16)
    dy = torch.zeros(2, 32, 0)
    g = _gpu_grad(inp, dy, None, dfinal)
    assert torch.count_nonzero(g["dA"]).item() == 0
    assert torch.count_nonzero(g["dD"]).item() == 0
    assert torch.count_nonzero(g["ddelta_bias"]).item() == 0
    assert torch.equal(g["dinitial_state"].cpu(), dfinal)


def test_scan_bwd_is_vjp_of_forward():
    """sum(dy * y(x + eps v)) - sum(dy * y(x - eps v)) over 2 eps equals <grad, v>
    for a random direction v in u, with the CUDA forward and backward alone: the
    two kernels agree with each other, not only with the oracle."""
    inp = inputs.scan_inputs(1, 32, 128, 16, 1, "f32", seed=77)
    dy = _dy((1, 32, 128), "f32", 78)
    g = _gpu_grad(inp, dy)
    v = torch.randn(1, 32, 128, generator=torch.Generator().manual_seed(79))
    eps = 0.5

    def loss(u):
        x = {k: (_dev(t) if isinstance(t, torch.Tensor) else t) for k, t in inp.items()}
        y, _ = binding.ssm_scan_fwd(u.cuda(), x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"],
                                    x["delta_bias"], True)
        return float((y.double().cpu() * dy.double()).sum())

    fd = (loss(inp["u"] + eps * v) - loss(inp["u"] - eps * v)) / (2 * eps)
    an = float((g["du"].double().cpu() * v.double()).sum())
    # y is linear in u, so the central difference is exact up to fp32 rounding
    assert abs(fd - an) <= 1e-3 * max(1.0, abs(an)), (fd, an)


def test_scan_bwd_full_size_properties():
    """8 x 1536 x 2048, the scan's benchmark workload, in its launch
    configuration.  (a) Channels are independent apart from the dB/dC sums:
    du, ddelta, dz, dinitial_state of channels 0..63 and their dA, dD,
    ddelta_bias match the oracle run on those channels alone.  (b) With dy zero
    after step 64, nothing flows back from later steps: every gradient at
    t >= 64 is exactly zero and dB, dC at t < 64 match the oracle on the first
    64 steps of all channels."""
    batch, dim, seqlen = 8, 1536, 2048
    inp = inputs.scan_inputs(batch, dim, seqlen, 16, 1, "bf16", seed=1002)
    dy = _dy((batch, dim, seqlen), "bf16", 1003)
    g = _gpu_grad(inp, dy, poison=False)
    cs = slice(0, 64)
    sl = {k: (v[:, cs].contiguous() if k in ("u", "delta", "z") else v) for k, v in inp.items()}
    sl["A"] = inp["A"][cs].contiguous()
    sl["D"] = inp["D"][cs].contiguous()
    sl["delta_bias"] = inp["delta_bias"][cs].contiguous()
    ref = _oracle_grad(sl, dy[:, cs].contiguous())
    for key, rkey, tol in KEYS:
        if key in ("dB", "dC") or ref[rkey] is None:
            continue
        got = g[key][:, cs] if g[key].dim() == 3 else g[key][cs]
        assert_close(got, ref[rkey], tol, key)

    T = 64
    dy2 = dy.clone()
    dy2[..., T:] = 0
    g2 = _gpu_grad(inp, dy2, poison=False)
    for key in ("du", "ddelta", "dz", "dB", "dC"):
        assert torch.count_nonzero(g2[key][..., T:]).item() == 0, key
    head = {k: (v[..., :T].contiguous() if k in ("u", "delta", "z", "B", "C") else v)
            for k, v in inp.items()}
    ref2 = _oracle_grad(head, dy2[..., :T].contiguous())
    assert_close(g2["dB"][..., :T], ref2["dB"], TOL_GRAD_SUM, "dB, first 64 steps")
    assert_close(g2["dC"][..., :T], ref2["dC"], TOL_GRAD_SUM, "dC, first 64 steps")
    assert_close(g2["du"][..., :T], ref2["du"], TOL_GRAD, "du, first 64 steps")


@pytest.mark.parametrize("name,grad", [("delta", "ddelta"), ("A", "dA"), ("B", "dB"), ("C", "dC"),
                                       ("z", "dz"), ("delta_bias", "ddelta_bias")])
def test_scan_bwd_directional_derivatives(name, grad):
    """<grad, v> against a central difference of sum(dy * y) through the CUDA
    forward, for a random direction v in one input (fp32 inputs): the two
    kernels agree with each other in every input, not only with the oracle."""
    inp = inputs.scan_inputs(1, 32, 160, 16, 1, "f32", seed=90, dskip="randn")
    dy = _dy((1, 32, 160), "f32", 91)
    g = _gpu_grad(inp, dy, poison=False)
    v = torch.randn(inp[name].shape, generator=torch.Generator().manual_seed(92))
    eps = 1e-2 if name in ("delta", "A", "z", "delta_bias") else 0.5

    def loss(t):
        x = {k: (_dev(u) if isinstance(u, torch.Tensor) else u) for k, u in inp.items()}
        x[name] = t.cuda()
        y, _ = binding.ssm_scan_fwd(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"],
                                    x["delta_bias"], True)
        return float((y.double().cpu() * dy.double()).sum())

    fd = (loss(inp[name] + eps * v) - loss(inp[name] - eps * v)) / (2 * eps)
    terms = g[grad].double().cpu() * v.double()
    an = float(terms.sum())
    # linear inputs (B, C): exact up to rounding; the others: O(eps^2) truncation.
    # The bound scales with sum |g v| as well as |<g, v>|: a random direction can
    # make the dot product cancel far below its terms (the difference quotient's
    # fp32 rounding does not cancel with it).
    assert abs(fd - an) <= 2e-3 * abs(an) + 1e-3 * float(terms.abs().sum()), (name, fd, an)


@pytest.mark.parametrize("shape", [(2, 96, 530, 2), (4, 5120, 256, 1)],
                         ids=["small", "640-blocks"])
@pytest.mark.parametrize("dt,out_dt", [("bf16", torch.float32), ("f32", torch.bfloat16)])
def test_scan_checkpoints_from_the_forward(dt, out_dt, shape):
    """ssm_scan_fwd with checkpoints gives the plain forward's y and final state
    bit for bit, and ssm_scan_bwd from those checkpoints gives the same bits as
    ssm_scan_bwd recomputing them.  The second shape has enough channel blocks
    for the forward kernels' 16-step prep groups (four CTAs per SM) in all three
    modes: plain, checkpointing and states only."""
    batch, dim, seqlen, ngroups = shape
    inp = inputs.scan_inputs(batch, dim, seqlen, 16, ngroups, dt, seed=140)
    x = {k: (_dev(v) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    h0 = torch.randn(batch, dim, 16, generator=torch.Generator().manual_seed(141)).cuda()
    args = (x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"], x["delta_bias"], True, h0)
    y0, f0 = binding.ssm_scan_fwd(*args, out_dtype=out_dt)
    ck = torch.full((binding.ssm_scan_checkpoint_bytes(batch, dim, seqlen) // 4,), float("nan"),
                    device="cuda")
    y1, f1 = binding.ssm_scan_fwd(*args, out_dtype=out_dt, checkpoints=ck)
    torch.cuda.synchronize()
    assert torch.equal(y0, y1) and torch.equal(f0, f1)
    assert not torch.isnan(ck).any()
    dy = _dy((batch, dim, seqlen), dt, 142).cuda()
    kw = dict(D=x["D"], z=x["z"], delta_bias=x["delta_bias"], delta_softplus=True,
              initial_state=h0)
    g0 = binding.ssm_scan_bwd(x["u"], x["delta"], x["A"], x["B"], x["C"], dy, **kw)
    g1 = binding.ssm_scan_bwd(x["u"], x["delta"], x["A"], x["B"], x["C"], dy, checkpoints=ck, **kw)
    torch.cuda.synchronize()
    for k, v in g0.items():
        if v is not None:
            assert torch.equal(v, g1[k]), k
