"""Parity of the Mamba-3 MIMO gradient (ssd_mamba3_mimo_bwd, through the C ABI)
with the fp64 oracle's reverse-mode derivative of the rank-R recurrence
("Mamba-3 NKI Kernels for AWS Neuron", section "Kernel details",
mamba3_mimo_ssd_kernel).

Tolerance: the SSD gradient's (1e-4 normwise per element, 5e-4 for dA_head),
the call being the tensor-core SSD gradient over sub-tokens plus fp32
elementwise kernels.
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


def _case(batch, seqlen, rank, nheads, ngroups, seed, h0, prev, dfinal):
    inp = inputs.mamba3_mimo_inputs(batch, seqlen, rank, nheads, 64, 128, ngroups, "bf16",
                                    seed=seed)
    gen = torch.Generator().manual_seed(seed + 1)
    dy = torch.randn(batch, seqlen, rank, nheads, 64, generator=gen).to(torch.bfloat16)
    df = torch.randn(batch, nheads, 64, 128, generator=gen) if dfinal else None
    if not h0:
        inp["h0"] = None
    if not prev:
        inp["prev_B"] = inp["prev_x"] = None
    return inp, dy, df


def _gpu(inp, dy, dfinal, ws_fill=0xAB):
    c = lambda t: None if t is None else t.cuda()
    batch, seqlen, rank, nheads, _ = inp["x"].shape
    need = binding.ssd_mamba3_mimo_bwd_workspace_bytes(batch, seqlen, rank, nheads, 64, 128,
                                                       inp["B"].shape[3])
    ws = torch.full((max(need, 256),), ws_fill, dtype=torch.uint8, device="cuda")
    g = binding.ssd_mamba3_mimo_bwd(c(inp["x"]), c(inp["dt"]), c(inp["lam"]), c(inp["A_head"]),
                                    c(inp["B"]), c(inp["C"]), c(dy), None, c(inp["h0"]),
                                    c(inp["prev_B"]), c(inp["prev_x"]), c(dfinal), workspace=ws)
    torch.cuda.synchronize()
    if seqlen > 0 and batch * nheads > 0:
        assert binding.ssm_last_device_status(ws) == 0
    return g


def _ref(inp, dy, dfinal):
    return oracle.mamba3_mimo_bwd(inp["x"], inp["dt"], inp["lam"], inp["A_head"], inp["B"],
                                  inp["C"], dy, inp["h0"], inp["prev_B"], inp["prev_x"], dfinal)


CASES = [  # batch, seqlen (steps), rank, nheads, ngroups, initial state, previous token, dfinal
    (1, 16, 4, 2, 1, False, False, False),   # 64 sub-tokens: one partial block
    (2, 32, 4, 4, 1, True, True, True),      # one full 128-row block
    (2, 64, 4, 4, 2, True, True, True),      # two blocks, 2 groups
    (1, 80, 4, 2, 1, False, True, True),     # 320 rows: two and a half blocks
    (2, 32, 2, 4, 4, True, True, False),     # rank 2: 64 rows, one head per group
    (2, 96, 2, 6, 3, True, True, True),      # rank 2: 192 rows, 3 groups
]


@pytest.mark.parametrize("case", CASES, ids=[
    f"B{c[0]}L{c[1]}R{c[2]}H{c[3]}G{c[4]}{'s' if c[5] else ''}{'p' if c[6] else ''}"
    f"{'f' if c[7] else ''}" for c in CASES])
def test_mimo_bwd_matches_oracle(case):
    batch, seqlen, rank, nheads, ngroups, h0, prev, df = case
    inp, dy, dfinal = _case(batch, seqlen, rank, nheads, ngroups, 600 + seqlen + rank, h0, prev,
                            df)
    g = _gpu(inp, dy, dfinal)
    ref = _ref(inp, dy, dfinal)
    for key, rkey, tol in KEYS:
        if ref[rkey] is None:
            assert g[key] is None, key
            continue
        assert_close(g[key], ref[rkey], tol, key)


def test_mimo_bwd_rank_one_is_the_siso_gradient():
    """Rank one through the MIMO entry point equals ssd_mamba3_bwd up to rounding."""
    inp, dy, dfinal = _case(2, 128, 1, 4, 2, 650, True, True, True)
    g = _gpu(inp, dy, dfinal)
    c = lambda t: t.cuda()
    s = binding.ssd_mamba3_bwd(c(inp["x"][:, :, 0]), c(inp["dt"]), c(inp["lam"]),
                               c(inp["A_head"]), c(inp["B"][:, :, 0]), c(inp["C"][:, :, 0]),
                               c(dy[:, :, 0]), 64, c(inp["h0"]), c(inp["prev_B"][:, 0]),
                               c(inp["prev_x"][:, 0]), c(dfinal))
    torch.cuda.synchronize()
    for key in ("dx", "dB", "dC"):
        assert_close(g[key][:, :, 0], s[key].double().cpu(), 1e-6, key)
    for key in ("dprev_B", "dprev_x"):
        assert_close(g[key][:, 0], s[key].double().cpu(), 1e-6, key)
    for key in ("ddt", "dlam", "dA_head", "dinitial_state"):
        assert_close(g[key], s[key].double().cpu(), 1e-6, key)


def test_mimo_bwd_deterministic_and_workspace_independent():
    inp, dy, dfinal = _case(2, 64, 4, 4, 1, 660, True, True, True)
    g1 = _gpu(inp, dy, dfinal, ws_fill=0x00)
    g2 = _gpu(inp, dy, dfinal, ws_fill=0xFF)
    for k, v in g1.items():
        if v is not None:
            assert torch.equal(v, g2[k]), k


def test_mimo_bwd_empty_sequence():
    inp, dy, dfinal = _case(2, 0, 4, 4, 1, 670, False, True, True)
    g = _gpu(inp, dy, dfinal)
    assert torch.count_nonzero(g["dA_head"]).item() == 0
    assert torch.equal(g["dinitial_state"].cpu(), dfinal)
    assert torch.count_nonzero(g["dprev_B"]).item() == 0
    assert torch.count_nonzero(g["dprev_x"]).item() == 0


@pytest.mark.parametrize("name,grad", [("dt", "ddt"), ("lam", "dlam")])
def test_mimo_bwd_directional_derivatives(name, grad):
    """<grad, v> against a central difference of sum(dy y) + sum(dfinal final_state)
    through the CUDA forward (ssd_mamba3_mimo_fwd) in dt and lambda."""
    inp, dy, dfinal = _case(1, 64, 4, 4, 1, 680, True, True, True)
    g = _gpu(inp, dy, dfinal)
    base = inp[name]
    v = torch.randn(base.shape, generator=torch.Generator().manual_seed(681)) * base.abs()
    eps = 1e-2

    def loss(t):
        d = {k: (None if u is None else u.cuda()) for k, u in inp.items()}
        d[name] = t.cuda()
        y, fs = binding.ssd_mamba3_mimo_fwd(d["x"], d["dt"], d["lam"], d["A_head"], d["B"],
                                            d["C"], 16, out_dtype=torch.float32,
                                            initial_state=d["h0"], prev_B=d["prev_B"],
                                            prev_x=d["prev_x"])
        return float((y.double().cpu() * dy.double()).sum() +
                     (fs.double().cpu() * dfinal.double()).sum())

    fd = (loss(base + eps * v) - loss(base - eps * v)) / (2 * eps)
    terms = g[grad].double().cpu() * v.double()
    an = float(terms.sum())
    assert abs(fd - an) <= 5e-3 * abs(an) + 1e-3 * float(terms.abs().sum()), (name, fd, an)


def test_mimo_block_states_from_the_forward():
    """ssd_mamba3_mimo_fwd keeping block states gives the plain forward's y and final
    state bit for bit, and ssd_mamba3_mimo_bwd from those states gives the same bits as
    ssd_mamba3_mimo_bwd recomputing them."""
    batch, seqlen, rank, nheads = 2, 80, 4, 4
    inp, dy, dfinal = _case(batch, seqlen, rank, nheads, 2, 690, True, True, True)
    d = {k: (None if v is None else v.cuda()) for k, v in inp.items()}
    args = (d["x"], d["dt"], d["lam"], d["A_head"], d["B"], d["C"])
    kw = dict(initial_state=d["h0"], prev_B=d["prev_B"], prev_x=d["prev_x"])
    y0, f0 = binding.ssd_mamba3_mimo_fwd(*args, 16, out_dtype=torch.float32, **kw)
    bs = torch.full((binding.ssd_chunked_checkpoint_bytes(batch, seqlen * rank, nheads) // 4,),
                    float("nan"), device="cuda")
    y1, f1 = binding.ssd_mamba3_mimo_fwd(*args, 16, out_dtype=torch.float32, block_states=bs,
                                         **kw)
    torch.cuda.synchronize()
    assert torch.equal(y0, y1) and torch.equal(f0, f1)
    assert not torch.isnan(bs).any()
    g0 = binding.ssd_mamba3_mimo_bwd(*args, dy.cuda(), 16, d["h0"], d["prev_B"], d["prev_x"],
                                     dfinal.cuda())
    g1 = binding.ssd_mamba3_mimo_bwd(*args, dy.cuda(), 16, d["h0"], d["prev_B"], d["prev_x"],
                                     dfinal.cuda(), block_states=bs)
    torch.cuda.synchronize()
    for k, v in g0.items():
        if v is not None:
            assert torch.equal(v, g1[k]), k
