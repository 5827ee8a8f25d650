"""Out-of-bounds writes and writes to inputs, caught without a sanitizer.

Every output buffer of every entry point is a view into a larger allocation
with 64 guard elements before and after it, filled with a canary value; the
outputs themselves start as NaN.  After each call the guards must still hold
the canary (no write outside the output), no output element may still be NaN
(every element written), and every input must be bit-for-bit unchanged (inputs
are never written, except the decode steps' state, which is itself guarded).
Shapes are small and ragged: scan lengths that are not a multiple of any tile,
chunked lengths that end half way through a 128-row block (a whole number of
chunks, as the chunked forms require), a decode head dimension that is not a
multiple of 32, several groups."""
import math

import pytest
import torch

from state_space_model_selective_gb300 import binding, inputs

pytestmark = pytest.mark.gpu

GUARD = 64  # elements: 256 B of fp32, 128 B of bf16, so every view stays 16-byte aligned
CANARY = -7.25e33


class Guarded:
    """A tensor of ``shape`` inside a buffer with canary guards on both sides."""

    def __init__(self, shape, dtype=torch.float32, fill=float("nan")):
        n = math.prod(shape)
        self.buf = torch.full((n + 2 * GUARD,), CANARY, dtype=dtype, device="cuda")
        self.ref = torch.full((GUARD,), CANARY, dtype=dtype, device="cuda")
        self.t = self.buf[GUARD:GUARD + n].view(shape)
        if isinstance(fill, torch.Tensor):
            self.t.copy_(fill)
        else:
            self.t.fill_(fill)

    def check(self, name, written=True):
        torch.cuda.synchronize()
        assert torch.equal(self.buf[:GUARD], self.ref), f"{name}: write before the buffer"
        assert torch.equal(self.buf[-GUARD:], self.ref), f"{name}: write past the buffer"
        if written:
            assert not torch.isnan(self.t).any(), f"{name}: elements left unwritten"


def _cuda(d):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


def _snapshot(d):
    return {k: v.clone() for k, v in d.items() if isinstance(v, torch.Tensor)}


def _unchanged(before, d):
    torch.cuda.synchronize()
    for k, v in before.items():
        assert torch.equal(v, d[k]), f"input {k} was written"


def _guarded_grads(fn, **kw):
    """Calls a gradient entry point once for its output shapes, then again with
    every output guarded; the guarded call must give the same bits."""
    g0 = fn(**kw)
    outs = {k: Guarded(tuple(v.shape)) for k, v in g0.items() if v is not None}
    g1 = fn(out={k: o.t for k, o in outs.items()}, **kw)
    for k, o in outs.items():
        o.check(k)
        assert torch.equal(g1[k], g0[k]), k
    return g1


@pytest.mark.parametrize("dt,out_dt", [("bf16", torch.float32), ("f32", torch.bfloat16)])
def test_scan_fwd_and_checkpoints_stay_in_bounds(dt, out_dt):
    batch, dim, seqlen, ngroups = 2, 96, 333, 2
    x = _cuda(inputs.scan_inputs(batch, dim, seqlen, 16, ngroups, dt, seed=170))
    h0 = 0.5 * torch.randn(batch, dim, 16, generator=torch.Generator().manual_seed(171)).cuda()
    before = _snapshot(x)
    y = Guarded((batch, dim, seqlen), out_dt)
    fs = Guarded((batch, dim, 16))
    ck = Guarded((binding.ssm_scan_checkpoint_bytes(batch, dim, seqlen) // 4,))
    binding.ssm_scan_fwd(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"],
                         x["delta_bias"], True, h0, out_dtype=out_dt, y=y.t, final_state=fs.t,
                         checkpoints=ck.t)
    y.check("y"), fs.check("final_state"), ck.check("checkpoints")
    _unchanged(before, x)
    y2 = Guarded((batch, dim, seqlen), out_dt)
    fs2 = Guarded((batch, dim, 16))
    binding.ssm_scan_fwd_noalloc(x["u"], x["delta"], x["A"], x["B"], x["C"], y2.t, fs2.t,
                                 x["D"], x["z"], x["delta_bias"], True, h0)
    y2.check("y (no-alloc)"), fs2.check("final_state (no-alloc)")
    assert torch.equal(y2.t, y.t) and torch.equal(fs2.t, fs.t)


def test_scan_bwd_stays_in_bounds():
    batch, dim, seqlen, ngroups = 2, 64, 300, 2
    x = _cuda(inputs.scan_inputs(batch, dim, seqlen, 16, ngroups, "bf16", seed=172))
    h0 = 0.5 * torch.randn(batch, dim, 16, generator=torch.Generator().manual_seed(173)).cuda()
    dy = torch.randn(batch, dim, seqlen, generator=torch.Generator().manual_seed(174)) \
        .to(torch.bfloat16).cuda()
    before = _snapshot(x)
    _guarded_grads(binding.ssm_scan_bwd, u=x["u"], delta=x["delta"], A=x["A"], B=x["B"],
                   C=x["C"], dy=dy, D=x["D"], z=x["z"], delta_bias=x["delta_bias"],
                   delta_softplus=True, initial_state=h0)
    _unchanged(before, x)


def test_ssd_fwd_bwd_stay_in_bounds():
    batch, seqlen, nheads, headdim, dstate, ngroups = 2, 192, 4, 64, 128, 2
    x = _cuda(inputs.ssd_inputs(batch, seqlen, nheads, headdim, dstate, ngroups, "bf16",
                                seed=175))
    h0 = 0.1 * torch.randn(batch, nheads, headdim, dstate,
                           generator=torch.Generator().manual_seed(176)).cuda()
    before = _snapshot(x)
    y = Guarded((batch, seqlen, nheads, headdim))
    fs = Guarded((batch, nheads, headdim, dstate))
    bs = Guarded((binding.ssd_chunked_checkpoint_bytes(batch, seqlen, nheads, headdim,
                                                       dstate) // 4,))
    binding.ssd_chunked_fwd(x["x"], x["dt"], x["A_head"], x["B"], x["C"], 64,
                            out_dtype=torch.float32, y=y.t, final_state=fs.t, initial_state=h0,
                            block_states=bs.t)
    y.check("y"), fs.check("final_state"), bs.check("block_states")
    _unchanged(before, x)
    dy = torch.randn(batch, seqlen, nheads, headdim,
                     generator=torch.Generator().manual_seed(177)).to(torch.bfloat16).cuda()
    _guarded_grads(binding.ssd_chunked_bwd, x=x["x"], dt=x["dt"], A_head=x["A_head"], B=x["B"],
                   C=x["C"], dy=dy, chunk=64, initial_state=h0, block_states=bs.t)
    _unchanged(before, x)


def test_mamba3_fwd_bwd_stay_in_bounds():
    batch, seqlen, nheads, headdim, dstate, ngroups = 2, 192, 4, 64, 128, 2
    x = _cuda(inputs.mamba3_inputs(batch, seqlen, nheads, headdim, dstate, ngroups, "bf16",
                                   seed=178))
    before = _snapshot(x)
    y = Guarded((batch, seqlen, nheads, headdim))
    fs = Guarded((batch, nheads, headdim, dstate))
    bs = Guarded((binding.ssd_chunked_checkpoint_bytes(batch, seqlen, nheads, headdim,
                                                       dstate) // 4,))
    binding.ssd_mamba3_fwd(x["x"], x["dt"], x["lam"], x["A_head"], x["B"], x["C"], 64,
                           out_dtype=torch.float32, y=y.t, final_state=fs.t,
                           initial_state=x["h0"], prev_B=x["prev_B"], prev_x=x["prev_x"],
                           block_states=bs.t)
    y.check("y"), fs.check("final_state"), bs.check("block_states")
    _unchanged(before, x)
    dy = torch.randn(batch, seqlen, nheads, headdim,
                     generator=torch.Generator().manual_seed(179)).to(torch.bfloat16).cuda()
    _guarded_grads(binding.ssd_mamba3_bwd, x=x["x"], dt=x["dt"], lam=x["lam"],
                   A_head=x["A_head"], B=x["B"], C=x["C"], dy=dy, chunk=64,
                   initial_state=x["h0"], prev_B=x["prev_B"], prev_x=x["prev_x"],
                   block_states=bs.t)
    _unchanged(before, x)


def test_mamba3_mimo_fwd_bwd_stay_in_bounds():
    batch, seqlen, rank, nheads, headdim, dstate, ngroups = 2, 48, 4, 4, 64, 128, 2
    x = _cuda(inputs.mamba3_mimo_inputs(batch, seqlen, rank, nheads, headdim, dstate, ngroups,
                                        "bf16", seed=180))
    before = _snapshot(x)
    y = Guarded((batch, seqlen, rank, nheads, headdim))
    fs = Guarded((batch, nheads, headdim, dstate))
    bs = Guarded((binding.ssd_chunked_checkpoint_bytes(batch, seqlen * rank, nheads, headdim,
                                                       dstate) // 4,))
    binding.ssd_mamba3_mimo_fwd(x["x"], x["dt"], x["lam"], x["A_head"], x["B"], x["C"], 16,
                                out_dtype=torch.float32, y=y.t, final_state=fs.t,
                                initial_state=x["h0"], prev_B=x["prev_B"], prev_x=x["prev_x"],
                                block_states=bs.t)
    y.check("y"), fs.check("final_state"), bs.check("block_states")
    _unchanged(before, x)
    dy = torch.randn(batch, seqlen, rank, nheads, headdim,
                     generator=torch.Generator().manual_seed(181)).to(torch.bfloat16).cuda()
    _guarded_grads(binding.ssd_mamba3_mimo_bwd, x=x["x"], dt=x["dt"], lam=x["lam"],
                   A_head=x["A_head"], B=x["B"], C=x["C"], dy=dy, chunk=16,
                   initial_state=x["h0"], prev_B=x["prev_B"], prev_x=x["prev_x"],
                   block_states=bs.t)
    _unchanged(before, x)


@pytest.mark.parametrize("form", ["mamba2", "mamba3", "mimo"])
def test_decode_steps_stay_in_bounds(form):
    batch, nheads, headdim, dstate, ngroups, rank = 3, 4, 100, 128, 2, 4
    g = torch.Generator().manual_seed(182)
    r = (lambda *s: torch.randn(*s, generator=g).cuda())  # noqa: E731
    state = Guarded((batch, nheads, headdim, dstate), fill=0.1 * r(batch, nheads, headdim, dstate))
    A = -(1.0 + 15.0 * torch.rand(nheads, generator=g)).cuda()
    D = r(nheads)
    dt = torch.nn.functional.softplus(r(batch, nheads) - 4.0)
    lam = torch.sigmoid(r(batch, nheads))
    if form == "mimo":
        xs = {"x": r(batch, rank, nheads, headdim), "z": r(batch, rank, nheads, headdim),
              "prev_x": r(batch, rank, nheads, headdim), "B": r(batch, rank, ngroups, dstate),
              "C": r(batch, rank, ngroups, dstate), "prev_B": r(batch, rank, ngroups, dstate)}
        y = Guarded((batch, rank, nheads, headdim))
    else:
        xs = {"x": r(batch, nheads, headdim), "z": r(batch, nheads, headdim),
              "prev_x": r(batch, nheads, headdim), "B": r(batch, ngroups, dstate),
              "C": r(batch, ngroups, dstate), "prev_B": r(batch, ngroups, dstate)}
        y = Guarded((batch, nheads, headdim))
    xs.update(A=A, D=D, dt=dt, lam=lam)
    before = _snapshot(xs)
    if form == "mamba2":
        binding.ssm_decode_step(state.t, xs["x"], dt, A, xs["B"], xs["C"], D, xs["z"], y=y.t)
    elif form == "mamba3":
        binding.ssm_decode_step_mamba3(state.t, xs["prev_B"], xs["prev_x"], xs["x"], dt, lam, A,
                                       xs["B"], xs["C"], D, xs["z"], y=y.t)
    else:
        binding.ssm_decode_step_mamba3_mimo(state.t, xs["prev_B"], xs["prev_x"], xs["x"], dt,
                                            lam, A, xs["B"], xs["C"], D, xs["z"], y=y.t)
    state.check("state"), y.check("y")
    _unchanged(before, xs)
