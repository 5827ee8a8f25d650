"""The allocation-free scan entry point (ssm_scan_fwd_noalloc).

It exists for callers that cannot allocate device memory when they run the
scan (an engine plug-in with a fixed memory budget, a real-time loop that may
not synchronise or wait on cudaMalloc, a C wrapper without an allocator), so
it keeps its scratch in a fixed array inside the library.  These tests call
it through the C ABI, twice in a row on the same problem (the second call
finds the array holding the first call's contents), and check that it gives
the bits of ssm_scan_fwd, which takes a caller-allocated workspace and runs
the same kernel with the same plan, and that it matches the oracle.  Its
device-side status (a look-back wait that ran out) is read back with
ssm_noalloc_last_status.

This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import pytest
import torch

import oracle
from state_space_model_selective_gb300 import binding, inputs
from tests.helpers import TOL_BF16, TOL_F32, assert_close

pytestmark = pytest.mark.gpu

OK, TIMEOUT, WORKSPACE = 0, 7, 6


def _dev(inp):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


# small_f32: one 128-step chunk of the sequence-parallel scan (no carry in the
# array); seqpar_lookback: 8 chunks joined by the look-back through the array;
# chained_bf16: 4 x 5120 channels in 640 blocks, more than the resident CTA
# slots of a 152-SM part, so the chained scan cuts L = 256 into chunks that
# carry their state through the array (3.9 MB of the 4 MiB)
CASES = [((2, 64, 128), "f32"), ((1, 256, 1000), "f32"), ((4, 5120, 256), "bf16")]
IDS = ["small_f32", "seqpar_lookback", "chained_bf16"]


@pytest.mark.parametrize("shape,dtype", CASES, ids=IDS)
def test_noalloc_gives_workspace_entry_bits_twice(shape, dtype):
    batch, dim, seqlen = shape
    inp = inputs.scan_inputs(batch, dim, seqlen, 16, 1, dtype, seed=77)
    d = _dev(inp)
    args = (d["u"], d["delta"], d["A"], d["B"], d["C"])
    kw = dict(D=d["D"], z=d["z"], delta_bias=d["delta_bias"], delta_softplus=True)
    y_ref, fs_ref = binding.ssm_scan_fwd(*args, out_dtype=torch.float32, **kw)
    for call in range(2):
        y = torch.full((batch, dim, seqlen), float("nan"), device="cuda")
        fs = torch.full((batch, dim, 16), float("nan"), device="cuda")
        binding.ssm_scan_fwd_noalloc(*args, y=y, final_state=fs, **kw)
        assert binding.ssm_noalloc_last_status() == OK
        assert torch.equal(y, y_ref), f"y, call {call}"
        assert torch.equal(fs, fs_ref), f"final_state, call {call}"
    if batch * dim <= 256:  # against the oracle too (small enough to run whole)
        yo, fo = oracle.scan(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"],
                             inp["z"], inp["delta_bias"], True)
        tol = TOL_F32 if dtype == "f32" else TOL_BF16
        assert_close(y, yo, tol, "y vs oracle")
        assert_close(fs, fo, tol, "final_state vs oracle")


@pytest.mark.parametrize("shape,dtype", CASES[1:], ids=IDS[1:])
def test_noalloc_reports_a_lookback_timeout(shape, dtype):
    """A wait that runs out (chunk 0 withholds its publish) is reported by
    ssm_noalloc_last_status; the next call is clean and gives the same bits.
    A timeout can only occur where chunks carry state through the array, so
    this also shows that both cases run as carried chunks."""
    batch, dim, seqlen = shape
    d = _dev(inputs.scan_inputs(batch, dim, seqlen, 16, 1, dtype, seed=78))
    args = (d["u"], d["delta"], d["A"], d["B"], d["C"])
    kw = dict(D=d["D"], z=d["z"], delta_bias=d["delta_bias"], delta_softplus=True)
    y = torch.empty((batch, dim, seqlen), device="cuda")
    fs = torch.empty((batch, dim, 16), device="cuda")
    binding.ssm_scan_fwd_noalloc(*args, y=y, final_state=fs, **kw)
    assert binding.ssm_noalloc_last_status() == OK
    y_ok, fs_ok = y.clone(), fs.clone()
    try:
        binding.ssm_debug_set_lookback(True, 2000)
        binding.ssm_scan_fwd_noalloc(*args, y=y, final_state=fs, **kw)
        status = binding.ssm_noalloc_last_status()
    finally:
        binding.ssm_debug_set_lookback()
    assert status == TIMEOUT
    binding.ssm_scan_fwd_noalloc(*args, y=y, final_state=fs, **kw)
    assert binding.ssm_noalloc_last_status() == OK
    assert torch.equal(y, y_ok) and torch.equal(fs, fs_ok)


def test_noalloc_rejects_problem_beyond_scratch():
    """batch 4, 5120 channels, L 16384 splits into chained chunks whose
    carried states need more than the 4 MiB of built-in scratch."""
    batch, dim, seqlen = 4, 5120, 16384
    u = torch.empty(batch, dim, seqlen, dtype=torch.bfloat16, device="cuda")
    Bm = torch.empty(batch, 1, 16, seqlen, dtype=torch.bfloat16, device="cuda")
    A = -torch.ones(dim, 16, device="cuda")
    y = torch.empty(batch, dim, seqlen, device="cuda")
    with pytest.raises(binding.SSMError) as e:
        binding.ssm_scan_fwd_noalloc(u, u, A, Bm, Bm, y=y)
    assert e.value.status == WORKSPACE
