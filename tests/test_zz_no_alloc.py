"""The allocation-free scan entry point (ssm_scan_fwd_noalloc).

It exists for callers that cannot allocate device memory when they run the
scan (an engine plug-in with a fixed memory budget, a real-time loop that may
not synchronise or wait on cudaMalloc, a C wrapper without an allocator), so
it keeps its scratch in a fixed array inside the library.  These tests call
it through the C ABI, twice in a row on the same problem (the second call
finds the array holding the first call's contents), and compare its output
with that of ssm_scan_fwd, which takes a caller-allocated workspace.

This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import pytest
import torch

from state_space_model_selective_gb300 import binding, inputs
from tests.helpers import TOL_BF16, TOL_F32, assert_close

pytestmark = pytest.mark.gpu

WORKSPACE = 6  # SSM_ERR_WORKSPACE


def _dev(inp):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


@pytest.mark.parametrize("shape,dtype", [((2, 64, 200), "f32"), ((4, 4096, 256), "bf16")],
                         ids=["small_f32", "chained_chunks_bf16"])
def test_noalloc_matches_workspace_entry_twice(shape, dtype):
    batch, dim, seqlen = shape
    d = _dev(inputs.scan_inputs(batch, dim, seqlen, 16, 1, dtype, seed=77))
    args = (d["u"], d["delta"], d["A"], d["B"], d["C"])
    kw = dict(D=d["D"], z=d["z"], delta_bias=d["delta_bias"], delta_softplus=True)
    y_ref, fs_ref = binding.ssm_scan_fwd(*args, out_dtype=torch.float32, **kw)
    tol = TOL_F32 if dtype == "f32" else TOL_BF16
    for call in range(2):
        y = torch.full((batch, dim, seqlen), float("nan"), device="cuda")
        fs = torch.full((batch, dim, 16), float("nan"), device="cuda")
        binding.ssm_scan_fwd_noalloc(*args, y=y, final_state=fs, **kw)
        torch.cuda.synchronize()
        assert_close(y, y_ref, tol, f"y, call {call}")
        assert_close(fs, fs_ref, tol, f"final_state, call {call}")


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
