"""The scan's bounded look-back wait, made to run out without a fault.

When the channel blocks outnumber the resident CTA slots the scan runs the
sequence as chunks chained through the state: chunk c of a block polls a flag
chunk c - 1 publishes (the decoupled look-back of Merrill and Garland's
single-pass prefix scan).  With chunk 0's publish withheld, chunk 1 polls a flag
that nothing sets; the wait must give up after its poll limit, record
SSM_ERR_TIMEOUT in the workspace and let the kernel finish, and the context must
stay usable: the next scan on it gives the bits of a clean run."""
import time

import pytest
import torch

from state_space_model_selective_gb300 import binding, inputs

pytestmark = pytest.mark.gpu

OK, TIMEOUT = 0, 7


def _scan(x, ws):
    return binding.ssm_scan_fwd(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"],
                                x["delta_bias"], True, out_dtype=torch.float32, workspace=ws)


def test_lookback_wait_runs_out_and_reports_timeout():
    # 4 x 5120 channels in 32-channel blocks: 640 blocks, more than the resident
    # CTA slots of a 152-SM part, so the 8 tiles of L = 512 run as chained chunks
    batch, dim, seqlen = 4, 5120, 512
    x = inputs.scan_inputs(batch, dim, seqlen, 16, 1, "bf16", seed=150, device="cuda")
    ws = torch.empty(binding.ssm_scan_workspace_bytes(batch, dim, seqlen, 16, 1),
                     dtype=torch.uint8, device="cuda")
    y_ref, fs_ref = _scan(x, ws)
    assert binding.ssm_last_device_status(ws) == OK
    try:
        binding.ssm_debug_set_lookback(True, 2000)
        t0 = time.perf_counter()
        _scan(x, ws)
        status = binding.ssm_last_device_status(ws)
        elapsed = time.perf_counter() - t0
    finally:
        binding.ssm_debug_set_lookback()
    assert status == TIMEOUT
    assert elapsed < 0.5, elapsed  # the shortened limit, not the default of about a second
    y, fs = _scan(x, ws)
    assert binding.ssm_last_device_status(ws) == OK
    assert torch.equal(y, y_ref) and torch.equal(fs, fs_ref)


def test_lookback_custom_limit_without_withheld_publish_is_clean():
    """A custom poll limit alone does not trip: every chunk publishes, the
    waits see their flags, and the result is the clean run's bits."""
    batch, dim, seqlen = 4, 5120, 512
    x = inputs.scan_inputs(batch, dim, seqlen, 16, 1, "bf16", seed=151, device="cuda")
    ws = torch.empty(binding.ssm_scan_workspace_bytes(batch, dim, seqlen, 16, 1),
                     dtype=torch.uint8, device="cuda")
    y_ref, fs_ref = _scan(x, ws)
    try:
        binding.ssm_debug_set_lookback(False, 1 << 20)
        y, fs = _scan(x, ws)
        status = binding.ssm_last_device_status(ws)
    finally:
        binding.ssm_debug_set_lookback()
    assert status == OK
    assert torch.equal(y, y_ref) and torch.equal(fs, fs_ref)


def test_seqpar_lookback_wait_runs_out_and_reports_timeout():
    """The sequence-parallel scan's look-back: chunk 0 withholds its inclusive
    state, so chunk 1 polls a flag that never reaches it; the bounded wait
    records SSM_ERR_TIMEOUT and the kernel finishes; the next scan on the same
    context gives the clean run's bits."""
    batch, dim, seqlen = 1, 64, 1024  # 64 channels: the sequence-parallel scan, 8 chunks
    x = inputs.scan_inputs(batch, dim, seqlen, 16, 1, "f32", seed=152, device="cuda")
    ws = torch.empty(binding.ssm_scan_workspace_bytes(batch, dim, seqlen, 16, 1),
                     dtype=torch.uint8, device="cuda")
    y_ref, fs_ref = _scan(x, ws)
    assert binding.ssm_last_device_status(ws) == OK
    try:
        binding.ssm_debug_set_lookback(True, 2000)
        t0 = time.perf_counter()
        _scan(x, ws)
        status = binding.ssm_last_device_status(ws)
        elapsed = time.perf_counter() - t0
    finally:
        binding.ssm_debug_set_lookback()
    assert status == TIMEOUT
    assert elapsed < 0.5, elapsed
    y, fs = _scan(x, ws)
    assert binding.ssm_last_device_status(ws) == OK
    assert torch.equal(y, y_ref) and torch.equal(fs, fs_ref)
