"""The stored tiny scan problem (tests/golden/scan_tiny.json, written by
tests/golden/make_golden.py from the oracle): the oracle still reproduces it,
and the CUDA scan matches it in fp32 and bf16 inputs (the values are exact
in bf16)."""
import json
import os

import numpy as np
import pytest

import oracle
from tests.helpers import TOL_F32, assert_close

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "scan_tiny.json")


def _load():
    d = json.load(open(GOLDEN))
    return {k: np.asarray(v, dtype=np.float64) for k, v in d.items() if k != "delta_softplus"}


def test_oracle_reproduces_golden():
    g = _load()
    y, hs = oracle.scan(g["u"], g["delta"], g["A"], g["B"], g["C"], g["D"], g["z"],
                        g["delta_bias"], True)
    np.testing.assert_allclose(y, g["y"], rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(hs, g["final_state"], rtol=1e-14, atol=1e-15)


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_cuda_scan_matches_golden(dtype):
    import torch
    from state_space_model_selective_gb300 import binding
    g = _load()
    td = torch.float32 if dtype == "f32" else torch.bfloat16
    t = {k: torch.tensor(g[k]).to(td).contiguous().cuda() for k in ("u", "delta", "B", "C", "z")}
    f = {k: torch.tensor(g[k]).float().contiguous().cuda() for k in ("A", "D", "delta_bias")}
    y, hs = binding.ssm_scan_fwd(t["u"], t["delta"], f["A"], t["B"], t["C"], f["D"], t["z"],
                                 f["delta_bias"], True, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert_close(y, g["y"], TOL_F32, "y")
    assert_close(hs, g["final_state"], TOL_F32, "final_state")
