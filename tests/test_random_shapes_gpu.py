"""Parity with the fp64 oracle on seeded random shapes: channel counts that are no
multiple of any tile, lengths around tile and chunk boundaries, mixed groups and
the optional inputs switched on and off.  The shape lists are drawn once from a
fixed seed, so every run checks the same problems."""
import numpy as np
import pytest
import torch

import oracle
from state_space_model_selective_gb300 import binding, inputs
from tests.helpers import TOL_BF16, TOL_F32, assert_close

pytestmark = pytest.mark.gpu


def _draw_scan(n, seed):
    rng = np.random.default_rng(seed)
    cases = []
    for _ in range(n):
        ngroups = int(rng.integers(1, 5))
        cases.append(dict(batch=int(rng.integers(1, 5)), ngroups=ngroups,
                          dim=ngroups * int(rng.integers(1, 121)),
                          seqlen=int(rng.choice([1, 2, 7, 31, 63, 64, 65, 127, 128, 129,
                                                 191, 256, 300, 513, 600])),
                          dtype=str(rng.choice(["f32", "bf16"])), gate=bool(rng.integers(2)),
                          dskip=str(rng.choice(["none", "ones", "randn"])),
                          softplus=bool(rng.integers(2)), h0=bool(rng.integers(2))))
    return cases


SCAN_CASES = _draw_scan(16, 2024)


@pytest.mark.parametrize("path", [(0, 0), (1, 0)], ids=["planned", "chained"])
@pytest.mark.parametrize("case", SCAN_CASES,
                         ids=[f"B{c['batch']}D{c['dim']}L{c['seqlen']}G{c['ngroups']}{c['dtype']}"
                              for c in SCAN_CASES])
def test_scan_random_shapes(case, path):
    c = case
    inp = inputs.scan_inputs(c["batch"], c["dim"], c["seqlen"], 16, c["ngroups"], c["dtype"],
                             seed=c["dim"] * 7 + c["seqlen"], gate=c["gate"], dskip=c["dskip"])
    inp["delta_softplus"] = c["softplus"]
    if not c["softplus"]:  # without softplus, delta + bias must stay positive
        inp["delta"] = (inp["delta"].float().abs() * 0.1).to(inp["delta"].dtype)
        inp["delta_bias"] = torch.full_like(inp["delta_bias"], 0.01)
    h0 = (torch.randn(c["batch"], c["dim"], 16, generator=torch.Generator().manual_seed(c["dim"]))
          * 0.5 if c["h0"] else None)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    binding.ssm_debug_set_scan_path(*path)
    try:
        y, fs = binding.ssm_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"],
                                     d["delta_bias"], c["softplus"],
                                     None if h0 is None else h0.cuda(), out_dtype=torch.float32)
        torch.cuda.synchronize()
    finally:
        binding.ssm_debug_set_scan_path()
    y_ref, fs_ref = oracle.scan(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"],
                                inp["z"], inp["delta_bias"], c["softplus"], h0)
    tol = TOL_F32 if c["dtype"] == "f32" else TOL_BF16
    assert_close(y, y_ref, tol, "y")
    assert_close(fs, fs_ref, tol, "final_state")


def _draw_ssd(n, seed):
    rng = np.random.default_rng(seed)
    cases = []
    for _ in range(n):
        ngroups = int(rng.integers(1, 4))
        cases.append(dict(batch=int(rng.integers(1, 4)), seqlen=64 * int(rng.integers(1, 11)),
                          ngroups=ngroups, nheads=ngroups * int(rng.integers(1, 4)),
                          h0=bool(rng.integers(2)), prev=bool(rng.integers(2))))
    return cases


SSD_CASES = _draw_ssd(8, 2025)


@pytest.mark.parametrize("case", SSD_CASES,
                         ids=[f"B{c['batch']}L{c['seqlen']}H{c['nheads']}G{c['ngroups']}"
                              for c in SSD_CASES])
def test_ssd_random_shapes(case):
    c = case
    inp = inputs.ssd_inputs(c["batch"], c["seqlen"], c["nheads"], 64, 128, c["ngroups"], "bf16",
                            seed=300 + c["seqlen"] + c["nheads"])
    h0 = (torch.randn(c["batch"], c["nheads"], 64, 128,
                      generator=torch.Generator().manual_seed(c["seqlen"])) * 0.3
          if c["h0"] else None)
    d = {k: v.cuda() for k, v in inp.items()}
    y = torch.full(d["x"].shape, float("nan"), device="cuda")
    fs = torch.full((c["batch"], c["nheads"], 64, 128), float("nan"), device="cuda")
    binding.ssd_chunked_fwd(d["x"], d["dt"], d["A_head"], d["B"], d["C"], 64,
                            out_dtype=torch.float32, y=y, final_state=fs,
                            initial_state=None if h0 is None else h0.cuda())
    torch.cuda.synchronize()
    y_ref, fs_ref = oracle.ssd_recurrence(inp["x"], inp["dt"], inp["A_head"], inp["B"], inp["C"],
                                          None if h0 is None else h0.double().numpy())
    assert_close(y, y_ref, TOL_BF16, "y")
    assert_close(fs, fs_ref, TOL_BF16, "final_state")


@pytest.mark.parametrize("case", SSD_CASES,
                         ids=[f"B{c['batch']}L{c['seqlen']}H{c['nheads']}G{c['ngroups']}"
                              for c in SSD_CASES])
def test_mamba3_prefill_random_shapes(case):
    c = case
    inp = inputs.mamba3_inputs(c["batch"], c["seqlen"], c["nheads"], 64, 128, c["ngroups"],
                               "bf16", seed=400 + c["seqlen"] + c["nheads"])
    h0 = inp["h0"] if c["h0"] else None
    d = {k: v.cuda() for k, v in inp.items()}
    y = torch.full(d["x"].shape, float("nan"), device="cuda")
    fs = torch.full((c["batch"], c["nheads"], 64, 128), float("nan"), device="cuda")
    binding.ssd_mamba3_fwd(d["x"], d["dt"], d["lam"], d["A_head"], d["B"], d["C"], 64,
                           out_dtype=torch.float32, y=y, final_state=fs,
                           initial_state=None if h0 is None else h0.cuda(),
                           prev_B=d["prev_B"] if c["prev"] else None,
                           prev_x=d["prev_x"] if c["prev"] else None)
    torch.cuda.synchronize()
    y_ref, fs_ref = oracle.mamba3_recurrence(
        inp["x"], inp["dt"], inp["lam"], inp["A_head"], inp["B"], inp["C"],
        None if h0 is None else h0.double().numpy(),
        inp["prev_B"] if c["prev"] else None, inp["prev_x"] if c["prev"] else None)
    assert_close(y, y_ref, TOL_BF16, "y")
    assert_close(fs, fs_ref, TOL_BF16, "final_state")


def _draw_decode(n, seed):
    rng = np.random.default_rng(seed)
    cases = []
    for _ in range(n):
        ngroups = int(rng.integers(1, 4))
        cases.append(dict(batch=int(rng.integers(1, 7)), ngroups=ngroups,
                          nheads=ngroups * int(rng.integers(1, 4)),
                          headdim=int(rng.integers(1, 131)),
                          dstate=int(rng.choice([16, 32, 64, 128, 256])),
                          dtype=str(rng.choice(["f32", "bf16"])), gate=bool(rng.integers(2)),
                          dskip=str(rng.choice(["none", "ones", "randn"]))))
    return cases


DECODE_CASES = _draw_decode(10, 2026)


@pytest.mark.parametrize("case", DECODE_CASES,
                         ids=[f"B{c['batch']}H{c['nheads']}P{c['headdim']}N{c['dstate']}"
                              f"G{c['ngroups']}{c['dtype']}" for c in DECODE_CASES])
def test_decode_random_shapes(case):
    c = case
    steps = 3
    inp = inputs.decode_inputs(c["batch"], c["nheads"], c["headdim"], c["dstate"], c["ngroups"],
                               steps, c["dtype"], seed=500 + c["headdim"], gate=c["gate"],
                               dskip=c["dskip"])
    state = inp["state"].cuda()
    ref_state = inp["state"]
    tol = TOL_F32 if c["dtype"] == "f32" else TOL_BF16
    D = inp["D"]
    for t in range(steps):
        z = inp["z"][t]
        y = binding.ssm_decode_step(state, inp["x"][t].cuda(), inp["dt"][t].cuda(),
                                    inp["A"].cuda(), inp["B"][t].cuda(), inp["C"][t].cuda(),
                                    None if D is None else D.cuda(),
                                    None if z is None else z.cuda())
        y_ref, ref_state = oracle.decode_step(ref_state, inp["x"][t], inp["dt"][t], inp["A"],
                                              inp["B"][t], inp["C"][t], D, z)
        if c["dtype"] == "f32":
            assert_close(y, y_ref, tol, f"y step {t}")
        else:  # bf16 y: the rounding of the exact result, within one bf16 ulp
            assert_close(y, y_ref, 2 ** -7, f"y step {t}")
        assert_close(state, ref_state, tol, f"state step {t}")


def _draw_mimo(n, seed):
    rng = np.random.default_rng(seed)
    cases = []
    for _ in range(n):
        rank = int(rng.choice([1, 2, 4]))
        chunk = 64 // rank
        ngroups = int(rng.integers(1, 3))
        cases.append(dict(batch=int(rng.integers(1, 3)), rank=rank,
                          seqlen=chunk * int(rng.integers(1, 9)), ngroups=ngroups,
                          nheads=ngroups * int(rng.integers(1, 4)), h0=bool(rng.integers(2)),
                          prev=bool(rng.integers(2))))
    return cases


MIMO_CASES = _draw_mimo(8, 2027)


@pytest.mark.parametrize("case", MIMO_CASES,
                         ids=[f"B{c['batch']}L{c['seqlen']}R{c['rank']}H{c['nheads']}"
                              f"G{c['ngroups']}" for c in MIMO_CASES])
def test_mimo_prefill_random_shapes(case):
    c = case
    inp = inputs.mamba3_mimo_inputs(c["batch"], c["seqlen"], c["rank"], c["nheads"], 64, 128,
                                    c["ngroups"], "bf16", seed=600 + c["seqlen"] + c["rank"])
    h0 = inp["h0"] if c["h0"] else None
    d = {k: v.cuda() for k, v in inp.items()}
    y = torch.full(d["x"].shape, float("nan"), device="cuda")
    fs = torch.full((c["batch"], c["nheads"], 64, 128), float("nan"), device="cuda")
    binding.ssd_mamba3_mimo_fwd(d["x"], d["dt"], d["lam"], d["A_head"], d["B"], d["C"],
                                64 // c["rank"], out_dtype=torch.float32, y=y, final_state=fs,
                                initial_state=None if h0 is None else h0.cuda(),
                                prev_B=d["prev_B"] if c["prev"] else None,
                                prev_x=d["prev_x"] if c["prev"] else None)
    torch.cuda.synchronize()
    y_ref, fs_ref = oracle.mamba3_mimo_recurrence(
        inp["x"], inp["dt"], inp["lam"], inp["A_head"], inp["B"], inp["C"],
        None if h0 is None else h0.double().numpy(),
        inp["prev_B"] if c["prev"] else None, inp["prev_x"] if c["prev"] else None)
    assert_close(y, y_ref, TOL_BF16, "y")
    assert_close(fs, fs_ref, TOL_BF16, "final_state")


def _draw_rope(n, seed):
    rng = np.random.default_rng(seed)
    cases = []
    for _ in range(n):
        ngroups = int(rng.integers(1, 4))
        cases.append(dict(batch=int(rng.integers(1, 4)), seqlen=int(rng.integers(1, 400)),
                          rank=int(rng.choice([1, 2, 3, 4])), ngroups=ngroups,
                          nheads=ngroups * int(rng.integers(1, 4)),
                          dstate=2 * int(rng.integers(1, 90)), a0=bool(rng.integers(2))))
    return cases


ROPE_CASES = _draw_rope(10, 2028)


@pytest.mark.parametrize("case", ROPE_CASES,
                         ids=[f"B{c['batch']}L{c['seqlen']}R{c['rank']}H{c['nheads']}"
                              f"G{c['ngroups']}N{c['dstate']}" for c in ROPE_CASES])
def test_rope_random_shapes(case):
    c = case
    g = torch.Generator().manual_seed(c["seqlen"] * 5 + c["dstate"])
    shape = ((c["batch"], c["seqlen"], c["ngroups"], c["dstate"]) if c["rank"] == 1 else
             (c["batch"], c["seqlen"], c["rank"], c["ngroups"], c["dstate"]))
    B = torch.randn(*shape, generator=g)
    C = torch.randn(*shape, generator=g)
    dt = torch.nn.functional.softplus(torch.randn(c["batch"], c["seqlen"], c["nheads"],
                                                  generator=g) - 4)
    r = inputs.rope_inputs(c["batch"], c["seqlen"], c["nheads"], c["dstate"],
                           seed=700 + c["seqlen"])
    a0 = r["angle0"] if c["a0"] else None
    Br, Cr, ang = binding.ssm_mamba3_rope(B.cuda(), C.cuda(), dt.cuda(), r["theta"].cuda(),
                                          None if a0 is None else a0.cuda())
    torch.cuda.synchronize()
    Br_ref, Cr_ref, ang_ref = oracle.mamba3_rope(B, C, dt, r["theta"], a0)
    assert_close(Br, Br_ref, TOL_F32, "B_rot")
    assert_close(Cr, Cr_ref, TOL_F32, "C_rot")
    np.testing.assert_allclose(ang.cpu().double().numpy(), ang_ref, rtol=2e-6, atol=2e-6)


@pytest.mark.parametrize("case", SCAN_CASES[:10],
                         ids=[f"B{c['batch']}D{c['dim']}L{c['seqlen']}G{c['ngroups']}{c['dtype']}"
                              for c in SCAN_CASES[:10]])
def test_scan_bwd_random_shapes(case):
    from tests.test_scan_bwd_gpu import _compare, _dy, _gpu_grad, _oracle_grad
    c = case
    inp = inputs.scan_inputs(c["batch"], c["dim"], c["seqlen"], 16, c["ngroups"], c["dtype"],
                             seed=c["dim"] * 3 + c["seqlen"], gate=c["gate"], dskip=c["dskip"])
    inp["delta_softplus"] = c["softplus"]
    if not c["softplus"]:
        inp["delta"] = (inp["delta"].float().abs() * 0.1).to(inp["delta"].dtype)
        inp["delta_bias"] = torch.full_like(inp["delta_bias"], 0.01)
    dy = _dy((c["batch"], c["dim"], c["seqlen"]), c["dtype"], 9 + c["seqlen"])
    gen = torch.Generator().manual_seed(c["dim"])
    h0 = torch.randn(c["batch"], c["dim"], 16, generator=gen) * 0.5 if c["h0"] else None
    dfinal = torch.randn(c["batch"], c["dim"], 16, generator=gen) if c["h0"] else None
    _compare(_gpu_grad(inp, dy, h0, dfinal), _oracle_grad(inp, dy, h0, dfinal))


@pytest.mark.parametrize("case", SSD_CASES[:6],
                         ids=[f"B{c['batch']}L{c['seqlen']}H{c['nheads']}G{c['ngroups']}"
                              for c in SSD_CASES[:6]])
def test_ssd_bwd_random_shapes(case):
    from tests.test_ssd_bwd_gpu import KEYS, _cotangents, _gpu, _ref
    c = case
    inp = inputs.ssd_inputs(c["batch"], c["seqlen"], c["nheads"], 64, 128, c["ngroups"], "bf16",
                            seed=800 + c["seqlen"] + c["nheads"])
    dy, dfinal = _cotangents(c["batch"], c["seqlen"], c["nheads"], 801 + c["seqlen"], c["h0"])
    h0 = (0.1 * torch.randn(c["batch"], c["nheads"], 64, 128,
                            generator=torch.Generator().manual_seed(c["nheads"]))
          if c["h0"] else None)
    g = _gpu(inp, dy, h0, dfinal)
    ref = _ref(inp, dy, h0, dfinal)
    for key, rkey, tol in KEYS:
        assert_close(g[key], ref[rkey], tol, key)


@pytest.mark.parametrize("case", SSD_CASES[:6],
                         ids=[f"B{c['batch']}L{c['seqlen']}H{c['nheads']}G{c['ngroups']}"
                              for c in SSD_CASES[:6]])
def test_mamba3_bwd_random_shapes(case):
    from tests.test_mamba3_bwd_gpu import KEYS, _case_inputs, _gpu, _ref
    c = case
    inp, dy, dfinal = _case_inputs(c["batch"], c["seqlen"], c["nheads"], c["ngroups"],
                                   900 + c["seqlen"] + c["nheads"], c["h0"], c["prev"], c["h0"])
    g = _gpu(inp, dy, dfinal)
    ref = _ref(inp, dy, dfinal)
    for key, rkey, tol in KEYS:
        if ref[rkey] is None:
            assert g[key] is None, key
            continue
        assert_close(g[key], ref[rkey], tol, key)


@pytest.mark.parametrize("case", MIMO_CASES[:6],
                         ids=[f"B{c['batch']}L{c['seqlen']}R{c['rank']}H{c['nheads']}"
                              f"G{c['ngroups']}" for c in MIMO_CASES[:6]])
def test_mimo_bwd_random_shapes(case):
    from tests.test_mamba3_mimo_bwd_gpu import KEYS, _case, _gpu, _ref
    c = case
    inp, dy, dfinal = _case(c["batch"], c["seqlen"], c["rank"], c["nheads"], c["ngroups"],
                            950 + c["seqlen"] + c["rank"], c["h0"], c["prev"], not c["h0"])
    g = _gpu(inp, dy, dfinal)
    ref = _ref(inp, dy, dfinal)
    for key, rkey, tol in KEYS:
        if ref[rkey] is None:
            assert g[key] is None, key
            continue
        assert_close(g[key], ref[rkey], tol, key)


@pytest.mark.parametrize("case", DECODE_CASES,
                         ids=[f"B{c['batch']}H{c['nheads']}P{c['headdim']}N{c['dstate']}"
                              f"G{c['ngroups']}{c['dtype']}" for c in DECODE_CASES])
def test_mamba3_decode_random_shapes(case):
    c = case
    steps = 3
    inp = inputs.decode_inputs(c["batch"], c["nheads"], c["headdim"], c["dstate"], c["ngroups"],
                               steps + 1, c["dtype"], seed=1500 + c["headdim"], gate=c["gate"],
                               dskip=c["dskip"])
    g = torch.Generator().manual_seed(c["headdim"])
    lams = [torch.sigmoid(torch.randn(c["batch"], c["nheads"], generator=g))
            for _ in range(steps)]
    tol = TOL_F32 if c["dtype"] == "f32" else TOL_BF16
    state = inp["state"].clone().cuda()
    st_ref = inp["state"].double().numpy()
    D = inp["D"]
    cu = lambda v: None if v is None else v.cuda()  # noqa: E731
    for t in range(1, steps + 1):  # step 0's x and B serve as the previous token
        y = binding.ssm_decode_step_mamba3(state, cu(inp["B"][t - 1]), cu(inp["x"][t - 1]),
                                           cu(inp["x"][t]), cu(inp["dt"][t]), cu(lams[t - 1]),
                                           inp["A"].cuda(), cu(inp["B"][t]), cu(inp["C"][t]),
                                           cu(D), cu(inp["z"][t]))
        torch.cuda.synchronize()
        y_ref, st_ref = oracle.mamba3_decode_step(st_ref, inp["B"][t - 1], inp["x"][t - 1],
                                                  inp["x"][t], inp["dt"][t], lams[t - 1],
                                                  inp["A"], inp["B"][t], inp["C"][t], D,
                                                  inp["z"][t])
        if c["dtype"] == "f32":
            assert_close(y, y_ref, tol, f"y step {t}")
        else:  # bf16 y: the rounding of the exact result, within one bf16 ulp
            assert_close(y, y_ref, 2 ** -7, f"y step {t}")
        assert_close(state, st_ref, tol, f"state step {t}")


def _draw_mimo_decode(n, seed):
    rng = np.random.default_rng(seed)
    cases = []
    for _ in range(n):
        ngroups = int(rng.integers(1, 4))
        cases.append(dict(batch=int(rng.integers(1, 5)), rank=int(rng.choice([2, 4])),
                          ngroups=ngroups, nheads=ngroups * int(rng.integers(1, 4)),
                          headdim=int(rng.integers(1, 150)),
                          dtype=str(rng.choice(["f32", "bf16"])), gate=bool(rng.integers(2)),
                          dskip=bool(rng.integers(2))))
    return cases


MIMO_DECODE_CASES = _draw_mimo_decode(8, 2029)


@pytest.mark.parametrize("case", MIMO_DECODE_CASES,
                         ids=[f"B{c['batch']}R{c['rank']}H{c['nheads']}P{c['headdim']}"
                              f"G{c['ngroups']}{c['dtype']}" for c in MIMO_DECODE_CASES])
def test_mimo_decode_random_shapes(case):
    c = case
    steps = 3
    inp = inputs.mamba3_mimo_inputs(c["batch"], steps + 1, c["rank"], c["nheads"], c["headdim"],
                                    128, c["ngroups"], c["dtype"], seed=1600 + c["headdim"])
    g = torch.Generator().manual_seed(c["headdim"] + 1)
    D = torch.randn(c["nheads"], generator=g) if c["dskip"] else None
    zs = [torch.randn(c["batch"], c["rank"], c["nheads"], c["headdim"],
                      generator=g).to(inp["x"].dtype) if c["gate"] else None
          for _ in range(steps + 1)]
    tol = TOL_F32 if c["dtype"] == "f32" else TOL_BF16
    state = inp["h0"].clone().cuda()
    st_ref = inp["h0"].double().numpy()
    cu = lambda v: None if v is None else v.contiguous().cuda()  # noqa: E731
    for t in range(1, steps + 1):
        y = binding.ssm_decode_step_mamba3_mimo(
            state, cu(inp["B"][:, t - 1]), cu(inp["x"][:, t - 1]), cu(inp["x"][:, t]),
            cu(inp["dt"][:, t]), cu(inp["lam"][:, t]), inp["A_head"].cuda(), cu(inp["B"][:, t]),
            cu(inp["C"][:, t]), cu(D), cu(zs[t]))
        torch.cuda.synchronize()
        y_ref, st_ref = oracle.mamba3_mimo_decode_step(
            st_ref, inp["B"][:, t - 1], inp["x"][:, t - 1], inp["x"][:, t], inp["dt"][:, t],
            inp["lam"][:, t], inp["A_head"], inp["B"][:, t], inp["C"][:, t], D, zs[t])
        if c["dtype"] == "f32":
            assert_close(y, y_ref, tol, f"y step {t}")
        else:
            assert_close(y, y_ref, 2 ** -7, f"y step {t}")
        assert_close(state, st_ref, tol, f"state step {t}")


@pytest.mark.parametrize("case", SCAN_CASES[:8],
                         ids=[f"B{c['batch']}D{c['dim']}L{c['seqlen']}G{c['ngroups']}{c['dtype']}"
                              for c in SCAN_CASES[:8]])
def test_scan_host_buffers_random_shapes(case):
    """ssm_scan_fwd_host on pinned host buffers gives ssm_scan_fwd's bits (these
    problems are small enough that both take the whole problem's kernel)."""
    c = case
    inp = inputs.scan_inputs(c["batch"], c["dim"], c["seqlen"], 16, c["ngroups"], c["dtype"],
                             seed=c["dim"] * 11 + c["seqlen"], gate=c["gate"], dskip=c["dskip"])
    h0 = (torch.randn(c["batch"], c["dim"], 16, generator=torch.Generator().manual_seed(3)) * 0.5
          if c["h0"] else None)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    y_dev, fs_dev = binding.ssm_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"],
                                         d["z"], d["delta_bias"], True,
                                         None if h0 is None else h0.cuda(),
                                         out_dtype=torch.float32)
    pin = {k: (v.pin_memory() if isinstance(v, torch.Tensor) and k in ("u", "delta", "z", "B", "C")
               else v) for k, v in inp.items()}
    y_h = torch.full((c["batch"], c["dim"], c["seqlen"]), float("nan")).pin_memory()
    fs_h = torch.full((c["batch"], c["dim"], 16), float("nan")).pin_memory()
    binding.ssm_scan_fwd_host(pin["u"], pin["delta"], d["A"], pin["B"], pin["C"], y_h, fs_h,
                              d["D"], pin["z"], d["delta_bias"], True,
                              None if h0 is None else h0.pin_memory())
    torch.cuda.synchronize()
    assert torch.equal(y_h, y_dev.cpu())
    assert torch.equal(fs_h, fs_dev.cpu())


def _draw_scan_chained(n, seed):
    """Problems whose 32-channel blocks fill every resident CTA slot, so the
    chained scan cuts the sequence into L-chunks carried through the workspace."""
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        ngroups = int(rng.choice([1, 2, 4]))
        dpg = int(rng.integers(5000, 6200)) // ngroups
        seqlen = int(rng.integers(65, 1300))
        if i % 2 == 0:  # rows 16-byte aligned for bf16: the TMA path (else plain loads)
            seqlen -= seqlen % 8
        cases.append(dict(batch=4, ngroups=ngroups, dim=ngroups * dpg, seqlen=seqlen,
                          dtype=str(rng.choice(["f32", "bf16"])), gate=bool(rng.integers(2)),
                          dskip=str(rng.choice(["none", "ones", "randn"])),
                          softplus=True, h0=bool(rng.integers(2))))
    return cases


SCAN_CHAINED_CASES = _draw_scan_chained(4, 2030)


@pytest.mark.parametrize("case", SCAN_CHAINED_CASES,
                         ids=[f"B{c['batch']}D{c['dim']}L{c['seqlen']}G{c['ngroups']}{c['dtype']}"
                              for c in SCAN_CHAINED_CASES])
def test_scan_chained_chunks_random_shapes(case):
    test_scan_random_shapes(case, (0, 0))
