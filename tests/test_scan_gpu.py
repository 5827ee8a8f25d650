"""Parity of the CUDA selective scan (through the C ABI) with the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from state_space_model_selective_gb300 import binding, inputs
from tests.helpers import TOL_BF16, TOL_F32, assert_close, assert_elementwise, to64

pytestmark = pytest.mark.gpu


def _to_dev(d):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


def _run(inp, out_dtype=torch.float32, initial_state=None, poison=True):
    x = _to_dev(inp)
    batch, dim, seqlen = x["u"].shape
    y = torch.empty((batch, dim, seqlen), dtype=out_dtype, device="cuda")
    fs = torch.empty((batch, dim, 16), dtype=torch.float32, device="cuda")
    if poison:  # catch elements the kernel never writes
        y.fill_(float("nan"))
        fs.fill_(float("nan"))
    need = binding.ssm_scan_workspace_bytes(batch, dim, seqlen, 16, x["B"].shape[1])
    ws = torch.full((need,), 0xAB, dtype=torch.uint8, device="cuda")
    binding.ssm_scan_fwd(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"],
                         x["delta_bias"], x["delta_softplus"],
                         None if initial_state is None else initial_state.cuda(),
                         out_dtype=out_dtype, y=y, final_state=fs, workspace=ws)
    torch.cuda.synchronize()
    assert binding.ssm_last_device_status(ws) == 0
    return y, fs


# the forward scan's two kernels (ssm_debug_set_scan_path): the chained scan,
# and the sequence-parallel scan with its planned or a forced segment count
PATHS = {"chained": (1, 0), "seqpar": (2, 0), "seqpar8": (2, 8), "seqpar16": (2, 16),
         "seqpar32": (2, 32)}


@pytest.fixture(params=["chained", "seqpar"])
def path(request):
    binding.ssm_debug_set_scan_path(*PATHS[request.param])
    yield request.param
    binding.ssm_debug_set_scan_path()


@pytest.fixture(params=["seqpar8", "seqpar16", "seqpar32"])
def seg_path(request):
    binding.ssm_debug_set_scan_path(*PATHS[request.param])
    yield request.param
    binding.ssm_debug_set_scan_path()


def _oracle(inp, initial_state=None):
    return oracle.scan(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"],
                       inp["delta_bias"], inp["delta_softplus"], initial_state)


CASES = [
    # batch, dim, seqlen, ngroups, dtype, gate, dskip, softplus
    (1, 32, 64, 1, "f32", True, "ones", True),       # one tile, one block
    (2, 64, 200, 1, "f32", True, "randn", True),     # ragged tail (200 % 64), TMA rows
    (2, 48, 333, 1, "f32", False, "none", False),    # odd L: plain-load path; partial block
    (3, 96, 256, 2, "bf16", True, "ones", True),     # groups
    (2, 40, 130, 4, "bf16", True, "randn", True),    # 10 channels per group: partial blocks
    (1, 32, 1000, 1, "bf16", False, "ones", True),   # bf16 rows 16B-aligned, ragged tail
    (2, 32, 77, 1, "bf16", True, "ones", False),     # odd L with bf16: plain-load path
    (1, 32, 1, 1, "f32", True, "randn", True),       # a single step
    (2, 32, 65, 1, "f32", True, "ones", True),       # one step past a tile, plain loads
    (2, 64, 72, 2, "bf16", True, "ones", True),      # one 8-step group past a tile, TMA rows
]


@pytest.mark.parametrize("case", CASES, ids=[f"B{c[0]}D{c[1]}L{c[2]}G{c[3]}{c[4]}" for c in CASES])
def test_scan_matches_oracle(case, path):
    batch, dim, seqlen, ngroups, dt, gate, dskip, softplus = case
    inp = inputs.scan_inputs(batch, dim, seqlen, 16, ngroups, dt, seed=100 + seqlen, gate=gate,
                             dskip=dskip)
    inp["delta_softplus"] = softplus
    if not softplus:  # without softplus, delta + bias must stay positive (a decaying state)
        inp["delta"] = (inp["delta"].float().abs() * 0.1).to(inp["delta"].dtype)
        inp["delta_bias"] = torch.full_like(inp["delta_bias"], 0.01)
    y, fs = _run(inp)
    y_ref, fs_ref = _oracle(inp)
    tol = TOL_F32 if dt == "f32" else TOL_BF16
    assert_close(y, y_ref, tol, "y")
    assert_close(fs, fs_ref, tol, "final_state")


def test_scan_initial_state_and_resume(path):
    """Scanning [0, k) then [k, L) from the first part's final state equals one scan."""
    inp = inputs.scan_inputs(2, 64, 384, 16, 1, "f32", seed=5)
    h0 = torch.randn(2, 64, 16, generator=torch.Generator().manual_seed(1)) * 0.5
    y, fs = _run(inp, initial_state=h0)
    y_ref, fs_ref = _oracle(inp, h0)
    assert_close(y, y_ref, TOL_F32, "y with initial state")
    assert_close(fs, fs_ref, TOL_F32, "final_state with initial state")
    k = 192
    first = {kk: (v[..., :k].contiguous() if kk in ("u", "delta", "z", "B", "C") else v)
             for kk, v in inp.items()}
    second = {kk: (v[..., k:].contiguous() if kk in ("u", "delta", "z", "B", "C") else v)
              for kk, v in inp.items()}
    y1, f1 = _run(first, initial_state=h0)
    y2, f2 = _run(second, initial_state=f1.cpu())
    assert_close(torch.cat([y1, y2], -1), y_ref, TOL_F32, "resumed y")
    assert_close(f2, fs_ref, TOL_F32, "resumed final_state")


def test_scan_bf16_output_is_rounded_fp32_output(path):
    inp = inputs.scan_inputs(2, 64, 256, 16, 1, "bf16", seed=9)
    y32, f32 = _run(inp, torch.float32)
    y16, f16 = _run(inp, torch.bfloat16)
    assert torch.equal(y16, y32.to(torch.bfloat16))
    assert torch.equal(f16, f32)


def test_scan_deterministic(path):
    inp = inputs.scan_inputs(2, 64, 300, 16, 1, "bf16", seed=11)
    a = _run(inp)
    b = _run(inp)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_scan_empty_and_zero_length(path):
    u = torch.zeros(2, 32, 0, device="cuda")
    A = -torch.ones(32, 16, device="cuda")
    B = torch.zeros(2, 1, 16, 0, device="cuda")
    h0 = torch.randn(2, 32, 16, device="cuda")
    y, fs = binding.ssm_scan_fwd(u, u, A, B, B, initial_state=h0)
    torch.cuda.synchronize()
    assert y.shape == (2, 32, 0) and torch.equal(fs, h0)
    y, fs = binding.ssm_scan_fwd(u, u, A, B, B)
    assert torch.count_nonzero(fs).item() == 0
    u0 = torch.zeros(0, 32, 10, device="cuda")
    B0 = torch.zeros(0, 1, 16, 10, device="cuda")
    y, fs = binding.ssm_scan_fwd(u0, u0, A, B0, B0)
    assert y.shape == (0, 32, 10)


WIDE_CASES = [
    # batch, dim, seqlen, ngroups, dtype, with initial state: a few hundred
    # 32-channel blocks of the chained scan, every output checked
    (2, 3840, 333, 2, "bf16", True),   # odd bf16 length: the plain-load path
    (1, 7680, 1000, 1, "f32", False),  # TMA rows, ragged last tile
    (3, 2560, 520, 4, "bf16", True),   # groups, 8 full tiles + 8 steps
]


@pytest.mark.parametrize("case", WIDE_CASES,
                         ids=[f"B{c[0]}D{c[1]}L{c[2]}G{c[3]}{c[4]}" for c in WIDE_CASES])
def test_scan_many_channels_match_oracle(case):
    """The chained scan on thousands of channels: every output against the
    oracle, and bf16 y exactly the fp32 y rounded."""
    batch, dim, seqlen, ngroups, dt, with_h0 = case
    inp = inputs.scan_inputs(batch, dim, seqlen, 16, ngroups, dt, seed=400 + seqlen)
    h0 = (torch.randn(batch, dim, 16, generator=torch.Generator().manual_seed(4)) * 0.5
          if with_h0 else None)
    y, fs = _run(inp, initial_state=h0)
    y_ref, fs_ref = _oracle(inp, h0)
    tol = TOL_F32 if dt == "f32" else TOL_BF16
    assert_close(y, y_ref, tol, "y")
    assert_close(fs, fs_ref, tol, "final_state")
    assert_elementwise(y, y_ref, "y")
    y16, fs16 = _run(inp, torch.bfloat16, initial_state=h0)
    assert torch.equal(y16, y.to(torch.bfloat16)) and torch.equal(fs16, fs)


def test_scan_chained_chunks_many_blocks():
    """Enough channel blocks that L is cut into chained chunks across CTAs."""
    inp = inputs.scan_inputs(4, 4096, 512, 16, 1, "bf16", seed=21)
    y, fs = _run(inp)
    rows = [(0, 0), (1, 1234), (2, 4095), (3, 2048), (3, 7), (0, 4000)]
    y_ref, fs_ref = oracle.scan_rows(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], rows,
                                     inp["D"], inp["z"], inp["delta_bias"], True)
    ys = torch.stack([y[b, d] for b, d in rows])
    fss = torch.stack([fs[b, d] for b, d in rows])
    assert_close(ys, y_ref, TOL_BF16, "y rows")
    assert_close(fss, fs_ref, TOL_BF16, "final_state rows")


# ------------------------------------------------- sequence-parallel scan

SEG_CASES = [
    # batch, dim, seqlen, ngroups, dtype: chunk counts 1 .. 41 (more than the
    # 32 chunks one look-back round examines), ragged last chunks and segments
    (1, 16, 5200, 1, "f32"),
    (2, 48, 1500, 3, "bf16"),
    (3, 20, 777, 1, "f32"),     # odd length: element loads; partial CTAs
    (1, 8, 4097, 1, "bf16"),    # one step into the 33rd chunk
    (2, 24, 129, 2, "f32"),     # one step into the second chunk
    (1, 4, 100, 1, "bf16"),     # a single partial chunk
]


@pytest.mark.parametrize("case", SEG_CASES,
                         ids=[f"B{c[0]}D{c[1]}L{c[2]}G{c[3]}{c[4]}" for c in SEG_CASES])
def test_seqpar_lookback_matches_oracle(case, seg_path):
    """Chunks joined by the decoupled look-back (aggregates composed with the
    associative operator) and segments joined by the in-warp shuffle scan give
    the recurrence, for every segment count."""
    batch, dim, seqlen, ngroups, dt = case
    inp = inputs.scan_inputs(batch, dim, seqlen, 16, ngroups, dt, seed=300 + seqlen)
    h0 = torch.randn(batch, dim, 16, generator=torch.Generator().manual_seed(seqlen)) * 0.5
    y, fs = _run(inp, initial_state=h0)
    y_ref, fs_ref = _oracle(inp, h0)
    tol = TOL_F32 if dt == "f32" else TOL_BF16
    assert_close(y, y_ref, tol, "y")
    assert_close(fs, fs_ref, tol, "final_state")
    assert_elementwise(y, y_ref, "y")


def test_seqpar_deterministic_and_resumable():
    """The look-back's result does not depend on which predecessor it stopped
    at, so repeated runs give the same bits; and a sequence scanned in pieces
    cut at multiples of 128 steps, each resumed from the previous final state,
    gives the bits of the whole scan (with the same segment count)."""
    inp = inputs.scan_inputs(2, 40, 1280, 16, 1, "bf16", seed=321)
    binding.ssm_debug_set_scan_path(2, 16)
    try:
        y, fs = _run(inp)
        for _ in range(3):
            y2, fs2 = _run(inp)
            assert torch.equal(y, y2) and torch.equal(fs, fs2)
        parts, state, ys = [(0, 384), (384, 1152), (1152, 1280)], None, []
        for a, b in parts:
            piece = {k: (v[..., a:b].contiguous() if k in ("u", "delta", "z", "B", "C") else v)
                     for k, v in inp.items()}
            yp, state = _run(piece, initial_state=None if state is None else state.cpu())
            ys.append(yp)
        assert torch.equal(torch.cat(ys, -1), y)
        assert torch.equal(state, fs)
    finally:
        binding.ssm_debug_set_scan_path()


def test_seqpar_and_chained_agree():
    """Both kernels on one problem: each within the tolerance of the oracle and
    of each other."""
    inp = inputs.scan_inputs(2, 64, 1000, 16, 2, "f32", seed=322)
    out = {}
    for name in ("chained", "seqpar"):
        binding.ssm_debug_set_scan_path(*PATHS[name])
        try:
            out[name] = _run(inp)
        finally:
            binding.ssm_debug_set_scan_path()
    y_ref, fs_ref = _oracle(inp)
    for name, (y, fs) in out.items():
        assert_close(y, y_ref, TOL_F32, f"y ({name})")
        assert_close(fs, fs_ref, TOL_F32, f"final_state ({name})")
    assert_close(out["seqpar"][0], out["chained"][0], 2 * TOL_F32, "y, one kernel vs the other")


# ------------------------------------------------------------------ workloads

def test_workload_scan_fp32_L128_D1536(path):
    """Selective scan fp32, batch 1, L 128, 1536 channels, N 16: every output."""
    inp = inputs.scan_inputs(1, 1536, 128, 16, 1, "f32", seed=1001)
    y, fs = _run(inp)
    y_ref, fs_ref = _oracle(inp)
    assert_close(y, y_ref, TOL_F32, "y")
    assert_close(fs, fs_ref, TOL_F32, "final_state")
    assert_elementwise(y, y_ref, "y")


@pytest.mark.parametrize("shape,seed", [((8, 1536, 2048), 1002), ((4, 5120, 16384), 1003)],
                         ids=["B8_D1536_L2048", "B4_D5120_L16384"])
def test_workload_scan_bf16_whole(shape, seed):
    """Full-size bf16 workloads, launched as the benchmark launches them; every
    output element checked against the oracle, one batch row at a time (the
    oracle's fp64 copies of a whole 5.4e9-element workload would not fit in
    host memory comfortably)."""
    batch, dim, seqlen = shape
    inp = inputs.scan_inputs(batch, dim, seqlen, 16, 1, "bf16", seed=seed)
    y, fs = _run(inp, poison=False)
    num_y = den_y = num_f = den_f = 0.0
    ew = 0.0
    for b in range(batch):
        sl = slice(b, b + 1)
        y_ref, fs_ref = oracle.scan(inp["u"][sl], inp["delta"][sl], inp["A"], inp["B"][sl],
                                    inp["C"][sl], inp["D"], inp["z"][sl], inp["delta_bias"], True)
        yb, fb = to64(y[sl]), to64(fs[sl])
        assert np.isfinite(yb).all() and np.isfinite(fb).all()
        num_y = max(num_y, float(np.max(np.abs(yb - y_ref))))
        den_y = max(den_y, float(np.max(np.abs(y_ref))))
        num_f = max(num_f, float(np.max(np.abs(fb - fs_ref))))
        den_f = max(den_f, float(np.max(np.abs(fs_ref))))
        ew = max(ew, assert_elementwise(yb, y_ref, f"y batch row {b}"))
        del y_ref, yb
    print(f"normwise y {num_y / den_y:.3e}, final_state {num_f / den_f:.3e}, "
          f"element-wise y {ew:.3e}")
    assert num_y / den_y <= TOL_BF16, num_y / den_y
    assert num_f / den_f <= TOL_BF16, num_f / den_f


@pytest.mark.parametrize("case", [(2, 64, 700, 1, "bf16", torch.float32, True),
                                  (1, 96, 1000, 2, "f32", torch.float32, False),
                                  (3, 40, 64, 4, "bf16", torch.bfloat16, True),
                                  (2, 32, 30, 1, "f32", torch.float32, True),
                                  (5, 64, 300, 1, "bf16", torch.float32, True),
                                  (9, 48, 130, 2, "f32", torch.float32, False),
                                  (4, 32, 64, 4, "bf16", torch.bfloat16, True),
                                  (2, 36, 200, 6, "f32", torch.float32, True),
                                  (1, 100, 300, 1, "bf16", torch.float32, True),
                                  (8, 4096, 64, 1, "f32", torch.float32, True)],
                         ids=["bf16-L700", "f32-L1000-G2", "bf16out-L64", "L30",
                              "B5-L300", "B9-G2-L130", "B4-bf16out-G4", "G6-whole-groups",
                              "part-groups-D100", "chained-segments"])
def test_scan_host_buffers_equal_device_scan(case):
    """ssm_scan_fwd_host (host-resident activations, copies pipelined over
    segments of the channels) gives the same bits as ssm_scan_fwd on device
    copies, and matches the oracle.  The cases cut segments at whole batches,
    whole groups (channel offsets that leave D and the bias unaligned) and
    inside a group.  All but the last are problems ssm_scan_fwd gives to the
    sequence-parallel scan; the last is a short sequence whose 4096-channel
    segments are too large for it, so every segment takes the chained scan,
    as the whole call does."""
    batch, dim, seqlen, ngroups, dt, out_dt, with_h0 = case
    inp = inputs.scan_inputs(batch, dim, seqlen, 16, ngroups, dt, seed=120 + seqlen)
    h0 = (torch.randn(batch, dim, 16, generator=torch.Generator().manual_seed(3)) * 0.5
          if with_h0 else None)
    y_dev, fs_dev = _run(inp, out_dtype=out_dt, initial_state=h0)
    pin = {k: (v.pin_memory() if isinstance(v, torch.Tensor) and k in ("u", "delta", "z", "B", "C")
               else v) for k, v in inp.items()}
    y_h = torch.full((batch, dim, seqlen), float("nan"), dtype=out_dt).pin_memory()
    fs_h = torch.full((batch, dim, 16), float("nan")).pin_memory()
    binding.ssm_scan_fwd_host(pin["u"], pin["delta"], inp["A"].cuda(), pin["B"], pin["C"], y_h,
                              fs_h, inp["D"].cuda(), pin["z"], inp["delta_bias"].cuda(), True,
                              None if h0 is None else h0.pin_memory())
    torch.cuda.synchronize()
    assert torch.equal(y_h, y_dev.cpu())
    assert torch.equal(fs_h, fs_dev.cpu())
    if out_dt == torch.float32:
        y_ref, fs_ref = _oracle(inp, h0)
        tol = TOL_F32 if dt == "f32" else TOL_BF16
        assert_close(y_h, y_ref, tol, "y")
        assert_close(fs_h, fs_ref, tol, "final_state")


def _piece(inp, h0, b, c0, c1):
    """The problem of batch row b's channels [c0, c1), all in one B/C group."""
    dim, ngroups = inp["u"].shape[1], inp["B"].shape[1]
    g = c0 // (dim // ngroups)
    assert (c1 - 1) // (dim // ngroups) == g
    x = dict(inp)
    for k in ("u", "delta", "z"):
        if inp[k] is not None:
            x[k] = inp[k][b:b + 1, c0:c1].contiguous()
    for k in ("B", "C"):
        x[k] = inp[k][b:b + 1, g:g + 1].contiguous()
    for k in ("A", "D", "delta_bias"):
        if inp[k] is not None:
            x[k] = inp[k][c0:c1].contiguous()
    return x, (None if h0 is None else h0[b:b + 1, c0:c1].contiguous())


@pytest.mark.parametrize("case", [
    # batch, dim, seqlen, dtype, out dtype, channels per device piece, forced segments per chunk
    (2, 2048, 256, "bf16", torch.float32, 2048, 16),
    (8, 4096, 1100, "bf16", torch.float32, 2048, 8),
], ids=["seqpar-segments", "capped-segments"])
def test_scan_host_sequence_parallel_segments(case):
    """Problems the chained scan takes whole, whose host-path segments each fit
    the sequence-parallel scan, have every segment scanned by that kernel with
    one segment count.  A channel's arithmetic then depends only on the kernel
    and that count: with the count forced, the host path gives the bits of
    ssm_scan_fwd run on device pieces of the channels; as planned it matches
    the oracle.  The second case is a long sequence whose segments, an eighth
    of the 32768 channels (4096) by default, are capped to fit the
    sequence-parallel scan (at most 3072 channels; here half a batch row)."""
    batch, dim, seqlen, dt, out_dt, piece, ts = case
    inp = inputs.scan_inputs(batch, dim, seqlen, 16, 1, dt, seed=160 + seqlen)
    h0 = torch.randn(batch, dim, 16, generator=torch.Generator().manual_seed(5)) * 0.5
    pin = {k: (v.pin_memory() if isinstance(v, torch.Tensor) and k in ("u", "delta", "z", "B", "C")
               else v) for k, v in inp.items()}

    def host():
        y_h = torch.full((batch, dim, seqlen), float("nan"), dtype=out_dt).pin_memory()
        fs_h = torch.full((batch, dim, 16), float("nan")).pin_memory()
        binding.ssm_scan_fwd_host(pin["u"], pin["delta"], inp["A"].cuda(), pin["B"], pin["C"],
                                  y_h, fs_h, inp["D"].cuda(), pin["z"], inp["delta_bias"].cuda(),
                                  True, h0.pin_memory())
        torch.cuda.synchronize()
        return y_h, fs_h

    binding.ssm_debug_set_scan_path(0, ts)
    try:
        y_h, fs_h = host()
        for b in range(batch):
            for c0 in range(0, dim, piece):
                x, h = _piece(inp, h0, b, c0, c0 + piece)
                y_p, fs_p = _run(x, out_dtype=out_dt, initial_state=h)
                assert torch.equal(y_h[b:b + 1, c0:c0 + piece], y_p.cpu()), (b, c0)
                assert torch.equal(fs_h[b:b + 1, c0:c0 + piece], fs_p.cpu()), (b, c0)
    finally:
        binding.ssm_debug_set_scan_path()
    y_h, fs_h = host()
    y_ref, fs_ref = _oracle(inp, h0)
    assert_close(y_h, y_ref, TOL_BF16, "y")
    assert_close(fs_h, fs_ref, TOL_BF16, "final_state")


@pytest.mark.parametrize("with_h0", [True, False])
def test_scan_host_empty_sequence(with_h0):
    """ssm_scan_fwd_host with seqlen 0: no rows to scan; the final state is the
    initial state (zeros without one), as ssm_scan_fwd gives."""
    batch, dim = 3, 40
    inp = inputs.scan_inputs(batch, dim, 0, 16, 2, "bf16", seed=7)
    h0 = torch.randn(batch, dim, 16, generator=torch.Generator().manual_seed(5)) if with_h0 else None
    pin = {k: (v.pin_memory() if isinstance(v, torch.Tensor) and k in ("u", "delta", "z", "B", "C")
               else v) for k, v in inp.items()}
    y_h = torch.empty((batch, dim, 0), dtype=torch.float32).pin_memory()
    fs_h = torch.full((batch, dim, 16), float("nan")).pin_memory()
    binding.ssm_scan_fwd_host(pin["u"], pin["delta"], inp["A"].cuda(), pin["B"], pin["C"], y_h,
                              fs_h, inp["D"].cuda(), pin["z"], inp["delta_bias"].cuda(), True,
                              None if h0 is None else h0.pin_memory())
    torch.cuda.synchronize()
    assert torch.equal(fs_h, h0 if with_h0 else torch.zeros_like(fs_h))
