"""The C ABI loads without a GPU, exports every symbol the header declares,
and rejects bad arguments on the host before anything is launched.

No call here reaches the GPU: every call carries an argument error that the
host-side checks catch first, and the pointers are fake addresses that are
never dereferenced.
"""
import ctypes
import os
import re

import pytest

from state_space_model_selective_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ssm.h")

OK, NULL, SHAPE, ALIGN, DTYPE, UNSUP, WS, TIMEOUT, CUDA, ALIAS = range(10)


@pytest.fixture(scope="module")
def L():
    return binding.lib()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b([a-z_][a-z0-9_]*)\s*\(", text)
    return sorted({n for n in names if n.startswith(("ssm_", "ssd_"))})


def test_header_symbols_exported(L):
    declared = _declared_functions()
    assert set(declared) == set(binding.EXPORTS), declared
    for name in declared:
        assert hasattr(L, name), f"libssm.so does not export {name}"


def test_lookback_debug_hook_is_host_only(L):
    # a process-wide setting read at enqueue time: setting and restoring it
    # touches no device
    assert L.ssm_debug_set_lookback(1, 2000) == OK
    assert L.ssm_debug_set_lookback(0, 0) == OK


def test_scan_path_debug_hook_is_host_only(L):
    # the forward scan's kernel choice, a process-wide setting read at enqueue
    # time; out-of-range values are rejected
    for path, segs in ((1, 0), (2, 8), (2, 16), (2, 32), (0, 0)):
        assert L.ssm_debug_set_scan_path(path, segs) == OK
    assert L.ssm_debug_set_scan_path(3, 0) == SHAPE
    assert L.ssm_debug_set_scan_path(-1, 0) == SHAPE
    assert L.ssm_debug_set_scan_path(2, 12) == SHAPE
    assert L.ssm_debug_set_scan_path(0, 0) == OK


def _t(*shape, dtype=None):
    import torch
    return torch.empty(shape, dtype=dtype or torch.float32)


def test_binding_rejects_mismatched_scan_shapes():
    """Every tensor handed to a scan entry point is checked against u's
    (batch, dim, seqlen), A's dstate and B's ngroups before the C call, so a
    short buffer can never be read or written past its end (pure shape
    logic: CPU tensors, no call reaches the library)."""
    b, d, l, n, g = 2, 8, 20, 16, 2
    good = dict(u=_t(b, d, l), delta=_t(b, d, l), A=_t(d, n), B=_t(b, g, n, l), C=_t(b, g, n, l),
                D=_t(d), z=_t(b, d, l), delta_bias=_t(d), initial_state=_t(b, d, n),
                y=_t(b, d, l), final_state=_t(b, d, n))
    assert binding._scan_shapes(**good) == (b, d, l, n, g)
    bad = {"delta": _t(b, d, l - 1), "A": _t(d + 1, n), "B": _t(b, g, n, l + 1),
           "C": _t(b, 1, n, l), "D": _t(d - 1), "z": _t(b, d + 1, l), "delta_bias": _t(2 * d),
           "initial_state": _t(b, d, n - 1), "y": _t(b, d, l - 5), "final_state": _t(1, d, n)}
    for name, t in bad.items():
        with pytest.raises(ValueError, match=name):
            binding._scan_shapes(**{**good, name: t})
    with pytest.raises(ValueError, match="dy"):
        binding._scan_shapes(**good, dy=_t(b, d, 1))
    with pytest.raises(ValueError, match="dfinal_state"):
        binding._scan_shapes(**good, dfinal_state=_t(b, 1, n))


def test_version_and_status_strings(L):
    assert binding.ssm_abi_version() == 4
    for code in range(10):
        s = binding.status_string(code)
        assert isinstance(s, str) and s
    assert binding.status_string(123) == "unknown status"


def test_workspace_bytes_pure_function():
    f = binding.ssm_scan_workspace_bytes
    assert f(8, 1536, 2048) == f(8, 1536, 2048) > 0
    assert f(1, 1536, 128) >= 256
    assert f(1, 10, 5, dstate=8) == 0            # unsupported dstate
    assert f(1, 10, 5, ngroups=3) == 0           # dim % ngroups != 0
    assert f(-1, 10, 5) == 0
    # grows with the problem
    assert f(4, 5120, 16384) > f(8, 1536, 2048)
    # few channels and many 128-step chunks: room for the sequence-parallel
    # scan's flags, aggregates and inclusive states of every chunk
    assert f(1, 64, 1024) >= 256 + 8 * 64 * (2 * 16 + 16) * 4


# fake, 16-byte aligned device addresses, far apart (never dereferenced)
def P(i):
    return ctypes.c_void_p(0x10000000 * (i + 1))


def scan_call(L, **kw):
    args = dict(u=P(0), delta=P(1), A=P(2), B=P(3), C=P(4), D=None, z=None, bias=None,
                softplus=1, h0=None, y=P(5), fs=P(6), batch=2, dim=32, seqlen=64, dstate=16,
                ngroups=1, in_dt=1, out_dt=0, ws=P(7), wsb=1 << 30, stream=None)
    args.update(kw)
    return L.ssm_scan_fwd(args["u"], args["delta"], args["A"], args["B"], args["C"], args["D"],
                          args["z"], args["bias"], args["softplus"], args["h0"], args["y"],
                          args["fs"], args["batch"], args["dim"], args["seqlen"], args["dstate"],
                          args["ngroups"], args["in_dt"], args["out_dt"], args["ws"], args["wsb"],
                          args["stream"])


def test_scan_argument_errors(L):
    assert scan_call(L, u=None) == NULL
    assert scan_call(L, y=None) == NULL
    assert scan_call(L, A=None) == NULL
    assert scan_call(L, batch=-1) == SHAPE
    assert scan_call(L, seqlen=-5) == SHAPE
    assert scan_call(L, ngroups=3) == SHAPE          # 32 % 3 != 0
    assert scan_call(L, ngroups=0) == SHAPE
    assert scan_call(L, dstate=8) == UNSUP
    assert scan_call(L, dstate=0) == SHAPE
    assert scan_call(L, in_dt=7) == DTYPE
    assert scan_call(L, out_dt=-1) == DTYPE
    assert scan_call(L, u=ctypes.c_void_p(0x10000008)) == ALIGN
    assert scan_call(L, fs=ctypes.c_void_p(0x70000004)) == ALIGN
    assert scan_call(L, ws=None) == WS
    assert scan_call(L, wsb=16) == WS
    assert scan_call(L, y=P(0)) == ALIAS             # y on top of u
    assert scan_call(L, fs=P(2)) == ALIAS            # final_state on top of A
    assert scan_call(L, ws=P(1)) == ALIAS            # workspace on top of delta
    # empty problems are valid and launch nothing
    assert scan_call(L, batch=0, u=None, y=None) == OK
    assert scan_call(L, dim=0, u=None, y=None) == OK


def ssd_call(L, **kw):
    args = dict(x=P(0), dt=P(1), A=P(2), B=P(3), C=P(4), chunk=64, h0=None, y=P(5), fs=P(6), batch=2,
                seqlen=128, nheads=4, headdim=64, dstate=128, ngroups=1, in_dt=1, out_dt=0,
                stream=None)
    args.update(kw)
    return L.ssd_chunked_fwd(args["x"], args["dt"], args["A"], args["B"], args["C"],
                             args["chunk"], args["h0"], args["y"], args["fs"], args["batch"],
                             args["seqlen"],
                             args["nheads"], args["headdim"], args["dstate"], args["ngroups"],
                             args["in_dt"], args["out_dt"], args["stream"])


def test_ssd_argument_errors(L):
    assert ssd_call(L, seqlen=100) == SHAPE           # seqlen % chunk != 0
    assert ssd_call(L, nheads=6, ngroups=4) == SHAPE
    assert ssd_call(L, chunk=0) == SHAPE
    assert ssd_call(L, batch=-1) == SHAPE
    assert ssd_call(L, in_dt=9) == DTYPE
    assert ssd_call(L, chunk=32) == UNSUP
    assert ssd_call(L, headdim=32) == UNSUP
    assert ssd_call(L, dstate=64) == UNSUP
    assert ssd_call(L, in_dt=0) == UNSUP
    assert ssd_call(L, x=None) == NULL
    assert ssd_call(L, y=P(3)) == ALIAS
    assert ssd_call(L, x=ctypes.c_void_p(0x10000002)) == ALIGN
    assert ssd_call(L, batch=0, x=None, y=None) == OK
    # the initial state may be the final state itself, nothing else that is written
    assert ssd_call(L, h0=P(5)) == ALIAS               # initial state on top of y
    assert ssd_call(L, h0=ctypes.c_void_p(0x70000000 + 4096)) == ALIAS  # inside final_state
    assert ssd_call(L, h0=ctypes.c_void_p(0x10000008)) == ALIGN


def decode_call(L, **kw):
    args = dict(state=P(0), x=P(1), dt=P(2), A=P(3), B=P(4), C=P(5), D=None, z=None, y=P(6),
                batch=4, nheads=8, headdim=64, dstate=128, ngroups=1, dtype=0, stream=None)
    args.update(kw)
    return L.ssm_decode_step(args["state"], args["x"], args["dt"], args["A"], args["B"],
                             args["C"], args["D"], args["z"], args["y"], args["batch"],
                             args["nheads"], args["headdim"], args["dstate"], args["ngroups"],
                             args["dtype"], args["stream"])


def test_decode_argument_errors(L):
    assert decode_call(L, state=None) == NULL
    assert decode_call(L, y=None) == NULL
    assert decode_call(L, nheads=6, ngroups=4) == SHAPE
    assert decode_call(L, dstate=48) == UNSUP
    assert decode_call(L, dstate=96) == UNSUP   # a multiple of 32 with no kernel build
    assert decode_call(L, dstate=512) == UNSUP
    assert decode_call(L, dtype=3) == DTYPE
    assert decode_call(L, x=ctypes.c_void_p(0x20000004)) == ALIGN
    assert decode_call(L, y=P(1)) == ALIAS
    assert decode_call(L, state=P(4)) == ALIAS
    assert decode_call(L, batch=0, state=None) == OK


def test_binding_refuses_cpu_tensors():
    import torch
    u = torch.zeros(1, 4, 8)
    with pytest.raises(TypeError):
        binding.ssm_scan_fwd(u, u, torch.zeros(4, 16), torch.zeros(1, 1, 16, 8),
                             torch.zeros(1, 1, 16, 8))


def m3_ssd_call(L, **kw):
    args = dict(x=P(0), dt=P(1), lam=P(7), A=P(2), B=P(3), C=P(4), chunk=64, h0=None, pB=None,
                px=None, y=P(5), fs=P(6), batch=2, seqlen=128, nheads=4, headdim=64, dstate=128,
                ngroups=1, in_dt=1, out_dt=0, stream=None)
    args.update(kw)
    a = args
    return L.ssd_mamba3_fwd(a["x"], a["dt"], a["lam"], a["A"], a["B"], a["C"], a["chunk"], a["h0"],
                            a["pB"], a["px"], a["y"], a["fs"], a["batch"], a["seqlen"],
                            a["nheads"], a["headdim"], a["dstate"], a["ngroups"], a["in_dt"],
                            a["out_dt"], a["stream"])


def test_mamba3_ssd_argument_errors(L):
    assert m3_ssd_call(L, seqlen=100) == SHAPE
    assert m3_ssd_call(L, lam=None) == NULL
    assert m3_ssd_call(L, pB=P(8)) == NULL              # prev_B without prev_x
    assert m3_ssd_call(L, px=P(8)) == NULL              # prev_x without prev_B
    assert m3_ssd_call(L, dstate=64) == UNSUP
    assert m3_ssd_call(L, lam=P(5)) == ALIAS            # lambda on top of y
    assert m3_ssd_call(L, lam=ctypes.c_void_p(0x80000004)) == ALIGN
    assert m3_ssd_call(L, batch=0, x=None, y=None) == OK


def m3_decode_call(L, **kw):
    args = dict(state=P(0), pB=P(1), px=P(2), x=P(3), dt=P(4), lam=P(5), A=P(6), B=P(7), C=P(8),
                D=None, z=None, y=P(9), batch=2, nheads=4, headdim=64, dstate=128, ngroups=1,
                dtype=0, stream=None)
    args.update(kw)
    a = args
    return L.ssm_decode_step_mamba3(a["state"], a["pB"], a["px"], a["x"], a["dt"], a["lam"],
                                    a["A"], a["B"], a["C"], a["D"], a["z"], a["y"], a["batch"],
                                    a["nheads"], a["headdim"], a["dstate"], a["ngroups"],
                                    a["dtype"], a["stream"])


def test_mamba3_decode_argument_errors(L):
    assert m3_decode_call(L, lam=None) == NULL
    assert m3_decode_call(L, pB=None) == NULL
    assert m3_decode_call(L, px=None) == NULL
    assert m3_decode_call(L, dstate=48) == UNSUP
    assert m3_decode_call(L, nheads=6, ngroups=4) == SHAPE
    assert m3_decode_call(L, px=P(0)) == ALIAS          # previous x inside the state
    assert m3_decode_call(L, y=P(1)) == ALIAS           # y on top of prev_B
    assert m3_decode_call(L, batch=0) == OK


def test_mimo_argument_errors(L):
    def ssd(**kw):
        a = dict(x=P(0), dt=P(1), lam=P(7), A=P(2), B=P(3), C=P(4), chunk=16, rank=4, h0=None,
                 pB=None, px=None, y=P(5), fs=P(6), batch=2, seqlen=32, nheads=4, headdim=64,
                 dstate=128, ngroups=1, in_dt=1, out_dt=0, stream=None)
        a.update(kw)
        return L.ssd_mamba3_mimo_fwd(a["x"], a["dt"], a["lam"], a["A"], a["B"], a["C"],
                                     a["chunk"], a["rank"], a["h0"], a["pB"], a["px"], a["y"],
                                     a["fs"], a["batch"], a["seqlen"], a["nheads"], a["headdim"],
                                     a["dstate"], a["ngroups"], a["in_dt"], a["out_dt"],
                                     a["stream"])
    assert ssd(rank=3, chunk=16) == UNSUP              # rank 3 unsupported
    assert ssd(chunk=64, seqlen=64) == UNSUP           # chunk * rank must be 64
    assert ssd(seqlen=40) == SHAPE                     # seqlen % chunk
    assert ssd(rank=0) == SHAPE
    assert ssd(lam=None) == NULL
    assert ssd(pB=P(8)) == NULL
    assert ssd(batch=0, x=None, y=None) == OK

    def dec(**kw):
        a = dict(state=P(0), pB=P(1), px=P(2), x=P(3), dt=P(4), lam=P(5), A=P(6), B=P(7),
                 C=P(8), D=None, z=None, y=P(9), batch=2, rank=4, nheads=4, headdim=64,
                 dstate=128, ngroups=1, dtype=0, stream=None)
        a.update(kw)
        return L.ssm_decode_step_mamba3_mimo(a["state"], a["pB"], a["px"], a["x"], a["dt"],
                                             a["lam"], a["A"], a["B"], a["C"], a["D"], a["z"],
                                             a["y"], a["batch"], a["rank"], a["nheads"],
                                             a["headdim"], a["dstate"], a["ngroups"], a["dtype"],
                                             a["stream"])
    assert dec(dstate=64) == UNSUP                     # MIMO decode runs dstate 128 only
    assert dec(rank=3) == UNSUP
    assert dec(rank=0) == SHAPE
    assert dec(lam=None) == NULL
    assert dec(y=P(1)) == ALIAS
    assert dec(batch=0) == OK


def bwd_call(L, **kw):
    args = dict(u=P(0), delta=P(1), A=P(2), B=P(3), C=P(4), D=None, z=None, bias=None,
                softplus=1, h0=None, dy=P(5), dfs=None, du=P(6), ddelta=P(7), dA=P(8), dB=P(9),
                dC=P(10), dD=None, dz=None, dbias=None, dh0=None, batch=2, dim=32, seqlen=64,
                dstate=16, ngroups=1, in_dt=1, ws=P(11), wsb=1 << 30, stream=None)
    args.update(kw)
    a = args
    return L.ssm_scan_bwd(a["u"], a["delta"], a["A"], a["B"], a["C"], a["D"], a["z"], a["bias"],
                          a["softplus"], a["h0"], a["dy"], a["dfs"], a.get("ck"), a["du"],
                          a["ddelta"],
                          a["dA"], a["dB"], a["dC"], a["dD"], a["dz"], a["dbias"], a["dh0"],
                          a["batch"], a["dim"], a["seqlen"], a["dstate"], a["ngroups"],
                          a["in_dt"], a["ws"], a["wsb"], a["stream"])


def test_scan_bwd_argument_errors(L):
    assert bwd_call(L, u=None) == NULL
    assert bwd_call(L, dy=None) == NULL
    assert bwd_call(L, du=None) == NULL
    assert bwd_call(L, dB=None) == NULL
    assert bwd_call(L, dA=None) == NULL
    assert bwd_call(L, z=P(12), dz=None) == NULL      # dz required with a gate
    assert bwd_call(L, batch=-1) == SHAPE
    assert bwd_call(L, ngroups=3) == SHAPE
    assert bwd_call(L, dstate=8) == UNSUP
    assert bwd_call(L, in_dt=5) == DTYPE
    assert bwd_call(L, dA=ctypes.c_void_p(0x90000004)) == ALIGN
    assert bwd_call(L, ws=None) == WS
    assert bwd_call(L, wsb=64) == WS
    assert bwd_call(L, du=P(0)) == ALIAS              # du on top of u
    assert bwd_call(L, dC=P(9)) == ALIAS              # two outputs on one buffer
    assert bwd_call(L, dD=P(13), dbias=P(13)) == ALIAS
    assert bwd_call(L, ws=P(5)) == ALIAS              # workspace on top of dy
    assert bwd_call(L, ws=P(8)) == ALIAS              # workspace on top of dA
    assert bwd_call(L, ck=ctypes.c_void_p(0x90000008)) == ALIGN
    assert bwd_call(L, du=P(12), ck=P(12)) == ALIAS    # checkpoints under an output
    # no channels: nothing to write, nothing launched
    assert bwd_call(L, dim=0, u=None, dA=None, du=None) == OK


def test_scan_bwd_workspace_bytes():
    f, fw = binding.ssm_scan_bwd_workspace_bytes, binding.ssm_scan_workspace_bytes
    assert f(8, 1536, 2048) == f(8, 1536, 2048) > fw(8, 1536, 2048)
    # checkpoints every 16 steps (64 bytes a channel) and the channel blocks' dB, dC partials
    assert f(8, 1536, 2048) >= fw(8, 1536, 2048) + 128 * 8 * 1536 * 64 + 48 * 8 * 2048 * 128
    assert f(1, 10, 5, dstate=8) == 0
    assert f(1, 10, 5, ngroups=3) == 0
    assert f(-1, 10, 5) == 0


def ssd_bwd_call(L, **kw):
    args = dict(x=P(0), dt=P(1), A=P(2), B=P(3), C=P(4), chunk=64, h0=None, dy=P(5), dfs=None,
                dx=P(6), ddt=P(7), dA=P(8), dB=P(9), dC=P(10), dh0=None, batch=2, seqlen=128,
                nheads=4, headdim=64, dstate=128, ngroups=1, in_dt=1, ws=P(11), wsb=1 << 30,
                stream=None)
    args.update(kw)
    a = args
    return L.ssd_chunked_bwd(a["x"], a["dt"], a["A"], a["B"], a["C"], a["chunk"], a["h0"], a["dy"],
                             a["dfs"], a.get("bs"), a["dx"], a["ddt"], a["dA"], a["dB"], a["dC"],
                             a["dh0"],
                             a["batch"], a["seqlen"], a["nheads"], a["headdim"], a["dstate"],
                             a["ngroups"], a["in_dt"], a["ws"], a["wsb"], a["stream"])


def test_ssd_bwd_argument_errors(L):
    assert ssd_bwd_call(L, x=None) == NULL
    assert ssd_bwd_call(L, dy=None) == NULL
    assert ssd_bwd_call(L, dC=None) == NULL
    assert ssd_bwd_call(L, dA=None) == NULL
    assert ssd_bwd_call(L, seqlen=100) == SHAPE       # not a multiple of the chunk
    assert ssd_bwd_call(L, ngroups=3) == SHAPE
    assert ssd_bwd_call(L, batch=-1) == SHAPE
    assert ssd_bwd_call(L, chunk=32, seqlen=128) == UNSUP
    assert ssd_bwd_call(L, headdim=32) == UNSUP
    assert ssd_bwd_call(L, dstate=64) == UNSUP
    assert ssd_bwd_call(L, in_dt=0) == UNSUP          # fp32 activations: not implemented
    assert ssd_bwd_call(L, in_dt=9) == DTYPE
    assert ssd_bwd_call(L, dx=ctypes.c_void_p(0x70000008)) == ALIGN
    assert ssd_bwd_call(L, ws=None) == WS
    assert ssd_bwd_call(L, wsb=1024) == WS
    assert ssd_bwd_call(L, dx=P(0)) == ALIAS           # dx on top of x
    assert ssd_bwd_call(L, dC=P(9)) == ALIAS           # dB and dC on one buffer
    assert ssd_bwd_call(L, ws=P(8)) == ALIAS           # workspace on top of dA
    assert ssd_bwd_call(L, bs=P(6)) == ALIAS           # block states under dx
    # no heads: nothing to write
    assert ssd_bwd_call(L, nheads=0, dA=None, x=None) == OK


def test_ssd_bwd_workspace_bytes():
    f = binding.ssd_chunked_bwd_workspace_bytes
    # block states (3 per (batch, head) for 256 steps) and the per-head dB, dC partials
    assert f(32, 256, 32) >= 32 * 32 * 3 * 64 * 128 * 4 + 2 * 32 * 32 * 256 * 128 * 4
    assert f(32, 256, 32) == f(32, 256, 32)
    assert f(1, 64, 2, headdim=32) == 0
    assert f(1, 64, 3, ngroups=2) == 0


def m3_bwd_call(L, **kw):
    args = dict(x=P(0), dt=P(1), lam=P(12), A=P(2), B=P(3), C=P(4), chunk=64, h0=None,
                pB=None, px=None, dy=P(5), dfs=None, dx=P(6), ddt=P(7), dlam=P(13), dA=P(8),
                dB=P(9), dC=P(10), dh0=None, dpB=None, dpx=None, batch=2, seqlen=128, nheads=4,
                headdim=64, dstate=128, ngroups=1, in_dt=1, ws=P(11), wsb=1 << 30, stream=None)
    args.update(kw)
    a = args
    return L.ssd_mamba3_bwd(a["x"], a["dt"], a["lam"], a["A"], a["B"], a["C"], a["chunk"],
                            a["h0"], a["pB"], a["px"], a["dy"], a["dfs"], a.get("bs"), a["dx"],
                            a["ddt"],
                            a["dlam"], a["dA"], a["dB"], a["dC"], a["dh0"], a["dpB"], a["dpx"],
                            a["batch"], a["seqlen"], a["nheads"], a["headdim"], a["dstate"],
                            a["ngroups"], a["in_dt"], a["ws"], a["wsb"], a["stream"])


def test_mamba3_bwd_argument_errors(L):
    assert m3_bwd_call(L, lam=None) == NULL
    assert m3_bwd_call(L, dlam=None) == NULL
    assert m3_bwd_call(L, dy=None) == NULL
    assert m3_bwd_call(L, pB=P(14)) == NULL              # prev_B without prev_x
    assert m3_bwd_call(L, pB=P(14), px=P(15)) == NULL    # previous token without its gradients
    assert m3_bwd_call(L, seqlen=100) == SHAPE
    assert m3_bwd_call(L, ngroups=3) == SHAPE
    assert m3_bwd_call(L, chunk=32) == UNSUP
    assert m3_bwd_call(L, dstate=64) == UNSUP
    assert m3_bwd_call(L, in_dt=0) == UNSUP
    assert m3_bwd_call(L, in_dt=9) == DTYPE
    assert m3_bwd_call(L, dlam=ctypes.c_void_p(0x70000008)) == ALIGN
    assert m3_bwd_call(L, ws=None) == WS
    assert m3_bwd_call(L, wsb=1024) == WS
    assert m3_bwd_call(L, dlam=P(12)) == ALIAS             # dlam on top of lam
    assert m3_bwd_call(L, dlam=P(7)) == ALIAS              # dlam and ddt on one buffer
    assert m3_bwd_call(L, pB=P(14), px=P(15), dpB=P(16), dpx=P(16)) == ALIAS
    assert m3_bwd_call(L, bs=P(6)) == ALIAS                # block states under dx
    assert m3_bwd_call(L, bs=ctypes.c_void_p(0x70000008)) == ALIGN
    assert m3_bwd_call(L, nheads=8192, ngroups=1) == UNSUP  # per-step shared memory
    assert m3_bwd_call(L, nheads=0, dA=None, x=None) == OK


def test_mamba3_bwd_workspace_bytes():
    f = binding.ssd_mamba3_bwd_workspace_bytes
    assert f(32, 256, 32) > binding.ssd_chunked_bwd_workspace_bytes(32, 256, 32)
    assert f(32, 256, 32) == f(32, 256, 32)
    assert f(1, 64, 2, headdim=32) == 0
    assert f(1, 64, 3, ngroups=2) == 0


def mimo_bwd_call(L, **kw):
    args = dict(x=P(0), dt=P(1), lam=P(12), A=P(2), B=P(3), C=P(4), chunk=16, rank=4, h0=None,
                pB=None, px=None, dy=P(5), dfs=None, dx=P(6), ddt=P(7), dlam=P(13), dA=P(8),
                dB=P(9), dC=P(10), dh0=None, dpB=None, dpx=None, batch=2, seqlen=64, nheads=4,
                headdim=64, dstate=128, ngroups=1, in_dt=1, ws=P(11), wsb=1 << 30, stream=None)
    args.update(kw)
    a = args
    return L.ssd_mamba3_mimo_bwd(a["x"], a["dt"], a["lam"], a["A"], a["B"], a["C"], a["chunk"],
                                 a["rank"], a["h0"], a["pB"], a["px"], a["dy"], a["dfs"],
                                 a.get("bs"), a["dx"],
                                 a["ddt"], a["dlam"], a["dA"], a["dB"], a["dC"], a["dh0"],
                                 a["dpB"], a["dpx"], a["batch"], a["seqlen"], a["nheads"],
                                 a["headdim"], a["dstate"], a["ngroups"], a["in_dt"], a["ws"],
                                 a["wsb"], a["stream"])


def test_mimo_bwd_argument_errors(L):
    assert mimo_bwd_call(L, lam=None) == NULL
    assert mimo_bwd_call(L, px=P(15)) == NULL            # prev_x without prev_B
    assert mimo_bwd_call(L, pB=P(14), px=P(15)) == NULL  # previous token without its gradients
    assert mimo_bwd_call(L, seqlen=60) == SHAPE          # not a multiple of the chunk
    assert mimo_bwd_call(L, rank=0) == SHAPE
    assert mimo_bwd_call(L, rank=3, chunk=16) == UNSUP
    assert mimo_bwd_call(L, rank=4, chunk=32) == UNSUP   # chunk * rank != 64
    assert mimo_bwd_call(L, in_dt=0) == UNSUP
    assert mimo_bwd_call(L, dx=ctypes.c_void_p(0x70000008)) == ALIGN
    assert mimo_bwd_call(L, wsb=1024) == WS
    assert mimo_bwd_call(L, dB=P(3)) == ALIAS             # dB on top of B
    assert mimo_bwd_call(L, nheads=512, ngroups=1) == UNSUP  # per-step shared memory
    assert mimo_bwd_call(L, nheads=0, dA=None, x=None) == OK


def test_mimo_bwd_workspace_bytes():
    f = binding.ssd_mamba3_mimo_bwd_workspace_bytes
    assert f(32, 256, 4, 32) > binding.ssd_chunked_bwd_workspace_bytes(32, 1024, 32)
    assert f(2, 64, 3, 4) == 0
    assert f(1, 64, 4, 3, ngroups=2) == 0


def host_call(L, **kw):
    args = dict(u=P(0), delta=P(1), A=P(2), B=P(3), C=P(4), D=None, z=None, bias=None,
                softplus=1, h0=None, y=P(5), fs=None, batch=2, dim=32, seqlen=64, dstate=16,
                ngroups=1, in_dt=1, out_dt=0, ws=P(7), wsb=1 << 30, stream=None)
    args.update(kw)
    a = args
    return L.ssm_scan_fwd_host(a["u"], a["delta"], a["A"], a["B"], a["C"], a["D"], a["z"],
                               a["bias"], a["softplus"], a["h0"], a["y"], a["fs"], a["batch"],
                               a["dim"], a["seqlen"], a["dstate"], a["ngroups"], a["in_dt"],
                               a["out_dt"], a["ws"], a["wsb"], a["stream"])


def test_scan_host_argument_errors(L):
    assert host_call(L, u=None) == NULL
    assert host_call(L, y=None) == NULL
    assert host_call(L, A=None) == NULL
    assert host_call(L, ws=None) == WS
    assert host_call(L, wsb=64) == WS
    assert host_call(L, batch=-1) == SHAPE
    assert host_call(L, ngroups=3) == SHAPE
    assert host_call(L, dstate=8) == UNSUP
    assert host_call(L, in_dt=4) == DTYPE
    assert host_call(L, A=ctypes.c_void_p(0x30000004)) == ALIGN
    assert host_call(L, dim=0, u=None, y=None) == OK    # no rows: nothing to do
    f = binding.ssm_scan_fwd_host_workspace_bytes
    assert f(8, 1536, 2048) == f(8, 1536, 2048) > 0
    # two slots of about an eighth of the sequence (u, delta, z, B, C in, y out)
    assert f(8, 1536, 2048) >= 2 * (8 * 1536 * 256 * (3 * 2 + 4))
    assert f(8, 1536, 2048, dstate=8) == 0


def test_scan_host_segments_capped_on_long_sequences():
    """On a long sequence the host path's segments are capped at the
    sequence-parallel scan's 3072 channels, whatever the problem's channel count;
    on a short one (a capped segment would move under 32 MB) a segment stays about
    an eighth of the (batch, channel) rows."""
    f = binding.ssm_scan_fwd_host_workspace_bytes
    # 16 x 4096 rows, 4 groups of 1024 channels, bf16 in / fp32 out: 10 bytes per
    # row-step.  Capped: segments of 3 groups (3072 rows) and 1 group.
    L = 4096
    capped = 4 * 3072 * L * 10 + binding.ssm_scan_workspace_bytes(1, 3072, L, 16, 3)
    assert 0 < f(16, 4096, L, ngroups=4) <= 1.05 * capped
    # an eighth of the rows (8192) per slot, as without the cap
    assert f(16, 4096, L, ngroups=4) < 4 * 8192 * L * 10
    # L 64: a 3072-row segment would move 2 MB, so segments stay 8192 rows
    assert f(16, 4096, 64, ngroups=4) >= 4 * 8192 * 64 * 10


def rope_call(L, **kw):
    args = dict(B=P(0), C=P(1), dt=P(2), theta=P(3), a0=None, Br=P(4), Cr=P(5), aout=P(6),
                batch=2, seqlen=8, rank=1, nheads=4, ngroups=2, dstate=16, dtype=1, stream=None)
    args.update(kw)
    return L.ssm_mamba3_rope(args["B"], args["C"], args["dt"], args["theta"], args["a0"],
                             args["Br"], args["Cr"], args["aout"], args["batch"],
                             args["seqlen"], args["rank"], args["nheads"], args["ngroups"],
                             args["dstate"], args["dtype"], args["stream"])


def test_rope_rejects_bad_arguments_on_the_host(L):
    assert rope_call(L, dstate=15) == SHAPE          # state pairs need an even dstate
    assert rope_call(L, ngroups=3) == SHAPE          # heads not a multiple of groups
    assert rope_call(L, rank=0) == SHAPE
    assert rope_call(L, batch=-1) == SHAPE
    assert rope_call(L, dtype=7) == DTYPE
    assert rope_call(L, B=None) == NULL
    assert rope_call(L, Cr=None) == NULL
    assert rope_call(L, theta=ctypes.c_void_p(0x10000008)) == ALIGN
    assert rope_call(L, Br=P(0)) == ALIAS            # output over an input
    assert rope_call(L, Cr=P(4)) == ALIAS            # the two outputs overlap
    assert rope_call(L, batch=0) == OK               # nothing to do, nothing launched
    # a tile's (step, rank, head) offsets must fit in int: 32 steps x 2^20 heads x 128
    far = [ctypes.c_void_p(0x10000000000 * (i + 1)) for i in range(7)]
    assert rope_call(L, B=far[0], C=far[1], dt=far[2], theta=far[3], Br=far[4], Cr=far[5],
                     aout=far[6], nheads=1 << 20, ngroups=1 << 20, dstate=128) == UNSUP
