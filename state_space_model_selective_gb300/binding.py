"""Thin Python binding of ``libssm.so`` (ctypes; argument marshalling only).

Every function here has the name of the C entry point it calls.  Tensors
are torch CUDA tensors; this module only checks that they are contiguous
CUDA tensors of the expected dtype, allocates outputs when the caller does
not pass them (PyTorch is the memory allocator), and passes raw pointers
and the current CUDA stream.  All arithmetic happens in the library's
kernels.  There is no fallback: if the library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libssm.so")

SSM_F32, SSM_BF16 = 0, 1
_DT = {torch.float32: SSM_F32, torch.bfloat16: SSM_BF16}
_TORCH_DT = {SSM_F32: torch.float32, SSM_BF16: torch.bfloat16}

STATUS_NAMES = {0: "SSM_OK", 1: "SSM_ERR_NULL", 2: "SSM_ERR_SHAPE", 3: "SSM_ERR_ALIGN",
                4: "SSM_ERR_DTYPE", 5: "SSM_ERR_UNSUPPORTED", 6: "SSM_ERR_WORKSPACE",
                7: "SSM_ERR_TIMEOUT", 8: "SSM_ERR_CUDA", 9: "SSM_ERR_ALIAS"}

# every symbol include/ssm.h declares
EXPORTS = ["ssm_abi_version", "ssm_status_string", "ssm_scan_workspace_bytes", "ssm_scan_fwd",
           "ssd_chunked_fwd", "ssd_mamba3_fwd", "ssd_mamba3_mimo_fwd", "ssm_decode_step",
           "ssm_decode_step_mamba3", "ssm_decode_step_mamba3_mimo", "ssm_last_device_status",
           "ssm_scan_fwd_noalloc", "ssm_scan_bwd_workspace_bytes", "ssm_scan_bwd",
           "ssd_chunked_bwd_workspace_bytes", "ssd_chunked_bwd", "ssm_scan_fwd_host_workspace_bytes",
           "ssm_scan_fwd_host", "ssm_scan_checkpoint_bytes", "ssm_scan_fwd_ckpt",
           "ssd_chunked_checkpoint_bytes", "ssd_chunked_fwd_ckpt", "ssd_mamba3_bwd_workspace_bytes",
           "ssd_mamba3_bwd", "ssd_mamba3_mimo_bwd_workspace_bytes", "ssd_mamba3_mimo_bwd",
           "ssd_mamba3_fwd_ckpt", "ssd_mamba3_mimo_fwd_ckpt", "ssm_debug_set_lookback",
           "ssm_debug_set_scan_path", "ssm_noalloc_last_status", "ssm_mamba3_rope"]


class SSMError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)} "
                         f"({status_string(status)})")


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it first "
                               "(python -c 'import __graft_entry__ as g; g.build()')")
        L = ctypes.CDLL(LIB_PATH)
        vp, i, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        L.ssm_abi_version.restype = i
        L.ssm_status_string.restype = ctypes.c_char_p
        L.ssm_status_string.argtypes = [i]
        L.ssm_scan_workspace_bytes.restype = sz
        L.ssm_scan_workspace_bytes.argtypes = [i] * 5
        L.ssm_scan_fwd.restype = i
        L.ssm_scan_fwd.argtypes = [vp] * 8 + [i] + [vp] * 3 + [i] * 7 + [vp, sz, vp]
        L.ssd_chunked_fwd.restype = i
        L.ssd_chunked_fwd.argtypes = [vp] * 5 + [i] + [vp] * 3 + [i] * 8 + [vp]
        L.ssm_decode_step.restype = i
        L.ssm_decode_step.argtypes = [vp] * 9 + [i] * 6 + [vp]
        L.ssd_mamba3_fwd.restype = i
        L.ssd_mamba3_fwd.argtypes = [vp] * 6 + [i] + [vp] * 5 + [i] * 8 + [vp]
        L.ssm_decode_step_mamba3.restype = i
        L.ssm_decode_step_mamba3.argtypes = [vp] * 12 + [i] * 6 + [vp]
        L.ssd_mamba3_mimo_fwd.restype = i
        L.ssd_mamba3_mimo_fwd.argtypes = [vp] * 6 + [i] * 2 + [vp] * 5 + [i] * 8 + [vp]
        L.ssm_decode_step_mamba3_mimo.restype = i
        L.ssm_decode_step_mamba3_mimo.argtypes = [vp] * 12 + [i] * 7 + [vp]
        L.ssm_scan_fwd_noalloc.restype = i
        L.ssm_scan_fwd_noalloc.argtypes = [vp] * 8 + [i] + [vp] * 3 + [i] * 7 + [vp]
        L.ssm_scan_bwd_workspace_bytes.restype = sz
        L.ssm_scan_bwd_workspace_bytes.argtypes = [i] * 5
        L.ssm_scan_bwd.restype = i
        L.ssm_scan_bwd.argtypes = [vp] * 8 + [i] + [vp] * 13 + [i] * 6 + [vp, sz, vp]
        L.ssm_scan_checkpoint_bytes.restype = sz
        L.ssm_scan_checkpoint_bytes.argtypes = [i] * 4
        L.ssm_scan_fwd_ckpt.restype = i
        L.ssm_scan_fwd_ckpt.argtypes = [vp] * 8 + [i] + [vp] * 4 + [i] * 7 + [vp, sz, vp]
        L.ssd_chunked_bwd_workspace_bytes.restype = sz
        L.ssd_chunked_bwd_workspace_bytes.argtypes = [i] * 6
        L.ssd_chunked_bwd.restype = i
        L.ssd_chunked_bwd.argtypes = [vp] * 5 + [i] + [vp] * 10 + [i] * 7 + [vp, sz, vp]
        L.ssd_mamba3_bwd_workspace_bytes.restype = sz
        L.ssd_mamba3_bwd_workspace_bytes.argtypes = [i] * 6
        L.ssd_mamba3_bwd.restype = i
        L.ssd_mamba3_bwd.argtypes = [vp] * 6 + [i] + [vp] * 15 + [i] * 7 + [vp, sz, vp]
        L.ssd_mamba3_fwd_ckpt.restype = i
        L.ssd_mamba3_fwd_ckpt.argtypes = [vp] * 6 + [i] + [vp] * 6 + [i] * 7 + [vp]
        L.ssd_mamba3_mimo_fwd_ckpt.restype = i
        L.ssd_mamba3_mimo_fwd_ckpt.argtypes = [vp] * 6 + [i, i] + [vp] * 6 + [i] * 7 + [vp]
        L.ssd_mamba3_mimo_bwd_workspace_bytes.restype = sz
        L.ssd_mamba3_mimo_bwd_workspace_bytes.argtypes = [i] * 7
        L.ssd_mamba3_mimo_bwd.restype = i
        L.ssd_mamba3_mimo_bwd.argtypes = [vp] * 6 + [i, i] + [vp] * 15 + [i] * 7 + [vp, sz, vp]
        L.ssd_chunked_checkpoint_bytes.restype = sz
        L.ssd_chunked_checkpoint_bytes.argtypes = [i] * 5
        L.ssd_chunked_fwd_ckpt.restype = i
        L.ssd_chunked_fwd_ckpt.argtypes = [vp] * 5 + [i] + [vp] * 4 + [i] * 8 + [vp]
        L.ssm_scan_fwd_host_workspace_bytes.restype = sz
        L.ssm_scan_fwd_host_workspace_bytes.argtypes = [i] * 7
        L.ssm_scan_fwd_host.restype = i
        L.ssm_scan_fwd_host.argtypes = [vp] * 8 + [i] + [vp] * 3 + [i] * 7 + [vp, sz, vp]
        L.ssm_last_device_status.restype = i
        L.ssm_last_device_status.argtypes = [vp, vp]
        L.ssm_debug_set_lookback.restype = i
        L.ssm_debug_set_lookback.argtypes = [i, ctypes.c_uint]
        L.ssm_debug_set_scan_path.restype = i
        L.ssm_debug_set_scan_path.argtypes = [i, i]
        L.ssm_noalloc_last_status.restype = i
        L.ssm_noalloc_last_status.argtypes = [vp]
        L.ssm_mamba3_rope.restype = i
        L.ssm_mamba3_rope.argtypes = [vp] * 8 + [i] * 7 + [vp]
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().ssm_status_string(int(status)).decode()


def ssm_abi_version() -> int:
    return int(lib().ssm_abi_version())


def _check(status: int, where: str):
    if status != 0:
        raise SSMError(status, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _req(t, name, dtype=None, ndim=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {t.dim()}")
    return t


def _opt(t, name, dtype=None, ndim=None):
    return None if t is None else _req(t, name, dtype, ndim)


def _shape(t, name, shape):
    """Raises ValueError unless tensor ``t`` (when given) has exactly ``shape``."""
    if t is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _scan_shapes(u, delta, A, B, C, D, z, delta_bias, initial_state, y, final_state,
                 dy=None, dfinal_state=None):
    """Checks every scan tensor against u's (batch, dim, seqlen), A's dstate and
    B's ngroups, so that no kernel reads or writes past a buffer the caller passed."""
    batch, dim, seqlen = u.shape
    if A.dim() != 2 or A.shape[0] != dim:
        raise ValueError(f"A must have shape ({dim}, dstate), got {tuple(A.shape)}")
    dstate = A.shape[1]
    if B.dim() != 4 or B.shape[0] != batch or B.shape[2] != dstate or B.shape[3] != seqlen:
        raise ValueError(f"B must have shape ({batch}, ngroups, {dstate}, {seqlen}), "
                         f"got {tuple(B.shape)}")
    ngroups = B.shape[1]
    act = (batch, dim, seqlen)
    _shape(delta, "delta", act)
    _shape(z, "z", act)
    _shape(y, "y", act)
    _shape(dy, "dy", act)
    _shape(C, "C", (batch, ngroups, dstate, seqlen))
    _shape(D, "D", (dim,))
    _shape(delta_bias, "delta_bias", (dim,))
    for t, name in ((initial_state, "initial_state"), (final_state, "final_state"),
                    (dfinal_state, "dfinal_state")):
        _shape(t, name, (batch, dim, dstate))
    return batch, dim, seqlen, dstate, ngroups


def _use_out(g, out):
    """Puts the caller's preallocated fp32 tensors (``out``: name -> tensor) in
    place of the gradient buffers ``g`` would allocate."""
    for k, t in (out or {}).items():
        if k not in g or g[k] is None:
            raise ValueError(f"out[{k!r}] is not an output of this call")
        _req(t, f"out[{k!r}]", torch.float32)
        if t.shape != g[k].shape:
            raise ValueError(f"out[{k!r}] must have shape {tuple(g[k].shape)}")
        g[k] = t


def ssm_scan_workspace_bytes(batch, dim, seqlen, dstate=16, ngroups=1) -> int:
    return int(lib().ssm_scan_workspace_bytes(batch, dim, seqlen, dstate, ngroups))


def ssm_scan_checkpoint_bytes(batch, dim, seqlen, dstate=16) -> int:
    return int(lib().ssm_scan_checkpoint_bytes(batch, dim, seqlen, dstate))


def ssm_scan_fwd(u, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus=False,
                 initial_state=None, out_dtype=None, y=None, final_state=None,
                 workspace=None, return_final_state=True, stream=None, checkpoints=None):
    """Selective scan.  u, delta, z: (batch, dim, seqlen); A: (dim, dstate) fp32;
    B, C: (batch, ngroups, dstate, seqlen); D, delta_bias: (dim,) fp32;
    initial_state: (batch, dim, dstate) fp32.  With ``checkpoints`` (a CUDA fp32
    tensor of ssm_scan_checkpoint_bytes bytes) the states ssm_scan_bwd needs are
    kept too (ssm_scan_fwd_ckpt).  Returns (y, final_state)."""
    _req(u, "u", ndim=3)
    in_dt = u.dtype
    if in_dt not in _DT:
        raise TypeError("u must be float32 or bfloat16")
    batch, dim, seqlen = u.shape
    _req(delta, "delta", in_dt)
    _req(A, "A", torch.float32, 2)
    dstate = A.shape[1]
    _req(B, "B", in_dt, 4)
    _req(C, "C", in_dt, 4)
    ngroups = B.shape[1]
    _opt(D, "D", torch.float32)
    _opt(z, "z", in_dt)
    _opt(delta_bias, "delta_bias", torch.float32)
    _opt(initial_state, "initial_state", torch.float32)
    out_dt = in_dt if out_dtype is None else out_dtype
    if y is None:
        y = torch.empty((batch, dim, seqlen), dtype=out_dt, device=u.device)
    _req(y, "y", out_dt)
    if final_state is None and return_final_state:
        final_state = torch.empty((batch, dim, dstate), dtype=torch.float32, device=u.device)
    _opt(final_state, "final_state", torch.float32)
    _scan_shapes(u, delta, A, B, C, D, z, delta_bias, initial_state, y, final_state)
    need = ssm_scan_workspace_bytes(batch, dim, seqlen, dstate, ngroups)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=u.device)
    _req(workspace, "workspace", torch.uint8)
    if checkpoints is not None:
        _req(checkpoints, "checkpoints", torch.float32)
        if checkpoints.numel() * 4 < ssm_scan_checkpoint_bytes(batch, dim, seqlen, dstate):
            raise ValueError("checkpoints is smaller than ssm_scan_checkpoint_bytes(...)")
        st = lib().ssm_scan_fwd_ckpt(_ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                                     _ptr(z), _ptr(delta_bias), int(bool(delta_softplus)),
                                     _ptr(initial_state), _ptr(y), _ptr(final_state),
                                     _ptr(checkpoints), batch, dim, seqlen, dstate, ngroups,
                                     _DT[in_dt], _DT[out_dt], _ptr(workspace), workspace.numel(),
                                     _stream(stream))
        _check(st, "ssm_scan_fwd_ckpt")
        return y, final_state
    st = lib().ssm_scan_fwd(_ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
                            _ptr(delta_bias), int(bool(delta_softplus)), _ptr(initial_state),
                            _ptr(y), _ptr(final_state), batch, dim, seqlen, dstate, ngroups,
                            _DT[in_dt], _DT[out_dt], _ptr(workspace), workspace.numel(),
                            _stream(stream))
    _check(st, "ssm_scan_fwd")
    return y, final_state


def ssm_scan_bwd_workspace_bytes(batch, dim, seqlen, dstate=16, ngroups=1) -> int:
    return int(lib().ssm_scan_bwd_workspace_bytes(batch, dim, seqlen, dstate, ngroups))


def ssm_scan_bwd(u, delta, A, B, C, dy, D=None, z=None, delta_bias=None, delta_softplus=False,
                 initial_state=None, dfinal_state=None, workspace=None, want_dD=None,
                 want_ddelta_bias=None, want_dinitial_state=True, out=None, stream=None,
                 checkpoints=None):
    """Gradient of ``ssm_scan_fwd`` for the loss sum(dy * y) + sum(dfinal_state *
    final_state).  Inputs as for ``ssm_scan_fwd``; dy (batch, dim, seqlen) in u's
    dtype; dfinal_state (batch, dim, dstate) fp32 or None.  Returns a dict of fp32
    tensors: du, ddelta, dz (batch, dim, seqlen); dA (dim, dstate); dB, dC
    (batch, ngroups, dstate, seqlen); dD, ddelta_bias (dim,); dinitial_state
    (batch, dim, dstate).  dz is None without z; dD / ddelta_bias are computed
    when D / delta_bias is given, or when want_dD / want_ddelta_bias is true.
    ``out`` may map any of these names to a preallocated fp32 tensor to write.
    ``checkpoints``: what ``ssm_scan_fwd(..., checkpoints=...)`` kept for the same
    inputs (the forward recurrence is then not run again)."""
    _req(u, "u", ndim=3)
    in_dt = u.dtype
    if in_dt not in _DT:
        raise TypeError("u must be float32 or bfloat16")
    batch, dim, seqlen = u.shape
    _req(delta, "delta", in_dt)
    _req(A, "A", torch.float32, 2)
    dstate = A.shape[1]
    _req(B, "B", in_dt, 4)
    _req(C, "C", in_dt, 4)
    ngroups = B.shape[1]
    _req(dy, "dy", in_dt, 3)
    _opt(D, "D", torch.float32)
    _opt(z, "z", in_dt)
    _opt(delta_bias, "delta_bias", torch.float32)
    _opt(initial_state, "initial_state", torch.float32)
    _opt(dfinal_state, "dfinal_state", torch.float32)
    _scan_shapes(u, delta, A, B, C, D, z, delta_bias, initial_state, None, None, dy=dy,
                 dfinal_state=dfinal_state)
    dev, f32 = u.device, torch.float32
    g = {"du": torch.empty((batch, dim, seqlen), dtype=f32, device=dev),
         "ddelta": torch.empty((batch, dim, seqlen), dtype=f32, device=dev),
         "dA": torch.empty((dim, dstate), dtype=f32, device=dev),
         "dB": torch.empty(tuple(B.shape), dtype=f32, device=dev),
         "dC": torch.empty(tuple(C.shape), dtype=f32, device=dev),
         "dD": None, "dz": None, "ddelta_bias": None, "dinitial_state": None}
    if D is not None or want_dD:
        g["dD"] = torch.empty(dim, dtype=f32, device=dev)
    if delta_bias is not None or want_ddelta_bias:
        g["ddelta_bias"] = torch.empty(dim, dtype=f32, device=dev)
    if z is not None:
        g["dz"] = torch.empty((batch, dim, seqlen), dtype=f32, device=dev)
    if want_dinitial_state:
        g["dinitial_state"] = torch.empty((batch, dim, dstate), dtype=f32, device=dev)
    _use_out(g, out)
    need = ssm_scan_bwd_workspace_bytes(batch, dim, seqlen, dstate, ngroups)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    _req(workspace, "workspace", torch.uint8)
    st = lib().ssm_scan_bwd(_ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
                            _ptr(delta_bias), int(bool(delta_softplus)), _ptr(initial_state),
                            _ptr(dy), _ptr(dfinal_state), _ptr(_opt(checkpoints, "checkpoints",
                                                                   torch.float32)),
                            _ptr(g["du"]), _ptr(g["ddelta"]),
                            _ptr(g["dA"]), _ptr(g["dB"]), _ptr(g["dC"]), _ptr(g["dD"]),
                            _ptr(g["dz"]), _ptr(g["ddelta_bias"]), _ptr(g["dinitial_state"]),
                            batch, dim, seqlen, dstate, ngroups, _DT[in_dt], _ptr(workspace),
                            workspace.numel(), _stream(stream))
    _check(st, "ssm_scan_bwd")
    return g


def ssm_scan_fwd_host_workspace_bytes(batch, dim, seqlen, dstate=16, ngroups=1,
                                      in_dtype=torch.bfloat16, out_dtype=torch.float32) -> int:
    return int(lib().ssm_scan_fwd_host_workspace_bytes(batch, dim, seqlen, dstate, ngroups,
                                                       _DT[in_dtype], _DT[out_dtype]))


def _pinned(t, name, dtype=None, ndim=None):
    # an empty tensor is never read or written, and may not be page-locked
    if (not isinstance(t, torch.Tensor) or t.is_cuda
            or (t.numel() > 0 and not t.is_pinned())):
        raise TypeError(f"{name} must be a pinned (page-locked) CPU tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {t.dim()}")
    return t


def ssm_scan_fwd_host(u, delta, A, B, C, y, final_state=None, D=None, z=None, delta_bias=None,
                      delta_softplus=False, initial_state=None, workspace=None, stream=None):
    """``ssm_scan_fwd`` on pinned host tensors: u, delta, z, B, C, initial_state, y and
    final_state are pinned CPU tensors (same layouts); A, D, delta_bias and the workspace
    are CUDA tensors.  The copies in and out are pipelined with the scan on the library's
    copy streams; the call returns once everything is enqueued on ``stream``."""
    _pinned(u, "u", ndim=3)
    in_dt = u.dtype
    if in_dt not in _DT:
        raise TypeError("u must be float32 or bfloat16")
    batch, dim, seqlen = u.shape
    _pinned(delta, "delta", in_dt)
    _req(A, "A", torch.float32, 2)
    dstate = A.shape[1]
    _pinned(B, "B", in_dt, 4)
    _pinned(C, "C", in_dt, 4)
    ngroups = B.shape[1]
    _opt(D, "D", torch.float32)
    _opt(delta_bias, "delta_bias", torch.float32)
    if z is not None:
        _pinned(z, "z", in_dt)
    if initial_state is not None:
        _pinned(initial_state, "initial_state", torch.float32)
    _pinned(y, "y")
    if y.dtype not in _DT:
        raise TypeError("y must be float32 or bfloat16")
    if final_state is not None:
        _pinned(final_state, "final_state", torch.float32)
    _scan_shapes(u, delta, A, B, C, D, z, delta_bias, initial_state, y, final_state)
    need = ssm_scan_fwd_host_workspace_bytes(batch, dim, seqlen, dstate, ngroups, in_dt, y.dtype)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=A.device)
    _req(workspace, "workspace", torch.uint8)
    st = lib().ssm_scan_fwd_host(_ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                                 _ptr(z), _ptr(delta_bias), int(bool(delta_softplus)),
                                 _ptr(initial_state), _ptr(y), _ptr(final_state), batch, dim,
                                 seqlen, dstate, ngroups, _DT[in_dt], _DT[y.dtype],
                                 _ptr(workspace), workspace.numel(), _stream(stream))
    _check(st, "ssm_scan_fwd_host")
    return y, final_state


def ssm_scan_fwd_noalloc(u, delta, A, B, C, y, final_state=None, D=None, z=None,
                         delta_bias=None, delta_softplus=False, initial_state=None, stream=None):
    """The selective scan without a workspace, for callers that cannot
    allocate: its scratch is a fixed array inside the library.  The caller
    passes every input and output (y, and final_state or None); nothing is
    allocated here or in the library.  Same layouts as ssm_scan_fwd."""
    _req(u, "u", ndim=3)
    in_dt = u.dtype
    if in_dt not in _DT:
        raise TypeError("u must be float32 or bfloat16")
    batch, dim, seqlen = u.shape
    _req(delta, "delta", in_dt)
    _req(A, "A", torch.float32, 2)
    _req(B, "B", in_dt, 4)
    _req(C, "C", in_dt, 4)
    _opt(D, "D", torch.float32)
    _opt(z, "z", in_dt)
    _opt(delta_bias, "delta_bias", torch.float32)
    _opt(initial_state, "initial_state", torch.float32)
    _req(y, "y")
    if y.dtype not in _DT:
        raise TypeError("y must be float32 or bfloat16")
    _opt(final_state, "final_state", torch.float32)
    _scan_shapes(u, delta, A, B, C, D, z, delta_bias, initial_state, y, final_state)
    st = lib().ssm_scan_fwd_noalloc(_ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                                    _ptr(z), _ptr(delta_bias), int(bool(delta_softplus)),
                                    _ptr(initial_state), _ptr(y), _ptr(final_state), batch, dim,
                                    seqlen, A.shape[1], B.shape[1], _DT[in_dt], _DT[y.dtype],
                                    _stream(stream))
    _check(st, "ssm_scan_fwd_noalloc")
    return y, final_state


def ssd_chunked_bwd_workspace_bytes(batch, seqlen, nheads, headdim=64, dstate=128,
                                    ngroups=1) -> int:
    return int(lib().ssd_chunked_bwd_workspace_bytes(batch, seqlen, nheads, headdim, dstate,
                                                     ngroups))


def ssd_chunked_checkpoint_bytes(batch, seqlen, nheads, headdim=64, dstate=128) -> int:
    return int(lib().ssd_chunked_checkpoint_bytes(batch, seqlen, nheads, headdim, dstate))


def ssd_chunked_bwd(x, dt, A_head, B, C, dy, chunk=64, initial_state=None, dfinal_state=None,
                    workspace=None, want_dinitial_state=True, out=None, stream=None,
                    block_states=None):
    """Gradient of ``ssd_chunked_fwd`` for the loss sum(dy * y) + sum(dfinal_state *
    final_state).  Inputs as for ``ssd_chunked_fwd``; dy like x (bf16); dfinal_state
    (batch, nheads, headdim, dstate) fp32 or None.  Returns a dict of fp32 tensors:
    dx (like x), ddt (like dt), dA_head (nheads,), dB, dC (like B) and dinitial_state
    (batch, nheads, headdim, dstate, or None).  ``out`` may map any of these names to
    a preallocated fp32 tensor to write.  ``block_states``: what
    ``ssd_chunked_fwd(..., block_states=...)`` kept for the same inputs."""
    _req(x, "x", torch.bfloat16, 4)
    batch, seqlen, nheads, headdim = x.shape
    _req(dt, "dt", torch.float32, 3)
    _req(A_head, "A_head", torch.float32, 1)
    _req(B, "B", torch.bfloat16, 4)
    _req(C, "C", torch.bfloat16, 4)
    _req(dy, "dy", torch.bfloat16, 4)
    ngroups, dstate = B.shape[2], B.shape[3]
    _opt(initial_state, "initial_state", torch.float32)
    _opt(dfinal_state, "dfinal_state", torch.float32)
    dev, f32 = x.device, torch.float32
    g = {"dx": torch.empty(tuple(x.shape), dtype=f32, device=dev),
         "ddt": torch.empty(tuple(dt.shape), dtype=f32, device=dev),
         "dA_head": torch.empty(nheads, dtype=f32, device=dev),
         "dB": torch.empty(tuple(B.shape), dtype=f32, device=dev),
         "dC": torch.empty(tuple(C.shape), dtype=f32, device=dev),
         "dinitial_state": (torch.empty((batch, nheads, headdim, dstate), dtype=f32, device=dev)
                            if want_dinitial_state else None)}
    _use_out(g, out)
    need = ssd_chunked_bwd_workspace_bytes(batch, seqlen, nheads, headdim, dstate, ngroups)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    _req(workspace, "workspace", torch.uint8)
    st = lib().ssd_chunked_bwd(_ptr(x), _ptr(dt), _ptr(A_head), _ptr(B), _ptr(C), int(chunk),
                               _ptr(initial_state), _ptr(dy), _ptr(dfinal_state),
                               _ptr(_opt(block_states, "block_states", torch.float32)),
                               _ptr(g["dx"]),
                               _ptr(g["ddt"]), _ptr(g["dA_head"]), _ptr(g["dB"]), _ptr(g["dC"]),
                               _ptr(g["dinitial_state"]), batch, seqlen, nheads, headdim, dstate,
                               ngroups, _DT[torch.bfloat16], _ptr(workspace), workspace.numel(),
                               _stream(stream))
    _check(st, "ssd_chunked_bwd")
    return g


def ssd_mamba3_bwd_workspace_bytes(batch, seqlen, nheads, headdim=64, dstate=128,
                                   ngroups=1) -> int:
    return int(lib().ssd_mamba3_bwd_workspace_bytes(batch, seqlen, nheads, headdim, dstate,
                                                    ngroups))


def ssd_mamba3_bwd(x, dt, lam, A_head, B, C, dy, chunk=64, initial_state=None, prev_B=None,
                   prev_x=None, dfinal_state=None, workspace=None, want_dinitial_state=True,
                   stream=None, block_states=None, out=None):
    """Gradient of ``ssd_mamba3_fwd`` for the loss sum(dy * y) + sum(dfinal_state *
    final_state).  Inputs as for ``ssd_mamba3_fwd`` (bf16 x, B, C, prev_B, prev_x);
    dy like x (bf16).  Returns a dict of fp32 tensors: dx, ddt, dlam, dA_head, dB, dC,
    dinitial_state (or None) and dprev_B, dprev_x (None without a previous token).
    ``out`` may map any of these names to a preallocated fp32 tensor to write."""
    _req(x, "x", torch.bfloat16, 4)
    batch, seqlen, nheads, headdim = x.shape
    _req(dt, "dt", torch.float32, 3)
    _req(lam, "lam", torch.float32, 3)
    _req(A_head, "A_head", torch.float32, 1)
    _req(B, "B", torch.bfloat16, 4)
    _req(C, "C", torch.bfloat16, 4)
    _req(dy, "dy", torch.bfloat16, 4)
    ngroups, dstate = B.shape[2], B.shape[3]
    _opt(initial_state, "initial_state", torch.float32)
    _opt(dfinal_state, "dfinal_state", torch.float32)
    _opt(prev_B, "prev_B", torch.bfloat16)
    _opt(prev_x, "prev_x", torch.bfloat16)
    has_prev = prev_B is not None
    dev, f32 = x.device, torch.float32
    g = {"dx": torch.empty(tuple(x.shape), dtype=f32, device=dev),
         "ddt": torch.empty(tuple(dt.shape), dtype=f32, device=dev),
         "dlam": torch.empty(tuple(dt.shape), dtype=f32, device=dev),
         "dA_head": torch.empty(nheads, dtype=f32, device=dev),
         "dB": torch.empty(tuple(B.shape), dtype=f32, device=dev),
         "dC": torch.empty(tuple(C.shape), dtype=f32, device=dev),
         "dinitial_state": (torch.empty((batch, nheads, headdim, dstate), dtype=f32, device=dev)
                            if want_dinitial_state else None),
         "dprev_B": (torch.empty((batch, ngroups, dstate), dtype=f32, device=dev)
                     if has_prev else None),
         "dprev_x": (torch.empty((batch, nheads, headdim), dtype=f32, device=dev)
                     if has_prev else None)}
    _use_out(g, out)
    need = ssd_mamba3_bwd_workspace_bytes(batch, seqlen, nheads, headdim, dstate, ngroups)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    _req(workspace, "workspace", torch.uint8)
    st = lib().ssd_mamba3_bwd(_ptr(x), _ptr(dt), _ptr(lam), _ptr(A_head), _ptr(B), _ptr(C),
                              int(chunk), _ptr(initial_state), _ptr(prev_B), _ptr(prev_x),
                              _ptr(dy), _ptr(dfinal_state),
                              _ptr(_opt(block_states, "block_states", torch.float32)),
                              _ptr(g["dx"]), _ptr(g["ddt"]),
                              _ptr(g["dlam"]), _ptr(g["dA_head"]), _ptr(g["dB"]), _ptr(g["dC"]),
                              _ptr(g["dinitial_state"]), _ptr(g["dprev_B"]), _ptr(g["dprev_x"]),
                              batch, seqlen, nheads, headdim, dstate, ngroups,
                              _DT[torch.bfloat16], _ptr(workspace), workspace.numel(),
                              _stream(stream))
    _check(st, "ssd_mamba3_bwd")
    return g


def ssd_mamba3_mimo_bwd_workspace_bytes(batch, seqlen, rank, nheads, headdim=64, dstate=128,
                                        ngroups=1) -> int:
    return int(lib().ssd_mamba3_mimo_bwd_workspace_bytes(batch, seqlen, rank, nheads, headdim,
                                                         dstate, ngroups))


def ssd_mamba3_mimo_bwd(x, dt, lam, A_head, B, C, dy, chunk=None, initial_state=None,
                        prev_B=None, prev_x=None, dfinal_state=None, workspace=None,
                        want_dinitial_state=True, stream=None, block_states=None, out=None):
    """Gradient of ``ssd_mamba3_mimo_fwd``.  x, dy: (batch, seqlen, rank, nheads,
    headdim) bf16; B, C: (batch, seqlen, rank, ngroups, dstate) bf16; prev_B (batch,
    rank, ngroups, dstate), prev_x (batch, rank, nheads, headdim) bf16 or None.
    ``chunk`` defaults to 64 // rank.  Returns a dict of fp32 tensors like
    ``ssd_mamba3_bwd``'s, with dx, dB, dC, dprev_B, dprev_x shaped like their inputs;
    ``out`` as for ``ssd_mamba3_bwd``."""
    _req(x, "x", torch.bfloat16, 5)
    batch, seqlen, rank, nheads, headdim = x.shape
    _req(dt, "dt", torch.float32, 3)
    _req(lam, "lam", torch.float32, 3)
    _req(A_head, "A_head", torch.float32, 1)
    _req(B, "B", torch.bfloat16, 5)
    _req(C, "C", torch.bfloat16, 5)
    _req(dy, "dy", torch.bfloat16, 5)
    ngroups, dstate = B.shape[3], B.shape[4]
    _opt(initial_state, "initial_state", torch.float32)
    _opt(dfinal_state, "dfinal_state", torch.float32)
    _opt(prev_B, "prev_B", torch.bfloat16)
    _opt(prev_x, "prev_x", torch.bfloat16)
    has_prev = prev_B is not None
    chunk = 64 // rank if chunk is None else chunk
    dev, f32 = x.device, torch.float32
    g = {"dx": torch.empty(tuple(x.shape), dtype=f32, device=dev),
         "ddt": torch.empty(tuple(dt.shape), dtype=f32, device=dev),
         "dlam": torch.empty(tuple(dt.shape), dtype=f32, device=dev),
         "dA_head": torch.empty(nheads, dtype=f32, device=dev),
         "dB": torch.empty(tuple(B.shape), dtype=f32, device=dev),
         "dC": torch.empty(tuple(C.shape), dtype=f32, device=dev),
         "dinitial_state": (torch.empty((batch, nheads, headdim, dstate), dtype=f32, device=dev)
                            if want_dinitial_state else None),
         "dprev_B": (torch.empty(tuple(prev_B.shape), dtype=f32, device=dev)
                     if has_prev else None),
         "dprev_x": (torch.empty(tuple(prev_x.shape), dtype=f32, device=dev)
                     if has_prev else None)}
    _use_out(g, out)
    need = ssd_mamba3_mimo_bwd_workspace_bytes(batch, seqlen, rank, nheads, headdim, dstate,
                                               ngroups)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    _req(workspace, "workspace", torch.uint8)
    st = lib().ssd_mamba3_mimo_bwd(_ptr(x), _ptr(dt), _ptr(lam), _ptr(A_head), _ptr(B), _ptr(C),
                                   int(chunk), int(rank), _ptr(initial_state), _ptr(prev_B),
                                   _ptr(prev_x), _ptr(dy), _ptr(dfinal_state),
                                   _ptr(_opt(block_states, "block_states", torch.float32)),
                                   _ptr(g["dx"]),
                                   _ptr(g["ddt"]), _ptr(g["dlam"]), _ptr(g["dA_head"]),
                                   _ptr(g["dB"]), _ptr(g["dC"]), _ptr(g["dinitial_state"]),
                                   _ptr(g["dprev_B"]), _ptr(g["dprev_x"]), batch, seqlen, nheads,
                                   headdim, dstate, ngroups, _DT[torch.bfloat16], _ptr(workspace),
                                   workspace.numel(), _stream(stream))
    _check(st, "ssd_mamba3_mimo_bwd")
    return g


def ssd_chunked_fwd(x, dt, A_head, B, C, chunk=64, out_dtype=None, y=None, final_state=None,
                    return_final_state=True, stream=None, initial_state=None, block_states=None):
    """Chunked SSD.  x: (batch, seqlen, nheads, headdim); dt: (batch, seqlen, nheads) fp32;
    A_head: (nheads,) fp32; B, C: (batch, seqlen, ngroups, dstate); initial_state (optional,
    may be ``final_state`` itself): (batch, nheads, headdim, dstate) fp32.
    Returns (y, final_state)."""
    _req(x, "x", ndim=4)
    in_dt = x.dtype
    if in_dt not in _DT:
        raise TypeError("x must be float32 or bfloat16")
    batch, seqlen, nheads, headdim = x.shape
    _req(dt, "dt", torch.float32, 3)
    _req(A_head, "A_head", torch.float32, 1)
    _req(B, "B", in_dt, 4)
    _req(C, "C", in_dt, 4)
    ngroups, dstate = B.shape[2], B.shape[3]
    out_dt = in_dt if out_dtype is None else out_dtype
    if y is None:
        y = torch.empty_like(x, dtype=out_dt)
    _req(y, "y", out_dt)
    if final_state is None and return_final_state:
        final_state = torch.empty((batch, nheads, headdim, dstate), dtype=torch.float32,
                                  device=x.device)
    _opt(final_state, "final_state", torch.float32)
    _opt(initial_state, "initial_state", torch.float32)
    _shape(dt, "dt", (batch, seqlen, nheads))
    _shape(A_head, "A_head", (nheads,))
    if B.shape[0] != batch or B.shape[1] != seqlen:
        raise ValueError(f"B must have shape ({batch}, {seqlen}, ngroups, dstate), "
                         f"got {tuple(B.shape)}")
    _shape(C, "C", tuple(B.shape))
    _shape(y, "y", tuple(x.shape))
    _shape(initial_state, "initial_state", (batch, nheads, headdim, dstate))
    _shape(final_state, "final_state", (batch, nheads, headdim, dstate))
    if block_states is not None:
        _req(block_states, "block_states", torch.float32)
        if block_states.numel() * 4 < ssd_chunked_checkpoint_bytes(batch, seqlen, nheads, headdim,
                                                                   dstate):
            raise ValueError("block_states is smaller than ssd_chunked_checkpoint_bytes(...)")
        st = lib().ssd_chunked_fwd_ckpt(_ptr(x), _ptr(dt), _ptr(A_head), _ptr(B), _ptr(C),
                                        int(chunk), _ptr(initial_state), _ptr(y),
                                        _ptr(final_state), _ptr(block_states), batch, seqlen,
                                        nheads, headdim, dstate, ngroups, _DT[in_dt], _DT[out_dt],
                                        _stream(stream))
        _check(st, "ssd_chunked_fwd_ckpt")
        return y, final_state
    st = lib().ssd_chunked_fwd(_ptr(x), _ptr(dt), _ptr(A_head), _ptr(B), _ptr(C), int(chunk),
                               _ptr(initial_state), _ptr(y), _ptr(final_state), batch, seqlen,
                               nheads, headdim, dstate,
                               ngroups, _DT[in_dt], _DT[out_dt], _stream(stream))
    _check(st, "ssd_chunked_fwd")
    return y, final_state


def ssm_decode_step(state, x, dt, A, B, C, D=None, z=None, y=None, stream=None):
    """One decode step; ``state`` (batch, nheads, headdim, dstate) fp32 is updated in place.
    x, z: (batch, nheads, headdim); dt: (batch, nheads) fp32; A, D: (nheads,) fp32;
    B, C: (batch, ngroups, dstate).  Returns y (batch, nheads, headdim)."""
    _req(state, "state", torch.float32, 4)
    batch, nheads, headdim, dstate = state.shape
    _req(x, "x", ndim=3)
    dt_ = x.dtype
    if dt_ not in _DT:
        raise TypeError("x must be float32 or bfloat16")
    _req(dt, "dt", torch.float32, 2)
    _req(A, "A", torch.float32, 1)
    _req(B, "B", dt_, 3)
    _req(C, "C", dt_, 3)
    ngroups = B.shape[1]
    _opt(D, "D", torch.float32)
    _opt(z, "z", dt_)
    if y is None:
        y = torch.empty_like(x)
    _req(y, "y", dt_)
    _shape(x, "x", (batch, nheads, headdim))
    _shape(z, "z", (batch, nheads, headdim))
    _shape(y, "y", (batch, nheads, headdim))
    _shape(dt, "dt", (batch, nheads))
    _shape(A, "A", (nheads,))
    _shape(D, "D", (nheads,))
    if B.shape[0] != batch or B.shape[2] != dstate:
        raise ValueError(f"B must have shape ({batch}, ngroups, {dstate}), got {tuple(B.shape)}")
    _shape(C, "C", tuple(B.shape))
    st = lib().ssm_decode_step(_ptr(state), _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C),
                               _ptr(D), _ptr(z), _ptr(y), batch, nheads, headdim, dstate,
                               ngroups, _DT[dt_], _stream(stream))
    _check(st, "ssm_decode_step")
    return y


def ssm_last_device_status(workspace, stream=None) -> int:
    """Device-side status recorded in a scan workspace (waits for the stream)."""
    return int(lib().ssm_last_device_status(_ptr(workspace), _stream(stream)))


def ssm_debug_set_lookback(drop_first_publish: bool = False, spin_limit: int = 0) -> None:
    """Test hook of the scan's chained L-chunks: chunk 0 withholds its publish
    (so chunk 1's bounded wait runs out and records SSM_ERR_TIMEOUT) and the
    wait gives up after ``spin_limit`` polls (0: the default).  Process-wide;
    call with no arguments to restore the defaults."""
    _check(lib().ssm_debug_set_lookback(1 if drop_first_publish else 0, int(spin_limit)),
           "ssm_debug_set_lookback")


def ssm_debug_set_scan_path(path: int = 0, segments: int = 0) -> None:
    """Test hook choosing the forward scan's kernel: path 0 as planned, 1 the
    chained scan, 2 the sequence-parallel scan (where batch * dim <= 3072);
    segments: the sequence-parallel scan's segments per 128-step chunk (8, 16,
    32; 0 = planned).  Process-wide; call with no arguments to restore."""
    _check(lib().ssm_debug_set_scan_path(int(path), int(segments)), "ssm_debug_set_scan_path")


def ssm_noalloc_last_status(stream=None) -> int:
    """Device-side status the last ``ssm_scan_fwd_noalloc`` on the current device
    recorded in its scratch array (waits for the stream)."""
    return int(lib().ssm_noalloc_last_status(_stream(stream)))


def ssm_mamba3_rope(B, C, dt, theta, angle0=None, B_rot=None, C_rot=None, angle_out=None,
                    return_angle=True, stream=None):
    """Mamba-3's data-dependent RoPE: angles -cumsum(dt * theta) (from angle0),
    B and C rotated by them pair by pair, one row per head.  B, C: (batch, L, G, N)
    or with a rank axis (batch, L, R, G, N); dt (batch, L, H) fp32; theta
    (batch, L, H, N/2) fp32; angle0 (batch, H, N/2) fp32 or None.  Returns
    (B_rot, C_rot, angle_out) with B_rot, C_rot (batch, L, [R,] H, N) in B's dtype;
    angle_out may be angle0 itself (updated in place)."""
    _req(B, "B")
    dt_ = B.dtype
    if dt_ not in _DT:
        raise TypeError("B must be float32 or bfloat16")
    siso = B.dim() == 4
    if B.dim() not in (4, 5):
        raise ValueError("B must have 4 dims (batch, L, G, N) or 5 (batch, L, R, G, N)")
    if siso:
        batch, seqlen, ngroups, dstate = B.shape
        rank = 1
    else:
        batch, seqlen, rank, ngroups, dstate = B.shape
    _req(C, "C", dt_)
    _shape(C, "C", tuple(B.shape))
    _req(dt, "dt", torch.float32, 3)
    nheads = dt.shape[2]
    _shape(dt, "dt", (batch, seqlen, nheads))
    _req(theta, "theta", torch.float32, 4)
    _shape(theta, "theta", (batch, seqlen, nheads, dstate // 2))
    _opt(angle0, "angle0", torch.float32)
    _shape(angle0, "angle0", (batch, nheads, dstate // 2))
    rot = (batch, seqlen, nheads, dstate) if siso else (batch, seqlen, rank, nheads, dstate)
    if B_rot is None:
        B_rot = torch.empty(rot, dtype=dt_, device=B.device)
    if C_rot is None:
        C_rot = torch.empty(rot, dtype=dt_, device=B.device)
    _req(B_rot, "B_rot", dt_)
    _req(C_rot, "C_rot", dt_)
    _shape(B_rot, "B_rot", rot)
    _shape(C_rot, "C_rot", rot)
    if angle_out is None and return_angle:
        angle_out = torch.empty((batch, nheads, dstate // 2), dtype=torch.float32,
                                device=B.device)
    _opt(angle_out, "angle_out", torch.float32)
    _shape(angle_out, "angle_out", (batch, nheads, dstate // 2))
    st = lib().ssm_mamba3_rope(_ptr(B), _ptr(C), _ptr(dt), _ptr(theta), _ptr(angle0),
                               _ptr(B_rot), _ptr(C_rot), _ptr(angle_out), batch, seqlen, rank,
                               nheads, ngroups, dstate, _DT[dt_], _stream(stream))
    _check(st, "ssm_mamba3_rope")
    return B_rot, C_rot, angle_out


def ssd_mamba3_fwd(x, dt, lam, A_head, B, C, chunk=64, out_dtype=None, y=None, final_state=None,
                   return_final_state=True, initial_state=None, prev_B=None, prev_x=None,
                   stream=None, block_states=None):
    """Mamba-3 SISO chunked prefill.  As ``ssd_chunked_fwd`` plus lam: (batch, seqlen,
    nheads) fp32 (lambda after sigmoid) and the token before the first, prev_B:
    (batch, ngroups, dstate) and prev_x: (batch, nheads, headdim) in x's dtype (both or
    neither).  B and C are taken already rotated.  ``block_states`` (fp32, at least
    ``ssd_chunked_checkpoint_bytes(batch, seqlen, nheads)`` bytes) also keeps the
    states ``ssd_mamba3_bwd`` starts from.  Returns (y, final_state)."""
    _req(x, "x", ndim=4)
    in_dt = x.dtype
    if in_dt not in _DT:
        raise TypeError("x must be float32 or bfloat16")
    batch, seqlen, nheads, headdim = x.shape
    _req(dt, "dt", torch.float32, 3)
    _req(lam, "lam", torch.float32, 3)
    _req(A_head, "A_head", torch.float32, 1)
    _req(B, "B", in_dt, 4)
    _req(C, "C", in_dt, 4)
    ngroups, dstate = B.shape[2], B.shape[3]
    out_dt = in_dt if out_dtype is None else out_dtype
    if y is None:
        y = torch.empty_like(x, dtype=out_dt)
    _req(y, "y", out_dt)
    if final_state is None and return_final_state:
        final_state = torch.empty((batch, nheads, headdim, dstate), dtype=torch.float32,
                                  device=x.device)
    _opt(final_state, "final_state", torch.float32)
    _opt(initial_state, "initial_state", torch.float32)
    _opt(prev_B, "prev_B", in_dt)
    _opt(prev_x, "prev_x", in_dt)
    if block_states is not None:
        _req(block_states, "block_states", torch.float32)
        if block_states.numel() * 4 < ssd_chunked_checkpoint_bytes(batch, seqlen, nheads, headdim,
                                                                   dstate):
            raise ValueError("block_states is smaller than ssd_chunked_checkpoint_bytes(...)")
        st = lib().ssd_mamba3_fwd_ckpt(_ptr(x), _ptr(dt), _ptr(lam), _ptr(A_head), _ptr(B),
                                       _ptr(C), int(chunk), _ptr(initial_state), _ptr(prev_B),
                                       _ptr(prev_x), _ptr(y), _ptr(final_state),
                                       _ptr(block_states), batch, seqlen, nheads, headdim,
                                       dstate, ngroups, _DT[in_dt], _DT[out_dt], _stream(stream))
        _check(st, "ssd_mamba3_fwd_ckpt")
        return y, final_state
    st = lib().ssd_mamba3_fwd(_ptr(x), _ptr(dt), _ptr(lam), _ptr(A_head), _ptr(B), _ptr(C),
                              int(chunk), _ptr(initial_state), _ptr(prev_B), _ptr(prev_x),
                              _ptr(y), _ptr(final_state), batch, seqlen, nheads, headdim, dstate,
                              ngroups, _DT[in_dt], _DT[out_dt], _stream(stream))
    _check(st, "ssd_mamba3_fwd")
    return y, final_state


def ssm_decode_step_mamba3(state, prev_B, prev_x, x, dt, lam, A, B, C, D=None, z=None, y=None,
                           stream=None):
    """One Mamba-3 SISO decode step; ``state`` (batch, nheads, headdim, dstate) fp32 is
    updated in place.  As ``ssm_decode_step`` plus lam: (batch, nheads) fp32 and the
    previous token's prev_B (batch, ngroups, dstate) and prev_x (batch, nheads, headdim).
    Returns y (batch, nheads, headdim)."""
    _req(state, "state", torch.float32, 4)
    batch, nheads, headdim, dstate = state.shape
    _req(x, "x", ndim=3)
    dt_ = x.dtype
    if dt_ not in _DT:
        raise TypeError("x must be float32 or bfloat16")
    _req(dt, "dt", torch.float32, 2)
    _req(lam, "lam", torch.float32, 2)
    _req(A, "A", torch.float32, 1)
    _req(B, "B", dt_, 3)
    _req(C, "C", dt_, 3)
    _req(prev_B, "prev_B", dt_, 3)
    _req(prev_x, "prev_x", dt_, 3)
    ngroups = B.shape[1]
    _opt(D, "D", torch.float32)
    _opt(z, "z", dt_)
    if y is None:
        y = torch.empty_like(x)
    _req(y, "y", dt_)
    st = lib().ssm_decode_step_mamba3(_ptr(state), _ptr(prev_B), _ptr(prev_x), _ptr(x),
                                      _ptr(dt), _ptr(lam), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                                      _ptr(z), _ptr(y), batch, nheads, headdim, dstate, ngroups,
                                      _DT[dt_], _stream(stream))
    _check(st, "ssm_decode_step_mamba3")
    return y


def ssd_mamba3_mimo_fwd(x, dt, lam, A_head, B, C, chunk=16, out_dtype=None, y=None,
                        final_state=None, return_final_state=True, initial_state=None,
                        prev_B=None, prev_x=None, stream=None, block_states=None):
    """Mamba-3 MIMO (rank R) chunked prefill.  x: (batch, seqlen, R, nheads, headdim);
    B, C: (batch, seqlen, R, ngroups, dstate); dt, lam: (batch, seqlen, nheads) fp32;
    prev_B: (batch, R, ngroups, dstate), prev_x: (batch, R, nheads, headdim) (both or
    neither).  ``block_states`` (fp32, at least ``ssd_chunked_checkpoint_bytes(batch,
    seqlen * R, nheads)`` bytes) also keeps the states ``ssd_mamba3_mimo_bwd`` starts
    from.  Returns (y (batch, seqlen, R, nheads, headdim), final_state)."""
    _req(x, "x", ndim=5)
    in_dt = x.dtype
    if in_dt not in _DT:
        raise TypeError("x must be float32 or bfloat16")
    batch, seqlen, rank, nheads, headdim = x.shape
    _req(dt, "dt", torch.float32, 3)
    _req(lam, "lam", torch.float32, 3)
    _req(A_head, "A_head", torch.float32, 1)
    _req(B, "B", in_dt, 5)
    _req(C, "C", in_dt, 5)
    ngroups, dstate = B.shape[3], B.shape[4]
    out_dt = in_dt if out_dtype is None else out_dtype
    if y is None:
        y = torch.empty_like(x, dtype=out_dt)
    _req(y, "y", out_dt)
    if final_state is None and return_final_state:
        final_state = torch.empty((batch, nheads, headdim, dstate), dtype=torch.float32,
                                  device=x.device)
    _opt(final_state, "final_state", torch.float32)
    _opt(initial_state, "initial_state", torch.float32)
    _opt(prev_B, "prev_B", in_dt)
    _opt(prev_x, "prev_x", in_dt)
    if block_states is not None:
        _req(block_states, "block_states", torch.float32)
        if block_states.numel() * 4 < ssd_chunked_checkpoint_bytes(batch, seqlen * rank, nheads,
                                                                   headdim, dstate):
            raise ValueError("block_states is smaller than ssd_chunked_checkpoint_bytes(...)")
        st = lib().ssd_mamba3_mimo_fwd_ckpt(_ptr(x), _ptr(dt), _ptr(lam), _ptr(A_head), _ptr(B),
                                            _ptr(C), int(chunk), int(rank), _ptr(initial_state),
                                            _ptr(prev_B), _ptr(prev_x), _ptr(y), _ptr(final_state),
                                            _ptr(block_states), batch, seqlen, nheads, headdim,
                                            dstate, ngroups, _DT[in_dt], _DT[out_dt],
                                            _stream(stream))
        _check(st, "ssd_mamba3_mimo_fwd_ckpt")
        return y, final_state
    st = lib().ssd_mamba3_mimo_fwd(_ptr(x), _ptr(dt), _ptr(lam), _ptr(A_head), _ptr(B), _ptr(C),
                                   int(chunk), int(rank), _ptr(initial_state), _ptr(prev_B),
                                   _ptr(prev_x), _ptr(y), _ptr(final_state), batch, seqlen,
                                   nheads, headdim, dstate, ngroups, _DT[in_dt], _DT[out_dt],
                                   _stream(stream))
    _check(st, "ssd_mamba3_mimo_fwd")
    return y, final_state


def ssm_decode_step_mamba3_mimo(state, prev_B, prev_x, x, dt, lam, A, B, C, D=None, z=None,
                                y=None, stream=None):
    """One Mamba-3 MIMO (rank R) decode step; ``state`` (batch, nheads, headdim, dstate)
    fp32 is updated in place.  x, z, prev_x: (batch, R, nheads, headdim); B, C, prev_B:
    (batch, R, ngroups, dstate); dt, lam: (batch, nheads) fp32; A, D: (nheads,) fp32.
    Returns y (batch, R, nheads, headdim)."""
    _req(state, "state", torch.float32, 4)
    batch, nheads, headdim, dstate = state.shape
    _req(x, "x", ndim=4)
    dt_ = x.dtype
    if dt_ not in _DT:
        raise TypeError("x must be float32 or bfloat16")
    rank = x.shape[1]
    _req(dt, "dt", torch.float32, 2)
    _req(lam, "lam", torch.float32, 2)
    _req(A, "A", torch.float32, 1)
    _req(B, "B", dt_, 4)
    _req(C, "C", dt_, 4)
    _req(prev_B, "prev_B", dt_, 4)
    _req(prev_x, "prev_x", dt_, 4)
    ngroups = B.shape[2]
    _opt(D, "D", torch.float32)
    _opt(z, "z", dt_)
    if y is None:
        y = torch.empty_like(x)
    _req(y, "y", dt_)
    st = lib().ssm_decode_step_mamba3_mimo(_ptr(state), _ptr(prev_B), _ptr(prev_x), _ptr(x),
                                           _ptr(dt), _ptr(lam), _ptr(A), _ptr(B), _ptr(C),
                                           _ptr(D), _ptr(z), _ptr(y), batch, rank, nheads,
                                           headdim, dstate, ngroups, _DT[dt_], _stream(stream))
    _check(st, "ssm_decode_step_mamba3_mimo")
    return y
