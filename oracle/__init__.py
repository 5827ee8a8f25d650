"""fp64 CPU oracle for the selective scan, the chunked SSD and the decode step.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  It shares no code
with the CUDA library: the arithmetic lives in ``oracle.c`` (plain C, double
precision, sequential within every row), compiled here with the host's gcc;
this module only converts numpy arrays to contiguous float64 and calls it.

Citations for every function are in ``oracle.c``.  Parity of the
functions exported here is pinned by ``tests/test_oracle.py`` against
closed forms, brute-force unrolling, invariants and textbook special cases.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
# A test may point the oracle at another build of oracle.c (the mutation test
# plants mistakes in a copy of the source to show that the pins catch them).
_LIB_OVERRIDE = os.environ.get("SSM_ORACLE_LIB")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` (gcc, -O2, OpenMP)."""
    stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            if _LIB_OVERRIDE:
                lib = ctypes.CDLL(_LIB_OVERRIDE)
            else:
                build()
                lib = ctypes.CDLL(_LIB)
            dp = ctypes.POINTER(ctypes.c_double)
            i = ctypes.c_int
            lib.oracle_scan.argtypes = [dp] * 8 + [i] + [dp] * 3 + [i] * 5
            lib.oracle_scan_pieces.argtypes = ([dp] * 8 + [i] + [dp] * 3 + [i] * 5
                                               + [ctypes.POINTER(ctypes.c_int), i])
            lib.oracle_ssd_recurrence.argtypes = [dp] * 8 + [i] * 6
            lib.oracle_ssd_chunked.argtypes = [dp] * 8 + [i] * 7
            lib.oracle_decode_step.argtypes = [dp] * 9 + [i] * 5
            lib.oracle_mamba3_recurrence.argtypes = [dp] * 11 + [i] * 6
            lib.oracle_mamba3_chunked.argtypes = [dp] * 11 + [i] * 7
            lib.oracle_mamba3_decode_step.argtypes = [dp] * 12 + [i] * 5
            lib.oracle_mamba3_mimo_recurrence.argtypes = [dp] * 11 + [i] * 7
            lib.oracle_mamba3_mimo_chunked.argtypes = [dp] * 11 + [i] * 8
            lib.oracle_mamba3_mimo_decode_step.argtypes = [dp] * 12 + [i] * 6
            lib.oracle_scan_bwd.argtypes = [dp] * 8 + [i] + [dp] * 12 + [i] * 5
            lib.oracle_ssd_bwd.argtypes = [dp] * 14 + [i] * 6
            lib.oracle_mamba3_bwd.argtypes = [dp] * 20 + [i] * 6
            lib.oracle_mamba3_mimo_bwd.argtypes = [dp] * 20 + [i] * 7
            lib.oracle_mamba3_rope.argtypes = [dp] * 8 + [i] * 6
            lib.oracle_combine.argtypes = [ctypes.c_double] * 4 + [dp, dp]
            lib.oracle_num_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(a):
    """Contiguous float64 copy (or view) of an array-like; None stays None."""
    if a is None:
        return None
    if hasattr(a, "detach"):  # torch tensor: exact upcast on the CPU
        a = a.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    if a is None:
        return ctypes.POINTER(ctypes.c_double)()
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def combine(a1, b1, a2, b2):
    """(a1, b1) o (a2, b2) = (a1 a2, a2 b1 + b2): first map, then second."""
    lib = _load()
    ao, bo = ctypes.c_double(), ctypes.c_double()
    lib.oracle_combine(float(a1), float(b1), float(a2), float(b2),
                       ctypes.byref(ao), ctypes.byref(bo))
    return ao.value, bo.value


def _scan_args(u, delta, A, B, C, D, z, delta_bias, h0):
    u, delta, A, B, C = (_f64(t) for t in (u, delta, A, B, C))
    D, z, delta_bias, h0 = (_f64(t) for t in (D, z, delta_bias, h0))
    batch, dim, seqlen = u.shape
    dstate = A.shape[1]
    ngroups = B.shape[1]
    assert delta.shape == u.shape and A.shape == (dim, dstate)
    assert B.shape == (batch, ngroups, dstate, seqlen) and C.shape == B.shape
    assert dim % ngroups == 0
    return (u, delta, A, B, C, D, z, delta_bias, h0), (batch, dim, seqlen, dstate, ngroups)


def scan(u, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus=False,
         h0=None):
    """Selective scan.  u, delta, z: (B, D, L); A: (D, N); B, C: (B, G, N, L).

    Returns (y (B, D, L), final_state (B, D, N)) in float64.
    """
    arrs, dims = _scan_args(u, delta, A, B, C, D, z, delta_bias, h0)
    batch, dim, seqlen, dstate, _ = dims
    y = np.empty((batch, dim, seqlen), np.float64)
    hs = np.empty((batch, dim, dstate), np.float64)
    _load().oracle_scan(*[_ptr(a) for a in arrs[:8]], int(bool(delta_softplus)),
                        _ptr(arrs[8]), _ptr(y), _ptr(hs), *dims)
    return y, hs


def scan_bwd(u, delta, A, B, C, dy, D=None, z=None, delta_bias=None, delta_softplus=False,
             h0=None, dfinal=None):
    """Gradient of ``scan`` for the loss sum(dy * y) + sum(dfinal * final_state).

    Returns a dict of float64 arrays: du, ddelta, dz (B, D, L); dA (D, N);
    dB, dC (B, G, N, L); dD, dbias (D,); dh0 (B, D, N).  dz, dD, dbias are None
    when z, D, delta_bias are."""
    arrs, dims = _scan_args(u, delta, A, B, C, D, z, delta_bias, h0)
    batch, dim, seqlen, dstate, ngroups = dims
    dy, dfinal = _f64(dy), _f64(dfinal)
    assert dy.shape == (batch, dim, seqlen)
    assert dfinal is None or dfinal.shape == (batch, dim, dstate)
    g = {"du": np.empty((batch, dim, seqlen)), "ddelta": np.empty((batch, dim, seqlen)),
         "dA": np.empty((dim, dstate)), "dB": np.empty((batch, ngroups, dstate, seqlen)),
         "dC": np.empty((batch, ngroups, dstate, seqlen)),
         "dD": np.empty(dim) if arrs[5] is not None else None,
         "dz": np.empty((batch, dim, seqlen)) if arrs[6] is not None else None,
         "dbias": np.empty(dim) if arrs[7] is not None else None,
         "dh0": np.empty((batch, dim, dstate))}
    _load().oracle_scan_bwd(*[_ptr(a) for a in arrs[:8]], int(bool(delta_softplus)),
                            _ptr(arrs[8]), _ptr(dy), _ptr(dfinal), _ptr(g["du"]),
                            _ptr(g["ddelta"]), _ptr(g["dA"]), _ptr(g["dB"]), _ptr(g["dC"]),
                            _ptr(g["dD"]), _ptr(g["dz"]), _ptr(g["dbias"]), _ptr(g["dh0"]),
                            *dims)
    return g


def scan_pieces(u, delta, A, B, C, cuts, D=None, z=None, delta_bias=None,
                delta_softplus=False, h0=None):
    """The scan evaluated piecewise: cut at ``cuts``, combined with the o operator."""
    arrs, dims = _scan_args(u, delta, A, B, C, D, z, delta_bias, h0)
    batch, dim, seqlen, dstate, _ = dims
    cuts = np.ascontiguousarray(np.asarray(cuts, dtype=np.int32))
    assert np.all(np.diff(cuts) > 0) and (cuts.size == 0 or (cuts[0] > 0 and cuts[-1] < seqlen))
    y = np.empty((batch, dim, seqlen), np.float64)
    hs = np.empty((batch, dim, dstate), np.float64)
    _load().oracle_scan_pieces(*[_ptr(a) for a in arrs[:8]], int(bool(delta_softplus)),
                               _ptr(arrs[8]), _ptr(y), _ptr(hs), *dims,
                               cuts.ctypes.data_as(ctypes.POINTER(ctypes.c_int)),
                               int(cuts.size))
    return y, hs


def _ssd_args(x, dt, A_head, B, C, h0):
    x, dt, A_head, B, C, h0 = (_f64(t) for t in (x, dt, A_head, B, C, h0))
    batch, seqlen, nheads, headdim = x.shape
    ngroups, dstate = B.shape[2], B.shape[3]
    assert dt.shape == (batch, seqlen, nheads) and A_head.shape == (nheads,)
    assert B.shape == (batch, seqlen, ngroups, dstate) and C.shape == B.shape
    assert nheads % ngroups == 0
    return (x, dt, A_head, B, C, h0), (batch, seqlen, nheads, headdim, dstate, ngroups)


def ssd_recurrence(x, dt, A_head, B, C, h0=None):
    """SSD as the step-by-step recurrence.  x: (B, L, H, P); dt: (B, L, H);
    A_head: (H,); B, C: (B, L, G, N).  Returns (y (B, L, H, P), state (B, H, P, N))."""
    arrs, dims = _ssd_args(x, dt, A_head, B, C, h0)
    batch, seqlen, nheads, headdim, dstate, _ = dims
    y = np.empty((batch, seqlen, nheads, headdim), np.float64)
    hs = np.empty((batch, nheads, headdim, dstate), np.float64)
    _load().oracle_ssd_recurrence(*[_ptr(a) for a in arrs], _ptr(y), _ptr(hs), *dims)
    return y, hs


def ssd_bwd(x, dt, A_head, B, C, dy, h0=None, dfinal=None):
    """Gradient of ``ssd_recurrence`` for the loss sum(dy * y) + sum(dfinal * final_state).

    Returns a dict of float64 arrays: dx (B, L, H, P), ddt (B, L, H), dA (H,),
    dB, dC (B, L, G, N), dh0 (B, H, P, N)."""
    arrs, dims = _ssd_args(x, dt, A_head, B, C, h0)
    batch, seqlen, nheads, headdim, dstate, ngroups = dims
    dy, dfinal = _f64(dy), _f64(dfinal)
    assert dy.shape == (batch, seqlen, nheads, headdim)
    assert dfinal is None or dfinal.shape == (batch, nheads, headdim, dstate)
    g = {"dx": np.empty((batch, seqlen, nheads, headdim)), "ddt": np.empty((batch, seqlen, nheads)),
         "dA": np.empty(nheads), "dB": np.empty((batch, seqlen, ngroups, dstate)),
         "dC": np.empty((batch, seqlen, ngroups, dstate)),
         "dh0": np.empty((batch, nheads, headdim, dstate))}
    _load().oracle_ssd_bwd(*[_ptr(a) for a in arrs], _ptr(dy), _ptr(dfinal), _ptr(g["dx"]),
                           _ptr(g["ddt"]), _ptr(g["dA"]), _ptr(g["dB"]), _ptr(g["dC"]),
                           _ptr(g["dh0"]), *dims)
    return g


def ssd_chunked(x, dt, A_head, B, C, chunk, h0=None):
    """SSD by the chunked algorithm (fp64 loops), for pinning against the recurrence."""
    arrs, dims = _ssd_args(x, dt, A_head, B, C, h0)
    batch, seqlen, nheads, headdim, dstate, _ = dims
    y = np.empty((batch, seqlen, nheads, headdim), np.float64)
    hs = np.empty((batch, nheads, headdim, dstate), np.float64)
    _load().oracle_ssd_chunked(*[_ptr(a) for a in arrs], _ptr(y), _ptr(hs), *dims, int(chunk))
    return y, hs


def _mamba3_args(x, dt, lam, A_head, B, C, h0, prev_B, prev_x):
    (x, dt, lam, A_head, B, C, h0, prev_B, prev_x) = (
        _f64(t) for t in (x, dt, lam, A_head, B, C, h0, prev_B, prev_x))
    batch, seqlen, nheads, headdim = x.shape
    ngroups, dstate = B.shape[2], B.shape[3]
    assert dt.shape == (batch, seqlen, nheads) and lam.shape == dt.shape
    assert A_head.shape == (nheads,) and C.shape == B.shape
    assert B.shape == (batch, seqlen, ngroups, dstate) and nheads % ngroups == 0
    assert (prev_B is None) == (prev_x is None)
    if prev_B is not None:
        assert prev_B.shape == (batch, ngroups, dstate)
        assert prev_x.shape == (batch, nheads, headdim)
    return ((x, dt, lam, A_head, B, C, h0, prev_B, prev_x),
            (batch, seqlen, nheads, headdim, dstate, ngroups))


def mamba3_recurrence(x, dt, lam, A_head, B, C, h0=None, prev_B=None, prev_x=None):
    """Mamba-3 SISO by the step-by-step recurrence (Eq. 9).  x: (B, L, H, P);
    dt, lam: (B, L, H) (dt after softplus, lam after sigmoid); A_head: (H,);
    B, C: (B, L, G, N); h0: (B, H, P, N); prev_B: (B, G, N) and prev_x: (B, H, P),
    the token before the first.  Returns (y (B, L, H, P), state (B, H, P, N))."""
    arrs, dims = _mamba3_args(x, dt, lam, A_head, B, C, h0, prev_B, prev_x)
    batch, seqlen, nheads, headdim, dstate, _ = dims
    y = np.empty((batch, seqlen, nheads, headdim), np.float64)
    hs = np.empty((batch, nheads, headdim, dstate), np.float64)
    _load().oracle_mamba3_recurrence(*[_ptr(a) for a in arrs], _ptr(y), _ptr(hs), *dims)
    return y, hs


def mamba3_bwd(x, dt, lam, A_head, B, C, dy, h0=None, prev_B=None, prev_x=None, dfinal=None):
    """Gradient of ``mamba3_recurrence`` for the loss sum(dy * y) + sum(dfinal *
    final_state).  Returns a dict of float64 arrays: dx (B, L, H, P), ddt, dlam
    (B, L, H), dA (H,), dB, dC (B, L, G, N), dh0 (B, H, P, N), and dprev_B (B, G, N),
    dprev_x (B, H, P) (None without a previous token)."""
    arrs, dims = _mamba3_args(x, dt, lam, A_head, B, C, h0, prev_B, prev_x)
    batch, seqlen, nheads, headdim, dstate, ngroups = dims
    dy, dfinal = _f64(dy), _f64(dfinal)
    assert dy.shape == (batch, seqlen, nheads, headdim)
    assert dfinal is None or dfinal.shape == (batch, nheads, headdim, dstate)
    has_prev = arrs[7] is not None
    g = {"dx": np.empty((batch, seqlen, nheads, headdim)), "ddt": np.empty((batch, seqlen, nheads)),
         "dlam": np.empty((batch, seqlen, nheads)), "dA": np.empty(nheads),
         "dB": np.empty((batch, seqlen, ngroups, dstate)),
         "dC": np.empty((batch, seqlen, ngroups, dstate)),
         "dh0": np.empty((batch, nheads, headdim, dstate)),
         "dprev_B": np.empty((batch, ngroups, dstate)) if has_prev else None,
         "dprev_x": np.empty((batch, nheads, headdim)) if has_prev else None}
    _load().oracle_mamba3_bwd(*[_ptr(a) for a in arrs], _ptr(dy), _ptr(dfinal), _ptr(g["dx"]),
                              _ptr(g["ddt"]), _ptr(g["dlam"]), _ptr(g["dA"]), _ptr(g["dB"]),
                              _ptr(g["dC"]), _ptr(g["dh0"]), _ptr(g["dprev_B"]),
                              _ptr(g["dprev_x"]), *dims)
    return g


def mamba3_chunked(x, dt, lam, A_head, B, C, chunk, h0=None, prev_B=None, prev_x=None):
    """Mamba-3 SISO by the chunked single-SSD form with the diagonal correction
    (fp64 loops), for pinning against the recurrence."""
    arrs, dims = _mamba3_args(x, dt, lam, A_head, B, C, h0, prev_B, prev_x)
    batch, seqlen, nheads, headdim, dstate, _ = dims
    y = np.empty((batch, seqlen, nheads, headdim), np.float64)
    hs = np.empty((batch, nheads, headdim, dstate), np.float64)
    _load().oracle_mamba3_chunked(*[_ptr(a) for a in arrs], _ptr(y), _ptr(hs), *dims,
                                  int(chunk))
    return y, hs


def mamba3_decode_step(state, prev_B, prev_x, x, dt, lam, A, B, C, D=None, z=None):
    """One Mamba-3 SISO decode step.  state: (B, H, P, N) (not modified; a new
    array is returned); prev_B, B, C: (B, G, N); prev_x, x, z: (B, H, P);
    dt, lam: (B, H); A, D: (H,).  Returns (y (B, H, P), new_state)."""
    st = _f64(state).copy()
    prev_B, prev_x, x, dt, lam, A, B, C, D, z = (
        _f64(t) for t in (prev_B, prev_x, x, dt, lam, A, B, C, D, z))
    batch, nheads, headdim, dstate = st.shape
    ngroups = B.shape[1]
    assert x.shape == (batch, nheads, headdim) and prev_x.shape == x.shape
    assert dt.shape == (batch, nheads) and lam.shape == dt.shape
    assert B.shape == (batch, ngroups, dstate) and C.shape == B.shape and prev_B.shape == B.shape
    y = np.empty((batch, nheads, headdim), np.float64)
    _load().oracle_mamba3_decode_step(_ptr(st), _ptr(prev_B), _ptr(prev_x), _ptr(x), _ptr(dt),
                                      _ptr(lam), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
                                      _ptr(y), batch, nheads, headdim, dstate, ngroups)
    return y, st


def _mimo_args(x, dt, lam, A_head, B, C, h0, prev_B, prev_x):
    (x, dt, lam, A_head, B, C, h0, prev_B, prev_x) = (
        _f64(t) for t in (x, dt, lam, A_head, B, C, h0, prev_B, prev_x))
    batch, seqlen, rank, nheads, headdim = x.shape
    ngroups, dstate = B.shape[3], B.shape[4]
    assert dt.shape == (batch, seqlen, nheads) and lam.shape == dt.shape
    assert A_head.shape == (nheads,) and C.shape == B.shape
    assert B.shape == (batch, seqlen, rank, ngroups, dstate) and nheads % ngroups == 0
    assert (prev_B is None) == (prev_x is None)
    if prev_B is not None:
        assert prev_B.shape == (batch, rank, ngroups, dstate)
        assert prev_x.shape == (batch, rank, nheads, headdim)
    return ((x, dt, lam, A_head, B, C, h0, prev_B, prev_x),
            (batch, seqlen, rank, nheads, headdim, dstate, ngroups))


def mamba3_mimo_recurrence(x, dt, lam, A_head, B, C, h0=None, prev_B=None, prev_x=None):
    """Mamba-3 MIMO (rank R) by the step-by-step recurrence.  x: (B, L, R, H, P);
    dt, lam: (B, L, H); A_head: (H,); B, C: (B, L, R, G, N); h0: (B, H, P, N);
    prev_B: (B, R, G, N) and prev_x: (B, R, H, P), the token before the first.
    Returns (y (B, L, R, H, P), state (B, H, P, N))."""
    arrs, dims = _mimo_args(x, dt, lam, A_head, B, C, h0, prev_B, prev_x)
    batch, seqlen, rank, nheads, headdim, dstate, _ = dims
    y = np.empty((batch, seqlen, rank, nheads, headdim), np.float64)
    hs = np.empty((batch, nheads, headdim, dstate), np.float64)
    _load().oracle_mamba3_mimo_recurrence(*[_ptr(a) for a in arrs], _ptr(y), _ptr(hs), *dims)
    return y, hs


def mamba3_mimo_bwd(x, dt, lam, A_head, B, C, dy, h0=None, prev_B=None, prev_x=None,
                    dfinal=None):
    """Gradient of ``mamba3_mimo_recurrence`` for the loss sum(dy * y) +
    sum(dfinal * final_state).  Returns a dict of float64 arrays: dx (like x), ddt,
    dlam (B, L, H), dA (H,), dB, dC (like B), dh0 (B, H, P, N), and dprev_B,
    dprev_x (like prev_B, prev_x; None without a previous token)."""
    arrs, dims = _mimo_args(x, dt, lam, A_head, B, C, h0, prev_B, prev_x)
    batch, seqlen, rank, nheads, headdim, dstate, ngroups = dims
    dy, dfinal = _f64(dy), _f64(dfinal)
    assert dy.shape == arrs[0].shape
    assert dfinal is None or dfinal.shape == (batch, nheads, headdim, dstate)
    has_prev = arrs[7] is not None
    g = {"dx": np.empty(arrs[0].shape), "ddt": np.empty((batch, seqlen, nheads)),
         "dlam": np.empty((batch, seqlen, nheads)), "dA": np.empty(nheads),
         "dB": np.empty(arrs[4].shape), "dC": np.empty(arrs[4].shape),
         "dh0": np.empty((batch, nheads, headdim, dstate)),
         "dprev_B": np.empty(arrs[7].shape) if has_prev else None,
         "dprev_x": np.empty(arrs[8].shape) if has_prev else None}
    _load().oracle_mamba3_mimo_bwd(*[_ptr(a) for a in arrs], _ptr(dy), _ptr(dfinal),
                                   _ptr(g["dx"]), _ptr(g["ddt"]), _ptr(g["dlam"]), _ptr(g["dA"]),
                                   _ptr(g["dB"]), _ptr(g["dC"]), _ptr(g["dh0"]),
                                   _ptr(g["dprev_B"]), _ptr(g["dprev_x"]), *dims)
    return g


def mamba3_mimo_chunked(x, dt, lam, A_head, B, C, chunk, h0=None, prev_B=None, prev_x=None):
    """Mamba-3 MIMO by the rank-flattened chunked form with the block-diagonal
    correction (fp64 loops; `chunk` counts steps), for pinning against the recurrence."""
    arrs, dims = _mimo_args(x, dt, lam, A_head, B, C, h0, prev_B, prev_x)
    batch, seqlen, rank, nheads, headdim, dstate, _ = dims
    y = np.empty((batch, seqlen, rank, nheads, headdim), np.float64)
    hs = np.empty((batch, nheads, headdim, dstate), np.float64)
    _load().oracle_mamba3_mimo_chunked(*[_ptr(a) for a in arrs], _ptr(y), _ptr(hs), *dims,
                                       int(chunk))
    return y, hs


def mamba3_mimo_decode_step(state, prev_B, prev_x, x, dt, lam, A, B, C, D=None, z=None):
    """One Mamba-3 MIMO decode step.  state: (B, H, P, N) (a new array is returned);
    prev_B, B, C: (B, R, G, N); prev_x, x, z: (B, R, H, P); dt, lam: (B, H); A, D: (H,).
    Returns (y (B, R, H, P), new_state)."""
    st = _f64(state).copy()
    prev_B, prev_x, x, dt, lam, A, B, C, D, z = (
        _f64(t) for t in (prev_B, prev_x, x, dt, lam, A, B, C, D, z))
    batch, nheads, headdim, dstate = st.shape
    rank, ngroups = B.shape[1], B.shape[2]
    assert x.shape == (batch, rank, nheads, headdim) and prev_x.shape == x.shape
    assert dt.shape == (batch, nheads) and lam.shape == dt.shape
    assert B.shape == (batch, rank, ngroups, dstate) and C.shape == B.shape
    assert prev_B.shape == B.shape
    y = np.empty((batch, rank, nheads, headdim), np.float64)
    _load().oracle_mamba3_mimo_decode_step(_ptr(st), _ptr(prev_B), _ptr(prev_x), _ptr(x),
                                           _ptr(dt), _ptr(lam), _ptr(A), _ptr(B), _ptr(C),
                                           _ptr(D), _ptr(z), _ptr(y), batch, rank, nheads,
                                           headdim, dstate, ngroups)
    return y, st


def decode_step(state, x, dt, A, B, C, D=None, z=None):
    """One decode step.  state: (B, H, P, N) (not modified; a new array is
    returned); x, z: (B, H, P); dt: (B, H); A, D: (H,); B, C: (B, G, N).
    Returns (y (B, H, P), new_state (B, H, P, N))."""
    st = _f64(state).copy()
    x, dt, A, B, C, D, z = (_f64(t) for t in (x, dt, A, B, C, D, z))
    batch, nheads, headdim, dstate = st.shape
    ngroups = B.shape[1]
    assert x.shape == (batch, nheads, headdim) and dt.shape == (batch, nheads)
    assert B.shape == (batch, ngroups, dstate) and C.shape == B.shape
    y = np.empty((batch, nheads, headdim), np.float64)
    _load().oracle_decode_step(_ptr(st), _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C),
                               _ptr(D), _ptr(z), _ptr(y),
                               batch, nheads, headdim, dstate, ngroups)
    return y, st


def scan_rows(u, delta, A, B, C, rows, D=None, z=None, delta_bias=None,
              delta_softplus=False):
    """Oracle scan of a subset of (batch, channel) rows of a large problem.

    ``rows`` is a list of (b, d) pairs.  Only those rows' inputs are gathered,
    so a sample of a multi-GB workload can be checked in seconds.  Returns
    (y (len(rows), L), final_state (len(rows), N)).
    """
    out_y, out_h = [], []
    ngroups = B.shape[1]
    dim = u.shape[1]
    dpg = dim // ngroups
    for (b, d) in rows:
        g = d // dpg
        sl = slice(d, d + 1)
        y, h = scan(u[b:b + 1, sl], delta[b:b + 1, sl], A[sl], B[b:b + 1, g:g + 1],
                    C[b:b + 1, g:g + 1],
                    None if D is None else D[sl], None if z is None else z[b:b + 1, sl],
                    None if delta_bias is None else delta_bias[sl], delta_softplus)
        out_y.append(y[0, 0])
        out_h.append(h[0, 0])
    return np.stack(out_y), np.stack(out_h)


def mamba3_rope(B, C, dt, theta, angle0=None):
    """Mamba-3's data-dependent RoPE (oracle.c, oracle_mamba3_rope): the angles
    -cumsum(dt * theta) along the sequence (from angle0), and B, C rotated by
    them pair by pair, one copy per head.

    B, C: (batch, L, G, N) or, with a rank axis, (batch, L, R, G, N); dt
    (batch, L, H); theta (batch, L, H, N/2); angle0 (batch, H, N/2) or None.
    Returns (B_rot, C_rot, angle_out): B_rot, C_rot (batch, L, H, N) or
    (batch, L, R, H, N), angle_out (batch, H, N/2), all float64.
    """
    B, C, dt, theta, angle0 = (_f64(t) for t in (B, C, dt, theta, angle0))
    siso = B.ndim == 4
    if siso:
        B, C = B[:, :, None], C[:, :, None]
    batch, seqlen, rank, ngroups, dstate = B.shape
    nheads = dt.shape[2]
    assert C.shape == B.shape and dstate % 2 == 0 and nheads % ngroups == 0
    assert dt.shape == (batch, seqlen, nheads)
    assert theta.shape == (batch, seqlen, nheads, dstate // 2)
    assert angle0 is None or angle0.shape == (batch, nheads, dstate // 2)
    B, C = np.ascontiguousarray(B), np.ascontiguousarray(C)
    Br = np.empty((batch, seqlen, rank, nheads, dstate))
    Cr = np.empty_like(Br)
    ang = np.empty((batch, nheads, dstate // 2))
    _load().oracle_mamba3_rope(_ptr(B), _ptr(C), _ptr(dt), _ptr(theta), _ptr(angle0), _ptr(Br),
                               _ptr(Cr), _ptr(ang), batch, seqlen, rank, nheads, ngroups, dstate)
    if siso:
        Br, Cr = Br[:, :, 0], Cr[:, :, 0]
    return Br, Cr, ang
