"""Pins for the fp64 oracle: nothing here calls the CUDA library.

The oracle is checked against things other than itself: closed forms,
brute-force unrolling written as explicit sums (not as the recurrence),
linearity, exact associativity of the combine on dyadic rationals,
textbook special cases (numpy.cumsum, scipy's expit, numpy's logaddexp),
the chunked SSD against the recurrence, the scan against the SSD through a
layout change, chained decode steps against the recurrence, and the
Mamba-3 three-term update (decode, Eq. 9 of "Mamba-3 NKI Kernels for AWS
Neuron", section "How it works") reduced at lambda = 1.
"""
import itertools

import numpy as np
import pytest
from scipy.special import expit

import oracle

RTOL = 1e-12


def _rng(seed):
    return np.random.default_rng(seed)


def _softplus_np(x):
    return np.logaddexp(0.0, x)


def _silu_np(z):
    return z * expit(z)


# ---------------------------------------------------------------- closed forms

@pytest.mark.parametrize("ngroups", [1, 2])
def test_scan_geometric_closed_form(ngroups):
    """Constant dt, A, B, C and u: h_t = dt*B*u*(1 - r^(t+1)) / (1 - r), r = e^(dt*a)."""
    batch, dim, seqlen, dstate = 2, 4, 40, 5
    dt, beta, c, xval = 0.07, 1.3, -0.6, 0.8
    a = -np.linspace(0.2, 3.0, dim * dstate).reshape(dim, dstate)
    u = np.full((batch, dim, seqlen), xval)
    delta = np.full_like(u, dt)
    B = np.full((batch, ngroups, dstate, seqlen), beta)
    C = np.full_like(B, c)
    y, hs = oracle.scan(u, delta, a, B, C)
    t = np.arange(seqlen)
    r = np.exp(dt * a)                                    # (dim, dstate)
    h = dt * beta * xval * (1 - r[..., None] ** (t + 1)) / (1 - r[..., None])  # (dim, N, L)
    y_ref = c * h.sum(axis=1)
    np.testing.assert_allclose(y, np.broadcast_to(y_ref, y.shape), rtol=RTOL)
    np.testing.assert_allclose(hs, np.broadcast_to(h[..., -1], hs.shape), rtol=RTOL)


def test_ssd_geometric_closed_form():
    batch, seqlen, nheads, headdim, dstate = 1, 33, 3, 2, 4
    dtv, beta, c, xval = 0.05, 0.9, 1.1, -1.5
    A_head = np.array([-1.0, -4.0, -9.5])
    x = np.full((batch, seqlen, nheads, headdim), xval)
    dt = np.full((batch, seqlen, nheads), dtv)
    B = np.full((batch, seqlen, 1, dstate), beta)
    C = np.full_like(B, c)
    t = np.arange(seqlen)
    r = np.exp(dtv * A_head)
    S = dtv * beta * xval * (1 - r[None, :] ** (t[:, None] + 1)) / (1 - r[None, :])  # (L, H)
    y_ref = dstate * c * S
    for fn in (lambda: oracle.ssd_recurrence(x, dt, A_head, B, C),
               lambda: oracle.ssd_chunked(x, dt, A_head, B, C, 8)):
        y, hs = fn()
        np.testing.assert_allclose(y[0], np.broadcast_to(y_ref[:, :, None], y[0].shape), rtol=RTOL)
        np.testing.assert_allclose(hs[0], np.broadcast_to(S[-1][:, None, None], hs[0].shape),
                                   rtol=RTOL)


# ------------------------------------------------------------ brute force

def _scan_bruteforce(u, delta, A, B, C, D, z, bias, softplus, h0):
    """y_t = gate_t * (sum_n C_t,n sum_{s<=t} exp(A_n sum_{k=s+1..t} dl_k) dl_s B_s,n u_s
    + exp(A_n sum_{k<=t} dl_k) h0_n) + D u_t), with explicit sums (O(L^2))."""
    batch, dim, seqlen = u.shape
    dstate = A.shape[1]
    ngroups = B.shape[1]
    dpg = dim // ngroups
    y = np.zeros_like(u)
    hs = np.zeros((batch, dim, dstate))
    for b in range(batch):
        for d in range(dim):
            g = d // dpg
            dl = delta[b, d] + (bias[d] if bias is not None else 0.0)
            if softplus:
                dl = _softplus_np(dl)
            cum = np.concatenate([[0.0], np.cumsum(dl)])  # cum[t+1] = sum_{k<=t}
            for t in range(seqlen):
                acc = 0.0
                for n in range(dstate):
                    hn = 0.0
                    for s in range(t + 1):
                        hn += np.exp(A[d, n] * (cum[t + 1] - cum[s + 1])) * dl[s] * B[b, g, n, s] * u[b, d, s]
                    if h0 is not None:
                        hn += np.exp(A[d, n] * cum[t + 1]) * h0[b, d, n]
                    acc += C[b, g, n, t] * hn
                    if t == seqlen - 1:
                        hs[b, d, n] = hn
                out = acc + (D[d] * u[b, d, t] if D is not None else 0.0)
                if z is not None:
                    out *= _silu_np(z[b, d, t])
                y[b, d, t] = out
    return y, hs


@pytest.mark.parametrize("softplus,use_z,use_D,use_h0,ngroups",
                         [(True, True, True, False, 1), (False, False, False, False, 2),
                          (True, False, True, True, 2), (False, True, False, True, 1)])
def test_scan_bruteforce(softplus, use_z, use_D, use_h0, ngroups):
    rng = _rng(7)
    batch, dim, seqlen, dstate = 2, 4, 17, 3
    u = rng.standard_normal((batch, dim, seqlen))
    delta = 0.5 * rng.standard_normal((batch, dim, seqlen)) + (0.0 if softplus else 0.6)
    A = -rng.uniform(0.1, 2.0, (dim, dstate))
    B = rng.standard_normal((batch, ngroups, dstate, seqlen))
    C = rng.standard_normal((batch, ngroups, dstate, seqlen))
    D = rng.standard_normal(dim) if use_D else None
    z = rng.standard_normal((batch, dim, seqlen)) if use_z else None
    bias = rng.standard_normal(dim) * 0.3
    h0 = rng.standard_normal((batch, dim, dstate)) if use_h0 else None
    y, hs = oracle.scan(u, delta, A, B, C, D, z, bias, softplus, h0)
    y_ref, hs_ref = _scan_bruteforce(u, delta, A, B, C, D, z, bias, softplus, h0)
    np.testing.assert_allclose(y, y_ref, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(hs, hs_ref, rtol=1e-11, atol=1e-13)


def test_ssd_bruteforce():
    """SSD: y_t[p] = sum_n C_t,n sum_{s<=t} exp(A_h sum_{k=s+1..t} dt_k) dt_s B_s,n x_s[p]."""
    rng = _rng(11)
    batch, seqlen, nheads, headdim, dstate, ngroups = 2, 9, 4, 3, 5, 2
    x = rng.standard_normal((batch, seqlen, nheads, headdim))
    dt = rng.uniform(0.01, 0.5, (batch, seqlen, nheads))
    A_head = -rng.uniform(0.5, 4.0, nheads)
    B = rng.standard_normal((batch, seqlen, ngroups, dstate))
    C = rng.standard_normal((batch, seqlen, ngroups, dstate))
    y_ref = np.zeros_like(x)
    hs_ref = np.zeros((batch, nheads, headdim, dstate))
    hpg = nheads // ngroups
    for b, h in itertools.product(range(batch), range(nheads)):
        g = h // hpg
        cum = np.concatenate([[0.0], np.cumsum(dt[b, :, h])])
        for t in range(seqlen):
            w = np.exp(A_head[h] * (cum[t + 1] - cum[1:t + 2])) * dt[b, :t + 1, h]  # (t+1,)
            S = np.einsum("s,sn,sp->pn", w, B[b, :t + 1, g], x[b, :t + 1, h])
            y_ref[b, t, h] = S @ C[b, t, g]
            if t == seqlen - 1:
                hs_ref[b, h] = S
    y, hs = oracle.ssd_recurrence(x, dt, A_head, B, C)
    np.testing.assert_allclose(y, y_ref, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(hs, hs_ref, rtol=1e-11, atol=1e-13)


# ------------------------------------------------------------- invariants

def test_scan_linear_in_u():
    rng = _rng(3)
    batch, dim, seqlen, dstate = 1, 3, 50, 4
    u1 = rng.standard_normal((batch, dim, seqlen))
    u2 = rng.standard_normal((batch, dim, seqlen))
    delta = 0.5 * rng.standard_normal((batch, dim, seqlen))
    A = -rng.uniform(0.5, 3, (dim, dstate))
    B = rng.standard_normal((batch, 1, dstate, seqlen))
    C = rng.standard_normal((batch, 1, dstate, seqlen))
    D = rng.standard_normal(dim)
    z = rng.standard_normal((batch, dim, seqlen))
    bias = rng.standard_normal(dim)
    al, be = 1.7, -0.4
    f = lambda uu: oracle.scan(uu, delta, A, B, C, D, z, bias, True)
    y12, h12 = f(al * u1 + be * u2)
    y1, h1 = f(u1)
    y2, h2 = f(u2)
    np.testing.assert_allclose(y12, al * y1 + be * y2, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(h12, al * h1 + be * h2, rtol=1e-11, atol=1e-12)


def _dyadic(rng, size):
    return rng.integers(-64, 65, size) / 64.0


def test_combine_is_composition_and_associative():
    """(a1,b1) o (a2,b2) is 'apply map 1, then map 2', and o is associative
    (exact in fp64 on dyadic rationals with few bits)."""
    rng = _rng(5)
    for _ in range(200):
        a1, b1, a2, b2, a3, b3, h = _dyadic(rng, 7)
        a12, b12 = oracle.combine(a1, b1, a2, b2)
        assert a12 * h + b12 == a2 * (a1 * h + b1) + b2
        left = oracle.combine(a12, b12, a3, b3)
        a23, b23 = oracle.combine(a2, b2, a3, b3)
        right = oracle.combine(a1, b1, a23, b23)
        assert left == right
    # identity element (1, 0) on both sides
    assert oracle.combine(1.0, 0.0, 0.375, -2.5) == (0.375, -2.5)
    assert oracle.combine(0.375, -2.5, 1.0, 0.0) == (0.375, -2.5)


def _small_scan_problem(seed, seqlen=13, dim=3, dstate=4, ngroups=1, batch=2):
    rng = _rng(seed)
    return dict(
        u=rng.standard_normal((batch, dim, seqlen)),
        delta=0.5 * rng.standard_normal((batch, dim, seqlen)),
        A=-rng.uniform(0.2, 3, (dim, dstate)),
        B=rng.standard_normal((batch, ngroups, dstate, seqlen)),
        C=rng.standard_normal((batch, ngroups, dstate, seqlen)),
        D=rng.standard_normal(dim),
        z=rng.standard_normal((batch, dim, seqlen)),
        delta_bias=rng.standard_normal(dim),
        delta_softplus=True,
        h0=rng.standard_normal((batch, dim, dstate)),
    )


def test_scan_pieces_every_split_point():
    p = _small_scan_problem(9)
    y, hs = oracle.scan(**p)
    L = p["u"].shape[-1]
    for cut in range(1, L):
        yp, hp = oracle.scan_pieces(cuts=[cut], **p)
        np.testing.assert_allclose(yp, y, rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(hp, hs, rtol=1e-13, atol=1e-14)
    rng = _rng(10)
    for _ in range(10):
        k = int(rng.integers(2, L - 1))
        cuts = np.sort(rng.choice(np.arange(1, L), size=k, replace=False))
        yp, hp = oracle.scan_pieces(cuts=cuts, **p)
        np.testing.assert_allclose(yp, y, rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(hp, hs, rtol=1e-13, atol=1e-14)


def test_scan_resume_from_final_state():
    """Scanning [0, k) and then [k, L) from the first part's final state equals one scan."""
    p = _small_scan_problem(12, seqlen=20)
    y, hs = oracle.scan(**p)
    k = 8
    first = {key: (v[..., :k] if key in ("u", "delta", "z", "B", "C") else v) for key, v in p.items()}
    second = {key: (v[..., k:] if key in ("u", "delta", "z", "B", "C") else v) for key, v in p.items()}
    y1, h1 = oracle.scan(**first)
    second["h0"] = h1
    y2, h2 = oracle.scan(**second)
    np.testing.assert_allclose(np.concatenate([y1, y2], axis=-1), y, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(h2, hs, rtol=1e-13, atol=1e-14)


# ------------------------------------------------------- special cases

def test_scan_reduces_to_cumsum():
    """A = 0, N = 1, B = C = 1, no softplus, gate or skip: y = cumsum(dt * u)."""
    rng = _rng(2)
    batch, dim, seqlen = 2, 3, 64
    u = rng.standard_normal((batch, dim, seqlen))
    delta = rng.uniform(0, 1, (batch, dim, seqlen))
    A = np.zeros((dim, 1))
    B = np.ones((batch, 1, 1, seqlen))
    y, hs = oracle.scan(u, delta, A, B, B)
    np.testing.assert_allclose(y, np.cumsum(delta * u, axis=-1), rtol=1e-13)
    np.testing.assert_allclose(hs[..., 0], np.sum(delta * u, axis=-1), rtol=1e-13)


def test_scan_zero_delta_is_skip_times_gate():
    rng = _rng(4)
    batch, dim, seqlen, dstate = 1, 4, 10, 3
    u = rng.standard_normal((batch, dim, seqlen))
    z = 3 * rng.standard_normal((batch, dim, seqlen))
    D = rng.standard_normal(dim)
    A = -rng.uniform(0.5, 2, (dim, dstate))
    B = rng.standard_normal((batch, 1, dstate, seqlen))
    y, hs = oracle.scan(u, np.zeros_like(u), A, B, B, D, z)
    np.testing.assert_allclose(y, D[None, :, None] * u * z * expit(z), rtol=1e-14)
    assert np.all(hs == 0.0)


def test_scan_single_step_and_softplus_bias_order():
    """L = 1: y = dl * u * sum_n B_n C_n + D u, with dl = softplus(delta + bias)."""
    rng = _rng(6)
    batch, dim, dstate = 2, 5, 4
    u = rng.standard_normal((batch, dim, 1))
    delta = rng.standard_normal((batch, dim, 1))
    bias = rng.standard_normal(dim)
    A = -rng.uniform(0.5, 2, (dim, dstate))
    B = rng.standard_normal((batch, 1, dstate, 1))
    C = rng.standard_normal((batch, 1, dstate, 1))
    D = rng.standard_normal(dim)
    bc = np.sum(B[:, 0, :, 0] * C[:, 0, :, 0], axis=-1)  # (batch,)
    for softplus in (True, False):
        dl = delta[..., 0] + bias[None, :]
        if softplus:
            dl = _softplus_np(dl)
        y, _ = oracle.scan(u, delta, A, B, C, D, None, bias, softplus)
        ref = dl * u[..., 0] * bc[:, None] + D[None, :] * u[..., 0]
        np.testing.assert_allclose(y[..., 0], ref, rtol=1e-13)


def test_softplus_large_arguments():
    """softplus stays finite and exact far out: softplus(800) = 800, softplus(-800) ~ e^-800 = 0."""
    u = np.ones((1, 2, 1))
    delta = np.array([[[800.0], [-800.0]]])
    A = np.zeros((2, 1))
    B = np.ones((1, 1, 1, 1))
    y, _ = oracle.scan(u, delta, A, B, B, delta_softplus=True)
    assert y[0, 0, 0] == 800.0
    assert y[0, 1, 0] == 0.0


# ------------------------------------------------------ cross-path pins

@pytest.mark.parametrize("chunk", [1, 2, 12, 24, 7])
def test_ssd_chunked_equals_recurrence(chunk):
    rng = _rng(13)
    batch, seqlen, nheads, headdim, dstate, ngroups = 2, 24, 4, 3, 6, 2
    x = rng.standard_normal((batch, seqlen, nheads, headdim))
    dt = _softplus_np(rng.standard_normal((batch, seqlen, nheads)) - 1.0)
    A_head = -rng.uniform(1, 16, nheads)
    B = rng.standard_normal((batch, seqlen, ngroups, dstate))
    C = rng.standard_normal((batch, seqlen, ngroups, dstate))
    h0 = rng.standard_normal((batch, nheads, headdim, dstate))
    y, hs = oracle.ssd_recurrence(x, dt, A_head, B, C, h0)
    yc, hc = oracle.ssd_chunked(x, dt, A_head, B, C, chunk, h0)
    np.testing.assert_allclose(yc, y, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(hc, hs, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("use_h0", [False, True])
def test_scan_with_head_constant_A_equals_ssd(use_h0):
    """Scan channels d = h*P + p with A[d, n] = A_h equal the SSD of (B, L, H, P),
    from zero or from a given initial state (the scan's initial-state path is
    pinned by brute force above)."""
    rng = _rng(17)
    batch, seqlen, nheads, headdim, dstate, ngroups = 2, 15, 4, 3, 5, 2
    x = rng.standard_normal((batch, seqlen, nheads, headdim))
    dt = rng.uniform(0.01, 0.3, (batch, seqlen, nheads))
    A_head = -rng.uniform(1, 8, nheads)
    B = rng.standard_normal((batch, seqlen, ngroups, dstate))
    C = rng.standard_normal((batch, seqlen, ngroups, dstate))
    h0 = rng.standard_normal((batch, nheads, headdim, dstate)) if use_h0 else None
    y_ssd, hs_ssd = oracle.ssd_recurrence(x, dt, A_head, B, C, h0)
    dim = nheads * headdim
    u = x.reshape(batch, seqlen, dim).transpose(0, 2, 1)
    delta = np.repeat(dt, headdim, axis=2).transpose(0, 2, 1)
    A = np.repeat(A_head, headdim)[:, None] * np.ones((1, dstate))
    Bs = B.transpose(0, 2, 3, 1)
    Cs = C.transpose(0, 2, 3, 1)
    h0s = None if h0 is None else h0.reshape(batch, dim, dstate)
    y_scan, hs_scan = oracle.scan(u, delta, A, Bs, Cs, h0=h0s)
    np.testing.assert_allclose(y_scan, y_ssd.reshape(batch, seqlen, dim).transpose(0, 2, 1),
                               rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(hs_scan, hs_ssd.reshape(batch, dim, dstate), rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("with_gate", [False, True])
def test_decode_chain_equals_recurrence(with_gate):
    rng = _rng(19)
    batch, T, nheads, headdim, dstate, ngroups = 2, 12, 4, 3, 5, 2
    x = rng.standard_normal((batch, T, nheads, headdim))
    dt = rng.uniform(0.01, 0.4, (batch, T, nheads))
    A_head = -rng.uniform(1, 8, nheads)
    B = rng.standard_normal((batch, T, ngroups, dstate))
    C = rng.standard_normal((batch, T, ngroups, dstate))
    D = rng.standard_normal(nheads) if with_gate else None
    z = rng.standard_normal((batch, T, nheads, headdim)) if with_gate else None
    h0 = rng.standard_normal((batch, nheads, headdim, dstate))
    y_ref, hs_ref = oracle.ssd_recurrence(x, dt, A_head, B, C, h0)
    state = h0.copy()
    for t in range(T):
        y, state = oracle.decode_step(state, x[:, t], dt[:, t], A_head, B[:, t], C[:, t], D,
                                      None if z is None else z[:, t])
        ref = y_ref[:, t]
        if with_gate:
            ref = (ref + D[None, :, None] * x[:, t]) * _silu_np(z[:, t])
        np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(state, hs_ref, rtol=1e-12, atol=1e-13)


def test_mamba3_three_term_update_reduces_at_lambda_one():
    """Eq. 9: h_t = alpha h_{t-1} + beta prev_Bx + gamma (B_t x_t), with
    alpha = exp(dt A), gamma = lambda dt, beta = (dt - gamma) alpha.  At
    lambda = 1, beta = 0 and gamma = dt: the decode step is this update."""
    rng = _rng(23)
    batch, T, nheads, headdim, dstate = 1, 10, 2, 3, 4
    x = rng.standard_normal((batch, T, nheads, headdim))
    dt = rng.uniform(0.01, 0.4, (batch, T, nheads))
    A_head = -rng.uniform(1, 8, nheads)
    B = rng.standard_normal((batch, T, 1, dstate))
    C = rng.standard_normal((batch, T, 1, dstate))

    def mamba3(lam):
        h = np.zeros((batch, nheads, headdim, dstate))
        prev_bx = np.zeros_like(h)
        ys = []
        for t in range(T):
            alpha = np.exp(dt[:, t] * A_head)[..., None, None]
            gamma = lam * dt[:, t][..., None, None]
            beta = (dt[:, t][..., None, None] - gamma) * alpha
            bx = np.einsum("bp,bn->bpn", x[:, t, 0], B[:, t, 0])[:, None] if nheads == 1 else \
                np.einsum("bhp,bn->bhpn", x[:, t], B[:, t, 0])
            h = alpha * h + beta * prev_bx + gamma * bx
            prev_bx = bx
            ys.append(np.einsum("bhpn,bn->bhp", h, C[:, t, 0]))
        return np.stack(ys, axis=1), h

    state = np.zeros((batch, nheads, headdim, dstate))
    ys = []
    for t in range(T):
        y, state = oracle.decode_step(state, x[:, t], dt[:, t], A_head, B[:, t], C[:, t])
        ys.append(y)
    y_m3, h_m3 = mamba3(1.0)
    np.testing.assert_allclose(np.stack(ys, axis=1), y_m3, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(state, h_m3, rtol=1e-12, atol=1e-13)
    y_half, _ = mamba3(0.5)
    assert np.max(np.abs(y_half - y_m3)) > 1e-3  # lambda matters away from 1


# ------------------------------------------------------ Mamba-3 SISO pins

def _mamba3_case(seed, batch=2, seqlen=13, nheads=4, headdim=3, dstate=5, ngroups=2,
                 lam_value=None):
    rng = _rng(seed)
    x = rng.standard_normal((batch, seqlen, nheads, headdim))
    dt = rng.uniform(0.02, 0.5, (batch, seqlen, nheads))
    if lam_value is None:
        lam = 1.0 / (1.0 + np.exp(-rng.standard_normal((batch, seqlen, nheads))))
    else:
        lam = np.full((batch, seqlen, nheads), float(lam_value))
    A_head = -rng.uniform(1, 8, nheads)
    B = rng.standard_normal((batch, seqlen, ngroups, dstate))
    C = rng.standard_normal((batch, seqlen, ngroups, dstate))
    h0 = rng.standard_normal((batch, nheads, headdim, dstate))
    prev_B = rng.standard_normal((batch, ngroups, dstate))
    prev_x = rng.standard_normal((batch, nheads, headdim))
    return dict(x=x, dt=dt, lam=lam, A_head=A_head, B=B, C=C, h0=h0, prev_B=prev_B,
                prev_x=prev_x)


def _mamba3_bruteforce(x, dt, lam, A_head, B, C, h0, prev_B, prev_x):
    """Eq. 9 unrolled with explicit products (O(L^2)):
    h_t = (prod_{k<=t} alpha_k) h0
          + sum_{s<=t} (prod_{s<k<=t} alpha_k) (gamma_s u_s + beta_s u_{s-1}),
    u_s = B_s (x) x_s, u_{-1} = prev_B (x) prev_x; y_t = C_t . h_t."""
    batch, seqlen, nheads, headdim = x.shape
    ngroups, dstate = B.shape[2], B.shape[3]
    hpg = nheads // ngroups
    y = np.zeros_like(x)
    hs = np.zeros((batch, nheads, headdim, dstate))
    for b in range(batch):
        for h in range(nheads):
            g = h // hpg
            alpha = np.exp(dt[b, :, h] * A_head[h])
            gamma = lam[b, :, h] * dt[b, :, h]
            beta = (dt[b, :, h] - gamma) * alpha
            u = [np.outer(x[b, s, h], B[b, s, g]) for s in range(seqlen)]
            u_prev = np.outer(prev_x[b, h], prev_B[b, g])
            for t in range(seqlen):
                ht = np.prod(alpha[:t + 1]) * h0[b, h]
                for s in range(t + 1):
                    carry = np.prod(alpha[s + 1:t + 1])
                    before = u[s - 1] if s > 0 else u_prev
                    ht = ht + carry * (gamma[s] * u[s] + beta[s] * before)
                y[b, t, h] = ht @ C[b, t, g]
                if t == seqlen - 1:
                    hs[b, h] = ht
    return y, hs


def test_mamba3_recurrence_bruteforce():
    c = _mamba3_case(101)
    y, hs = oracle.mamba3_recurrence(**c)
    y_ref, hs_ref = _mamba3_bruteforce(**c)
    np.testing.assert_allclose(y, y_ref, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(hs, hs_ref, rtol=1e-11, atol=1e-12)


def test_mamba3_lambda_one_is_mamba2():
    """lambda = 1: gamma = dt, beta = 0, the previous token drops out and Eq. 9
    is the Mamba-2 update of ssd_recurrence."""
    c = _mamba3_case(103, lam_value=1.0)
    y, hs = oracle.mamba3_recurrence(**c)
    y2, hs2 = oracle.ssd_recurrence(c["x"], c["dt"], c["A_head"], c["B"], c["C"], c["h0"])
    np.testing.assert_allclose(y, y2, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(hs, hs2, rtol=1e-12, atol=1e-13)


def test_mamba3_lambda_zero_is_shifted_mamba2():
    """lambda = 0: gamma = 0, beta = dt alpha, so h_t = alpha_t h_{t-1} +
    dt_t (alpha_t u_{t-1}): the Mamba-2 recurrence on the inputs shifted one
    step later (x'_t = alpha_t x_{t-1}, B'_t = B_{t-1}, the first from the
    previous token)."""
    c = _mamba3_case(107, lam_value=0.0)
    y, hs = oracle.mamba3_recurrence(**c)
    alpha = np.exp(c["dt"] * c["A_head"][None, None, :])
    xs = np.concatenate([c["prev_x"][:, None], c["x"][:, :-1]], axis=1) * alpha[..., None]
    Bs = np.concatenate([c["prev_B"][:, None], c["B"][:, :-1]], axis=1)
    y2, hs2 = oracle.ssd_recurrence(xs, c["dt"], c["A_head"], Bs, c["C"], c["h0"])
    np.testing.assert_allclose(y, y2, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(hs, hs2, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("chunk", [1, 2, 5, 13, 64])
@pytest.mark.parametrize("with_prev", [False, True])
def test_mamba3_chunked_single_ssd_equals_recurrence(chunk, with_prev):
    c = _mamba3_case(109)
    if not with_prev:
        c["prev_B"] = c["prev_x"] = None
        c["h0"] = None
    y, hs = oracle.mamba3_recurrence(**c)
    yc, hc = oracle.mamba3_chunked(chunk=chunk, **c)
    np.testing.assert_allclose(yc, y, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(hc, hs, rtol=1e-11, atol=1e-12)


def test_mamba3_decode_chain_equals_recurrence():
    c = _mamba3_case(113, seqlen=9)
    y_ref, hs_ref = oracle.mamba3_recurrence(**c)
    state, pB, px = c["h0"].copy(), c["prev_B"], c["prev_x"]
    for t in range(c["x"].shape[1]):
        y, state = oracle.mamba3_decode_step(state, pB, px, c["x"][:, t], c["dt"][:, t],
                                             c["lam"][:, t], c["A_head"], c["B"][:, t],
                                             c["C"][:, t])
        np.testing.assert_allclose(y, y_ref[:, t], rtol=1e-12, atol=1e-13)
        pB, px = c["B"][:, t], c["x"][:, t]
    np.testing.assert_allclose(state, hs_ref, rtol=1e-12, atol=1e-13)


def test_mamba3_decode_skip_and_gate():
    """D skip then silu gate on top of the state read-out, as in the Mamba-2 decode."""
    c = _mamba3_case(127, seqlen=1)
    rng = _rng(128)
    D = rng.standard_normal(c["A_head"].shape)
    z = rng.standard_normal(c["prev_x"].shape)
    args = (c["h0"], c["prev_B"], c["prev_x"], c["x"][:, 0], c["dt"][:, 0], c["lam"][:, 0],
            c["A_head"], c["B"][:, 0], c["C"][:, 0])
    y0, s0 = oracle.mamba3_decode_step(*args)
    y1, s1 = oracle.mamba3_decode_step(*args, D=D, z=z)
    np.testing.assert_array_equal(s0, s1)
    np.testing.assert_allclose(y1, (y0 + D[None, :, None] * c["x"][:, 0]) * _silu_np(z),
                               rtol=1e-13, atol=1e-14)


# ------------------------------------------------------ Mamba-3 MIMO pins

def _mimo_case(seed, batch=2, seqlen=7, rank=3, nheads=4, headdim=3, dstate=5, ngroups=2):
    rng = _rng(seed)
    return dict(
        x=rng.standard_normal((batch, seqlen, rank, nheads, headdim)),
        dt=rng.uniform(0.02, 0.5, (batch, seqlen, nheads)),
        lam=1.0 / (1.0 + np.exp(-rng.standard_normal((batch, seqlen, nheads)))),
        A_head=-rng.uniform(1, 8, nheads),
        B=rng.standard_normal((batch, seqlen, rank, ngroups, dstate)),
        C=rng.standard_normal((batch, seqlen, rank, ngroups, dstate)),
        h0=rng.standard_normal((batch, nheads, headdim, dstate)),
        prev_B=rng.standard_normal((batch, rank, ngroups, dstate)),
        prev_x=rng.standard_normal((batch, rank, nheads, headdim)))


def test_mimo_is_a_sum_of_siso_paths():
    """The state update is linear in the inputs, so output rank r of MIMO equals
    the sum over input ranks r' of the SISO recurrence driven by (B[.,r'], x[.,r'])
    and read out by C[.,r] (the initial state carried by one of them)."""
    c = _mimo_case(131)
    y, hs = oracle.mamba3_mimo_recurrence(**c)
    rank = c["x"].shape[2]
    for r in range(rank):
        y_sum = 0.0
        hs_sum = 0.0
        for rp in range(rank):
            ys, hss = oracle.mamba3_recurrence(
                c["x"][:, :, rp], c["dt"], c["lam"], c["A_head"], c["B"][:, :, rp],
                c["C"][:, :, r], c["h0"] if rp == 0 else None,
                c["prev_B"][:, rp], c["prev_x"][:, rp])
            y_sum = y_sum + ys
            hs_sum = hs_sum + hss
        np.testing.assert_allclose(y[:, :, r], y_sum, rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(hs, hs_sum, rtol=1e-11, atol=1e-12)


def test_mimo_rank_one_is_siso():
    c = _mimo_case(137, rank=1)
    y, hs = oracle.mamba3_mimo_recurrence(**c)
    ys, hss = oracle.mamba3_recurrence(c["x"][:, :, 0], c["dt"], c["lam"], c["A_head"],
                                       c["B"][:, :, 0], c["C"][:, :, 0], c["h0"],
                                       c["prev_B"][:, 0], c["prev_x"][:, 0])
    np.testing.assert_allclose(y[:, :, 0], ys, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(hs, hss, rtol=1e-13, atol=1e-14)


def test_mimo_bruteforce():
    """Explicit rank sums and products, O(L^2), written independently."""
    c = _mimo_case(139, batch=1, nheads=2, ngroups=1)
    y, hs = oracle.mamba3_mimo_recurrence(**c)
    x, dt, lam, A = c["x"], c["dt"], c["lam"], c["A_head"]
    B, C = c["B"], c["C"]
    _, L, R, H, P = x.shape
    for h in range(H):
        alpha = np.exp(dt[0, :, h] * A[h])
        gamma = lam[0, :, h] * dt[0, :, h]
        beta = (dt[0, :, h] - gamma) * alpha
        U = [sum(np.outer(B[0, t, r, 0], x[0, t, r, h]) for r in range(R)) for t in range(L)]
        U_prev = sum(np.outer(c["prev_B"][0, r, 0], c["prev_x"][0, r, h]) for r in range(R))
        for t in range(L):
            ht = np.prod(alpha[:t + 1]) * c["h0"][0, h].T
            for s in range(t + 1):
                ht = ht + np.prod(alpha[s + 1:t + 1]) * (
                    gamma[s] * U[s] + beta[s] * (U[s - 1] if s > 0 else U_prev))
            for r in range(R):
                np.testing.assert_allclose(y[0, t, r, h], C[0, t, r, 0] @ ht,
                                           rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(hs[0, h], ht.T, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("chunk", [1, 2, 3, 7, 16])
def test_mimo_flattened_chunked_equals_recurrence(chunk):
    c = _mimo_case(149)
    y, hs = oracle.mamba3_mimo_recurrence(**c)
    yc, hc = oracle.mamba3_mimo_chunked(chunk=chunk, **c)
    np.testing.assert_allclose(yc, y, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(hc, hs, rtol=1e-11, atol=1e-12)


def test_mimo_decode_chain_equals_recurrence():
    c = _mimo_case(151, seqlen=5)
    rng = _rng(152)
    D = rng.standard_normal(c["A_head"].shape)
    y_ref, hs_ref = oracle.mamba3_mimo_recurrence(**c)
    state, pB, px = c["h0"].copy(), c["prev_B"], c["prev_x"]
    for t in range(c["x"].shape[1]):
        y, state = oracle.mamba3_mimo_decode_step(state, pB, px, c["x"][:, t], c["dt"][:, t],
                                                  c["lam"][:, t], c["A_head"], c["B"][:, t],
                                                  c["C"][:, t], D)
        ref = y_ref[:, t] + D[None, None, :, None] * c["x"][:, t]
        np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-13)
        pB, px = c["B"][:, t], c["x"][:, t]
    np.testing.assert_allclose(state, hs_ref, rtol=1e-12, atol=1e-13)


# ------------------------------------------------------ scan backward pins

_BWD_INPUTS = ("u", "delta", "A", "B", "C", "D", "z", "delta_bias", "h0")


def _bwd_case(seed, softplus, use_z, use_D, use_bias, use_h0, ngroups=1):
    rng = _rng(seed)
    batch, dim, seqlen, dstate = 2, 4, 6, 3
    c = dict(u=rng.standard_normal((batch, dim, seqlen)),
             delta=0.5 * rng.standard_normal((batch, dim, seqlen)) + (0.0 if softplus else 0.6),
             A=-rng.uniform(0.5, 2.0, (dim, dstate)),
             B=rng.standard_normal((batch, ngroups, dstate, seqlen)),
             C=rng.standard_normal((batch, ngroups, dstate, seqlen)),
             D=rng.standard_normal(dim) if use_D else None,
             z=rng.standard_normal((batch, dim, seqlen)) if use_z else None,
             delta_bias=0.3 * rng.standard_normal(dim) if use_bias else None,
             h0=rng.standard_normal((batch, dim, dstate)) if use_h0 else None)
    dy = rng.standard_normal((batch, dim, seqlen))
    dfinal = rng.standard_normal((batch, dim, dstate))
    return c, dy, dfinal


def _loss(c, dy, dfinal, softplus):
    y, hs = oracle.scan(c["u"], c["delta"], c["A"], c["B"], c["C"], c["D"], c["z"],
                        c["delta_bias"], softplus, c["h0"])
    return float(np.sum(dy * y) + np.sum(dfinal * hs))


@pytest.mark.parametrize("softplus,use_z,use_D,use_bias,use_h0,ngroups",
                         [(True, True, True, True, True, 1), (False, False, False, False, False, 2),
                          (True, False, True, False, True, 4), (False, True, False, True, False, 1)])
def test_scan_bwd_equals_finite_differences(softplus, use_z, use_D, use_bias, use_h0, ngroups):
    """Every gradient entry against a central difference of the forward oracle's
    loss sum(dy y) + sum(dfinal final_state), step 1e-6 (fp64)."""
    c, dy, dfinal = _bwd_case(211, softplus, use_z, use_D, use_bias, use_h0, ngroups)
    g = oracle.scan_bwd(c["u"], c["delta"], c["A"], c["B"], c["C"], dy, c["D"], c["z"],
                        c["delta_bias"], softplus, c["h0"], dfinal)
    names = {"u": "du", "delta": "ddelta", "A": "dA", "B": "dB", "C": "dC", "D": "dD",
             "z": "dz", "delta_bias": "dbias", "h0": "dh0"}
    eps = 1e-6
    for k in _BWD_INPUTS:
        if c[k] is None:
            continue
        grad = g[names[k]]
        fd = np.zeros_like(c[k])
        for idx in np.ndindex(c[k].shape):
            cp = {kk: (None if vv is None else vv.copy()) for kk, vv in c.items()}
            cp[k][idx] += eps
            lp = _loss(cp, dy, dfinal, softplus)
            cp[k][idx] -= 2 * eps
            lm = _loss(cp, dy, dfinal, softplus)
            fd[idx] = (lp - lm) / (2 * eps)
        np.testing.assert_allclose(grad, fd, rtol=1e-6, atol=1e-7, err_msg=k)


def test_scan_bwd_is_linear_in_dy():
    """The gradient is linear in the output cotangent: g(dy1 + 2 dy2) = g(dy1) + 2 g(dy2)."""
    c, dy, _ = _bwd_case(223, True, True, True, True, True)
    dy2 = _rng(224).standard_normal(dy.shape)
    args = (c["u"], c["delta"], c["A"], c["B"], c["C"])
    kw = dict(D=c["D"], z=c["z"], delta_bias=c["delta_bias"], delta_softplus=True, h0=c["h0"])
    g1 = oracle.scan_bwd(*args, dy, **kw)
    g2 = oracle.scan_bwd(*args, dy2, **kw)
    g3 = oracle.scan_bwd(*args, dy + 2 * dy2, **kw)
    for k in ("du", "dB", "dC", "dD", "dh0"):
        np.testing.assert_allclose(g3[k], g1[k] + 2 * g2[k], rtol=1e-11, atol=1e-12, err_msg=k)


# ------------------------------------------------------- SSD backward pins

def _ssd_bwd_case(seed, ngroups, use_h0):
    rng = _rng(seed)
    batch, seqlen, nheads, headdim, dstate = 2, 5, 4, 3, 4
    c = dict(x=rng.standard_normal((batch, seqlen, nheads, headdim)),
             dt=rng.uniform(0.05, 0.6, (batch, seqlen, nheads)),
             A_head=-rng.uniform(0.5, 2.0, nheads),
             B=rng.standard_normal((batch, seqlen, ngroups, dstate)),
             C=rng.standard_normal((batch, seqlen, ngroups, dstate)),
             h0=rng.standard_normal((batch, nheads, headdim, dstate)) if use_h0 else None)
    dy = rng.standard_normal((batch, seqlen, nheads, headdim))
    dfinal = rng.standard_normal((batch, nheads, headdim, dstate))
    return c, dy, dfinal


def _ssd_loss(c, dy, dfinal):
    y, hs = oracle.ssd_recurrence(c["x"], c["dt"], c["A_head"], c["B"], c["C"], c["h0"])
    return float(np.sum(dy * y) + np.sum(dfinal * hs))


@pytest.mark.parametrize("ngroups,use_h0", [(1, True), (2, False), (4, True)])
def test_ssd_bwd_equals_finite_differences(ngroups, use_h0):
    """Every entry of the SSD gradient against a central difference of the
    forward recurrence oracle's loss sum(dy y) + sum(dfinal final_state)."""
    c, dy, dfinal = _ssd_bwd_case(301 + ngroups, ngroups, use_h0)
    g = oracle.ssd_bwd(c["x"], c["dt"], c["A_head"], c["B"], c["C"], dy, c["h0"], dfinal)
    names = {"x": "dx", "dt": "ddt", "A_head": "dA", "B": "dB", "C": "dC", "h0": "dh0"}
    eps = 1e-6
    for k, gk in names.items():
        if c[k] is None:
            continue
        fd = np.zeros_like(c[k])
        for idx in np.ndindex(c[k].shape):
            cp = {kk: (None if vv is None else vv.copy()) for kk, vv in c.items()}
            cp[k][idx] += eps
            lp = _ssd_loss(cp, dy, dfinal)
            cp[k][idx] -= 2 * eps
            lm = _ssd_loss(cp, dy, dfinal)
            fd[idx] = (lp - lm) / (2 * eps)
        np.testing.assert_allclose(g[gk], fd, rtol=1e-6, atol=1e-7, err_msg=k)


def test_ssd_bwd_is_the_scan_gradient_with_head_constant_A():
    """The SSD is the selective scan with channels (h, p), A constant over a
    head's channels and states, delta = dt without softplus or bias.  Its
    gradient is then the scan gradient with the layouts exchanged, dt's
    gradient summed over p and A's over (p, n): checked against the scan
    gradient oracle (itself pinned by finite differences)."""
    c, dy, dfinal = _ssd_bwd_case(331, 2, True)
    x, dt, Ah, B, C, h0 = c["x"], c["dt"], c["A_head"], c["B"], c["C"], c["h0"]
    batch, seqlen, nheads, headdim = x.shape
    dstate = B.shape[3]
    u = x.transpose(0, 2, 3, 1).reshape(batch, nheads * headdim, seqlen)
    delta = np.repeat(dt.transpose(0, 2, 1), headdim, axis=1)
    A = np.repeat(Ah, headdim)[:, None] * np.ones((1, dstate))
    Bs, Cs = B.transpose(0, 2, 3, 1), C.transpose(0, 2, 3, 1)
    dys = dy.transpose(0, 2, 3, 1).reshape(batch, nheads * headdim, seqlen)
    gs = oracle.scan_bwd(u, delta, A, Bs, Cs, dys, None, None, None, False,
                         h0.reshape(batch, nheads * headdim, dstate),
                         dfinal.reshape(batch, nheads * headdim, dstate))
    g = oracle.ssd_bwd(x, dt, Ah, B, C, dy, h0, dfinal)
    tol = dict(rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(
        g["dx"], gs["du"].reshape(batch, nheads, headdim, seqlen).transpose(0, 3, 1, 2), **tol)
    np.testing.assert_allclose(
        g["ddt"], gs["ddelta"].reshape(batch, nheads, headdim, seqlen).sum(2).transpose(0, 2, 1),
        **tol)
    np.testing.assert_allclose(g["dA"], gs["dA"].reshape(nheads, headdim, dstate).sum((1, 2)),
                               **tol)
    np.testing.assert_allclose(g["dB"], gs["dB"].transpose(0, 3, 1, 2), **tol)
    np.testing.assert_allclose(g["dC"], gs["dC"].transpose(0, 3, 1, 2), **tol)
    np.testing.assert_allclose(g["dh0"], gs["dh0"].reshape(batch, nheads, headdim, dstate), **tol)


def test_ssd_bwd_is_linear_in_the_cotangents():
    c, dy, dfinal = _ssd_bwd_case(341, 1, True)
    r = _rng(342)
    dy2, df2 = r.standard_normal(dy.shape), r.standard_normal(dfinal.shape)
    args = (c["x"], c["dt"], c["A_head"], c["B"], c["C"])
    g1 = oracle.ssd_bwd(*args, dy, c["h0"], dfinal)
    g2 = oracle.ssd_bwd(*args, dy2, c["h0"], df2)
    g3 = oracle.ssd_bwd(*args, dy + 2 * dy2, c["h0"], dfinal + 2 * df2)
    for k in g1:
        np.testing.assert_allclose(g3[k], g1[k] + 2 * g2[k], rtol=1e-11, atol=1e-12, err_msg=k)


# --------------------------------------------------- Mamba-3 backward pins

def _m3_bwd_case(seed, ngroups, use_h0, use_prev):
    rng = _rng(seed)
    batch, seqlen, nheads, headdim, dstate = 2, 5, 4, 3, 4
    c = dict(x=rng.standard_normal((batch, seqlen, nheads, headdim)),
             dt=rng.uniform(0.05, 0.6, (batch, seqlen, nheads)),
             lam=rng.uniform(0.05, 0.95, (batch, seqlen, nheads)),
             A_head=-rng.uniform(0.5, 2.0, nheads),
             B=rng.standard_normal((batch, seqlen, ngroups, dstate)),
             C=rng.standard_normal((batch, seqlen, ngroups, dstate)),
             h0=rng.standard_normal((batch, nheads, headdim, dstate)) if use_h0 else None,
             prev_B=rng.standard_normal((batch, ngroups, dstate)) if use_prev else None,
             prev_x=rng.standard_normal((batch, nheads, headdim)) if use_prev else None)
    dy = rng.standard_normal((batch, seqlen, nheads, headdim))
    dfinal = rng.standard_normal((batch, nheads, headdim, dstate))
    return c, dy, dfinal


def _m3_loss(c, dy, dfinal):
    y, hs = oracle.mamba3_recurrence(c["x"], c["dt"], c["lam"], c["A_head"], c["B"], c["C"],
                                     c["h0"], c["prev_B"], c["prev_x"])
    return float(np.sum(dy * y) + np.sum(dfinal * hs))


@pytest.mark.parametrize("ngroups,use_h0,use_prev", [(1, True, True), (2, False, True),
                                                     (4, True, False)])
def test_mamba3_bwd_equals_finite_differences(ngroups, use_h0, use_prev):
    """Every entry of the Mamba-3 gradient (x, dt, lambda, A, B, C, h0 and the
    previous token) against a central difference of the Eq. 9 recurrence
    oracle's loss sum(dy y) + sum(dfinal final_state)."""
    c, dy, dfinal = _m3_bwd_case(401 + ngroups, ngroups, use_h0, use_prev)
    g = oracle.mamba3_bwd(c["x"], c["dt"], c["lam"], c["A_head"], c["B"], c["C"], dy, c["h0"],
                          c["prev_B"], c["prev_x"], dfinal)
    names = {"x": "dx", "dt": "ddt", "lam": "dlam", "A_head": "dA", "B": "dB", "C": "dC",
             "h0": "dh0", "prev_B": "dprev_B", "prev_x": "dprev_x"}
    eps = 1e-6
    for k, gk in names.items():
        if c[k] is None:
            continue
        fd = np.zeros_like(c[k])
        for idx in np.ndindex(c[k].shape):
            cp = {kk: (None if vv is None else vv.copy()) for kk, vv in c.items()}
            cp[k][idx] += eps
            lp = _m3_loss(cp, dy, dfinal)
            cp[k][idx] -= 2 * eps
            lm = _m3_loss(cp, dy, dfinal)
            fd[idx] = (lp - lm) / (2 * eps)
        np.testing.assert_allclose(g[gk], fd, rtol=1e-6, atol=1e-7, err_msg=k)


def test_mamba3_bwd_at_lambda_one_is_the_ssd_gradient():
    """At lambda = 1 (beta = 0, gamma = dt) and no previous token, Eq. 9 is the
    Mamba-2 recurrence: the gradients match the SSD gradient oracle's, and the
    lambda gradient is the derivative through gamma and beta alone."""
    c, dy, dfinal = _m3_bwd_case(431, 2, True, False)
    lam1 = np.ones_like(c["lam"])
    g = oracle.mamba3_bwd(c["x"], c["dt"], lam1, c["A_head"], c["B"], c["C"], dy, c["h0"],
                          None, None, dfinal)
    s = oracle.ssd_bwd(c["x"], c["dt"], c["A_head"], c["B"], c["C"], dy, c["h0"], dfinal)
    tol = dict(rtol=1e-11, atol=1e-12)
    for k, sk in (("dx", "dx"), ("ddt", "ddt"), ("dA", "dA"), ("dB", "dB"), ("dC", "dC"),
                  ("dh0", "dh0")):
        np.testing.assert_allclose(g[k], s[sk], err_msg=k, **tol)


# ---------------------------------------------- Mamba-3 MIMO backward pins

def _mimo_bwd_case(seed, rank, ngroups, use_h0, use_prev):
    rng = _rng(seed)
    batch, seqlen, nheads, headdim, dstate = 2, 4, 4, 2, 3
    c = dict(x=rng.standard_normal((batch, seqlen, rank, nheads, headdim)),
             dt=rng.uniform(0.05, 0.6, (batch, seqlen, nheads)),
             lam=rng.uniform(0.05, 0.95, (batch, seqlen, nheads)),
             A_head=-rng.uniform(0.5, 2.0, nheads),
             B=rng.standard_normal((batch, seqlen, rank, ngroups, dstate)),
             C=rng.standard_normal((batch, seqlen, rank, ngroups, dstate)),
             h0=rng.standard_normal((batch, nheads, headdim, dstate)) if use_h0 else None,
             prev_B=rng.standard_normal((batch, rank, ngroups, dstate)) if use_prev else None,
             prev_x=rng.standard_normal((batch, rank, nheads, headdim)) if use_prev else None)
    dy = rng.standard_normal((batch, seqlen, rank, nheads, headdim))
    dfinal = rng.standard_normal((batch, nheads, headdim, dstate))
    return c, dy, dfinal


def _mimo_loss(c, dy, dfinal):
    y, hs = oracle.mamba3_mimo_recurrence(c["x"], c["dt"], c["lam"], c["A_head"], c["B"],
                                          c["C"], c["h0"], c["prev_B"], c["prev_x"])
    return float(np.sum(dy * y) + np.sum(dfinal * hs))


@pytest.mark.parametrize("rank,ngroups,use_h0,use_prev", [(2, 1, True, True), (4, 2, False, True),
                                                          (2, 4, True, False)])
def test_mimo_bwd_equals_finite_differences(rank, ngroups, use_h0, use_prev):
    """Every entry of the Mamba-3 MIMO gradient (x, dt, lambda, A, B, C, h0 and the
    previous token, every rank) against a central difference of the rank-R
    recurrence oracle's loss sum(dy y) + sum(dfinal final_state)."""
    c, dy, dfinal = _mimo_bwd_case(501 + rank + ngroups, rank, ngroups, use_h0, use_prev)
    g = oracle.mamba3_mimo_bwd(c["x"], c["dt"], c["lam"], c["A_head"], c["B"], c["C"], dy,
                               c["h0"], c["prev_B"], c["prev_x"], dfinal)
    names = {"x": "dx", "dt": "ddt", "lam": "dlam", "A_head": "dA", "B": "dB", "C": "dC",
             "h0": "dh0", "prev_B": "dprev_B", "prev_x": "dprev_x"}
    eps = 1e-6
    for k, gk in names.items():
        if c[k] is None:
            assert g[gk] is None or k == "h0", k
            continue
        fd = np.zeros_like(c[k])
        for idx in np.ndindex(c[k].shape):
            cp = {kk: (None if vv is None else vv.copy()) for kk, vv in c.items()}
            cp[k][idx] += eps
            lp = _mimo_loss(cp, dy, dfinal)
            cp[k][idx] -= 2 * eps
            lm = _mimo_loss(cp, dy, dfinal)
            fd[idx] = (lp - lm) / (2 * eps)
        np.testing.assert_allclose(g[gk], fd, rtol=1e-6, atol=1e-7, err_msg=k)


def test_mimo_bwd_rank_one_is_the_siso_gradient():
    """At rank one the MIMO recurrence is the SISO one (Eq. 9): every gradient
    equals the SISO gradient oracle's under the layout exchange."""
    c, dy, dfinal = _mimo_bwd_case(521, 1, 2, True, True)
    g = oracle.mamba3_mimo_bwd(c["x"], c["dt"], c["lam"], c["A_head"], c["B"], c["C"], dy,
                               c["h0"], c["prev_B"], c["prev_x"], dfinal)
    s = oracle.mamba3_bwd(c["x"][:, :, 0], c["dt"], c["lam"], c["A_head"], c["B"][:, :, 0],
                          c["C"][:, :, 0], dy[:, :, 0], c["h0"], c["prev_B"][:, 0],
                          c["prev_x"][:, 0], dfinal)
    tol = dict(rtol=1e-12, atol=1e-13)
    for k in ("dx", "dB", "dC"):
        np.testing.assert_allclose(g[k][:, :, 0], s[k], err_msg=k, **tol)
    for k in ("dprev_B", "dprev_x"):
        np.testing.assert_allclose(g[k][:, 0], s[k], err_msg=k, **tol)
    for k in ("ddt", "dlam", "dA", "dh0"):
        np.testing.assert_allclose(g[k], s[k], err_msg=k, **tol)


def test_mimo_bwd_is_linear_in_the_cotangents():
    c, dy, dfinal = _mimo_bwd_case(531, 2, 1, True, True)
    r = _rng(532)
    dy2, df2 = r.standard_normal(dy.shape), r.standard_normal(dfinal.shape)
    args = (c["x"], c["dt"], c["lam"], c["A_head"], c["B"], c["C"])
    extra = (c["h0"], c["prev_B"], c["prev_x"])
    g1 = oracle.mamba3_mimo_bwd(*args, dy, *extra, dfinal)
    g2 = oracle.mamba3_mimo_bwd(*args, dy2, *extra, df2)
    g3 = oracle.mamba3_mimo_bwd(*args, dy + 2 * dy2, *extra, dfinal + 2 * df2)
    for k in g1:
        np.testing.assert_allclose(g3[k], g1[k] + 2 * g2[k], rtol=1e-11, atol=1e-12, err_msg=k)


# ---------------------------------------------------------------- Mamba-3 RoPE
# "Mamba-3 NKI Kernels for AWS Neuron", section "How it works", Phase 1:
# cum_angles = -cumsum(dt * theta), then RoPE on B and C; the page's feature
# list calls the result a complex-valued state.

def _rope_inputs(seed, batch=2, seqlen=11, rank=None, nheads=4, ngroups=2, dstate=6):
    rng = _rng(seed)
    shape = ((batch, seqlen, ngroups, dstate) if rank is None
             else (batch, seqlen, rank, ngroups, dstate))
    B = rng.normal(size=shape)
    C = rng.normal(size=shape)
    dt = rng.uniform(0.02, 0.3, size=(batch, seqlen, nheads))
    theta = rng.normal(size=(batch, seqlen, nheads, dstate // 2)) * 2.0
    angle0 = rng.uniform(-3, 3, size=(batch, nheads, dstate // 2))
    return B, C, dt, theta, angle0


def _per_head(X, nheads):
    """(..., G, N) -> (..., H, N): each head takes its group's row."""
    ngroups = X.shape[-2]
    return np.repeat(X, nheads // ngroups, axis=-2)


@pytest.mark.parametrize("rank", [None, 3])
def test_rope_equals_complex_rotation_by_numpy_cumsum(rank):
    """Each pair (B[2k], B[2k+1]) as the complex number B[2k] + i B[2k+1],
    multiplied by exp(i phi), phi = angle0 - numpy.cumsum(dt theta) over the
    steps: written with numpy's complex arithmetic and cumsum, not the
    oracle's sin/cos loop."""
    B, C, dt, theta, angle0 = _rope_inputs(21, rank=rank)
    nheads = dt.shape[2]
    phi = angle0[:, None] - np.cumsum(dt[..., None] * theta, axis=1)  # (b, L, H, N/2)
    if rank is not None:
        phi_r = phi[:, :, None]
    else:
        phi_r = phi
    got_B, got_C, ang = oracle.mamba3_rope(B, C, dt, theta, angle0)
    for X, got in ((B, got_B), (C, got_C)):
        Xh = _per_head(X, nheads)
        z = (Xh[..., 0::2] + 1j * Xh[..., 1::2]) * np.exp(1j * phi_r)
        np.testing.assert_allclose(got[..., 0::2], z.real, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(got[..., 1::2], z.imag, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(ang, phi[:, -1], rtol=1e-13, atol=1e-13)


def test_rope_zero_rate_is_identity_and_keeps_the_angle():
    B, C, dt, theta, angle0 = _rope_inputs(22)
    got_B, got_C, ang = oracle.mamba3_rope(B, C, dt, np.zeros_like(theta))
    np.testing.assert_array_equal(got_B, _per_head(B, dt.shape[2]))
    np.testing.assert_array_equal(got_C, _per_head(C, dt.shape[2]))
    np.testing.assert_array_equal(ang, 0.0)
    _, _, ang = oracle.mamba3_rope(B, C, dt, np.zeros_like(theta), angle0)
    np.testing.assert_array_equal(ang, angle0)


def test_rope_preserves_each_pair_norm():
    B, C, dt, theta, angle0 = _rope_inputs(23)
    got_B, _, _ = oracle.mamba3_rope(B, C, dt, theta, angle0)
    Bh = _per_head(B, dt.shape[2])
    n_in = Bh[..., 0::2] ** 2 + Bh[..., 1::2] ** 2
    n_out = got_B[..., 0::2] ** 2 + got_B[..., 1::2] ** 2
    np.testing.assert_allclose(n_out, n_in, rtol=1e-12)


def test_rope_constant_rate_closed_form():
    """dt theta = w for every step and pair, B = (1, 0) pairs: step t's pair is
    (cos(-w (t + 1)), sin(-w (t + 1)))."""
    batch, seqlen, nheads, dstate, w = 1, 9, 2, 4, 0.37
    B = np.zeros((batch, seqlen, 1, dstate))
    B[..., 0::2] = 1.0
    dt = np.full((batch, seqlen, nheads), 0.5)
    theta = np.full((batch, seqlen, nheads, dstate // 2), w / 0.5)
    got_B, _, ang = oracle.mamba3_rope(B, B, dt, theta)
    t = np.arange(1, seqlen + 1)[None, :, None, None]
    np.testing.assert_allclose(got_B[..., 0::2], np.broadcast_to(np.cos(-w * t), got_B[..., 0::2].shape), atol=1e-13)
    np.testing.assert_allclose(got_B[..., 1::2], np.broadcast_to(np.sin(-w * t), got_B[..., 1::2].shape), atol=1e-13)
    np.testing.assert_allclose(ang, -w * seqlen, atol=1e-13)


def test_rope_resumes_from_its_final_angle():
    B, C, dt, theta, angle0 = _rope_inputs(24, seqlen=12)
    whole_B, whole_C, whole_ang = oracle.mamba3_rope(B, C, dt, theta, angle0)
    k = 5
    B1, C1, a1 = oracle.mamba3_rope(B[:, :k], C[:, :k], dt[:, :k], theta[:, :k], angle0)
    B2, C2, a2 = oracle.mamba3_rope(B[:, k:], C[:, k:], dt[:, k:], theta[:, k:], a1)
    np.testing.assert_allclose(np.concatenate([B1, B2], 1), whole_B, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(np.concatenate([C1, C2], 1), whole_C, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(a2, whole_ang, rtol=1e-12, atol=1e-12)


def _complex_ssm(x, dt, A_head, B, C, theta):
    """The complex-valued SSM the rotation encodes, written directly: per
    (batch, head, p) and state pair k, with z_t = B_t[2k] + i B_t[2k+1],
    H_t = exp(dt_t A + i dt_t theta_t) H_{t-1} + dt_t x_t z_t, and
    y_t = sum_k Re(conj(c_t) H_t), c_t = C_t[2k] + i C_t[2k+1]."""
    batch, seqlen, nheads, headdim = x.shape
    Bh, Ch = _per_head(B, nheads), _per_head(C, nheads)
    zb = Bh[..., 0::2] + 1j * Bh[..., 1::2]
    zc = Ch[..., 0::2] + 1j * Ch[..., 1::2]
    y = np.zeros(x.shape)
    H = np.zeros((batch, nheads, headdim, zb.shape[-1]), dtype=complex)
    for t in range(seqlen):
        eig = np.exp(dt[:, t, :, None] * (A_head[None, :, None] + 1j * theta[:, t]))  # (b, H, N/2)
        H = eig[:, :, None, :] * H + (dt[:, t, :, None, None] * x[:, t, :, :, None]) * zb[:, t, :, None, :]
        y[:, t] = np.real(np.sum(np.conj(zc[:, t, :, None, :]) * H, axis=-1))
    return y


def test_rope_then_real_recurrence_is_the_complex_ssm():
    """The Mamba-2 recurrence (oracle.ssd_recurrence, lambda = 1 of Mamba-3)
    on the rotated B and C equals the complex-valued SSM with eigenvalues
    exp(dt (A + i theta)), written out with numpy complex numbers; with a zero
    initial state the angle the sequence starts from does not matter."""
    rng = _rng(25)
    batch, seqlen, nheads, headdim, ngroups, dstate = 2, 13, 4, 3, 2, 6
    B, C, dt, theta, angle0 = _rope_inputs(25, batch, seqlen, None, nheads, ngroups, dstate)
    x = rng.normal(size=(batch, seqlen, nheads, headdim))
    A_head = -rng.uniform(0.5, 2.0, size=nheads)
    want = _complex_ssm(x, dt, A_head, B, C, theta)
    for a0 in (None, angle0):
        Br, Cr, _ = oracle.mamba3_rope(B, C, dt, theta, a0)
        y, _ = oracle.ssd_recurrence(x, dt, A_head, Br, Cr)
        np.testing.assert_allclose(y, want, rtol=1e-10, atol=1e-11)
