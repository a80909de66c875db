"""Pins for the fp64 oracle: results fixed by the mathematics, not by the oracle.

Each ``check_*`` function takes a loaded oracle library (the real one, or a
deliberately broken copy in the mutation test) and raises ``AssertionError``
when the oracle disagrees with a closed form, an invariant or an independent
brute-force evaluation.  None of them re-types the oracle's loop: the expected
values come from geometric-series sums, a causal convolution via
``numpy.convolve``, explicit products over time, library softplus/sigmoid
(``numpy.logaddexp``, ``scipy.special.expit``), or from the oracle itself
under a transformation that must leave the answer unchanged (splitting the
sequence, permuting channels or batches, linearity in u, a chain of decode
steps).

Steps pinned (see the page sections cited in ``oracle/scan_oracle.c``):
  A = -exp(A_log), Abar = exp(dt*A), Bbar = dt*B, h_t = Abar h_{t-1} + Bbar u,
  y = sum_n C h + D u, SiLU(z) gate, dt = softplus(delta + bias), zero h0,
  a given h0, the state restarting at document boundaries (reset mask), the
  gradients (finite differences), and the causal depthwise conv1d + SiLU in
  front of the scan (numpy.convolve, impulse response, SiLU values, state
  chaining).
"""
from __future__ import annotations

import numpy as np
from scipy.special import expit

import oracle

RTOL = 1e-12


def _close(got, want, rtol=RTOL, atol=0.0, what=""):
    cplx = np.iscomplexobj(got) or np.iscomplexobj(want)
    got = np.asarray(got, dtype=np.complex128 if cplx else np.float64)
    want = np.asarray(want, dtype=np.complex128 if cplx else np.float64)
    assert got.shape == want.shape, f"{what}: shape {got.shape} != {want.shape}"
    scale = max(float(np.max(np.abs(want))) if want.size else 0.0, 1e-300)
    err = float(np.max(np.abs(got - want))) if want.size else 0.0
    assert err <= rtol * scale + atol, f"{what}: max abs err {err:.3e} (scale {scale:.3e})"


def _softplus_inv(dt):
    """raw such that log(1 + e^raw) == dt (inverse softplus, by expm1)."""
    return np.log(np.expm1(dt))


def _silu(z):
    return z * expit(z)


def _rng(seed):
    return np.random.default_rng(seed)


# --------------------------------------------------------------------------
def check_delta_zero_limit(lib):
    """dt = 0 (softplus off, zero delta, no bias): Abar = 1 and Bbar = 0, so the
    state never leaves zero and out = D*u*SiLU(z) exactly."""
    r = _rng(1)
    b, d, L, N = 2, 3, 9, 4
    u, z = r.normal(size=(b, d, L)), r.normal(size=(b, d, L))
    B, C = r.normal(size=(b, L, N)), r.normal(size=(b, L, N))
    D = r.normal(size=d)
    A_log = np.log(r.uniform(0.5, 8, size=(d, N)))
    y, hL, _ = oracle.selective_scan(u, np.zeros_like(u), A_log, B, C, D=D, z=z,
                                     softplus=False, lib=lib)
    assert np.all(hL == 0.0), "state must stay exactly zero when dt = 0"
    _close(y, D[None, :, None] * u * _silu(z), rtol=1e-14, what="dt=0 output")


def check_single_step(lib):
    """L = 1 from a zero state: h = dt*B*u, out = (sum_n C h + D u) SiLU(z).
    dt is fixed through the inverse softplus, with a nonzero bias, and spans
    both softplus branches (dt below and above log 2)."""
    r = _rng(2)
    b, d, N = 3, 4, 5
    dt = np.array([1e-4, 0.05, 0.9, 3.0])                 # per channel
    bias = r.normal(size=d)
    raw = np.broadcast_to((_softplus_inv(dt) - bias)[None, :, None], (b, d, 1)).copy()
    u, z = r.normal(size=(b, d, 1)), r.normal(size=(b, d, 1))
    B, C = r.normal(size=(b, 1, N)), r.normal(size=(b, 1, N))
    D = r.normal(size=d)
    A_log = r.normal(size=(d, N))
    y, hL, _ = oracle.selective_scan(u, raw, A_log, B, C, D=D, z=z, delta_bias=bias,
                                     softplus=True, lib=lib)
    h = dt[None, :, None] * B[:, 0, None, :] * u[:, :, 0, None]      # [b, d, N]
    _close(hL, h, rtol=1e-12, what="single-step state")
    out = (np.einsum("bn,bdn->bd", C[:, 0, :], h) + D[None, :] * u[:, :, 0]) * _silu(z[:, :, 0])
    _close(y[:, :, 0], out, rtol=1e-12, what="single-step output")


def check_geometric_series(lib):
    """Constant dt, B, C, u: h_t = Bbar u (1 - a^(t+1)) / (1 - a) with
    a = exp(-dt k) for A_log = log k, and out_t = sum_n C_n h_t + D u.  B and C
    differ per state and per batch; dt differs per channel (through the bias)
    and softplus is off here, so dt is used as given."""
    b, d, L, N = 2, 3, 300, 4
    k = np.array([[1.0, 2.0, 3.0, 4.0], [0.5, 1.5, 7.0, 16.0], [1.0, 1.0, 2.0, 64.0]])
    dt = np.array([0.05, 0.002, 0.3])
    Bn = np.array([[0.7, -1.1, 0.3, 2.0], [-0.4, 0.9, 1.3, -0.2]])      # per batch, state
    Cn = np.array([[1.2, 0.5, -0.8, 0.1], [0.3, -1.5, 0.6, 1.1]])
    uc = np.array([[0.9, -0.6, 1.7], [-1.3, 0.4, 0.8]])                 # per batch, channel
    D = np.array([0.25, -1.0, 2.0])
    u = np.repeat(uc[:, :, None], L, axis=2)
    B = np.repeat(Bn[:, None, :], L, axis=1)
    C = np.repeat(Cn[:, None, :], L, axis=1)
    bias = dt.copy()
    y, hL, _ = oracle.selective_scan(u, np.zeros((b, d, L)), np.log(k), B, C, D=D,
                                     delta_bias=bias, softplus=False, lib=lib)
    a = np.exp(-dt[:, None] * k)                                          # [d, N]
    t = np.arange(L)
    bu = dt[None, :, None] * Bn[:, None, :] * uc[:, :, None]              # [b, d, N]
    h = bu[:, :, None, :] * (1 - a[None, :, None, :] ** (t[None, None, :, None] + 1)) \
        / (1 - a[None, :, None, :])                                       # [b, d, L, N]
    _close(hL, h[:, :, -1, :], rtol=1e-11, what="geometric final state")
    out = np.einsum("bn,bdtn->bdt", Cn, h) + D[None, :, None] * u
    _close(y, out, rtol=1e-11, what="geometric outputs")


def check_steady_state(lib):
    """A long constant input drives the state to its fixed point Bbar u / (1 - a)."""
    d, N, L = 2, 3, 20000
    k = np.array([[1.0, 2.0, 3.0], [4.0, 5.0, 6.0]])
    dt = np.array([0.01, 0.02])
    Bn, uc = np.array([0.5, -1.0, 2.0]), np.array([1.5, -0.5])
    u = np.repeat(uc[None, :, None], L, axis=2)
    B = np.repeat(Bn[None, None, :], L, axis=1)
    _, hL, _ = oracle.selective_scan(u, np.repeat(dt[None, :, None], L, axis=2), np.log(k), B,
                                     np.ones((1, L, N)), softplus=False, lib=lib)
    h_inf = dt[:, None] * Bn[None, :] * uc[:, None] / (1 - np.exp(-dt[:, None] * k))
    _close(hL[0], h_inf, rtol=1e-10, what="steady state")


def check_lti_convolution(lib):
    """Time-invariant case (constant dt, B, C; random u): the recurrence equals
    the causal convolution y_t = sum_{j<=t} K_j u_{t-j} + D u_t with the kernel
    K_j = sum_n C_n a_n^j dt B_n (the recurrence/convolution equivalence of the
    mhpn.cn article, section 3).  Evaluated with numpy.convolve."""
    r = _rng(3)
    b, d, L, N = 2, 3, 128, 6
    k = r.uniform(0.5, 10.0, size=(d, N))
    dt = np.array([0.03, 0.3, 0.001])
    Bn, Cn = r.normal(size=(b, N)), r.normal(size=(b, N))
    u = r.normal(size=(b, d, L))
    D = r.normal(size=d)
    B = np.repeat(Bn[:, None, :], L, axis=1)
    C = np.repeat(Cn[:, None, :], L, axis=1)
    raw = np.broadcast_to(_softplus_inv(dt)[None, :, None], (b, d, L)).copy()
    y, _, _ = oracle.selective_scan(u, raw, np.log(k), B, C, D=D, softplus=True, lib=lib)
    j = np.arange(L)
    for bi in range(b):
        for di in range(d):
            a = np.exp(-dt[di] * k[di])                                      # [N]
            K = (Cn[bi] * dt[di] * Bn[bi] * a[None, :] ** j[:, None]).sum(axis=1)
            want = np.convolve(u[bi, di], K)[:L] + D[di] * u[bi, di]
            _close(y[bi, di], want, rtol=1e-11, what=f"convolution b={bi} d={di}")


def check_bruteforce_unrolled(lib):
    """Everything time-varying, tiny sizes: the state written as an explicit
    sum h_t = sum_{s<=t} (prod_{s<r<=t} Abar_r) Bbar_s u_s, with softplus via
    numpy.logaddexp and the gate via scipy's expit."""
    r = _rng(4)
    b, d, L, N = 2, 3, 7, 3
    u, z, raw = r.normal(size=(b, d, L)), r.normal(size=(b, d, L)), r.normal(size=(b, d, L))
    B, C = r.normal(size=(b, L, N)), r.normal(size=(b, L, N))
    A_log, D, bias = r.normal(size=(d, N)), r.normal(size=d), r.normal(size=d)
    y, hL, _ = oracle.selective_scan(u, raw, A_log, B, C, D=D, z=z, delta_bias=bias,
                                     softplus=True, lib=lib)
    want_y = np.zeros((b, d, L))
    want_h = np.zeros((b, d, N))
    for bi in range(b):
        for di in range(d):
            dt = np.logaddexp(0.0, raw[bi, di] + bias[di])                 # [L]
            A = -np.exp(A_log[di])                                         # [N]
            for t in range(L):
                h = np.zeros(N)
                for s in range(t + 1):
                    decay = np.ones(N)
                    for rr in range(s + 1, t + 1):
                        decay = decay * np.exp(dt[rr] * A)
                    h = h + decay * dt[s] * B[bi, s] * u[bi, di, s]
                yt = float(np.dot(C[bi, t], h)) + D[di] * u[bi, di, t]
                want_y[bi, di, t] = yt * z[bi, di, t] * expit(z[bi, di, t])
                if t == L - 1:
                    want_h[bi, di] = h
    _close(hL, want_h, rtol=1e-12, what="unrolled final state")
    _close(y, want_y, rtol=1e-12, what="unrolled outputs")


def check_linearity_in_u(lib):
    """For fixed dt, B, C, z the map u -> (y, h_L) is linear."""
    r = _rng(5)
    b, d, L, N = 2, 4, 40, 4
    raw, z = r.normal(size=(b, d, L)), r.normal(size=(b, d, L))
    B, C = r.normal(size=(b, L, N)), r.normal(size=(b, L, N))
    A_log, D, bias = r.normal(size=(d, N)), r.normal(size=d), r.normal(size=d)
    u1, u2 = r.normal(size=(b, d, L)), r.normal(size=(b, d, L))
    al, be = 0.75, -1.25
    run = lambda uu: oracle.selective_scan(uu, raw, A_log, B, C, D=D, z=z, delta_bias=bias,
                                           lib=lib)
    y1, h1, _ = run(u1)
    y2, h2, _ = run(u2)
    y3, h3, _ = run(al * u1 + be * u2)
    _close(y3, al * y1 + be * y2, rtol=1e-12, what="linearity y")
    _close(h3, al * h1 + be * h2, rtol=1e-12, what="linearity state")


def check_split_invariance(lib):
    """Scanning [0, L) equals scanning [0, L1) and then [L1, L) from the state
    reached at L1 (the chunk-carry property the GPU relies on)."""
    r = _rng(6)
    b, d, L, N, L1 = 2, 3, 50, 4, 19
    u, z, raw = r.normal(size=(b, d, L)), r.normal(size=(b, d, L)), r.normal(size=(b, d, L))
    B, C = r.normal(size=(b, L, N)), r.normal(size=(b, L, N))
    A_log, D, bias = r.normal(size=(d, N)), r.normal(size=d), r.normal(size=d)
    kw = dict(D=D, delta_bias=bias, softplus=True, lib=lib)
    y, hL, _ = oracle.selective_scan(u, raw, A_log, B, C, z=z, **kw)
    ya, ha, _ = oracle.selective_scan(u[..., :L1], raw[..., :L1], A_log, B[:, :L1], C[:, :L1],
                                      z=z[..., :L1], **kw)
    yb, hb, _ = oracle.selective_scan(u[..., L1:], raw[..., L1:], A_log, B[:, L1:], C[:, L1:],
                                      z=z[..., L1:], h0=ha, **kw)
    _close(y, np.concatenate([ya, yb], axis=-1), rtol=1e-12, what="split outputs")
    _close(hL, hb, rtol=1e-12, what="split final state")


def check_decode_chain(lib):
    """L single-token decode steps from a zero state reproduce the scan."""
    r = _rng(7)
    b, d, L, N = 2, 3, 12, 4
    u, z, raw = r.normal(size=(b, d, L)), r.normal(size=(b, d, L)), r.normal(size=(b, d, L))
    B, C = r.normal(size=(b, L, N)), r.normal(size=(b, L, N))
    A_log, D, bias = r.normal(size=(d, N)), r.normal(size=d), r.normal(size=d)
    y, hL, _ = oracle.selective_scan(u, raw, A_log, B, C, D=D, z=z, delta_bias=bias, lib=lib)
    st = np.zeros((b, d, N))
    ys = []
    for t in range(L):
        out, st = oracle.selective_state_update(st, u[..., t], raw[..., t], A_log, B[:, t], C[:, t],
                                                D=D, z=z[..., t], dt_bias=bias, lib=lib)
        ys.append(out)
    _close(np.stack(ys, axis=-1), y, rtol=1e-12, what="decode chain outputs")
    _close(st, hL, rtol=1e-12, what="decode chain state")


def check_decode_single_step(lib):
    """One decode step from a known state: h' = exp(-dt k) h + dt B x and
    out = (sum_n C h' + D x) SiLU(z), dt fixed through the inverse softplus."""
    b, d, N = 2, 2, 3
    k = np.array([[1.0, 2.0, 3.0], [0.5, 4.0, 9.0]])
    dt = np.array([0.02, 1.5])
    bias = np.array([0.3, -0.7])
    x = np.array([[1.0, -2.0], [0.5, 3.0]])
    z = np.array([[0.4, -1.2], [2.0, 0.0]])
    B = np.array([[0.5, -1.0, 2.0], [1.5, 0.2, -0.3]])
    C = np.array([[1.0, 0.25, -0.5], [-2.0, 0.5, 1.0]])
    D = np.array([0.1, -0.4])
    h = np.arange(b * d * N, dtype=np.float64).reshape(b, d, N) * 0.1 - 0.5
    raw = np.broadcast_to(_softplus_inv(dt)[None, :] - bias[None, :], (b, d)).copy()
    out, h1 = oracle.selective_state_update(h, x, raw,
                                            np.log(k), B, C, D=D, z=z, dt_bias=bias, lib=lib)
    want_h = np.exp(-dt[None, :, None] * k[None]) * h + dt[None, :, None] * B[:, None, :] * x[..., None]
    _close(h1, want_h, rtol=1e-12, what="decode state")
    want = (np.einsum("bn,bdn->bd", C, want_h) + D[None, :] * x) * _silu(z)
    _close(out, want, rtol=1e-12, what="decode output")


def check_permutations(lib):
    """Permuting channels (u, delta, z, A_log, D, bias together) permutes the
    outputs; swapping batches (u, delta, z, B, C together) swaps them."""
    r = _rng(8)
    b, d, L, N = 3, 5, 16, 4
    u, z, raw = r.normal(size=(b, d, L)), r.normal(size=(b, d, L)), r.normal(size=(b, d, L))
    B, C = r.normal(size=(b, L, N)), r.normal(size=(b, L, N))
    A_log, D, bias = r.normal(size=(d, N)), r.normal(size=d), r.normal(size=d)
    y, hL, _ = oracle.selective_scan(u, raw, A_log, B, C, D=D, z=z, delta_bias=bias, lib=lib)
    p = np.array([3, 0, 4, 1, 2])
    yp, hp, _ = oracle.selective_scan(u[:, p], raw[:, p], A_log[p], B, C, D=D[p], z=z[:, p],
                                      delta_bias=bias[p], lib=lib)
    _close(yp, y[:, p], rtol=1e-14, what="channel permutation y")
    _close(hp, hL[:, p], rtol=1e-14, what="channel permutation state")
    q = np.array([2, 0, 1])
    yq, hq, _ = oracle.selective_scan(u[q], raw[q], A_log, B[q], C[q], D=D, z=z[q],
                                      delta_bias=bias, lib=lib)
    _close(yq, y[q], rtol=1e-14, what="batch permutation y")
    _close(hq, hL[q], rtol=1e-14, what="batch permutation state")


def check_optional_inputs(lib):
    """No z: no gate.  No D: no skip.  No bias: delta used alone.  Each optional
    input, when absent, must act like its neutral value supplied explicitly
    (a gate that passes y through is z -> infinity; emulate with the explicit
    ungated closed form instead)."""
    r = _rng(9)
    b, d, L, N = 1, 3, 10, 4
    u, raw = r.normal(size=(b, d, L)), r.normal(size=(b, d, L))
    B, C = r.normal(size=(b, L, N)), r.normal(size=(b, L, N))
    A_log = r.normal(size=(d, N))
    y0, h0, _ = oracle.selective_scan(u, raw, A_log, B, C, lib=lib)
    y1, h1, _ = oracle.selective_scan(u, raw, A_log, B, C, D=np.zeros(d), delta_bias=np.zeros(d),
                                      lib=lib)
    _close(y0, y1, rtol=0, what="absent D/bias == zero D/bias")
    _close(h0, h1, rtol=0, what="absent D/bias state")
    z = r.normal(size=(b, d, L))
    y2, _, _ = oracle.selective_scan(u, raw, A_log, B, C, z=z, lib=lib)
    _close(y2, y0 * _silu(z), rtol=1e-13, what="gate multiplies the ungated output")


def check_reset_splits_documents(lib):
    """A reset mask cuts each batch row into documents: the scan must equal the
    concatenation of independent scans of the documents, the first started
    from h0 and every later one from a zero state (codechina.net overview,
    section 3.2: resetting the hidden state isolates documents).  The masks
    differ between batch rows, and one boundary sits on the last step."""
    r = _rng(10)
    b, d, L, N = 2, 3, 30, 4
    u, z, raw = r.normal(size=(b, d, L)), r.normal(size=(b, d, L)), r.normal(size=(b, d, L))
    B, C = r.normal(size=(b, L, N)), r.normal(size=(b, L, N))
    A_log, D, bias = r.normal(size=(d, N)), r.normal(size=d), r.normal(size=d)
    h0 = r.normal(size=(b, d, N))
    starts = {0: [7, 8, 20], 1: [13, 29]}
    reset = np.zeros((b, L), dtype=np.uint8)
    for bi, ss in starts.items():
        reset[bi, ss] = 1
    kw = dict(D=D, delta_bias=bias, softplus=True, lib=lib)
    y, hL, _ = oracle.selective_scan(u, raw, A_log, B, C, z=z, h0=h0, reset=reset, **kw)
    for bi, ss in starts.items():
        edges = [0, *ss, L]
        ys, h = [], None
        for k, (t0, t1) in enumerate(zip(edges[:-1], edges[1:])):
            yk, h, _ = oracle.selective_scan(u[bi:bi + 1, :, t0:t1], raw[bi:bi + 1, :, t0:t1],
                                             A_log, B[bi:bi + 1, t0:t1], C[bi:bi + 1, t0:t1],
                                             z=z[bi:bi + 1, :, t0:t1],
                                             h0=h0[bi:bi + 1] if k == 0 else None, **kw)
            ys.append(yk)
        _close(y[bi:bi + 1], np.concatenate(ys, axis=-1), rtol=1e-12, what=f"documents b={bi}")
        _close(hL[bi:bi + 1], h, rtol=1e-12, what=f"last document state b={bi}")


def check_reset_every_step_is_memoryless(lib):
    """A reset at every step leaves no memory: h_t = dt_t B_t u_t, so
    y_t = (sum_n C_tn dt_t B_tn u_t + D u_t) SiLU(z_t), whatever h0 was."""
    r = _rng(11)
    b, d, L, N = 2, 2, 6, 3
    u, z, raw = r.normal(size=(b, d, L)), r.normal(size=(b, d, L)), r.normal(size=(b, d, L))
    B, C = r.normal(size=(b, L, N)), r.normal(size=(b, L, N))
    A_log, D, bias = r.normal(size=(d, N)), r.normal(size=d), r.normal(size=d)
    y, hL, _ = oracle.selective_scan(u, raw, A_log, B, C, D=D, z=z, delta_bias=bias,
                                     h0=r.normal(size=(b, d, N)), reset=np.ones((b, L)), lib=lib)
    dt = np.logaddexp(0.0, raw + bias[None, :, None])                     # [b, d, L]
    h = dt[..., None] * B[:, None] * u[..., None]                         # [b, d, L, N]
    want = (np.einsum("btn,bdtn->bdt", C, h) + D[None, :, None] * u) * _silu(z)
    _close(y, want, rtol=1e-12, what="memoryless outputs")
    _close(hL, h[:, :, -1], rtol=1e-12, what="memoryless final state")


def check_reset_at_start_ignores_h0(lib):
    """A document boundary on step 0 discards the given initial state."""
    r = _rng(12)
    b, d, L, N = 2, 3, 12, 4
    u, raw = r.normal(size=(b, d, L)), r.normal(size=(b, d, L))
    B, C = r.normal(size=(b, L, N)), r.normal(size=(b, L, N))
    A_log = r.normal(size=(d, N))
    reset = np.zeros((b, L), dtype=np.uint8)
    reset[:, 0] = 1
    y0, h0, _ = oracle.selective_scan(u, raw, A_log, B, C, lib=lib)
    y1, h1, _ = oracle.selective_scan(u, raw, A_log, B, C, h0=r.normal(size=(b, d, N)),
                                      reset=reset, lib=lib)
    _close(y1, y0, rtol=0, what="outputs after a reset on step 0")
    _close(h1, h0, rtol=0, what="state after a reset on step 0")


def _fd_check(lib, softplus, with_opt, seed, ex=False, dlast=False):
    """Central differences of the forward oracle's loss sum(dout * y) with
    respect to every element of every input must equal the gradients of the
    backward oracle (fp64: steps of 1e-6 leave errors near 1e-9).  With
    ``ex`` the scans also start from a random h0 (its gradient checked too)
    and carry document boundaries (a reset inside each batch row).  With
    ``dlast`` the loss adds sum(w * last_state), w passed as dlast_state."""
    r = _rng(seed)
    b, d, L, N = 2, 2, 5, 3
    x = dict(u=r.normal(size=(b, d, L)), delta=r.normal(size=(b, d, L)),
             A_log=r.normal(size=(d, N)) * 0.5, B=r.normal(size=(b, L, N)),
             C=r.normal(size=(b, L, N)))
    if not softplus:  # keep dt positive and moderate
        x["delta"] = np.abs(x["delta"]) * 0.3 + 0.05
    if with_opt:
        x.update(D=r.normal(size=d), z=r.normal(size=(b, d, L)), delta_bias=r.normal(size=d))
    reset = None
    if ex:
        x["h0"] = r.normal(size=(b, d, N))
        reset = np.zeros((b, L), dtype=np.uint8)
        reset[0, 2] = reset[1, 3] = 1
    dout = r.normal(size=(b, d, L))
    w = r.normal(size=(b, d, N)) if dlast else None

    def loss(xx):
        y, hl, _ = oracle.selective_scan(xx["u"], xx["delta"], xx["A_log"], xx["B"], xx["C"],
                                         D=xx.get("D"), z=xx.get("z"),
                                         delta_bias=xx.get("delta_bias"), softplus=softplus,
                                         h0=xx.get("h0"), reset=reset, nthreads=1, lib=lib)
        return float(np.sum(dout * y)) + (float(np.sum(w * hl)) if dlast else 0.0)

    g = oracle.selective_scan_bwd(x["u"], x["delta"], x["A_log"], x["B"], x["C"], dout,
                                  D=x.get("D"), z=x.get("z"), delta_bias=x.get("delta_bias"),
                                  softplus=softplus, h0=x.get("h0"), reset=reset,
                                  dlast_state=w, lib=lib)
    names = {"u": "du", "delta": "ddelta", "A_log": "dA_log", "B": "dB", "C": "dC", "D": "dD",
             "z": "dz", "delta_bias": "ddelta_bias", "h0": "dh0"}
    eps = 1e-6
    for k, gk in names.items():
        if k not in x:
            assert gk not in g, f"{gk} returned without its input"
            continue
        fd = np.zeros_like(x[k])
        for idx in np.ndindex(x[k].shape):
            xp = {kk: vv.copy() for kk, vv in x.items()}
            xm = {kk: vv.copy() for kk, vv in x.items()}
            xp[k][idx] += eps
            xm[k][idx] -= eps
            fd[idx] = (loss(xp) - loss(xm)) / (2 * eps)
        _close(g[gk], fd, rtol=1e-6, atol=1e-8, what=f"{gk} vs finite differences")


def check_backward_finite_differences(lib):
    _fd_check(lib, softplus=True, with_opt=True, seed=13)


def check_backward_finite_differences_plain(lib):
    """The other branches: softplus off, no gate, no skip, no bias."""
    _fd_check(lib, softplus=False, with_opt=False, seed=14)


# --------------------------------------------------------------------------
# causal depthwise conv1d (+ SiLU) in front of the scan
def check_conv_against_numpy_convolve(lib):
    """Without the activation, each channel is numpy's full convolution of the
    zero-padded input with the channel's filter (PyTorch's Conv1d is a
    cross-correlation, so the filter is reversed for np.convolve), keeping the
    first L outputs; widths 1 to 6, with and without a bias."""
    r = _rng(40)
    for width in (1, 2, 3, 4, 6):
        b, d, L = 2, 3, 17
        x, w = r.normal(size=(b, d, L)), r.normal(size=(d, width))
        bias = r.normal(size=d) if width % 2 == 0 else None
        out, _ = oracle.causal_conv1d(x, w, bias=bias, silu=False, lib=lib)
        want = np.empty_like(x)
        for bi in range(b):
            for di in range(d):
                full = np.convolve(x[bi, di], w[di][::-1], mode="full")[:L]
                want[bi, di] = full + (bias[di] if bias is not None else 0.0)
        _close(out, want, rtol=1e-13, what=f"conv width {width}")


def check_conv_impulse_response(lib):
    """A unit impulse at step t0 (no bias, no activation) comes out as the
    filter read backwards: out[t0 + j] = w[width-1-j] for j < width, zero
    elsewhere -- the current input meets the last tap, and nothing leaks
    before t0 (causality)."""
    L, t0, width = 12, 5, 4
    w = np.array([[0.5, -1.25, 2.0, 3.5]])
    x = np.zeros((1, 1, L))
    x[0, 0, t0] = 1.0
    out, _ = oracle.causal_conv1d(x, w, silu=False, lib=lib)
    want = np.zeros(L)
    for j in range(width):
        want[t0 + j] = w[0, width - 1 - j]
    assert np.array_equal(out[0, 0], want), (out[0, 0], want)


def check_conv_silu_closed_forms(lib):
    """A pass-through filter (last tap 1, bias 0) leaves SiLU(x) = x/(1+e^-x):
    SiLU(0) = 0, SiLU(1) = 1/(1+e^-1) = 0.7310585786300049, SiLU(-1) =
    -0.2689414213699951, SiLU(40) = 40 to double precision; the bias enters
    before the activation (SiLU(0 + 1) for a zero input)."""
    x = np.array([[[0.0, 1.0, -1.0, 40.0]]])
    w = np.array([[0.0, 0.0, 0.0, 1.0]])
    out, _ = oracle.causal_conv1d(x, w, silu=True, lib=lib)
    _close(out[0, 0], [0.0, 0.7310585786300049, -0.2689414213699951, 40.0], rtol=1e-15,
           what="SiLU values")
    out, _ = oracle.causal_conv1d(np.zeros((1, 1, 3)), w, bias=np.array([1.0]), silu=True, lib=lib)
    _close(out[0, 0], [0.7310585786300049] * 3, rtol=1e-15, what="bias before SiLU")


def check_conv_state_chaining(lib):
    """Cutting a sequence into blocks and passing each block's final state as
    the next block's initial state gives the unsplit result, outputs and final
    state; the final state is the last width-1 inputs (also when a block is
    shorter than width-1)."""
    r = _rng(41)
    b, d, L, width = 2, 4, 23, 4
    x, w, bias = r.normal(size=(b, d, L)), r.normal(size=(d, width)), r.normal(size=d)
    st0 = r.normal(size=(b, d, width - 1))
    ref, fin = oracle.causal_conv1d(x, w, bias=bias, initial_state=st0, lib=lib)
    _close(fin, x[:, :, L - (width - 1):], rtol=0.0, what="final state = last inputs")
    outs, st = [], st0
    for lo, hi in ((0, 2), (2, 3), (3, 11), (11, 23)):
        o, st = oracle.causal_conv1d(x[:, :, lo:hi], w, bias=bias, initial_state=st, lib=lib)
        outs.append(o)
    _close(np.concatenate(outs, axis=2), ref, rtol=0.0, what="chained blocks")
    _close(st, fin, rtol=0.0, what="chained final state")


def check_conv_initial_state_reaches_first_outputs_only(lib):
    """The initial state is the input before step 0: with zero x it alone
    drives out[t] for t < width-1 (out[t] = sum_k w[k] st[t+k] over the taps
    that reach back before the sequence), and outputs from step width-1 on
    equal the bias."""
    width = 4
    w = np.array([[1.0, 10.0, 100.0, 1000.0]])
    st = np.array([[[2.0, 3.0, 5.0]]])
    out, _ = oracle.causal_conv1d(np.zeros((1, 1, 6)), w, bias=np.array([0.25]),
                                  initial_state=st, silu=False, lib=lib)
    want = [1 * 2 + 10 * 3 + 100 * 5, 1 * 3 + 10 * 5, 1 * 5, 0.0, 0.0, 0.0]
    _close(out[0, 0], np.array(want) + 0.25, rtol=1e-15, what="initial state")


def check_conv_channels_and_batches_are_independent(lib):
    """Each (batch, channel) row uses only its own input and its channel's
    filter: permuting channels (with their filters and biases) or batch rows
    permutes the output the same way."""
    r = _rng(42)
    b, d, L, width = 3, 5, 9, 4
    x, w, bias = r.normal(size=(b, d, L)), r.normal(size=(d, width)), r.normal(size=d)
    st = r.normal(size=(b, d, width - 1))
    ref, fin = oracle.causal_conv1d(x, w, bias=bias, initial_state=st, lib=lib)
    pd, pb = r.permutation(d), r.permutation(b)
    out, f2 = oracle.causal_conv1d(x[pb][:, pd], w[pd], bias=bias[pd],
                                   initial_state=st[pb][:, pd], lib=lib)
    _close(out, ref[pb][:, pd], rtol=0.0, what="permuted rows")
    _close(f2, fin[pb][:, pd], rtol=0.0, what="permuted final state")


# --------------------------------------------------------------------------
# complex-state (S4D-Lin) scan
def _cplx(r, shape):
    return r.normal(size=shape) + 1j * r.normal(size=shape)


def check_complex_with_real_parameters_is_the_real_scan(lib):
    """A_im = 0 and real B, C: every state stays real and the complex scan is
    the real scan (same dt, D, gate), output and final state."""
    r = _rng(50)
    b, d, L, N = 2, 3, 21, 4
    u, delta, z = r.normal(size=(b, d, L)), r.normal(size=(b, d, L)), r.normal(size=(b, d, L))
    A_log = np.log(r.uniform(0.5, 4, size=(d, N)))
    B, C = r.normal(size=(b, L, N)), r.normal(size=(b, L, N))
    D, bias = r.normal(size=d), r.normal(size=d)
    yc, hc = oracle.selective_scan_complex(u, delta, A_log, np.zeros((d, N)), B + 0j, C + 0j,
                                           D=D, z=z, delta_bias=bias, lib=lib)
    yr, hr, _ = oracle.selective_scan(u, delta, A_log, B, C, D=D, z=z, delta_bias=bias)
    _close(yc, yr, rtol=1e-13, what="complex vs real output")
    _close(hc.real, hr, rtol=1e-13, what="complex vs real state")
    assert np.all(hc.imag == 0.0)


def check_complex_impulse_response_closed_form(lib):
    """S4D-Lin A = -0.5 + i*n (and one channel with Re A ~ 0: a pure
    rotation), a unit impulse at t = 0, constant dt, B and C: h_t = dt B a^t
    with a = exp(dt A), so y_t = Re(sum_n C_n dt B_n a_n^t) + D [t == 0], from
    complex powers (no recurrence); for the rotation, |h_t| stays |dt B| and
    the phase advances by dt * Im A per step."""
    r = _rng(51)
    b, d, L, N = 1, 2, 30, 5
    dt = 0.3
    A_log = np.stack([np.full(N, np.log(0.5)), np.full(N, -60.0)])  # Re A = -0.5 and ~ -1e-26
    A_im = np.tile(np.arange(N, dtype=float), (d, 1))
    B0, C0 = _cplx(r, N), _cplx(r, N)
    B = np.broadcast_to(B0, (b, L, N)).copy()
    C = np.broadcast_to(C0, (b, L, N)).copy()
    u = np.zeros((b, d, L))
    u[:, :, 0] = 1.0
    D = np.array([0.7, -1.1])
    y, hL = oracle.selective_scan_complex(u, np.full((b, d, L), dt), A_log, A_im, B, C, D=D,
                                          softplus=False, lib=lib)
    t = np.arange(L)
    for di in range(d):
        a = np.exp(dt * (-np.exp(A_log[di]) + 1j * A_im[di]))
        ht = dt * B0[None, :] * a[None, :] ** t[:, None]           # [L, N]
        want = (ht * C0[None, :]).sum(axis=1).real + D[di] * u[0, di]
        _close(y[0, di], want, rtol=1e-12, what=f"impulse response, channel {di}")
        _close(hL[0, di], ht[-1], rtol=1e-12, what=f"final state, channel {di}")
    rot = hL[0, 1]
    _close(np.abs(rot), np.abs(dt * B0), rtol=1e-12, what="rotation keeps the modulus")
    _close(np.exp(1j * (np.angle(rot) - np.angle(dt * B0))),
           np.exp(1j * dt * A_im[1] * (L - 1)), rtol=1e-11, what="rotation phase")


def check_complex_geometric_series(lib):
    """Constant u, dt and B: h_L = dt B u (1 - a^L) / (1 - a), a = exp(dt A)."""
    r = _rng(52)
    b, d, L, N = 1, 3, 40, 4
    dt, uval = 0.2, 1.5
    A_log = np.log(r.uniform(0.2, 2.0, size=(d, N)))
    A_im = r.uniform(-6, 6, size=(d, N))
    B0 = _cplx(r, N)
    B = np.broadcast_to(B0, (b, L, N)).copy()
    y, hL = oracle.selective_scan_complex(np.full((b, d, L), uval), np.full((b, d, L), dt),
                                          A_log, A_im, B, _cplx(r, (b, L, N)), softplus=False,
                                          lib=lib)
    a = np.exp(dt * (-np.exp(A_log) + 1j * A_im))
    want = dt * B0[None, :] * uval * (1 - a ** L) / (1 - a)
    _close(hL[0], want, rtol=1e-12, what="geometric series")


def check_complex_bruteforce_unrolled(lib):
    """Everything time-varying (complex B and C per step, any A_im), tiny
    sizes: the complex state written as the explicit sum
    h_t = sum_{s<=t} (prod_{s<r<=t} exp(dt_r A)) dt_s B_s u_s with numpy's
    complex exp, y_t = (Re sum_n C_tn h_tn + D u_t) * SiLU(z_t)."""
    r = _rng(54)
    b, d, L, N = 2, 2, 6, 3
    u, z, raw = r.normal(size=(b, d, L)), r.normal(size=(b, d, L)), r.normal(size=(b, d, L))
    A_log, A_im = r.normal(size=(d, N)) * 0.5, r.normal(size=(d, N)) * 3.0
    B, C = _cplx(r, (b, L, N)), _cplx(r, (b, L, N))
    D, bias = r.normal(size=d), r.normal(size=d)
    y, hL = oracle.selective_scan_complex(u, raw, A_log, A_im, B, C, D=D, z=z, delta_bias=bias,
                                          lib=lib)
    want_y = np.zeros((b, d, L))
    want_h = np.zeros((b, d, N), dtype=complex)
    for bi in range(b):
        for di in range(d):
            dt = np.logaddexp(0.0, raw[bi, di] + bias[di])
            A = -np.exp(A_log[di]) + 1j * A_im[di]
            for t in range(L):
                h = np.zeros(N, dtype=complex)
                for s_ in range(t + 1):
                    decay = np.ones(N, dtype=complex)
                    for rr in range(s_ + 1, t + 1):
                        decay = decay * np.exp(dt[rr] * A)
                    h = h + decay * dt[s_] * B[bi, s_] * u[bi, di, s_]
                yt = float(np.sum(C[bi, t] * h).real) + D[di] * u[bi, di, t]
                want_y[bi, di, t] = yt * z[bi, di, t] * expit(z[bi, di, t])
                if t == L - 1:
                    want_h[bi, di] = h
    _close(hL, want_h, rtol=1e-12, what="complex unrolled final state")
    _close(y, want_y, rtol=1e-12, what="complex unrolled outputs")


def check_complex_conjugation_symmetry(lib):
    """Conjugating A, B and C conjugates every state and leaves the real
    output unchanged."""
    r = _rng(53)
    b, d, L, N = 2, 2, 17, 3
    args = dict(u=r.normal(size=(b, d, L)), delta=r.normal(size=(b, d, L)),
                A_log_re=np.log(r.uniform(0.3, 3, size=(d, N))))
    A_im, B, C = r.normal(size=(d, N)) * 3, _cplx(r, (b, L, N)), _cplx(r, (b, L, N))
    z = r.normal(size=(b, d, L))
    y1, h1 = oracle.selective_scan_complex(A_im=A_im, B=B, C=C, z=z, lib=lib, **args)
    y2, h2 = oracle.selective_scan_complex(A_im=-A_im, B=B.conj(), C=C.conj(), z=z, lib=lib,
                                           **args)
    _close(y2, y1, rtol=1e-12, what="conjugated output")
    _close(h2, h1.conj(), rtol=1e-12, what="conjugated state")


def check_backward_finite_differences_h0_reset(lib):
    _fd_check(lib, softplus=True, with_opt=True, seed=15, ex=True)


def check_backward_reset_splits_documents(lib):
    """A document boundary at step L1 makes the backward of the whole row equal
    the backwards of the two documents taken alone (the second from a zero
    state): per-element gradients and dB/dC per step match piecewise, the
    summed dA_log, dD and bias gradients add up, and no gradient reaches h0
    from the second document."""
    r = _rng(16)
    b, d, L, N, L1 = 1, 3, 12, 4, 5
    x = dict(u=r.normal(size=(b, d, L)), delta=r.normal(size=(b, d, L)),
             A_log=r.normal(size=(d, N)) * 0.5, B=r.normal(size=(b, L, N)),
             C=r.normal(size=(b, L, N)), dout=r.normal(size=(b, d, L)))
    kw = dict(D=r.normal(size=d), z=r.normal(size=(b, d, L)), delta_bias=r.normal(size=d))
    h0 = r.normal(size=(b, d, N))
    reset = np.zeros((b, L))
    reset[0, L1] = 1
    whole = oracle.selective_scan_bwd(x["u"], x["delta"], x["A_log"], x["B"], x["C"], x["dout"],
                                      h0=h0, reset=reset, lib=lib, **kw)

    def piece(lo, hi, start):
        t = lambda a: a[:, :, lo:hi] if a.ndim == 3 and a.shape[2] == L else a
        return oracle.selective_scan_bwd(
            t(x["u"]), t(x["delta"]), x["A_log"], x["B"][:, lo:hi], x["C"][:, lo:hi],
            t(x["dout"]), D=kw["D"], z=t(kw["z"]), delta_bias=kw["delta_bias"], h0=start,
            lib=lib)

    first, second = piece(0, L1, h0), piece(L1, L, np.zeros_like(h0))
    for k in ("du", "ddelta", "dz"):
        _close(whole[k], np.concatenate([first[k], second[k]], axis=2), rtol=1e-12, what=k)
    for k in ("dB", "dC"):
        _close(whole[k], np.concatenate([first[k], second[k]], axis=1), rtol=1e-12, what=k)
    for k in ("dA_log", "dD", "ddelta_bias"):
        _close(whole[k], first[k] + second[k], rtol=1e-12, what=k)
    _close(whole["dh0"], first["dh0"], rtol=1e-12, what="dh0")


def check_backward_final_state_gradient(lib):
    """A loss on the final state as well as on y (its gradient given as
    dlast_state): every gradient, dh0 included, against central differences,
    from a random h0 and across document boundaries."""
    _fd_check(lib, softplus=True, with_opt=True, seed=18, ex=True, dlast=True)


def check_backward_chains_across_blocks(lib):
    """A sequence cut into two blocks, the second started from the first's
    final state (block-by-block processing of a long sequence), trained block
    by block -- the second block's dh0 passed as the first block's gradient on
    its final state -- gives the gradients of one backward over the whole
    sequence: per-step gradients concatenated, summed ones added, the same
    dh0.  A boundary inside each block and a loss on the final state too."""
    r = _rng(19)
    b, d, L, N, L1 = 2, 3, 11, 4, 5
    x = dict(u=r.normal(size=(b, d, L)), delta=r.normal(size=(b, d, L)),
             A_log=r.normal(size=(d, N)) * 0.5, B=r.normal(size=(b, L, N)),
             C=r.normal(size=(b, L, N)), dout=r.normal(size=(b, d, L)))
    kw = dict(D=r.normal(size=d), z=r.normal(size=(b, d, L)), delta_bias=r.normal(size=d))
    h0, w = r.normal(size=(b, d, N)), r.normal(size=(b, d, N))
    reset = np.zeros((b, L), dtype=np.uint8)
    reset[0, 7] = reset[1, 2] = 1
    whole = oracle.selective_scan_bwd(x["u"], x["delta"], x["A_log"], x["B"], x["C"], x["dout"],
                                      h0=h0, reset=reset, dlast_state=w, lib=lib, **kw)

    def cut(lo, hi):
        t = lambda a: a[:, :, lo:hi]
        return (t(x["u"]), t(x["delta"]), x["A_log"], x["B"][:, lo:hi], x["C"][:, lo:hi]), \
            dict(kw, z=t(kw["z"])), t(x["dout"]), reset[:, lo:hi]

    a1, k1, g1out, r1 = cut(0, L1)
    a2, k2, g2out, r2 = cut(L1, L)
    _, h_mid, _ = oracle.selective_scan(*a1, h0=h0, reset=r1, lib=lib, **k1)
    second = oracle.selective_scan_bwd(*a2, g2out, h0=h_mid, reset=r2, dlast_state=w, lib=lib,
                                       **k2)
    first = oracle.selective_scan_bwd(*a1, g1out, h0=h0, reset=r1,
                                      dlast_state=second["dh0"], lib=lib, **k1)
    for k in ("du", "ddelta", "dz"):
        _close(whole[k], np.concatenate([first[k], second[k]], axis=2), rtol=1e-12, what=k)
    for k in ("dB", "dC"):
        _close(whole[k], np.concatenate([first[k], second[k]], axis=1), rtol=1e-12, what=k)
    for k in ("dA_log", "dD", "ddelta_bias"):
        _close(whole[k], first[k] + second[k], rtol=1e-12, what=k)
    _close(whole["dh0"], first["dh0"], rtol=1e-12, what="dh0")


def check_backward_reset_at_start_cuts_h0(lib):
    """A reset at step 0 discards h0: its gradient is exactly zero and every
    other gradient equals that of the scan started from zero."""
    r = _rng(17)
    b, d, L, N = 2, 2, 9, 3
    a = [r.normal(size=(b, d, L)), r.normal(size=(b, d, L)), r.normal(size=(d, N)),
         r.normal(size=(b, L, N)), r.normal(size=(b, L, N)), r.normal(size=(b, d, L))]
    reset = np.zeros((b, L))
    reset[:, 0] = 1
    g = oracle.selective_scan_bwd(*a, h0=r.normal(size=(b, d, N)), reset=reset, lib=lib)
    g0 = oracle.selective_scan_bwd(*a, lib=lib)
    assert np.all(g["dh0"] == 0.0)
    for k in g0:
        _close(g[k], g0[k], rtol=1e-12, what=k)


ALL_CHECKS = [
    check_delta_zero_limit,
    check_single_step,
    check_geometric_series,
    check_steady_state,
    check_lti_convolution,
    check_bruteforce_unrolled,
    check_linearity_in_u,
    check_split_invariance,
    check_decode_chain,
    check_decode_single_step,
    check_permutations,
    check_optional_inputs,
    check_reset_splits_documents,
    check_reset_every_step_is_memoryless,
    check_reset_at_start_ignores_h0,
    check_backward_finite_differences,
    check_backward_finite_differences_plain,
    check_backward_finite_differences_h0_reset,
    check_backward_reset_splits_documents,
    check_backward_reset_at_start_cuts_h0,
    check_backward_final_state_gradient,
    check_backward_chains_across_blocks,
    check_conv_against_numpy_convolve,
    check_conv_impulse_response,
    check_conv_silu_closed_forms,
    check_conv_state_chaining,
    check_conv_initial_state_reaches_first_outputs_only,
    check_conv_channels_and_batches_are_independent,
    check_complex_with_real_parameters_is_the_real_scan,
    check_complex_impulse_response_closed_form,
    check_complex_geometric_series,
    check_complex_conjugation_symmetry,
    check_complex_bruteforce_unrolled,
]
