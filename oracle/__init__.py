"""fp64 CPU oracle for the Mamba selective scan -- TEST INFRASTRUCTURE ONLY.

The arithmetic lives in ``scan_oracle.c`` (plain C, double precision, one
sequential loop per (batch, channel) chain).  This module only compiles that
file with gcc and marshals numpy arrays into it.

Who may use it: the tests, the smoke check in ``__graft_entry__`` and the CPU
baseline leg of ``bench.py``.  The CUDA library never imports, links or calls
anything here, and nothing here imports the CUDA package.

Every function takes float64 numpy arrays in the layouts documented in
``scan_oracle.c`` (u/delta/z/y: [batch, dim, seqlen]; B/C: [batch, seqlen,
dstate]; A_log: [dim, dstate]; D/delta_bias: [dim]; states: [batch, dim,
dstate]).  bf16 or fp32 inputs are widened to float64 by the caller, so the
oracle sees exactly the values the GPU sees.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "scan_oracle.c")
_LIB = os.path.join(_HERE, "liboracle_scan.so")
_lock = threading.Lock()
_lib = None

# No fast-math and no FMA contraction: every fp64 operation rounds as written.
GCC_FLAGS = ["-O2", "-fPIC", "-shared", "-std=c11", "-ffp-contract=off", "-fno-fast-math"]


def build(src: str = _SRC, out: str = _LIB, extra_flags=()) -> str:
    """Compile ``src`` into the shared library ``out`` with gcc; return ``out``."""
    cmd = ["gcc", *GCC_FLAGS, *extra_flags, "-o", out, src, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return out


def _declare(lib):
    dp = ctypes.POINTER(ctypes.c_double)
    i64 = ctypes.c_int64
    lib.oracle_selective_scan_f64.restype = ctypes.c_int
    lib.oracle_selective_scan_f64.argtypes = [dp, dp, dp, dp, dp, dp, dp, dp, ctypes.c_int,
                                              dp, ctypes.c_void_p, dp, dp, i64, i64, i64, i64,
                                              ctypes.c_int]
    lib.oracle_selective_state_update_f64.restype = ctypes.c_int
    lib.oracle_selective_state_update_f64.argtypes = [dp, dp, dp, dp, dp, dp, dp, dp, dp,
                                                      ctypes.c_int, dp, i64, i64, i64]
    lib.oracle_selective_scan_bwd_f64.restype = ctypes.c_int
    lib.oracle_selective_scan_bwd_f64.argtypes = [dp, dp, dp, dp, dp, dp, dp, dp, ctypes.c_int,
                                                  dp, dp, dp, dp, dp, dp, dp, dp, dp,
                                                  i64, i64, i64, i64]
    lib.oracle_selective_scan_bwd_ex_f64.restype = ctypes.c_int
    lib.oracle_selective_scan_bwd_ex_f64.argtypes = [dp, dp, dp, dp, dp, dp, dp, dp, ctypes.c_int,
                                                     dp, ctypes.c_void_p, dp, dp, dp, dp, dp, dp,
                                                     dp, dp, dp, dp, dp, i64, i64, i64, i64]
    lib.oracle_causal_conv1d_f64.restype = ctypes.c_int
    lib.oracle_causal_conv1d_f64.argtypes = [dp, dp, dp, dp, ctypes.c_int, dp, dp,
                                             i64, i64, i64, i64]
    lib.oracle_selective_scan_complex_f64.restype = ctypes.c_int
    lib.oracle_selective_scan_complex_f64.argtypes = [dp, dp, dp, dp, dp, dp, dp, dp, dp,
                                                      ctypes.c_int, dp, dp, i64, i64, i64, i64]
    lib.oracle_hw_threads.restype = ctypes.c_int
    lib.oracle_hw_threads.argtypes = []
    return lib


def load(path: str | None = None):
    """Load (building first if needed) the oracle library.

    ``path`` selects another build of the same source (the mutation tests use
    this to load deliberately broken copies); the default is the oracle itself.
    """
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            if (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
                build()
            _lib = _declare(ctypes.CDLL(_LIB))
    return _lib


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _f64(a):
    if a is None:
        return None
    return np.ascontiguousarray(a, dtype=np.float64)


def hw_threads(lib=None) -> int:
    return (lib or load()).oracle_hw_threads()


def selective_scan(u, delta, A_log, B, C, D=None, z=None, delta_bias=None, softplus=True,
                   h0=None, reset=None, nthreads: int = 0, lib=None):
    """Run the fp64 recurrence; return ``(y, last_state, threads_used)``.

    Shapes: u/delta/z [batch, dim, L]; B/C [batch, L, N]; A_log [dim, N];
    D/delta_bias [dim]; h0 (optional) [batch, dim, N]; reset (optional)
    [batch, L], non-zero where a new document starts (the state restarts
    from zero before that step).
    """
    lib = lib or load()
    u, delta, A_log, B, C = map(_f64, (u, delta, A_log, B, C))
    D, z, delta_bias, h0 = map(_f64, (D, z, delta_bias, h0))
    batch, dim, L = u.shape
    N = A_log.shape[1]
    assert delta.shape == u.shape and A_log.shape == (dim, N)
    assert B.shape == (batch, L, N) and C.shape == (batch, L, N)
    assert z is None or z.shape == u.shape
    assert D is None or D.shape == (dim,)
    assert delta_bias is None or delta_bias.shape == (dim,)
    assert h0 is None or h0.shape == (batch, dim, N)
    if reset is not None:
        reset = np.ascontiguousarray(np.asarray(reset) != 0, dtype=np.uint8)
        assert reset.shape == (batch, L)
    y = np.empty((batch, dim, L), dtype=np.float64)
    hL = np.empty((batch, dim, N), dtype=np.float64)
    used = lib.oracle_selective_scan_f64(
        _ptr(u), _ptr(delta), _ptr(A_log), _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(delta_bias),
        int(bool(softplus)), _ptr(h0), None if reset is None else reset.ctypes.data,
        _ptr(y), _ptr(hL), batch, dim, L, N, int(nthreads))
    if used < 0:
        raise ValueError(f"oracle_selective_scan_f64 rejected its arguments ({used})")
    return y, hL, used


def selective_scan_bwd(u, delta, A_log, B, C, dout, D=None, z=None, delta_bias=None,
                       softplus=True, h0=None, reset=None, dlast_state=None, lib=None):
    """Gradients of the scan for the output gradient ``dout`` [batch, dim, L].
    Returns a dict with du, ddelta, dA_log, dB, dC and, when the matching input
    is given, dD, dz, ddelta_bias and dh0 (float64 arrays in the layouts of the
    inputs).  ``h0`` [batch, dim, N] is the state before step 0 (zero if None);
    ``reset`` [batch, L] marks document starts as in :func:`selective_scan`;
    ``dlast_state`` [batch, dim, N] is the loss's gradient on the final state
    (none if None)."""
    lib = lib or load()
    u, delta, A_log, B, C, dout = map(_f64, (u, delta, A_log, B, C, dout))
    D, z, delta_bias, h0, dlast_state = map(_f64, (D, z, delta_bias, h0, dlast_state))
    batch, dim, L = u.shape
    N = A_log.shape[1]
    assert dout.shape == u.shape and B.shape == (batch, L, N) and C.shape == (batch, L, N)
    assert h0 is None or h0.shape == (batch, dim, N)
    assert dlast_state is None or dlast_state.shape == (batch, dim, N)
    if reset is not None:
        reset = np.ascontiguousarray(np.asarray(reset) != 0, dtype=np.uint8)
        assert reset.shape == (batch, L)
    g = {k: np.zeros((batch, dim, L)) for k in ("du", "ddelta", "dz")}
    g["dB"], g["dC"] = np.zeros((batch, L, N)), np.zeros((batch, L, N))
    g["dA_log"] = np.zeros((dim, N))
    g["dD"], g["ddelta_bias"] = np.zeros(dim), np.zeros(dim)
    g["dh0"] = np.zeros((batch, dim, N))
    if h0 is None and reset is None and dlast_state is None:
        rc = lib.oracle_selective_scan_bwd_f64(
            _ptr(u), _ptr(delta), _ptr(A_log), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
            _ptr(delta_bias), int(bool(softplus)), _ptr(dout), _ptr(g["du"]), _ptr(g["ddelta"]),
            _ptr(g["dA_log"]), _ptr(g["dB"]), _ptr(g["dC"]), _ptr(g["dD"]),
            _ptr(g["dz"] if z is not None else None), _ptr(g["ddelta_bias"]), batch, dim, L, N)
    else:
        rc = lib.oracle_selective_scan_bwd_ex_f64(
            _ptr(u), _ptr(delta), _ptr(A_log), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
            _ptr(delta_bias), int(bool(softplus)), _ptr(h0),
            None if reset is None else reset.ctypes.data, _ptr(dout), _ptr(dlast_state),
            _ptr(g["du"]),
            _ptr(g["ddelta"]), _ptr(g["dA_log"]), _ptr(g["dB"]), _ptr(g["dC"]), _ptr(g["dD"]),
            _ptr(g["dz"] if z is not None else None), _ptr(g["ddelta_bias"]), _ptr(g["dh0"]),
            batch, dim, L, N)
    if rc != 0:
        raise ValueError(f"oracle_selective_scan_bwd_f64 rejected its arguments ({rc})")
    if z is None:
        del g["dz"]
    if D is None:
        del g["dD"]
    if delta_bias is None:
        del g["ddelta_bias"]
    if h0 is None:
        del g["dh0"]
    return g


def selective_scan_complex(u, delta, A_log_re, A_im, B, C, D=None, z=None, delta_bias=None,
                           softplus=True, lib=None):
    """Complex-state scan: A = -exp(A_log_re) + i*A_im [dim, N]; B, C complex
    [batch, L, N] (numpy complex arrays, or real arrays [batch, L, N, 2] of
    (re, im) pairs).  Returns ``(y [batch, dim, L] real, last_state [batch,
    dim, N] complex)``."""
    lib = lib or load()

    def pairs(a):
        a = np.asarray(a)
        if np.iscomplexobj(a):
            a = np.stack([a.real, a.imag], axis=-1)
        return _f64(a)

    u, delta, A_log_re, A_im = map(_f64, (u, delta, A_log_re, A_im))
    B, C = pairs(B), pairs(C)
    D, z, delta_bias = map(_f64, (D, z, delta_bias))
    batch, dim, L = u.shape
    N = A_log_re.shape[1]
    assert A_im.shape == (dim, N) and B.shape == (batch, L, N, 2) and C.shape == B.shape
    y = np.empty((batch, dim, L), dtype=np.float64)
    hL = np.empty((batch, dim, N, 2), dtype=np.float64)
    rc = lib.oracle_selective_scan_complex_f64(
        _ptr(u), _ptr(delta), _ptr(A_log_re), _ptr(A_im), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
        _ptr(delta_bias), int(bool(softplus)), _ptr(y), _ptr(hL), batch, dim, L, N)
    if rc != 0:
        raise ValueError(f"oracle_selective_scan_complex_f64 rejected its arguments ({rc})")
    return y, hL[..., 0] + 1j * hL[..., 1]


def causal_conv1d(x, weight, bias=None, initial_state=None, silu=True, lib=None):
    """Causal depthwise conv1d (one filter per channel), then SiLU if ``silu``.

    x [batch, dim, L]; weight [dim, width]; bias [dim]; initial_state
    [batch, dim, width-1] (the inputs before step 0, oldest first; zeros if
    None).  Returns ``(out [batch, dim, L], final_state [batch, dim, width-1])``
    where final_state holds the last width-1 inputs."""
    lib = lib or load()
    x, weight, bias, initial_state = map(_f64, (x, weight, bias, initial_state))
    batch, dim, L = x.shape
    width = weight.shape[1]
    assert weight.shape == (dim, width) and width >= 1
    assert bias is None or bias.shape == (dim,)
    assert initial_state is None or initial_state.shape == (batch, dim, width - 1)
    out = np.empty((batch, dim, L), dtype=np.float64)
    fin = np.empty((batch, dim, width - 1), dtype=np.float64)
    rc = lib.oracle_causal_conv1d_f64(_ptr(x), _ptr(weight), _ptr(bias), _ptr(initial_state),
                                      int(bool(silu)), _ptr(out), _ptr(fin), batch, dim, L, width)
    if rc != 0:
        raise ValueError(f"oracle_causal_conv1d_f64 rejected its arguments ({rc})")
    return out, fin


def selective_state_update(state, x, dt, A_log, B, C, D=None, z=None, dt_bias=None,
                           softplus=True, lib=None):
    """One decode step.  Returns ``(out, new_state)``; the input is not modified.

    Shapes: state [batch, dim, N]; x/dt/z [batch, dim]; B/C [batch, N];
    A_log [dim, N]; D/dt_bias [dim].
    """
    lib = lib or load()
    st = np.array(state, dtype=np.float64, copy=True, order="C")
    x, dt, A_log, B, C = map(_f64, (x, dt, A_log, B, C))
    D, z, dt_bias = map(_f64, (D, z, dt_bias))
    batch, dim, N = st.shape
    assert x.shape == (batch, dim) and dt.shape == (batch, dim)
    assert B.shape == (batch, N) and C.shape == (batch, N) and A_log.shape == (dim, N)
    out = np.empty((batch, dim), dtype=np.float64)
    rc = lib.oracle_selective_state_update_f64(
        _ptr(st), _ptr(x), _ptr(dt), _ptr(A_log), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
        _ptr(dt_bias), int(bool(softplus)), _ptr(out), batch, dim, N)
    if rc != 0:
        raise ValueError(f"oracle_selective_state_update_f64 rejected its arguments ({rc})")
    return out, st
