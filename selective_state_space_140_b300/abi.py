"""Thin ctypes binding of libmamba_scan.so (declared in include/mamba_scan.h).

The functions here carry the C entry points' names and do argument
marshalling only: device pointers, sizes, the io dtype and the current CUDA
stream go straight into the C call, and a non-zero status raises
``MambaError``.  Every step of the scan runs in the library's CUDA kernels;
there is no fallback of any kind, and a missing library raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libmamba_scan.so")

MAMBA_F32, MAMBA_BF16 = 0, 1
STATUS = {0: "MAMBA_OK", 1: "MAMBA_ERR_NULL", 2: "MAMBA_ERR_SIZE", 3: "MAMBA_ERR_DSTATE",
          4: "MAMBA_ERR_ALIGN", 5: "MAMBA_ERR_DTYPE", 6: "MAMBA_ERR_LAUNCH",
          7: "MAMBA_ERR_TIMEOUT", 8: "MAMBA_ERR_ALIAS", 9: "MAMBA_ERR_SCRATCH"}
MAX_DSTATE = 256

# Every symbol include/mamba_scan.h declares.
EXPORTED = ("mamba_selective_scan_fwd", "mamba_selective_scan_fwd_noalloc",
            "mamba_selective_scan_fwd_ex", "mamba_selective_scan_bwd",
            "mamba_selective_scan_bwd_ex",
            "mamba_selective_scan_complex_fwd",
            "mamba_causal_conv1d_fwd", "mamba_causal_conv1d_update",
            "mamba_selective_state_update", "mamba_device_status", "mamba_status_string",
            "mamba_abi_version")

# Test-only symbols, declared in include/mamba_scan_testing.h.
TESTING_EXPORTED = ("mamba_test_bounded_wait",)

_lib = None


class MambaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


def _declare(lib):
    vp, fp, i64, ci = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    for name in ("mamba_selective_scan_fwd", "mamba_selective_scan_fwd_noalloc"):
        getattr(lib, name).restype = ci
        getattr(lib, name).argtypes = [vp, vp, fp, vp, vp, fp, vp, fp, ci, vp, fp,
                                       i64, i64, i64, i64, ci, vp]
    lib.mamba_selective_scan_fwd_ex.restype = ci
    lib.mamba_selective_scan_fwd_ex.argtypes = [vp, vp, fp, vp, vp, fp, vp, fp, ci, fp, vp, vp, fp,
                                                i64, i64, i64, i64, ci, vp]
    lib.mamba_selective_scan_bwd.restype = ci
    lib.mamba_selective_scan_bwd.argtypes = [vp, vp, fp, vp, vp, fp, vp, fp, ci, vp, vp, vp, vp,
                                             fp, fp, fp, fp, fp, i64, i64, i64, i64, ci, vp]
    lib.mamba_selective_scan_bwd_ex.restype = ci
    lib.mamba_selective_scan_bwd_ex.argtypes = [vp, vp, fp, vp, vp, fp, vp, fp, ci, fp, vp, vp, fp,
                                                vp, vp, vp, fp, fp, fp, fp, fp, fp, i64, i64, i64,
                                                i64, ci, vp]
    lib.mamba_selective_scan_complex_fwd.restype = ci
    lib.mamba_selective_scan_complex_fwd.argtypes = [vp, vp, fp, fp, vp, vp, fp, vp, fp, ci, vp,
                                                     fp, i64, i64, i64, i64, ci, vp]
    lib.mamba_causal_conv1d_fwd.restype = ci
    lib.mamba_causal_conv1d_fwd.argtypes = [vp, fp, fp, vp, ci, vp, vp, i64, i64, i64, i64, ci, vp]
    lib.mamba_causal_conv1d_update.restype = ci
    lib.mamba_causal_conv1d_update.argtypes = [vp, vp, fp, fp, ci, vp, i64, i64, i64, ci, vp]
    lib.mamba_selective_state_update.restype = ci
    lib.mamba_selective_state_update.argtypes = [fp, vp, vp, fp, vp, vp, fp, vp, fp, ci, vp,
                                                 i64, i64, i64, ci, vp]
    lib.mamba_status_string.restype = ctypes.c_char_p
    lib.mamba_status_string.argtypes = [ci]
    lib.mamba_abi_version.restype = ci
    lib.mamba_abi_version.argtypes = []
    lib.mamba_device_status.restype = ci
    lib.mamba_device_status.argtypes = [vp]
    lib.mamba_test_bounded_wait.restype = ci
    lib.mamba_test_bounded_wait.argtypes = [ci, vp]
    return lib


def load(path: str = LIB_PATH):
    """Load the CUDA library; raise if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with "
                               "`python -m selective_state_space_140_b300.build`")
        _lib = _declare(ctypes.CDLL(path))
    return _lib


def status_string(status: int) -> str:
    return load().mamba_status_string(int(status)).decode()


def abi_version() -> int:
    return load().mamba_abi_version()


def mamba_device_status(stream=None, device=None) -> int:
    """Synchronise the stream and return (and clear) the device-side status:
    0, or MAMBA_ERR_TIMEOUT (7) if an on-device bounded wait gave up."""
    dev = device or torch.device("cuda", torch.cuda.current_device())
    return load().mamba_device_status(_stream(stream, dev))


def mamba_test_bounded_wait(polls: int, stream=None, device=None) -> None:
    """Test hook (include/mamba_scan_testing.h): queue a wait that nothing
    completes, given up after ``polls`` polls; the next ``mamba_device_status``
    reports MAMBA_ERR_TIMEOUT."""
    dev = device or torch.device("cuda", torch.cuda.current_device())
    rc = load().mamba_test_bounded_wait(int(polls), _stream(stream, dev))
    if rc != 0:
        raise MambaError(rc, "mamba_test_bounded_wait")


def _io_dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return MAMBA_F32
    if t.dtype == torch.bfloat16:
        return MAMBA_BF16
    raise TypeError(f"io tensors must be float32 or bfloat16, got {t.dtype}")


def _ptr(t):
    return None if t is None else t.data_ptr()


def _check(t, name, device, dtype=None):
    if t is None:
        return
    if not t.is_cuda or t.device != device:
        raise ValueError(f"{name} must be on {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")


def _stream(stream, device):
    if stream is None:
        return torch.cuda.current_stream(device).cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def mamba_selective_scan_fwd(u, delta, A_log, B, C, D=None, z=None, delta_bias=None,
                             softplus=True, y=None, last_state=None, want_last_state=True,
                             stream=None):
    """Launch the fused forward scan; return ``(y, last_state)``.

    u, delta, z: [batch, dim, seqlen]; B, C: [batch, seqlen, dstate] (same io
    dtype, float32 or bfloat16); A_log [dim, dstate], D and delta_bias [dim] are
    float32.  ``y`` / ``last_state`` are allocated when not given
    (``last_state`` only if ``want_last_state``).  Runs on ``stream`` (default:
    the current stream) and does not synchronise.
    """
    return _scan_fwd("mamba_selective_scan_fwd", u, delta, A_log, B, C, D, z, delta_bias,
                     softplus, y, last_state, want_last_state, stream)


def mamba_selective_scan_fwd_noalloc(u, delta, A_log, B, C, D=None, z=None, delta_bias=None,
                                     softplus=True, y=None, last_state=None,
                                     want_last_state=True, stream=None):
    """``mamba_selective_scan_fwd`` through the C entry point that never
    allocates (a split keeps its carried states in the library's fixed 4 MiB
    device buffer; calls overlapping in time race on it).  ``y`` and
    ``last_state`` are allocated here by PyTorch when not given, so pass them
    in to keep the whole call free of allocation."""
    return _scan_fwd("mamba_selective_scan_fwd_noalloc", u, delta, A_log, B, C, D, z, delta_bias,
                     softplus, y, last_state, want_last_state, stream)


def mamba_selective_scan_fwd_ex(u, delta, A_log, B, C, D=None, z=None, delta_bias=None,
                                softplus=True, h0=None, reset=None, y=None, last_state=None,
                                want_last_state=True, stream=None):
    """``mamba_selective_scan_fwd`` from a starting state ``h0`` ([batch, dim,
    dstate] float32; may be the same tensor as ``last_state`` to continue a
    stream in place) with document boundaries ``reset`` ([batch, seqlen]
    uint8 or bool; non-zero at a token that starts a new document: the state
    restarts from zero before it).  Returns ``(y, last_state)``."""
    dev = u.device
    _check(h0, "h0", dev, torch.float32)
    if reset is not None:
        _check(reset, "reset", dev)
        if reset.dtype == torch.bool:
            reset = reset.view(torch.uint8)
        if reset.dtype != torch.uint8 or reset.shape != (u.shape[0], u.shape[2]):
            raise TypeError("reset must be uint8 or bool of shape [batch, seqlen]")
    return _scan_fwd("mamba_selective_scan_fwd_ex", u, delta, A_log, B, C, D, z, delta_bias,
                     softplus, y, last_state, want_last_state, stream, h0=h0, reset=reset)


def _scan_fwd(entry, u, delta, A_log, B, C, D, z, delta_bias, softplus, y, last_state,
              want_last_state, stream, h0=None, reset=None):
    dev = u.device
    batch, dim, seqlen = u.shape
    dstate = A_log.shape[-1]
    io = _io_dtype(u)
    for t, n in ((u, "u"), (delta, "delta"), (z, "z"), (B, "B"), (C, "C"), (y, "y")):
        _check(t, n, dev, u.dtype)
    for t, n in ((A_log, "A_log"), (D, "D"), (delta_bias, "delta_bias"),
                 (last_state, "last_state")):
        _check(t, n, dev, torch.float32)
    if y is None:
        y = torch.empty_like(u)
    if last_state is None and want_last_state:
        last_state = torch.empty((batch, dim, dstate), device=dev, dtype=torch.float32)
    ext = (_ptr(h0), _ptr(reset)) if entry.endswith("_ex") else ()
    rc = getattr(load(), entry)(
        _ptr(u), _ptr(delta), _ptr(A_log), _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(delta_bias),
        int(bool(softplus)), *ext, _ptr(y), _ptr(last_state), batch, dim, seqlen, dstate, io,
        _stream(stream, dev))
    if rc != 0:
        raise MambaError(rc, entry)
    return y, last_state


def mamba_selective_scan_bwd(u, delta, A_log, B, C, dout, D=None, z=None, delta_bias=None,
                             softplus=True, want_dD=True, want_ddelta_bias=True, grads=None,
                             stream=None, h0=None, reset=None, want_dh0=None,
                             dlast_state=None):
    """Gradients of ``mamba_selective_scan_fwd`` (zero initial state) for the
    output gradient ``dout``; returns a dict with ``du``, ``ddelta``,
    ``dA_log``, ``dB``, ``dC`` and, when wanted, ``dz`` (iff ``z`` is given),
    ``dD`` and ``ddelta_bias``.

    du/ddelta/dz have the io dtype of ``u``; dA_log [dim, dstate], dB/dC
    [batch, seqlen, dstate], dD/ddelta_bias [dim] are float32 (dB and dC sum
    over the channels).  ``grads`` may hold preallocated outputs by the same
    names.  Runs on ``stream`` and does not synchronise.

    ``h0`` [batch, dim, dstate] float32 (the state before step 0) and ``reset``
    [batch, seqlen] uint8 or bool (non-zero at a document start) select the
    backward of ``mamba_selective_scan_fwd_ex`` (C entry
    ``mamba_selective_scan_bwd_ex``); ``dh0``, the gradient of h0, is
    returned when h0 is given (or ``want_dh0``).  ``dlast_state`` [batch,
    dim, dstate] float32 is the loss's gradient on the final state (e.g. the
    ``dh0`` of the next block of the same sequence)."""
    dev = u.device
    batch, dim, seqlen = u.shape
    dstate = A_log.shape[-1]
    io = _io_dtype(u)
    for t, n in ((u, "u"), (delta, "delta"), (z, "z"), (B, "B"), (C, "C"), (dout, "dout")):
        _check(t, n, dev, u.dtype)
    for t, n in ((A_log, "A_log"), (D, "D"), (delta_bias, "delta_bias")):
        _check(t, n, dev, torch.float32)
    g = dict(grads or {})
    f32 = torch.float32
    shapes = {"du": (u.shape, u.dtype), "ddelta": (u.shape, u.dtype),
              "dA_log": ((dim, dstate), f32), "dB": ((batch, seqlen, dstate), f32),
              "dC": ((batch, seqlen, dstate), f32)}
    if z is not None:
        shapes["dz"] = (u.shape, u.dtype)
    if want_dD:
        shapes["dD"] = ((dim,), f32)
    if want_ddelta_bias:
        shapes["ddelta_bias"] = ((dim,), f32)
    for k, (shape, dtype) in shapes.items():
        if g.get(k) is None:
            g[k] = torch.empty(shape, device=dev, dtype=dtype)
        _check(g[k], k, dev, dtype)
        if tuple(g[k].shape) != tuple(shape):
            raise TypeError(f"{k} must have shape {tuple(shape)}")
    if want_dh0 is None:
        want_dh0 = h0 is not None
    _check(h0, "h0", dev, torch.float32)
    _check(dlast_state, "dlast_state", dev, torch.float32)
    if dlast_state is not None and tuple(dlast_state.shape) != (batch, dim, dstate):
        raise TypeError("dlast_state must have shape [batch, dim, dstate]")
    if reset is not None:
        _check(reset, "reset", dev)
        if reset.dtype == torch.bool:
            reset = reset.view(torch.uint8)
        if reset.dtype != torch.uint8 or reset.shape != (batch, seqlen):
            raise TypeError("reset must be uint8 or bool of shape [batch, seqlen]")
    if want_dh0:
        shapes["dh0"] = ((batch, dim, dstate), f32)
        if g.get("dh0") is None:
            g["dh0"] = torch.empty((batch, dim, dstate), device=dev, dtype=f32)
        _check(g["dh0"], "dh0", dev, f32)
    if h0 is None and reset is None and dlast_state is None and not want_dh0:
        rc = load().mamba_selective_scan_bwd(
            _ptr(u), _ptr(delta), _ptr(A_log), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
            _ptr(delta_bias), int(bool(softplus)), _ptr(dout), _ptr(g["du"]), _ptr(g["ddelta"]),
            _ptr(g.get("dz")), _ptr(g["dA_log"]), _ptr(g["dB"]), _ptr(g["dC"]), _ptr(g.get("dD")),
            _ptr(g.get("ddelta_bias")), batch, dim, seqlen, dstate, io, _stream(stream, dev))
        entry = "mamba_selective_scan_bwd"
    else:
        rc = load().mamba_selective_scan_bwd_ex(
            _ptr(u), _ptr(delta), _ptr(A_log), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
            _ptr(delta_bias), int(bool(softplus)), _ptr(h0), _ptr(reset), _ptr(dout),
            _ptr(dlast_state), _ptr(g["du"]), _ptr(g["ddelta"]), _ptr(g.get("dz")),
            _ptr(g["dA_log"]), _ptr(g["dB"]),
            _ptr(g["dC"]), _ptr(g.get("dD")), _ptr(g.get("ddelta_bias")), _ptr(g.get("dh0")),
            batch, dim, seqlen, dstate, io, _stream(stream, dev))
        entry = "mamba_selective_scan_bwd_ex"
    if rc != 0:
        raise MambaError(rc, entry)
    return {k: g[k] for k in shapes}


def mamba_selective_scan_complex_fwd(u, delta, A_log_re, A_im, B, C, D=None, z=None,
                                     delta_bias=None, softplus=True, y=None, last_state=None,
                                     want_last_state=True, stream=None):
    """Complex-state scan.  B, C: [batch, seqlen, dstate, 2] (re, im) pairs in
    the io dtype of ``u``; A_log_re, A_im [dim, dstate] float32.  Returns
    ``(y, last_state)`` with last_state [batch, dim, dstate, 2] float32."""
    dev = u.device
    batch, dim, seqlen = u.shape
    dstate = A_log_re.shape[-1]
    io = _io_dtype(u)
    for t, n in ((u, "u"), (delta, "delta"), (z, "z"), (B, "B"), (C, "C"), (y, "y")):
        _check(t, n, dev, u.dtype)
    for t, n in ((A_log_re, "A_log_re"), (A_im, "A_im"), (D, "D"), (delta_bias, "delta_bias"),
                 (last_state, "last_state")):
        _check(t, n, dev, torch.float32)
    if B.shape != (batch, seqlen, dstate, 2) or C.shape != B.shape:
        raise TypeError("B and C must be [batch, seqlen, dstate, 2]")
    if y is None:
        y = torch.empty_like(u)
    if last_state is None and want_last_state:
        last_state = torch.empty((batch, dim, dstate, 2), device=dev, dtype=torch.float32)
    rc = load().mamba_selective_scan_complex_fwd(
        _ptr(u), _ptr(delta), _ptr(A_log_re), _ptr(A_im), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
        _ptr(delta_bias), int(bool(softplus)), _ptr(y), _ptr(last_state), batch, dim, seqlen,
        dstate, io, _stream(stream, dev))
    if rc != 0:
        raise MambaError(rc, "mamba_selective_scan_complex_fwd")
    return y, last_state


def mamba_causal_conv1d_fwd(x, weight, bias=None, initial_state=None, silu=True, out=None,
                            final_state=None, want_final_state=False, stream=None):
    """Causal depthwise conv1d (+ SiLU) of ``x`` [batch, dim, L] with
    ``weight`` [dim, width] (float32) and ``bias`` [dim]; ``initial_state`` /
    ``final_state`` [batch, dim, width-1] hold the last width-1 inputs before /
    after the block (io dtype).  Returns ``(out, final_state)``."""
    dev = x.device
    batch, dim, L = x.shape
    width = weight.shape[-1]
    io = _io_dtype(x)
    for t, n in ((x, "x"), (initial_state, "initial_state"), (out, "out"),
                 (final_state, "final_state")):
        _check(t, n, dev, x.dtype)
    for t, n in ((weight, "weight"), (bias, "bias")):
        _check(t, n, dev, torch.float32)
    if out is None:
        out = torch.empty_like(x)
    if final_state is None and want_final_state:
        final_state = torch.empty((batch, dim, width - 1), device=dev, dtype=x.dtype)
    rc = load().mamba_causal_conv1d_fwd(_ptr(x), _ptr(weight), _ptr(bias), _ptr(initial_state),
                                        int(bool(silu)), _ptr(out), _ptr(final_state), batch, dim,
                                        L, width, io, _stream(stream, dev))
    if rc != 0:
        raise MambaError(rc, "mamba_causal_conv1d_fwd")
    return out, final_state


def mamba_causal_conv1d_update(conv_state, x, weight, bias=None, silu=True, out=None,
                               stream=None):
    """One decode token per row: ``x`` [batch, dim]; ``conv_state`` [batch, dim,
    width-1] (io dtype) is shifted in place.  Returns ``out`` [batch, dim]."""
    dev = x.device
    batch, dim = x.shape
    width = weight.shape[-1]
    io = _io_dtype(x)
    for t, n in ((x, "x"), (conv_state, "conv_state"), (out, "out")):
        _check(t, n, dev, x.dtype)
    for t, n in ((weight, "weight"), (bias, "bias")):
        _check(t, n, dev, torch.float32)
    if out is None:
        out = torch.empty_like(x)
    rc = load().mamba_causal_conv1d_update(_ptr(conv_state), _ptr(x), _ptr(weight), _ptr(bias),
                                           int(bool(silu)), _ptr(out), batch, dim, width, io,
                                           _stream(stream, dev))
    if rc != 0:
        raise MambaError(rc, "mamba_causal_conv1d_update")
    return out


def mamba_selective_state_update(state, x, dt, A_log, B, C, D=None, z=None, dt_bias=None,
                                 softplus=True, out=None, stream=None):
    """One decode step; ``state`` [batch, dim, dstate] fp32 is updated in place.

    x, dt, z: [batch, dim]; B, C: [batch, dstate] (float32 or bfloat16).
    Returns ``out`` [batch, dim].
    """
    dev = state.device
    batch, dim, dstate = state.shape
    io = _io_dtype(x)
    _check(state, "state", dev, torch.float32)
    for t, n in ((x, "x"), (dt, "dt"), (z, "z"), (B, "B"), (C, "C"), (out, "out")):
        _check(t, n, dev, x.dtype)
    for t, n in ((A_log, "A_log"), (D, "D"), (dt_bias, "dt_bias")):
        _check(t, n, dev, torch.float32)
    if out is None:
        out = torch.empty_like(x)
    rc = load().mamba_selective_state_update(
        _ptr(state), _ptr(x), _ptr(dt), _ptr(A_log), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
        _ptr(dt_bias), int(bool(softplus)), _ptr(out), batch, dim, dstate, io,
        _stream(stream, dev))
    if rc != 0:
        raise MambaError(rc, "mamba_selective_state_update")
    return out


def raw_scan_fwd(u, delta, A_log, B, C, D, z, delta_bias, softplus_flag, y, last_state,
                 batch, dim, seqlen, dstate, io_dtype, stream) -> int:
    """The C entry point with plain integers as pointers; returns the status code.

    Lets tests exercise the C validation (NULL pointers, bad sizes, misaligned
    addresses) without building tensors.  No pointer is dereferenced on the
    host; argument errors return before any CUDA call.
    """
    return load().mamba_selective_scan_fwd(u, delta, A_log, B, C, D, z, delta_bias,
                                           softplus_flag, y, last_state, batch, dim, seqlen,
                                           dstate, io_dtype, stream)


def raw_scan_fwd_noalloc(u, delta, A_log, B, C, D, z, delta_bias, softplus_flag, y, last_state,
                         batch, dim, seqlen, dstate, io_dtype, stream) -> int:
    """``mamba_selective_scan_fwd_noalloc`` with plain integers as pointers."""
    return load().mamba_selective_scan_fwd_noalloc(u, delta, A_log, B, C, D, z, delta_bias,
                                                   softplus_flag, y, last_state, batch, dim,
                                                   seqlen, dstate, io_dtype, stream)


def raw_scan_fwd_ex(u, delta, A_log, B, C, D, z, delta_bias, softplus_flag, h0, reset, y,
                    last_state, batch, dim, seqlen, dstate, io_dtype, stream) -> int:
    """``mamba_selective_scan_fwd_ex`` with plain integers as pointers."""
    return load().mamba_selective_scan_fwd_ex(u, delta, A_log, B, C, D, z, delta_bias,
                                              softplus_flag, h0, reset, y, last_state, batch, dim,
                                              seqlen, dstate, io_dtype, stream)


def raw_state_update(state, x, dt, A_log, B, C, D, z, dt_bias, softplus_flag, out, batch, dim,
                     dstate, io_dtype, stream) -> int:
    """``mamba_selective_state_update`` with plain integers as pointers."""
    return load().mamba_selective_state_update(state, x, dt, A_log, B, C, D, z, dt_bias,
                                               softplus_flag, out, batch, dim, dstate, io_dtype,
                                               stream)


def raw_scan_bwd(u, delta, A_log, B, C, D, z, delta_bias, softplus_flag, dout, du, ddelta, dz,
                 dA_log, dB, dC, dD, ddelta_bias, batch, dim, seqlen, dstate, io_dtype,
                 stream) -> int:
    """``mamba_selective_scan_bwd`` with plain integers as pointers."""
    return load().mamba_selective_scan_bwd(u, delta, A_log, B, C, D, z, delta_bias,
                                           softplus_flag, dout, du, ddelta, dz, dA_log, dB, dC,
                                           dD, ddelta_bias, batch, dim, seqlen, dstate, io_dtype,
                                           stream)


def raw_conv1d_fwd(x, weight, bias, initial_state, silu_flag, out, final_state, batch, dim,
                   seqlen, width, io_dtype, stream) -> int:
    """``mamba_causal_conv1d_fwd`` with plain integers as pointers."""
    return load().mamba_causal_conv1d_fwd(x, weight, bias, initial_state, silu_flag, out,
                                          final_state, batch, dim, seqlen, width, io_dtype, stream)


def raw_conv1d_update(conv_state, x, weight, bias, silu_flag, out, batch, dim, width, io_dtype,
                      stream) -> int:
    """``mamba_causal_conv1d_update`` with plain integers as pointers."""
    return load().mamba_causal_conv1d_update(conv_state, x, weight, bias, silu_flag, out, batch,
                                             dim, width, io_dtype, stream)


def raw_scan_complex_fwd(u, delta, A_log_re, A_im, B, C, D, z, delta_bias, softplus_flag, y,
                         last_state, batch, dim, seqlen, dstate, io_dtype, stream) -> int:
    """``mamba_selective_scan_complex_fwd`` with plain integers as pointers."""
    return load().mamba_selective_scan_complex_fwd(u, delta, A_log_re, A_im, B, C, D, z,
                                                   delta_bias, softplus_flag, y, last_state, batch,
                                                   dim, seqlen, dstate, io_dtype, stream)


def raw_scan_bwd_ex(u, delta, A_log, B, C, D, z, delta_bias, softplus_flag, h0, reset, dout, du,
                    ddelta, dz, dA_log, dB, dC, dD, ddelta_bias, dh0, batch, dim, seqlen, dstate,
                    io_dtype, stream, dlast_state=None) -> int:
    """``mamba_selective_scan_bwd_ex`` with plain integers as pointers."""
    return load().mamba_selective_scan_bwd_ex(u, delta, A_log, B, C, D, z, delta_bias,
                                              softplus_flag, h0, reset, dout, dlast_state, du,
                                              ddelta, dz, dA_log, dB, dC, dD, ddelta_bias, dh0,
                                              batch, dim, seqlen, dstate, io_dtype, stream)
