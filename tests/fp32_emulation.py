"""fp32 evaluation of the selective scan in numpy -- test infrastructure only.

This is not the oracle (the oracle is fp64, ``oracle/``) and not the kernel:
it is the scan evaluated step by step with correctly rounded fp32 numpy
operations (exp, log1p, products and sums each rounded to fp32), in the order
the recurrence is written.  Its distance to the fp64 oracle is what correct
fp32 arithmetic reaches on a given input, so the parity tests use it to
derive bounds from the arithmetic where a fixed bound cannot hold for any
fp32 evaluation (e.g. states whose memory exceeds the sequence, where the
state is a long running sum that rounds at every step).

``dt_rel_err`` scales every step size by (1 + dt_rel_err): the worst case of
a step computed with that relative error in one direction.  ``out_bf16``
rounds y to bf16 (nearest even) as the bf16-io kernels store it.
Elementary functions (exp, log1p) are evaluated in fp64 and rounded to fp32,
i.e. correctly rounded up to a rare double rounding.

``fp32_envelope`` runs four evaluations of the same recurrence that differ
only in rounding: the state update Abar * h + dt * u * B rounded after the
product and again after the sum, or once (a fused multiply-add: the product
of two fp32 numbers is exact in fp64, and the fp64 sum is rounded to fp32);
and the elementary functions correctly rounded, or numpy's float32 versions
(within 2-3 ulp, as GPU elementary functions are).  On inputs whose outputs
cancel (a few slow states holding values 100x the output), the largest
relative error on small elements is one element's rounding noise, and these
equally correct evaluations spread over a factor of 2-3 either way on it, so
a bound taken from the arithmetic uses the largest of them.
"""
from __future__ import annotations

import numpy as np
import torch


def _emulate(x: dict, dt_rel_err: float, out_bf16: bool, variants):
    """The scan in fp32 for each (fused_state, rounded_math) in ``variants``,
    all carried through time together as one stacked array."""
    f32, f64 = np.float32, np.float64
    u = x["u"].float().numpy()
    dl = x["delta"].float().numpy()
    z = None if x["z"] is None else x["z"].float().numpy()
    B = x["B"].float().numpy()
    C = x["C"].float().numpy()
    A = (-np.exp(x["A_log"].numpy().astype(f64))).astype(f32)
    batch, dim, L = u.shape
    N = A.shape[1]
    V = len(variants)
    D = np.zeros(dim, f32) if x["D"] is None else x["D"].numpy().astype(f32)
    bias = np.zeros(dim, f32) if x["delta_bias"] is None else x["delta_bias"].numpy().astype(f32)
    scale = f32(1.0 + dt_rel_err)
    fused = np.array([fs for fs, _ in variants])[:, None, None, None]
    rounded = [rm for _, rm in variants]

    def fn(f, arg, rm):  # an elementary function in fp32
        return f(arg.astype(f64)).astype(f32) if rm else f(arg).astype(f32)

    def per_variant(f, arg):  # [V, ...] from one fp32 argument
        out = {rm: fn(f, arg, rm) for rm in set(rounded)}
        return np.stack([out[rm] for rm in rounded])

    h = np.zeros((V, batch, dim, N), f32)
    y = np.zeros((V, batch, dim, L), f32)
    for t in range(L):
        raw = (dl[:, :, t] + bias[None, :]).astype(f32)
        if x["softplus"]:
            e = per_variant(np.exp, np.minimum(raw, f32(20)))
            sp = np.stack([fn(np.log1p, e[v], rounded[v]) for v in range(V)])
            dt = np.where(raw[None] > 20, raw[None], sp).astype(f32)
        else:
            dt = np.broadcast_to(raw[None], (V,) + raw.shape)
        dt = (dt * scale).astype(f32)
        arg = (dt[..., None] * A[None, None]).astype(f32)
        a = np.stack([fn(np.exp, arg[v], rounded[v]) for v in range(V)])
        du = (dt * u[None, :, :, t]).astype(f32)
        bu = (du[..., None] * B[None, :, None, t, :]).astype(f32)
        h = np.where(fused, (a.astype(f64) * h + bu).astype(f32),
                     ((a * h).astype(f32) + bu).astype(f32))
        acc = np.zeros((V, batch, dim), f32)
        for n in range(N):
            acc = (acc + (C[None, :, None, t, n] * h[..., n]).astype(f32)).astype(f32)
        v = (acc + (D[None, None, :] * u[None, :, :, t]).astype(f32)).astype(f32)
        if z is not None:
            zz = z[:, :, t]
            den = (f32(1) + per_variant(np.exp, -zz)).astype(f32)
            v = ((v * zz[None]).astype(f32) / den).astype(f32)
        y[:, :, :, t] = v
    if out_bf16:
        y = torch.from_numpy(y).to(torch.bfloat16).float().numpy()
    return [(y[i].astype(f64), h[i].astype(f64)) for i in range(V)]


def emulate_scan_f32(x: dict, dt_rel_err: float = 0.0, out_bf16: bool = False,
                     fused_state: bool = False):
    """Return (y, last_state) as float64 arrays for the inputs ``x`` of
    ``workloads.make_scan_inputs`` (CPU tensors): the state update rounded per
    operation (or fused), elementary functions correctly rounded."""
    return _emulate(x, dt_rel_err, out_bf16, [(fused_state, True)])[0]


def fp32_envelope(x: dict, out_bf16: bool = False):
    """The four fp32 evaluations (state update per operation or fused;
    elementary functions correctly rounded or numpy float32), as a list of
    (y, last_state)."""
    return _emulate(x, 0.0, out_bf16, [(False, True), (True, True), (False, False), (True, False)])
