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
"""
from __future__ import annotations

import numpy as np
import torch


def emulate_scan_f32(x: dict, dt_rel_err: float = 0.0, out_bf16: bool = False):
    """Return (y, last_state) as float64 arrays for the inputs ``x`` of
    ``workloads.make_scan_inputs`` (CPU tensors)."""
    f32 = np.float32
    u = x["u"].float().numpy()
    dl = x["delta"].float().numpy()
    z = None if x["z"] is None else x["z"].float().numpy()
    B = x["B"].float().numpy()
    C = x["C"].float().numpy()
    A = (-np.exp(x["A_log"].numpy().astype(np.float64))).astype(f32)
    batch, dim, L = u.shape
    N = A.shape[1]
    D = np.zeros(dim, f32) if x["D"] is None else x["D"].numpy().astype(f32)
    bias = np.zeros(dim, f32) if x["delta_bias"] is None else x["delta_bias"].numpy().astype(f32)
    scale = f32(1.0 + dt_rel_err)
    h = np.zeros((batch, dim, N), f32)
    y = np.zeros((batch, dim, L), f32)
    for t in range(L):
        raw = (dl[:, :, t] + bias[None, :]).astype(f32)
        if x["softplus"]:
            dt = np.where(raw > 20, raw, np.log1p(np.exp(np.minimum(raw, 20)))).astype(f32)
        else:
            dt = raw
        dt = (dt * scale).astype(f32)
        a = np.exp((dt[..., None] * A[None]).astype(f32)).astype(f32)
        du = (dt * u[:, :, t]).astype(f32)
        h = (a * h + (du[..., None] * B[:, None, t, :]).astype(f32)).astype(f32)
        acc = np.zeros((batch, dim), f32)
        for n in range(N):
            acc = (acc + (C[:, None, t, n] * h[..., n]).astype(f32)).astype(f32)
        v = (acc + (D[None, :] * u[:, :, t]).astype(f32)).astype(f32)
        if z is not None:
            zz = z[:, :, t]
            v = ((v * zz).astype(f32) / (f32(1) + np.exp(-zz)).astype(f32)).astype(f32)
        y[:, :, t] = v
    if out_bf16:
        y = torch.from_numpy(y).to(torch.bfloat16).float().numpy()
    return y.astype(np.float64), h.astype(np.float64)
