"""Shared pieces of the GPU-vs-oracle parity tests.

Error metric (one number per output tensor, y and last_state separately):

    err = max_i |gpu_i - ref_i| / max(|ref_i|, FLOOR * rms(ref)),  FLOOR = 0.1

Tolerances: 1e-4 for fp32 io, 2e-2 for bf16 io (the oracle is fed the same
bf16-rounded inputs; the GPU's bf16 output is compared unrounded against the
fp64 result).  The floor keeps the ratio meaningful where an output crosses
zero: an fp32 evaluation of the same recurrence in the same order, emulated
with numpy on 16 channels of the large-state case (L=8192, N=64), reaches
3.7e-4 with a 1e-3 floor but 1.0e-5 with the 0.1 floor, so 0.1 is the
smallest decade floor at which correct fp32 arithmetic sits 10x inside 1e-4.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from selective_state_space_140_b300 import abi, workloads

FLOOR = 0.1
TOL = {"f32": 1e-4, "bf16": 2e-2}


def rel_err(gpu, ref, floor: float = FLOOR) -> float:
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape
    if ref.size == 0:
        return 0.0
    assert np.all(np.isfinite(gpu)), "non-finite GPU output"
    rms = float(np.sqrt(np.mean(ref * ref)))
    den = np.maximum(np.abs(ref), floor * rms)
    den = np.where(den > 0, den, 1.0)
    return float(np.max(np.abs(gpu - ref) / den))


def normwise(gpu, ref) -> float:
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    nr = float(np.linalg.norm(ref))
    return float(np.linalg.norm(gpu - ref)) / nr if nr > 0 else float(np.linalg.norm(gpu))


def to_device(x: dict, device) -> dict:
    out = {}
    for k, v in x.items():
        out[k] = v.to(device) if isinstance(v, torch.Tensor) else v
    return out


def gpu_scan(xd: dict, **kw):
    """Run the CUDA scan on device tensors; return (y, last_state) device tensors."""
    return abi.mamba_selective_scan_fwd(xd["u"], xd["delta"], xd["A_log"], xd["B"], xd["C"],
                                        D=xd["D"], z=xd["z"], delta_bias=xd["delta_bias"],
                                        softplus=xd["softplus"], **kw)


def oracle_scan(x: dict, chains=None, nthreads: int = 0):
    """fp64 oracle on CPU inputs.  ``chains``: optional list of (b, d) to
    evaluate alone (for full-size configs); returns arrays [len, L] / [len, N]."""
    f = workloads.to_f64
    if chains is None:
        y, h, _ = oracle.selective_scan(f(x["u"]), f(x["delta"]), f(x["A_log"]), f(x["B"]),
                                        f(x["C"]), D=f(x["D"]), z=f(x["z"]),
                                        delta_bias=f(x["delta_bias"]), softplus=x["softplus"],
                                        nthreads=nthreads)
        return y, h
    ys, hs = [], []
    for b, d in chains:
        sl = lambda t: None if t is None else t[b:b + 1, d:d + 1]
        sd = lambda t: None if t is None else t[d:d + 1]
        y, h, _ = oracle.selective_scan(f(sl(x["u"])), f(sl(x["delta"])), f(x["A_log"][d:d + 1]),
                                        f(x["B"][b:b + 1]), f(x["C"][b:b + 1]), D=f(sd(x["D"])),
                                        z=f(sl(x["z"])), delta_bias=f(sd(x["delta_bias"])),
                                        softplus=x["softplus"], nthreads=1)
        ys.append(y[0, 0])
        hs.append(h[0, 0])
    return np.stack(ys), np.stack(hs)


def sample_chains(batch: int, dim: int, k: int, seed: int = 0):
    """k distinct (b, d) chains, always including the first and the last one."""
    r = np.random.default_rng(seed)
    picks = {(0, 0), (batch - 1, dim - 1)}
    while len(picks) < min(k, batch * dim):
        picks.add((int(r.integers(batch)), int(r.integers(dim))))
    return sorted(picks)
