"""Shared pieces of the GPU-vs-oracle parity tests.

Error metric (one number per output tensor, y and last_state separately):

    err = max_i |gpu_i - ref_i| / max(|ref_i|, FLOOR * rms(ref)),  FLOOR = 0.1

Tolerances: 1e-4 for fp32 io, 2e-2 for bf16 io (the oracle is fed the same
bf16-rounded inputs; the GPU's bf16 output is compared unrounded against the
fp64 result).  The floor keeps the ratio meaningful where an output crosses
zero: an fp32 evaluation of the same recurrence in the same order, emulated
with numpy on 16 channels of the large-state case (L=8192, N=64), reaches
2.8e-4 with a 1e-3 floor but 1.0e-5 with the 0.1 floor, so 0.1 is the
smallest decade floor at which correct fp32 arithmetic sits 10x inside 1e-4.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from selective_state_space_140_b300 import abi, workloads

FLOOR = 0.1
TOL = {"f32": 1e-4, "bf16": 2e-2}

# The same metric at a floor of 1e-3 * rms bounds the error on small elements
# too.  Bounds from the arithmetic (fp32_emulation, checked in
# test_fp32_emulation.py): correct fp32 evaluation of the three scan workloads
# reaches 2.0e-4 .. 2.8e-4 there (up to 4.4e-4 over the four rounding patterns
# of fp32_envelope), hence 1e-3 for fp32 io; bf16 io adds the
# output's rounding (2^-8 relative) and the bf16 path's softplus error (at
# most 2e-5 relative in dt; taken in one direction at every step the
# emulation reaches 4.6e-2), hence 1e-1.
FINE_FLOOR = 1e-3
FINE_TOL = {"f32": 1e-3, "bf16": 1e-1}


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


def blockwise_rel_err(blocks, pair_fn, floors=(FLOOR, FINE_FLOOR), workers: int = 1):
    """``rel_err`` over outputs too large to hold whole in fp64.

    ``pair_fn(block)`` returns ``{name: (gpu, ref)}`` for one block of
    independent chains.  The rms that sets the floor is over all blocks, so the
    references are computed twice: a first pass sums their squares, a second
    takes the largest relative error.  Returns ``{name: [err per floor]}``.
    ``workers`` > 1 runs blocks on threads (the oracle's ctypes calls release
    the GIL)."""
    from concurrent.futures import ThreadPoolExecutor

    def sums(blk):
        return {k: (float(np.sum(np.square(np.asarray(r, np.float64)))), np.size(r))
                for k, (_, r) in pair_fn(blk).items()}

    ss, cnt = {}, {}
    with ThreadPoolExecutor(workers) as ex:
        for res in ex.map(sums, blocks):
            for k, (s, n) in res.items():
                ss[k] = ss.get(k, 0.0) + s
                cnt[k] = cnt.get(k, 0) + n
    rms = {k: (ss[k] / cnt[k]) ** 0.5 if cnt[k] else 0.0 for k in ss}

    def errs(blk):
        out = {}
        for k, (g, r) in pair_fn(blk).items():
            g = np.asarray(g, np.float64)
            r = np.asarray(r, np.float64)
            assert g.shape == r.shape and np.all(np.isfinite(g)), k
            e = []
            for fl in floors:
                den = np.maximum(np.abs(r), fl * rms[k])
                den = np.where(den > 0, den, 1.0)
                e.append(float(np.max(np.abs(g - r) / den)) if r.size else 0.0)
            out[k] = e
        return out

    worst = {}
    with ThreadPoolExecutor(workers) as ex:
        for res in ex.map(errs, blocks):
            for k, e in res.items():
                worst[k] = [max(a, b) for a, b in zip(worst.get(k, [0.0] * len(e)), e)]
    return worst


def channel_blocks(batch: int, dim: int, block: int):
    """(b, d0, d1) blocks covering every chain of a [batch, dim] grid."""
    return [(b, d0, min(dim, d0 + block)) for b in range(batch) for d0 in range(0, dim, block)]


def full_size_errors(x, y, h, h0=None, reset=None, block=None, emulate=False):
    """Every chain of a full-size launch against the oracle, channel block by
    channel block (the fp64 arrays of a whole workload would not fit at
    once); returns {"y": [err at FLOOR, err at FINE_FLOOR], "h": [...]}.
    With ``emulate`` the same for the four fp32 evaluations of the scan on
    the same blocks (fp32_envelope), under "y_emu0".."y_emu3" and
    "h_emu0".."h_emu3" (what correct fp32 arithmetic reaches on these inputs;
    computed once per block)."""
    batch, dim, L = x["u"].shape
    block = block or max(1, min(dim, (1 << 24) // max(L, 1)))
    ycpu, hcpu = y.cpu(), h.cpu()
    f = workloads.to_f64
    emu_cache = {}

    def pair(blk):
        b, d0, d1 = blk
        sl = lambda t: None if t is None else t[b:b + 1, d0:d1]
        sd = lambda t: None if t is None else t[d0:d1]
        yr, hr, _ = oracle.selective_scan(
            f(sl(x["u"])), f(sl(x["delta"])), f(x["A_log"][d0:d1]), f(x["B"][b:b + 1]),
            f(x["C"][b:b + 1]), D=f(sd(x["D"])), z=f(sl(x["z"])),
            delta_bias=f(sd(x["delta_bias"])), softplus=x["softplus"],
            h0=None if h0 is None else h0[b:b + 1, d0:d1].astype(np.float64),
            reset=None if reset is None else reset[b:b + 1])
        out = {"y": (ycpu[b:b + 1, d0:d1].double().numpy(), yr),
               "h": (hcpu[b:b + 1, d0:d1].double().numpy(), hr)}
        if emulate:
            from fp32_emulation import fp32_envelope
            if blk not in emu_cache:
                xs = {k: (sl(v) if k in ("u", "delta", "z") else
                          sd(v) if k in ("D", "delta_bias") else
                          v[d0:d1] if k == "A_log" else
                          v[b:b + 1] if k in ("B", "C") else v) for k, v in x.items()}
                emu_cache[blk] = fp32_envelope(xs, out_bf16=x["io_dtype"] == "bf16")
            for i, (ye, he) in enumerate(emu_cache[blk]):
                out[f"y_emu{i}"], out[f"h_emu{i}"] = (ye, yr), (he, hr)
        return out

    # the emulation's blocks run two at a time (numpy releases the GIL)
    return blockwise_rel_err(channel_blocks(batch, dim, block), pair,
                             workers=2 if emulate else 1)


def assert_full_size(io, errs, what):
    """The parity bound at the 0.1 * rms floor, and at the 1e-3 * rms floor
    FINE_TOL -- or, where the emulation was run, twice what correct fp32
    arithmetic reaches on the same inputs (the largest of its four
    evaluations) if that is more: FINE_TOL comes from
    channel subsets, and the largest relative error over a whole tensor grows
    with its element count."""
    for k in ("y", "h"):
        e, fe = errs[k]
        ftol = FINE_TOL[io]
        for i in range(4):
            if f"{k}_emu{i}" in errs:
                ftol = max(ftol, 2 * errs[f"{k}_emu{i}"][1])
        assert e <= TOL[io] and fe <= ftol, (
            f"{what} {k}: err {e:.3e} (tol {TOL[io]}), at the {FINE_FLOOR} floor {fe:.3e} "
            f"(tol {ftol:.3e})")
