"""Seeded synthetic inputs for the selective scan.

This module only draws random numbers and lays them out; it contains none of
the scan's arithmetic, so both the CUDA path and the fp64 oracle can be fed
from it.  Values follow the Mamba-shaped recipe:

* u, z, B, C, delta_raw ~ N(0, 1) (B and C are per (batch, time, state) and
  shared by every channel);
* per-channel step dt_d ~ log-uniform[1e-3, 1e-1], folded into the bias as
  bias_d = softplus^-1(dt_d) = dt_d + log(1 - exp(-dt_d)), with softplus on, so
  delta = softplus(delta_raw + bias_d) (the dt projection has a bias: codechina
  overview section 2.1, highthink.cn dt_proj with use_bias=True);
* A_log[d, n] = log(n + 1), the S4D-Real initialisation A = -(n + 1)
  (codechina overview section 4.1);
* D = 1 for the Mamba-shaped layers, N(0, 1) for the small and large-state
  cases.

Draws are made in fp32 with a CPU ``torch.Generator`` and then rounded once
(round-to-nearest-even) to the io dtype, so the oracle can be given exactly the
values the GPU reads.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class ScanConfig:
    name: str
    batch: int
    dim: int
    seqlen: int
    dstate: int
    io_dtype: str  # "f32" or "bf16"
    seed: int
    d_mode: str = "ones"  # "ones" or "normal"
    description: str = ""


@dataclasses.dataclass(frozen=True)
class DecodeConfig:
    name: str
    batch: int
    dim: int
    dstate: int
    io_dtype: str
    seed: int
    description: str = ""


SCAN_CONFIGS = {
    "tiny_f32": ScanConfig("tiny_f32", 1, 16, 64, 4, "f32", 0, "normal",
                           "tiny fp32 scan: batch 1, 16 channels, L=64, N=4"),
    "mamba130m_bf16": ScanConfig("mamba130m_bf16", 8, 1536, 2048, 16, "bf16", 1, "ones",
                                 "Mamba-130M-style layer: batch 8, d_inner 1536, L=2048, N=16, bf16"),
    "mamba1p4b_bf16": ScanConfig("mamba1p4b_bf16", 4, 4096, 4096, 16, "bf16", 2, "ones",
                                 "Mamba-1.4B-style layer: batch 4, d_inner 4096, L=4096, N=16, bf16"),
    "dna_long_bf16": ScanConfig("dna_long_bf16", 1, 1536, 131072, 16, "bf16", 3, "ones",
                                "long-sequence DNA-like scan: batch 1, d_inner 1536, L=131072, N=16, bf16"),
    "large_state_f32": ScanConfig("large_state_f32", 2, 2048, 8192, 64, "f32", 4, "normal",
                                  "large-state scan: batch 2, d_inner 2048, L=8192, N=64, fp32"),
}

DECODE_CONFIGS = {
    "decode_bf16": DecodeConfig("decode_bf16", 256, 4096, 16, "bf16", 5,
                                "single-token state update: batch 256, d_inner 4096, N=16, "
                                "bf16 x/dt/B/C/z, fp32 state ~ N(0,1)"),
}

TORCH_DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


def _dt_bias(gen: torch.Generator, dim: int, dt_min=1e-3, dt_max=1e-1) -> torch.Tensor:
    """bias_d = softplus^-1(dt_d), dt_d log-uniform in [dt_min, dt_max]."""
    r = torch.rand(dim, generator=gen, dtype=torch.float64)
    dt = torch.exp(r * (np.log(dt_max) - np.log(dt_min)) + np.log(dt_min))
    return (dt + torch.log(-torch.expm1(-dt))).to(torch.float32)


def make_scan_inputs(batch: int, dim: int, seqlen: int, dstate: int, io_dtype: str = "bf16",
                     seed: int = 0, d_mode: str = "ones", with_z: bool = True,
                     with_D: bool = True, with_bias: bool = True) -> dict:
    """Draw one set of scan inputs as CPU tensors.

    u, delta, z: [batch, dim, seqlen] io dtype; B, C: [batch, seqlen, dstate]
    io dtype; A_log: [dim, dstate] fp32; D, delta_bias: [dim] fp32.  Optional
    inputs that are switched off are returned as ``None``.
    """
    gen = torch.Generator().manual_seed(int(seed))
    tdt = TORCH_DTYPES[io_dtype]
    shape = (batch, dim, seqlen)
    u = torch.randn(shape, generator=gen, dtype=torch.float32).to(tdt)
    delta = torch.randn(shape, generator=gen, dtype=torch.float32).to(tdt)
    z = torch.randn(shape, generator=gen, dtype=torch.float32).to(tdt)
    B = torch.randn((batch, seqlen, dstate), generator=gen, dtype=torch.float32).to(tdt)
    C = torch.randn((batch, seqlen, dstate), generator=gen, dtype=torch.float32).to(tdt)
    bias = _dt_bias(gen, dim)
    if d_mode == "ones":
        D = torch.ones(dim, dtype=torch.float32)
    else:
        D = torch.randn(dim, generator=gen, dtype=torch.float32)
    A_log = torch.log(torch.arange(1, dstate + 1, dtype=torch.float32)).repeat(dim, 1).contiguous()
    return {
        "u": u, "delta": delta, "z": z if with_z else None, "B": B, "C": C,
        "A_log": A_log, "D": D if with_D else None,
        "delta_bias": bias if with_bias else None, "softplus": True,
        "io_dtype": io_dtype,
    }


def wide_a_log(dim: int, dstate: int, seed: int) -> torch.Tensor:
    """A_log [dim, dstate] fp32 with |A| = exp(A_log) log-uniform over [1e-2, 1e2]
    per (channel, state): the spread of a trained layer, whose slow states
    (|A| * dt far below 1/L) keep their whole history."""
    g = torch.Generator().manual_seed(int(seed))
    lo, hi = np.log(1e-2), np.log(1e2)
    return (torch.rand(dim, dstate, generator=g, dtype=torch.float64) * (hi - lo) + lo).float()


def make_config_inputs(cfg: ScanConfig) -> dict:
    return make_scan_inputs(cfg.batch, cfg.dim, cfg.seqlen, cfg.dstate, cfg.io_dtype, cfg.seed,
                            cfg.d_mode)


def make_decode_inputs(batch: int, dim: int, dstate: int, io_dtype: str = "bf16", seed: int = 5,
                       with_z: bool = True, with_D: bool = True, with_bias: bool = True) -> dict:
    """Draw one decode step: state [batch, dim, dstate] fp32 ~ N(0,1);
    x, dt, z [batch, dim] io dtype; B, C [batch, dstate] io dtype."""
    gen = torch.Generator().manual_seed(int(seed))
    tdt = TORCH_DTYPES[io_dtype]
    state = torch.randn((batch, dim, dstate), generator=gen, dtype=torch.float32)
    x = torch.randn((batch, dim), generator=gen, dtype=torch.float32).to(tdt)
    dt = torch.randn((batch, dim), generator=gen, dtype=torch.float32).to(tdt)
    z = torch.randn((batch, dim), generator=gen, dtype=torch.float32).to(tdt)
    B = torch.randn((batch, dstate), generator=gen, dtype=torch.float32).to(tdt)
    C = torch.randn((batch, dstate), generator=gen, dtype=torch.float32).to(tdt)
    bias = _dt_bias(gen, dim)
    D = torch.ones(dim, dtype=torch.float32)
    A_log = torch.log(torch.arange(1, dstate + 1, dtype=torch.float32)).repeat(dim, 1).contiguous()
    return {
        "state": state, "x": x, "dt": dt, "z": z if with_z else None, "B": B, "C": C,
        "A_log": A_log, "D": D if with_D else None, "dt_bias": bias if with_bias else None,
        "softplus": True, "io_dtype": io_dtype,
    }


def make_complex_inputs(batch: int, dim: int, seqlen: int, dstate: int, io_dtype: str = "bf16",
                        seed: int = 30, with_z: bool = True, with_D: bool = True,
                        with_bias: bool = True) -> dict:
    """Inputs of the complex-state scan as CPU tensors: u, delta, z [batch,
    dim, seqlen] ~ N(0, 1); B, C [batch, seqlen, dstate, 2] (re, im) ~ N(0, 1/2)
    each part (unit complex variance) in the io dtype; S4D-Lin A = -0.5 + i*n:
    A_log_re = log 0.5 and A_im = n; D ~ N(0, 1); the step bias as for the
    real scan (dt in [1e-3, 1e-1])."""
    gen = torch.Generator().manual_seed(int(seed))
    tdt = TORCH_DTYPES[io_dtype]
    shape = (batch, dim, seqlen)
    u = torch.randn(shape, generator=gen, dtype=torch.float32).to(tdt)
    delta = torch.randn(shape, generator=gen, dtype=torch.float32).to(tdt)
    z = torch.randn(shape, generator=gen, dtype=torch.float32).to(tdt)
    s = math.sqrt(0.5)
    B = (torch.randn((batch, seqlen, dstate, 2), generator=gen, dtype=torch.float32) * s).to(tdt)
    C = (torch.randn((batch, seqlen, dstate, 2), generator=gen, dtype=torch.float32) * s).to(tdt)
    bias = _dt_bias(gen, dim)
    D = torch.randn(dim, generator=gen, dtype=torch.float32)
    A_log_re = torch.full((dim, dstate), math.log(0.5), dtype=torch.float32)
    A_im = torch.arange(dstate, dtype=torch.float32).repeat(dim, 1).contiguous()
    return {"u": u, "delta": delta, "z": z if with_z else None, "B": B, "C": C,
            "A_log_re": A_log_re, "A_im": A_im, "D": D if with_D else None,
            "delta_bias": bias if with_bias else None, "softplus": True, "io_dtype": io_dtype}


def make_conv_inputs(batch: int, dim: int, seqlen: int, width: int = 4, io_dtype: str = "bf16",
                     seed: int = 20, with_bias: bool = True, with_state: bool = False) -> dict:
    """Draw inputs of the causal depthwise conv1d as CPU tensors: x [batch,
    dim, seqlen] ~ N(0, 1) in the io dtype; weight [dim, width] and bias [dim]
    fp32 ~ U(-1/sqrt(width), 1/sqrt(width)) (the default initialisation of a
    depthwise Conv1d, fan-in = width); initial_state [batch, dim, width-1]
    ~ N(0, 1) in the io dtype when ``with_state``."""
    gen = torch.Generator().manual_seed(int(seed))
    tdt = TORCH_DTYPES[io_dtype]
    bound = 1.0 / math.sqrt(width)
    x = torch.randn((batch, dim, seqlen), generator=gen, dtype=torch.float32).to(tdt)
    w = (torch.rand((dim, width), generator=gen, dtype=torch.float32) * 2 - 1) * bound
    bias = (torch.rand(dim, generator=gen, dtype=torch.float32) * 2 - 1) * bound
    st = torch.randn((batch, dim, width - 1), generator=gen, dtype=torch.float32).to(tdt)
    return {"x": x, "weight": w.contiguous(), "bias": bias if with_bias else None,
            "initial_state": st if with_state else None, "io_dtype": io_dtype}


def to_f64(t):
    """Widen a CPU tensor (bf16 / fp32) to a float64 numpy array, or pass None."""
    if t is None:
        return None
    return t.detach().to("cpu", torch.float64).numpy()
