"""Where the parity bounds come from (CPU only).

The fp32 emulation (``fp32_emulation.py``) evaluates the scan with correctly
rounded fp32 operations; its distance to the fp64 oracle is what correct
fp32 arithmetic reaches.  These checks pin the bounds the GPU tests use to
that arithmetic, on channel subsets of the workloads (same shapes per chain,
same value distributions and seeds):

* at the 0.1 * rms floor correct fp32 sits at least 5x inside the fp32 bound
  (1e-4) on the S4D-Real workloads;
* at the 1e-3 * rms floor it reaches at most half of FINE_TOL["f32"];
* bf16 output rounding plus the bf16 path's softplus error bound (2e-5
  relative in dt, in one direction at every step) stays inside the bf16
  bound (2e-2) and half of FINE_TOL["bf16"];
* with |A| spread over [1e-2, 1e2] (trained layers drift to small |A|) the
  states' memory exceeds the sequence: fp32 arithmetic whose exponentials
  are a few ulp off (numpy's float32 ones, as a GPU's are) exceeds 1e-4 at
  L = 4096, and with correctly rounded exponentials it lands within 2x of
  it, so a fixed fp32 bound cannot hold there, which is why that GPU test
  bounds the kernel by the emulation's own error;
* the S4D-Real bounds hold for the state update rounded per operation and
  fused, and the four evaluations of the envelope all round differently, so
  the envelope the GPU tests take over them is not one pattern counted
  several times.
"""
import numpy as np
import pytest
import torch

import oracle
from fp32_emulation import emulate_scan_f32, fp32_envelope
from parity_util import FINE_FLOOR, FINE_TOL, TOL, rel_err
from selective_state_space_140_b300 import workloads


def _oracle(x):
    f = workloads.to_f64
    y, h, _ = oracle.selective_scan(f(x["u"]), f(x["delta"]), f(x["A_log"]), f(x["B"]),
                                    f(x["C"]), D=f(x["D"]), z=f(x["z"]),
                                    delta_bias=f(x["delta_bias"]), softplus=x["softplus"])
    return y, h


def _errs(got, want):
    return [rel_err(g, w) for g, w in zip(got, want)], \
        [rel_err(g, w, FINE_FLOOR) for g, w in zip(got, want)]


CASES = [("large_state_f32", 16, 8192), ("mamba1p4b_bf16", 64, 4096), ("dna_long_bf16", 8, 8192)]


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("name,dim,L", CASES)
def test_correct_fp32_sits_inside_the_fp32_bounds(name, dim, L, fused):
    cfg = workloads.SCAN_CONFIGS[name]
    x = workloads.make_scan_inputs(min(cfg.batch, 2), dim, L, cfg.dstate, cfg.io_dtype,
                                   seed=cfg.seed, d_mode=cfg.d_mode)
    coarse, fine = _errs(emulate_scan_f32(x, fused_state=fused), _oracle(x))
    assert max(coarse) <= TOL["f32"] / 5, coarse
    assert max(fine) <= FINE_TOL["f32"] / 2, fine


@pytest.mark.parametrize("name,dim,L", CASES)
def test_bf16_rounding_and_softplus_error_sit_inside_the_bf16_bounds(name, dim, L):
    cfg = workloads.SCAN_CONFIGS[name]
    x = workloads.make_scan_inputs(min(cfg.batch, 2), dim, L, cfg.dstate, "bf16",
                                   seed=cfg.seed, d_mode=cfg.d_mode)
    coarse, fine = _errs(emulate_scan_f32(x, dt_rel_err=2e-5, out_bf16=True), _oracle(x))
    assert max(coarse) <= TOL["bf16"], coarse
    assert max(fine) <= FINE_TOL["bf16"] / 2, fine


def test_long_memory_states_exceed_a_fixed_fp32_bound():
    x = workloads.make_scan_inputs(2, 32, 4096, 16, "f32", seed=77, d_mode="normal")
    x["A_log"] = workloads.wide_a_log(32, 16, 77)
    want = _oracle(x)
    env = fp32_envelope(x)
    coarse = [max(_errs(got, want)[0]) for got in env]
    # exponentials correctly rounded (0, 1) or numpy float32 (2, 3)
    assert min(coarse[2:]) > TOL["f32"], coarse
    assert min(coarse[:2]) > TOL["f32"] / 2, coarse
    # the evaluations round differently (four samples, not one)
    for i in range(4):
        for j in range(i):
            assert not np.array_equal(env[i][1], env[j][1])
            assert not np.array_equal(env[i][0], env[j][0])
