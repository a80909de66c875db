"""GPU complex-state (S4D-Lin) scan vs the fp64 oracle, through the C ABI.

Error metric and tolerances as for the real scan (``parity_util``: 1e-4 for
fp32 io, 2e-2 for bf16 io); the state is compared as (re, im) pairs with the
same metric.  The angle dt * Im A reaches hundreds of radians for large steps
and fast rotations, so an angle formed in fp32 would carry an absolute error
of |dt * Im A| * 2^-24 per step (and the step dt's own rounding on top); the
fp32-io kernel therefore forms dt and the angle in fp64 and the plain 1e-4
bound applies to every case here, large angles included.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from parity_util import TOL, blockwise_rel_err, channel_blocks, rel_err, to_device
from selective_state_space_140_b300 import abi, workloads

pytestmark = pytest.mark.gpu


def _gpu(x, device, **kw):
    xd = to_device(x, device)
    y, h = abi.mamba_selective_scan_complex_fwd(xd["u"], xd["delta"], xd["A_log_re"], xd["A_im"],
                                                xd["B"], xd["C"], D=xd["D"], z=xd["z"],
                                                delta_bias=xd["delta_bias"],
                                                softplus=xd["softplus"], **kw)
    torch.cuda.synchronize()
    return y.float().cpu().numpy(), h.cpu().numpy()


def _ref(x):
    f = workloads.to_f64
    y, h = oracle.selective_scan_complex(f(x["u"]), f(x["delta"]), f(x["A_log_re"]),
                                         f(x["A_im"]), f(x["B"]), f(x["C"]), D=f(x["D"]),
                                         z=f(x["z"]), delta_bias=f(x["delta_bias"]),
                                         softplus=x["softplus"])
    return y, np.stack([h.real, h.imag], axis=-1)


def _theta_max(x):
    f = workloads.to_f64
    raw = f(x["delta"]) + (0.0 if x["delta_bias"] is None else f(x["delta_bias"])[None, :, None])
    dt = np.logaddexp(0.0, raw) if x["softplus"] else raw
    if dt.size == 0:
        return 0.0
    return float(np.max(np.abs(dt).max(axis=(0, 2)) * np.abs(f(x["A_im"])).max(axis=1)))


def _check(x, got, want, what):
    tol = TOL[x["io_dtype"]]
    ey, eh = rel_err(got[0], want[0]), rel_err(got[1], want[1])
    assert ey <= tol and eh <= tol, f"{what}: y err {ey:.2e}, state err {eh:.2e}, tol {tol}"


SHAPES = [
    (1, 1, 1, 16, "f32"), (1, 3, 15, 4, "f32"), (2, 7, 17, 16, "bf16"), (1, 33, 33, 16, "f32"),
    (2, 37, 100, 16, "bf16"), (1, 9, 63, 1, "f32"), (1, 6, 65, 3, "f32"), (2, 10, 70, 8, "f32"),
    (1, 5, 70, 17, "f32"), (1, 6, 50, 32, "bf16"), (1, 6, 50, 64, "f32"), (1, 4, 40, 100, "f32"),
    (1, 3, 30, 256, "f32"), (1, 130, 40, 8, "bf16"), (2, 70, 1000, 16, "f32"),
    (2, 70, 1000, 16, "bf16"), (1, 16, 2049, 16, "f32"),
    # bf16 (packed pairs of states) at every tile width, with padded lanes
    (1, 9, 63, 3, "bf16"), (1, 5, 70, 17, "bf16"), (1, 6, 50, 64, "bf16"),
    (1, 4, 40, 100, "bf16"), (1, 3, 30, 256, "bf16"),
]


@pytest.mark.parametrize("batch,dim,L,N,io", SHAPES, ids=lambda v: str(v))
def test_shapes_match_oracle(cuda, batch, dim, L, N, io):
    x = workloads.make_complex_inputs(batch, dim, L, N, io, seed=batch + dim + L + N)
    _check(x, _gpu(x, cuda), _ref(x), str((batch, dim, L, N, io)))


@pytest.mark.parametrize("with_z,with_D,with_bias", [(False, True, True), (True, False, True),
                                                      (True, True, False), (False, False, False)])
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_optional_inputs(cuda, with_z, with_D, with_bias, io):
    x = workloads.make_complex_inputs(2, 21, 150, 16, io, seed=31, with_z=with_z, with_D=with_D,
                                      with_bias=with_bias)
    _check(x, _gpu(x, cuda), _ref(x), f"z={with_z} D={with_D} bias={with_bias}")


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_softplus_off(cuda, io):
    x = workloads.make_complex_inputs(1, 12, 200, 16, io, seed=32, with_bias=False)
    x["delta"] = (x["delta"].float().abs() * 0.05).to(x["delta"].dtype)
    x["softplus"] = False
    _check(x, _gpu(x, cuda), _ref(x), "softplus off")


def test_large_steps_and_fast_rotations(cuda):
    """Biases up to +25 and Im A up to 40: dt * Im A reaches ~1000 rad, which
    the range reduction must bring back to [-pi, pi] accurately."""
    x = workloads.make_complex_inputs(1, 8, 64, 16, "f32", seed=33)
    x["delta_bias"] = torch.linspace(-3.0, 25.0, 8)
    x["A_im"] = (torch.arange(16, dtype=torch.float32) * 2.7).repeat(8, 1).contiguous()
    assert _theta_max(x) > 500.0  # the angles this test is about
    _check(x, _gpu(x, cuda), _ref(x), "large steps")


def test_real_parameters_match_the_real_scan_kernel(cuda):
    """A_im = 0 and zero imaginary parts: the complex kernel gives the real
    scan's output (within fp32 rounding) and a real final state."""
    x = workloads.make_complex_inputs(2, 40, 300, 16, "f32", seed=34)
    x["A_im"] = torch.zeros_like(x["A_im"])
    x["B"][..., 1] = 0
    x["C"][..., 1] = 0
    yc, hc = _gpu(x, cuda)
    xd = to_device(x, cuda)
    yr, hr = abi.mamba_selective_scan_fwd(xd["u"], xd["delta"], xd["A_log_re"],
                                          xd["B"][..., 0].contiguous(), xd["C"][..., 0].contiguous(),
                                          D=xd["D"], z=xd["z"], delta_bias=xd["delta_bias"])
    torch.cuda.synchronize()
    assert rel_err(yc, yr.cpu().numpy()) <= 1e-5
    assert rel_err(hc[..., 0], hr.cpu().numpy()) <= 1e-5 and not np.any(hc[..., 1])


def test_empty_and_no_state(cuda):
    x = workloads.make_complex_inputs(2, 3, 0, 16, "f32", seed=35)
    y, h = _gpu(x, cuda)
    assert y.shape == (2, 3, 0) and not np.any(h)
    x = workloads.make_complex_inputs(1, 5, 40, 16, "bf16", seed=36)
    xd = to_device(x, cuda)
    y, h = abi.mamba_selective_scan_complex_fwd(xd["u"], xd["delta"], xd["A_log_re"], xd["A_im"],
                                                xd["B"], xd["C"], D=xd["D"], z=xd["z"],
                                                delta_bias=xd["delta_bias"],
                                                want_last_state=False)
    torch.cuda.synchronize()
    assert h is None
    assert rel_err(y.float().cpu().numpy(), _ref(x)[0]) <= TOL["bf16"]


def test_full_size_layer_every_chain(cuda):
    """Complex variant of the Mamba-130M-style layer (batch 8, d_inner 1536,
    L = 2048, N = 16, bf16): every chain against the oracle, channel block by
    channel block on the host's cores."""
    x = workloads.make_complex_inputs(8, 1536, 2048, 16, "bf16", seed=37)
    y, h = _gpu(x, cuda)
    f = workloads.to_f64

    def pair(blk):
        b, d0, d1 = blk
        sl = lambda t: None if t is None else t[b:b + 1, d0:d1]
        sd = lambda t: None if t is None else t[d0:d1]
        yr, hr = oracle.selective_scan_complex(
            f(sl(x["u"])), f(sl(x["delta"])), f(x["A_log_re"][d0:d1]), f(x["A_im"][d0:d1]),
            f(x["B"][b:b + 1]), f(x["C"][b:b + 1]), D=f(sd(x["D"])), z=f(sl(x["z"])),
            delta_bias=f(sd(x["delta_bias"])))
        return {"y": (y[b:b + 1, d0:d1], yr),
                "h": (h[b:b + 1, d0:d1], np.stack([hr.real, hr.imag], -1))}

    errs = blockwise_rel_err(channel_blocks(8, 1536, 128), pair, floors=(0.1,),
                             workers=os.cpu_count() or 1)
    for k, (e,) in errs.items():
        assert e <= TOL["bf16"], (k, e)
