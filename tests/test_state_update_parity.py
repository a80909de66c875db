"""GPU decode step vs the fp64 oracle, and decode chains vs the GPU scan."""
import numpy as np
import pytest
import torch

import oracle
from parity_util import TOL, gpu_scan, normwise, rel_err, to_device
from selective_state_space_140_b300 import abi, workloads

pytestmark = pytest.mark.gpu


def _gpu_step(xd):
    st = xd["state"].clone()
    out = abi.mamba_selective_state_update(st, xd["x"], xd["dt"], xd["A_log"], xd["B"], xd["C"],
                                           D=xd["D"], z=xd["z"], dt_bias=xd["dt_bias"],
                                           softplus=xd["softplus"])
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), st.cpu().numpy()


def _oracle_step(x):
    f = workloads.to_f64
    return oracle.selective_state_update(f(x["state"]), f(x["x"]), f(x["dt"]), f(x["A_log"]),
                                         f(x["B"]), f(x["C"]), D=f(x["D"]), z=f(x["z"]),
                                         dt_bias=f(x["dt_bias"]), softplus=x["softplus"])


def _check(x, yg, hg, yr, hr, what):
    tol = TOL[x["io_dtype"]]
    ey, eh = rel_err(yg, yr), rel_err(hg, hr)
    assert ey <= tol and eh <= tol, f"{what}: out {ey:.3e} ({normwise(yg, yr):.2e}) state {eh:.3e}"


def test_decode_config_full(cuda):
    cfg = workloads.DECODE_CONFIGS["decode_bf16"]
    x = workloads.make_decode_inputs(cfg.batch, cfg.dim, cfg.dstate, cfg.io_dtype, cfg.seed)
    yg, hg = _gpu_step(to_device(x, cuda))
    yr, hr = _oracle_step(x)
    _check(x, yg, hg, yr, hr, "decode config")


@pytest.mark.parametrize("batch,dim,N,io", [(1, 1, 1, "f32"), (3, 7, 3, "f32"), (2, 9, 4, "bf16"),
                                            (5, 13, 5, "f32"), (4, 33, 16, "bf16"),
                                            (2, 10, 17, "f32"), (3, 6, 64, "f32"),
                                            (2, 5, 100, "bf16"), (2, 3, 256, "f32"),
                                            (1, 4, 255, "f32"), (3, 65, 16, "bf16"),
                                            (5, 300, 16, "f32"), (2, 257, 8, "bf16"),
                                            (3, 1000, 64, "bf16"), (70, 3, 16, "f32")])
def test_decode_shapes(cuda, batch, dim, N, io):
    x = workloads.make_decode_inputs(batch, dim, N, io, seed=batch + dim + N)
    yg, hg = _gpu_step(to_device(x, cuda))
    yr, hr = _oracle_step(x)
    _check(x, yg, hg, yr, hr, f"{(batch, dim, N, io)}")


@pytest.mark.parametrize("with_z,with_D,with_bias", [(False, False, False), (True, False, True),
                                                      (False, True, False)])
def test_decode_optional_inputs(cuda, with_z, with_D, with_bias):
    x = workloads.make_decode_inputs(3, 20, 16, "f32", seed=21, with_z=with_z, with_D=with_D,
                                     with_bias=with_bias)
    yg, hg = _gpu_step(to_device(x, cuda))
    yr, hr = _oracle_step(x)
    _check(x, yg, hg, yr, hr, "optional inputs")


def test_decode_element_aligned_state(cuda):
    """A state that starts 4 bytes past a 16-byte boundary takes the scalar
    path and gives the same answer as an aligned one."""
    x = to_device(workloads.make_decode_inputs(4, 16, 16, "bf16", seed=22), cuda)
    st0 = x["state"].clone()
    o0 = abi.mamba_selective_state_update(st0, x["x"], x["dt"], x["A_log"], x["B"], x["C"],
                                          D=x["D"], z=x["z"], dt_bias=x["dt_bias"])
    buf = torch.empty(st0.numel() + 1, device=cuda)
    st1 = buf[1:].view(st0.shape)
    st1.copy_(x["state"])
    o1 = abi.mamba_selective_state_update(st1, x["x"], x["dt"], x["A_log"], x["B"], x["C"],
                                          D=x["D"], z=x["z"], dt_bias=x["dt_bias"])
    torch.cuda.synchronize()
    assert torch.equal(o0, o1) and torch.equal(st0, st1)


@pytest.mark.parametrize("io,N", [("f32", 16), ("bf16", 16), ("f32", 64)])
def test_decode_chain_reproduces_the_scan(cuda, io, N):
    """L decode steps from a zero state equal one scan of length L (GPU vs GPU
    and both vs the oracle)."""
    batch, dim, L = 2, 24, 40
    x = workloads.make_scan_inputs(batch, dim, L, N, io, seed=23, d_mode="normal")
    xd = to_device(x, cuda)
    y_scan, h_scan = gpu_scan(xd)
    st = torch.zeros((batch, dim, N), device=cuda)
    outs = []
    for t in range(L):
        outs.append(abi.mamba_selective_state_update(
            st, xd["u"][..., t].contiguous(), xd["delta"][..., t].contiguous(), xd["A_log"],
            xd["B"][:, t].contiguous(), xd["C"][:, t].contiguous(), D=xd["D"],
            z=xd["z"][..., t].contiguous(), dt_bias=xd["delta_bias"]))
    y_dec = torch.stack(outs, dim=-1)
    torch.cuda.synchronize()
    tol = TOL[io]
    assert rel_err(y_dec.float().cpu().numpy(), y_scan.float().cpu().numpy()) <= tol
    assert rel_err(st.cpu().numpy(), h_scan.cpu().numpy()) <= tol
    f = workloads.to_f64
    yr, hr, _ = oracle.selective_scan(f(x["u"]), f(x["delta"]), f(x["A_log"]), f(x["B"]), f(x["C"]),
                                      D=f(x["D"]), z=f(x["z"]), delta_bias=f(x["delta_bias"]))
    assert rel_err(y_dec.float().cpu().numpy(), yr) <= tol
    assert rel_err(st.cpu().numpy(), hr) <= tol


@pytest.mark.parametrize("io,N,batch,dim", [("bf16", 16, 3, 512), ("f32", 16, 2, 768),
                                            ("bf16", 4, 2, 2048), ("f32", 8, 3, 1024),
                                            ("bf16", 32, 2, 256), ("f32", 64, 3, 128),
                                            ("bf16", 128, 2, 64), ("f32", 128, 1, 96),
                                            ("bf16", 16, 2, 300)])
def test_decode_ring_matches_the_plain_kernel(cuda, io, N, batch, dim, monkeypatch):
    """dstate 4..128 (powers of two) with dim a multiple of the 16 KB tile and
    16-byte aligned rows take the bulk-copy ring kernel (persistent CTAs,
    3-stage ring); MAMBA_DECODE_PATH=plain forces one state access per thread
    (the last shape, dim 300, always does).  Both must match the oracle and
    each other bit for bit (same arithmetic)."""
    x = workloads.make_decode_inputs(batch, dim, N, io, seed=41 + N)
    for opt in ({}, dict(with_z=False, with_D=False, with_bias=False)):
        if opt:
            x = workloads.make_decode_inputs(batch, dim, N, io, seed=43 + N, **opt)
        xd = to_device(x, cuda)
        yr, hr = _oracle_step(x)
        monkeypatch.delenv("MAMBA_DECODE_PATH", raising=False)
        y0, h0 = _gpu_step(xd)
        monkeypatch.setenv("MAMBA_DECODE_PATH", "plain")
        y1, h1 = _gpu_step(xd)
        _check(x, y0, h0, yr, hr, f"ring {opt}")
        _check(x, y1, h1, yr, hr, f"plain {opt}")
        assert np.array_equal(y0, y1) and np.array_equal(h0, h1)
    assert abi.mamba_device_status() == 0
