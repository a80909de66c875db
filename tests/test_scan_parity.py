"""GPU forward scan vs the fp64 oracle, element by element, through the C ABI."""
import numpy as np
import pytest
import torch

from golden_io import load_tiny_f32
from fp32_emulation import fp32_envelope
from parity_util import (FINE_FLOOR, FINE_TOL, TOL, assert_full_size, full_size_errors, gpu_scan,
                         normwise, oracle_scan, rel_err, to_device)
from selective_state_space_140_b300 import abi, workloads

pytestmark = pytest.mark.gpu


def _run(x, device, **kw):
    xd = to_device(x, device)
    y, h = gpu_scan(xd, **kw)
    torch.cuda.synchronize()
    return y.float().cpu().numpy(), h.cpu().numpy()


def _assert_close(x, yg, hg, yr, hr, tol=None, what=""):
    """The parity bound at the 0.1 * rms floor, and the bound for small
    elements at the 1e-3 * rms floor (both from parity_util)."""
    tol = TOL[x["io_dtype"]] if tol is None else tol
    ey, eh = rel_err(yg, yr), rel_err(hg, hr)
    assert ey <= tol and eh <= tol, (f"{what}: y err {ey:.3e} (normwise {normwise(yg, yr):.2e}), "
                                     f"state err {eh:.3e}, tol {tol}")
    fy, fh = rel_err(yg, yr, FINE_FLOOR), rel_err(hg, hr, FINE_FLOOR)
    ftol = FINE_TOL[x["io_dtype"]]
    assert fy <= ftol and fh <= ftol, (f"{what}: at the {FINE_FLOOR} floor y err {fy:.3e}, "
                                       f"state err {fh:.3e}, tol {ftol}")
    return ey, eh


def test_tiny_config_matches_oracle_and_stored_fixture(cuda):
    x = workloads.make_config_inputs(workloads.SCAN_CONFIGS["tiny_f32"])
    yg, hg = _run(x, cuda)
    yr, hr = oracle_scan(x)
    _assert_close(x, yg, hg, yr, hr, what="tiny")
    yf, hf = load_tiny_f32()
    _assert_close(x, yg, hg, yf, hf, what="tiny vs fixture")


SHAPES = [
    # batch, dim, L, N, io
    (1, 1, 1, 16, "bf16"), (1, 5, 2, 16, "f32"), (1, 3, 3, 4, "f32"), (2, 37, 33, 16, "bf16"),
    (1, 33, 31, 4, "f32"), (2, 9, 63, 1, "f32"), (1, 3, 65, 3, "f32"), (1, 17, 2047, 16, "bf16"),
    (1, 8, 2049, 16, "f32"), (2, 7, 100, 5, "bf16"), (1, 5, 70, 17, "f32"), (1, 6, 50, 64, "f32"),
    (1, 4, 40, 100, "f32"), (1, 3, 30, 256, "f32"), (1, 130, 40, 8, "bf16"),
    (3, 2, 129, 32, "bf16"), (2, 70, 1000, 16, "bf16"), (2, 70, 1000, 16, "f32"),
    (1, 64, 4096, 16, "bf16"), (2, 40, 777, 64, "f32"),
]


@pytest.mark.parametrize("batch,dim,L,N,io", SHAPES, ids=lambda v: str(v))
def test_shapes_match_oracle(cuda, batch, dim, L, N, io):
    x = workloads.make_scan_inputs(batch, dim, L, N, io, seed=batch * 1000 + dim + L + N,
                                   d_mode="normal")
    yg, hg = _run(x, cuda)
    yr, hr = oracle_scan(x)
    _assert_close(x, yg, hg, yr, hr, what=f"{(batch, dim, L, N, io)}")


@pytest.mark.parametrize("with_z,with_D,with_bias", [(False, True, True), (True, False, True),
                                                      (True, True, False), (False, False, False)])
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_optional_inputs(cuda, with_z, with_D, with_bias, io):
    x = workloads.make_scan_inputs(2, 21, 150, 16, io, seed=7, d_mode="normal", with_z=with_z,
                                   with_D=with_D, with_bias=with_bias)
    yg, hg = _run(x, cuda)
    yr, hr = oracle_scan(x)
    _assert_close(x, yg, hg, yr, hr, what=f"z={with_z} D={with_D} bias={with_bias}")


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_softplus_off_uses_delta_as_given(cuda, io):
    x = workloads.make_scan_inputs(1, 12, 200, 16, io, seed=8, d_mode="normal", with_bias=False)
    x["delta"] = (x["delta"].float().abs() * 0.05).to(x["delta"].dtype)
    x["softplus"] = False
    yg, hg = _run(x, cuda)
    yr, hr = oracle_scan(x)
    _assert_close(x, yg, hg, yr, hr, what="softplus off")


def test_large_steps_take_the_upper_softplus_branch(cuda):
    x = workloads.make_scan_inputs(1, 8, 64, 16, "f32", seed=9, d_mode="normal")
    x["delta_bias"] = torch.linspace(-3.0, 25.0, 8)
    yg, hg = _run(x, cuda)
    yr, hr = oracle_scan(x)
    _assert_close(x, yg, hg, yr, hr, what="large dt")


def test_zero_steps_leave_the_state_zero(cuda):
    """dt = 0 limit: out = D*u*SiLU(z) and the final state is exactly zero."""
    x = workloads.make_scan_inputs(2, 10, 77, 16, "f32", seed=10, d_mode="normal",
                                   with_bias=False)
    x["delta"] = torch.zeros_like(x["delta"])
    x["softplus"] = False
    yg, hg = _run(x, cuda)
    assert np.all(hg == 0.0)
    yr, hr = oracle_scan(x)
    _assert_close(x, yg, hg, yr, hr, what="dt=0")


def test_empty_sequence_zeroes_the_state(cuda):
    x = workloads.make_scan_inputs(2, 5, 0, 16, "bf16", seed=11)
    xd = to_device(x, cuda)
    h = torch.full((2, 5, 16), float("nan"), device=cuda)
    y, h = gpu_scan(xd, last_state=h)
    torch.cuda.synchronize()
    assert y.numel() == 0 and torch.all(h == 0)


def test_results_are_deterministic(cuda):
    x = workloads.make_scan_inputs(2, 64, 513, 16, "bf16", seed=12)
    y1, h1 = _run(x, cuda)
    y2, h2 = _run(x, cuda)
    assert np.array_equal(y1, y2) and np.array_equal(h1, h2)


def test_output_is_linear_in_u(cuda):
    """With dt, B, C and z held fixed, the recurrence and the gated output are
    linear in u: scanning al*u1 + be*u2 gives al*y1 + be*y2 and the same
    combination of the final states.  Each of the three fp32 runs sits well
    inside the 1e-4 parity bound of its exact result, so the residual is at
    most (1 + |al| + |be|) times that; 1e-3 leaves room while any place where
    u enters non-linearly (the step size, the gate) gives errors of order one."""
    x1 = workloads.make_scan_inputs(2, 19, 300, 16, "f32", seed=18, d_mode="normal")
    u2 = workloads.make_scan_inputs(2, 19, 300, 16, "f32", seed=19)["u"]
    al, be = 0.75, -1.25
    y1, h1 = _run(x1, cuda)
    y2, h2 = _run(dict(x1, u=u2), cuda)
    y3, h3 = _run(dict(x1, u=al * x1["u"] + be * u2), cuda)
    assert rel_err(y3, al * y1 + be * y2) <= 1e-3
    assert rel_err(h3, al * h1 + be * h2) <= 1e-3


def test_permuting_channels_and_batches_permutes_the_outputs(cuda):
    """Chains are independent: permuting channels (u, dt, z with their A_log
    rows, D and bias) and batches (with their B, C) permutes y and the final
    state the same way.  A_log gets a per-channel offset so that a row taken
    from the wrong channel shows.  Every chain goes through the same
    arithmetic wherever it sits in the grid, so the bound is a tenth of the
    fp32 parity bound."""
    x = workloads.make_scan_inputs(3, 45, 257, 16, "f32", seed=20, d_mode="normal")
    g = torch.Generator().manual_seed(20)
    x["A_log"] = (x["A_log"] + 0.5 * torch.rand(45, 1, generator=g)).contiguous()
    yg, hg = _run(x, cuda)
    p = torch.randperm(45, generator=g)
    q = torch.tensor([2, 0, 1])
    xp = dict(x)
    for k in ("u", "delta", "z"):
        xp[k] = x[k][q][:, p].contiguous()
    for k in ("B", "C"):
        xp[k] = x[k][q].contiguous()
    for k in ("A_log", "D", "delta_bias"):
        xp[k] = x[k][p].contiguous()
    yp, hp = _run(xp, cuda)
    pn, qn = p.numpy(), q.numpy()
    assert rel_err(yp, yg[qn][:, pn]) <= 1e-5
    assert rel_err(hp, hg[qn][:, pn]) <= 1e-5
    yr, hr = oracle_scan(xp)
    _assert_close(xp, yp, hp, yr, hr, what="permuted")


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_element_aligned_buffers_give_the_same_result(cuda, io):
    """Inputs that start one element past a 16-byte boundary take the scalar
    path and must give bitwise the same answer as aligned ones."""
    x = workloads.make_scan_inputs(2, 24, 96, 16, io, seed=13)
    xd = to_device(x, cuda)
    y0, h0 = gpu_scan(xd)
    shifted = {}
    for k in ("u", "delta", "z", "B", "C"):
        t = xd[k]
        buf = torch.empty(t.numel() + 1, dtype=t.dtype, device=cuda)
        v = buf[1:].view(t.shape)
        v.copy_(t)
        shifted[k] = v
    xs = dict(xd, **shifted)
    ybuf = torch.empty(y0.numel() + 1, dtype=y0.dtype, device=cuda)
    y1, h1 = gpu_scan(xs, y=ybuf[1:].view(y0.shape))
    torch.cuda.synchronize()
    assert torch.equal(y0, y1) and torch.equal(h0, h1)


def test_runs_on_a_side_stream(cuda):
    x = workloads.make_scan_inputs(1, 32, 300, 16, "bf16", seed=14)
    xd = to_device(x, cuda)
    y0, h0 = gpu_scan(xd)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        y1, h1 = gpu_scan(xd)
    s.synchronize()
    assert torch.equal(y0, y1) and torch.equal(h0, h1)


def test_reports_alias_error(cuda):
    x = to_device(workloads.make_scan_inputs(1, 4, 16, 4, "f32", seed=15), cuda)
    with pytest.raises(abi.MambaError, match="ALIAS"):
        gpu_scan(x, y=x["u"])


@pytest.mark.parametrize("name", ["mamba130m_bf16", "mamba1p4b_bf16", "dna_long_bf16",
                                  "large_state_f32"])
def test_full_size_configs_every_chain(cuda, name):
    """Full-size launch as the benchmark runs it; the oracle recomputes every
    chain (whole sequences, every element of y and every final state), so
    partial CTAs, segment edges and wave tails at full size are all checked."""
    cfg = workloads.SCAN_CONFIGS[name]
    x = workloads.make_config_inputs(cfg)
    xd = to_device(x, cuda)
    y, h = gpu_scan(xd)
    torch.cuda.synchronize()
    assert torch.isfinite(y).all() and torch.isfinite(h).all()
    errs = full_size_errors(x, y, h, emulate=cfg.io_dtype == "f32")
    assert_full_size(cfg.io_dtype, errs, name)


@pytest.mark.parametrize("split", ["planned", "unsplit"])
@pytest.mark.parametrize("io,L", [("f32", 1000), ("f32", 4096), ("bf16", 4096)])
def test_wide_range_a_log(cuda, io, L, split, monkeypatch):
    """|A| log-uniform over [1e-2, 1e2] per (channel, state), as a trained
    layer drifts: at small dt the decay Abar = 2^(dt * A * log2 e) comes within
    1e-5 of 1, where an error in the exponential is amplified by the state's
    memory 1/(1 - Abar).  The bound is the larger of the fixed one and twice
    what correctly rounded fp32 arithmetic reaches on the same inputs, taken
    over four fp32 evaluations that differ only in rounding (fp32_envelope):
    slow states that keep their whole history are long fp32 running sums,
    which fp32 arithmetic with exponentials a few ulp off (as the GPU's are)
    does not hold to 1e-4 at L = 4096, and the largest error on small
    elements is one cancelling element's rounding noise, which spreads over a
    factor of 2-3 between equally correct evaluations
    (test_fp32_emulation.py).  These 96 chains take the time-split path as
    planned, and the one-pass tile when the split is switched off."""
    if split == "unsplit":
        monkeypatch.setenv("MAMBA_SCAN_SEGMENTS", "1")
    x = workloads.make_scan_inputs(2, 48, L, 16, io, seed=78 + L, d_mode="normal")
    x["A_log"] = workloads.wide_a_log(48, 16, 78 + L)
    yg, hg = _run(x, cuda)
    yr, hr = oracle_scan(x)
    env = fp32_envelope(x, out_bf16=io == "bf16")
    for what, g, r, k in (("y", yg, yr, 0), ("state", hg, hr, 1)):
        for floor, fixed in ((0.1, TOL[io]), (FINE_FLOOR, FINE_TOL[io])):
            bound = max(fixed, 2 * max(rel_err(e[k], r, floor) for e in env))
            err = rel_err(g, r, floor)
            assert err <= bound, f"{what} at floor {floor}: {err:.3e} > {bound:.3e}"


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("L,dim", [(336, 50), (4096, 33), (333, 50)])
def test_all_tile_shapes_give_the_same_scan(cuda, io, L, dim, monkeypatch):
    """dstate = 16 has several tile shapes: one chain x 8 states per thread
    with separate recurrence and element warps (default; 32 chains per CTA, or
    16 with one warp of each role), the same without the split, one chain x 4
    states, two chains x 4 states.  Each must match the oracle and the others
    (odd channel counts leave half-used pairs)."""
    x = workloads.make_scan_inputs(2, dim, L, 16, io, seed=16, d_mode="normal")
    yr, hr = oracle_scan(x)
    outs = []
    for tile in ("0", "1", "2", "3", "4", "5", "6", "7", "8"):
        monkeypatch.setenv("MAMBA_SCAN_TILE", tile)
        y, h = _run(x, cuda)
        _assert_close(x, y, h, yr, hr, what=f"tile {tile}")
        outs.append((y, h))
    tol = TOL[io]
    for y, h in outs[1:]:
        assert rel_err(y, outs[0][0]) <= tol and rel_err(h, outs[0][1]) <= tol


@pytest.mark.parametrize("io,N", [("bf16", 16), ("f32", 16), ("f32", 64), ("bf16", 4), ("f32", 200),
                                  ("bf16", 8), ("f32", 32), ("bf16", 128)])
def test_register_path_matches_tensor_map_path(cuda, io, N, monkeypatch):
    """Rows that are 16-byte aligned go through the tensor-map (TMA) kernel;
    the register-prefetch kernel is the fallback.  Forcing the fallback on the
    same aligned inputs must give the same scan (ragged tail included)."""
    x = workloads.make_scan_inputs(2, 37, 1000, N, io, seed=17, d_mode="normal")
    y0, h0 = _run(x, cuda)
    monkeypatch.setenv("MAMBA_SCAN_PATH", "reg")
    y1, h1 = _run(x, cuda)
    yr, hr = oracle_scan(x)
    _assert_close(x, y0, h0, yr, hr, what="tma path")
    _assert_close(x, y1, h1, yr, hr, what="register path")


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("batch,dim,L,nseg", [(2, 40, 1000, 2), (1, 70, 2048, 3), (2, 33, 1504, 7),
                                              (1, 32, 4096, 16)])
def test_segmented_scan_matches_oracle(cuda, io, batch, dim, L, nseg, monkeypatch):
    """A sequence split along time (summary pass, carry pass, full pass) must
    give the oracle's scan, ragged last segment and partial CTAs included, and
    agree with the unsplit kernel."""
    x = workloads.make_scan_inputs(batch, dim, L, 16, io, seed=18 + nseg, d_mode="normal")
    yr, hr = oracle_scan(x)
    monkeypatch.setenv("MAMBA_SCAN_SEGMENTS", "1")
    y1, h1 = _run(x, cuda)
    monkeypatch.setenv("MAMBA_SCAN_SEGMENTS", str(nseg))
    ys, hs = _run(x, cuda)
    _assert_close(x, ys, hs, yr, hr, what=f"{nseg} segments")
    _assert_close(x, y1, h1, yr, hr, what="unsplit")
    assert rel_err(ys, y1) <= TOL[io] and rel_err(hs, h1) <= TOL[io]


def test_segmented_scan_without_softplus_and_optional_inputs(cuda, monkeypatch):
    x = workloads.make_scan_inputs(1, 50, 1200, 16, "bf16", seed=23, d_mode="normal",
                                   with_z=False, with_D=False, with_bias=False)
    x["delta"] = (x["delta"].float().abs() * 0.05).to(x["delta"].dtype)
    x["softplus"] = False
    monkeypatch.setenv("MAMBA_SCAN_SEGMENTS", "5")
    yg, hg = _run(x, cuda)
    yr, hr = oracle_scan(x)
    _assert_close(x, yg, hg, yr, hr, what="segmented, no z/D/bias, softplus off")


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("batch,dim,L", [(2, 40, 1000), (1, 16, 336), (3, 33, 4096)])
def test_dstate64_tiles_agree(cuda, io, batch, dim, L, monkeypatch):
    """dstate 64: MAMBA_SCAN_TILE=4 selects the warp-specialised tile (16
    states x 4 lanes per chain, 16 chains per CTA), 3 the paired-chain tile
    (the default).  Both must match the oracle and each other (partial CTAs
    and a ragged last chunk included)."""
    x = workloads.make_scan_inputs(batch, dim, L, 64, io, seed=50 + L, d_mode="normal")
    yr, hr = oracle_scan(x)
    monkeypatch.setenv("MAMBA_SCAN_TILE", "4")
    y0, h0 = _run(x, cuda)
    monkeypatch.setenv("MAMBA_SCAN_TILE", "3")
    y1, h1 = _run(x, cuda)
    _assert_close(x, y0, h0, yr, hr, what="warp-specialised")
    _assert_close(x, y1, h1, yr, hr, what="paired")
    assert rel_err(y0, y1) <= TOL[io] and rel_err(h0, h1) <= TOL[io]
