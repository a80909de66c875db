"""mamba_selective_scan_fwd_ex: a starting state and document boundaries.

The oracle (oracle.selective_scan with h0 / reset) restarts every state of a
batch row from zero before a token whose reset byte is set, and starts from h0
when given; the GPU must match it element by element on the warp-specialised
tile, on the split (summary / carry / full) path with boundaries inside and at
the edges of segments, and on the register-prefetch path that other shapes
take.
"""
import numpy as np
import pytest
import torch

import oracle
from parity_util import TOL, assert_full_size, full_size_errors, rel_err, to_device
from selective_state_space_140_b300 import abi, workloads

pytestmark = pytest.mark.gpu


def _mask(batch, L, seed, density=0.02, extra=()):
    r = np.random.default_rng(seed)
    m = (r.random((batch, L)) < density).astype(np.uint8)
    for bi, t in extra:
        m[bi, t] = 1
    return m


def _oracle(x, h0, reset):
    f = workloads.to_f64
    y, h, _ = oracle.selective_scan(f(x["u"]), f(x["delta"]), f(x["A_log"]), f(x["B"]), f(x["C"]),
                                    D=f(x["D"]), z=f(x["z"]), delta_bias=f(x["delta_bias"]),
                                    softplus=x["softplus"], h0=h0, reset=reset)
    return y, h


def _gpu(xd, h0=None, reset=None, **kw):
    y, h = abi.mamba_selective_scan_fwd_ex(xd["u"], xd["delta"], xd["A_log"], xd["B"], xd["C"],
                                           D=xd["D"], z=xd["z"], delta_bias=xd["delta_bias"],
                                           softplus=xd["softplus"], h0=h0, reset=reset, **kw)
    torch.cuda.synchronize()
    return y, h


def _check(x, y, h, yr, hr, what):
    tol = TOL[x["io_dtype"]]
    ey, eh = rel_err(y.float().cpu().numpy(), yr), rel_err(h.cpu().numpy(), hr)
    assert ey <= tol and eh <= tol, f"{what}: y {ey:.3e} state {eh:.3e} (tol {tol})"


@pytest.mark.parametrize("io", ["bf16", "f32"])
@pytest.mark.parametrize("batch,dim,L,N,segs", [
    (2, 40, 1000, 16, "1"),      # warp-specialised tile, ragged last chunk, partial CTA
    (1, 70, 2048, 16, "4"),      # split: 4 segments of 512 steps
    (2, 33, 1504, 16, "7"),      # split: ragged last segment
    (2, 37, 999, 16, "1"),       # rows not 16-byte aligned: register-prefetch kernel
    (2, 21, 640, 8, "1"),        # dstate 8: register-prefetch kernel
    (1, 12, 512, 64, "1"),       # dstate 64: register-prefetch kernel
])
def test_reset_and_initial_state_match_the_oracle(cuda, io, batch, dim, L, N, segs, monkeypatch):
    monkeypatch.setenv("MAMBA_SCAN_SEGMENTS", segs)
    x = workloads.make_scan_inputs(batch, dim, L, N, io, seed=60 + L + N, d_mode="normal")
    r = np.random.default_rng(61)
    h0 = r.normal(size=(batch, dim, N)).astype(np.float32)
    seg = (L + int(segs) - 1) // int(segs)
    seg = (seg + 15) // 16 * 16
    extra = [(0, 0), (batch - 1, L - 1), (0, min(seg, L - 1)), (batch - 1, min(seg + 5, L - 1))]
    reset = _mask(batch, L, 62 + L, extra=extra)
    xd = to_device(x, cuda)
    y, h = _gpu(xd, torch.from_numpy(h0).to(cuda), torch.from_numpy(reset).to(cuda))
    yr, hr = _oracle(x, h0.astype(np.float64), reset)
    _check(x, y, h, yr, hr, f"reset + h0 {batch}x{dim}x{L}x{N} segs {segs}")
    # h0 alone, and a mask alone
    y, h = _gpu(xd, h0=torch.from_numpy(h0).to(cuda))
    yr, hr = _oracle(x, h0.astype(np.float64), None)
    _check(x, y, h, yr, hr, "h0 only")
    y, h = _gpu(xd, reset=torch.from_numpy(reset).to(cuda).bool())
    yr, hr = _oracle(x, None, reset)
    _check(x, y, h, yr, hr, "reset only (bool mask)")
    assert abi.mamba_device_status() == 0


@pytest.mark.parametrize("batch,dim,L,N", [(2, 40, 1000, 16), (2, 37, 999, 16), (1, 12, 512, 64)])
def test_without_state_or_mask_equals_the_plain_entry(cuda, batch, dim, L, N):
    x = workloads.make_scan_inputs(batch, dim, L, N, "bf16", seed=63, d_mode="normal")
    xd = to_device(x, cuda)
    y0, h0 = abi.mamba_selective_scan_fwd(xd["u"], xd["delta"], xd["A_log"], xd["B"], xd["C"],
                                          D=xd["D"], z=xd["z"], delta_bias=xd["delta_bias"])
    y1, h1 = _gpu(xd)
    assert torch.equal(y0, y1) and torch.equal(h0, h1)


@pytest.mark.parametrize("io", ["bf16", "f32"])
def test_streaming_in_blocks_in_place(cuda, io):
    """A long sequence processed in three blocks, each started from the state
    the previous block left in the same buffer (h0 is last_state), with a
    document boundary inside the second block, equals one scan of the whole."""
    batch, dim, L, N = 2, 64, 3072, 16
    x = workloads.make_scan_inputs(batch, dim, L, N, io, seed=64, d_mode="normal")
    reset = _mask(batch, L, 65, density=0.0, extra=[(0, 1500), (1, 2047)])
    yr, hr = _oracle(x, None, reset)
    xd = to_device(x, cuda)
    rd = torch.from_numpy(reset).to(cuda)
    state = torch.zeros((batch, dim, N), device=cuda)
    ys = []
    for t0, t1 in ((0, 1024), (1024, 2048), (2048, 3072)):
        blk = {k: (v[..., t0:t1].contiguous() if k in ("u", "delta", "z") else
                   v[:, t0:t1].contiguous() if k in ("B", "C") else v) for k, v in xd.items()}
        y, _ = _gpu(blk, h0=state, reset=rd[:, t0:t1].contiguous(), last_state=state)
        ys.append(y)
    y = torch.cat(ys, dim=-1)
    _check(x, y, state, yr, hr, "three in-place blocks")


def test_empty_sequence_copies_the_initial_state(cuda):
    x = workloads.make_scan_inputs(2, 5, 0, 16, "bf16", seed=66)
    xd = to_device(x, cuda)
    h0 = torch.randn((2, 5, 16), device=cuda)
    y, h = _gpu(xd, h0=h0)
    assert y.numel() == 0 and torch.equal(h, h0)


def test_full_size_layer_with_state_and_boundaries_every_chain(cuda):
    """The Mamba-1.4B-style layer (batch 4, d_inner 4096, L 4096, N 16, bf16)
    from a starting state with a document boundary every 512 tokens (offset
    per batch row), the launch the benchmark times through this entry; the
    oracle recomputes every chain."""
    cfg = workloads.SCAN_CONFIGS["mamba1p4b_bf16"]
    x = workloads.make_config_inputs(cfg)
    h0 = np.random.default_rng(67).normal(size=(cfg.batch, cfg.dim, cfg.dstate)).astype(np.float32)
    reset = np.zeros((cfg.batch, cfg.seqlen), dtype=np.uint8)
    for b in range(cfg.batch):
        reset[b, (97 * b) % 512::512] = 1
    xd = to_device(x, cuda)
    y, h = _gpu(xd, torch.from_numpy(h0).to(cuda), torch.from_numpy(reset).to(cuda))
    torch.cuda.synchronize()
    assert torch.isfinite(y).all() and torch.isfinite(h).all()
    assert_full_size("bf16", full_size_errors(x, y, h, h0=h0, reset=reset), "h0 + boundaries")


def test_beyond_a_million_tokens_in_one_launch_and_in_blocks(cuda):
    """2^20 + 4104 tokens on 4 channels (N 16, fp32, two document boundaries):
    one launch, which the planner splits along time into about a thousand
    segments, and the same sequence streamed as three blocks through h0 into
    the same state buffer, both match the oracle element by element."""
    batch, dim, L, N = 1, 4, (1 << 20) + 4104, 16
    x = workloads.make_scan_inputs(batch, dim, L, N, "f32", seed=68, d_mode="normal")
    reset = _mask(batch, L, 69, density=0.0, extra=[(0, 300001), (0, 777777)])
    yr, hr = _oracle(x, None, reset)
    xd = to_device(x, cuda)
    rd = torch.from_numpy(reset).to(cuda)
    y, h = _gpu(xd, reset=rd)
    _check(x, y, h, yr, hr, "one launch")
    state = torch.zeros((batch, dim, N), device=cuda)
    ys = []
    for t0, t1 in ((0, 400000), (400000, 800000), (800000, L)):
        blk = {k: (v[..., t0:t1].contiguous() if k in ("u", "delta", "z") else
                   v[:, t0:t1].contiguous() if k in ("B", "C") else v) for k, v in xd.items()}
        yb, _ = _gpu(blk, h0=state, reset=rd[:, t0:t1].contiguous(), last_state=state)
        ys.append(yb)
    _check(x, torch.cat(ys, dim=-1), state, yr, hr, "three streamed blocks")


@pytest.mark.parametrize("io", ["bf16", "f32"])
@pytest.mark.parametrize("batch,dim,L,N", [(2, 128, 2048, 16), (1, 72, 1537, 16)])
def test_zero_state_and_empty_mask_equal_the_stateless_scan(cuda, io, batch, dim, L, N):
    """A zero h0 and an all-zero reset mask change nothing: the scan that is
    given them (general tile) equals, bit for bit, the one that is not (the
    tile compiled for a gated softplus scan without state or mask)."""
    x = workloads.make_scan_inputs(batch, dim, L, N, io, seed=66, d_mode="normal")
    xd = to_device(x, cuda)
    y0, h0 = _gpu(xd)
    zero = torch.zeros((batch, dim, N), device=cuda)
    none = torch.zeros((batch, L), dtype=torch.uint8, device=cuda)
    y1, h1 = _gpu(xd, h0=zero, reset=none)
    assert torch.equal(y0, y1) and torch.equal(h0, h1)
    y2, h2 = _gpu(xd, h0=zero)
    assert torch.equal(y0, y2) and torch.equal(h0, h2)
