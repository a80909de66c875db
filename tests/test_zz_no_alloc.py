"""mamba_selective_scan_fwd_noalloc against mamba_selective_scan_fwd.

The no-allocation entry point is for callers that cannot call the CUDA
allocator (a framework that owns all device memory, a serving loop that must
not allocate mid-request).  It runs the same kernels; when it splits a scan
along time its carried states live in the library's fixed device buffer.
This file is collected last so that it runs both on its own and after every
other test, on a process whose GPU state the other tests have already used.
"""
import pytest
import torch

from parity_util import TOL, oracle_scan, rel_err, sample_chains, to_device
from selective_state_space_140_b300 import abi, workloads

pytestmark = pytest.mark.gpu


def _call(fn, xd, y=None, h=None):
    return fn(xd["u"], xd["delta"], xd["A_log"], xd["B"], xd["C"], D=xd["D"], z=xd["z"],
              delta_bias=xd["delta_bias"], softplus=xd["softplus"], y=y, last_state=h)


@pytest.mark.parametrize("io,batch,dim,L,segments", [("bf16", 1, 96, 8192, None),
                                                     ("f32", 2, 48, 4096, None),
                                                     ("bf16", 2, 64, 2048, "4")])
def test_noalloc_matches_the_allocating_entry_on_two_calls_in_a_row(cuda, io, batch, dim, L,
                                                                    segments, monkeypatch):
    """Few chains and a long sequence: both entry points split the scan (the
    planner's choice, or a forced segment count so that the split and hence
    the fixed scratch is used whatever the planner decides), so the no-alloc
    calls use the fixed scratch.  Two no-alloc calls back to back on one
    stream reuse it; each must equal the allocating entry point bit for bit
    and match the oracle."""
    if segments is not None:
        monkeypatch.setenv("MAMBA_SCAN_SEGMENTS", segments)
    x = workloads.make_scan_inputs(batch, dim, L, 16, io, seed=31, d_mode="normal")
    xd = to_device(x, cuda)
    y_ref, h_ref = _call(abi.mamba_selective_scan_fwd, xd)
    y1, h1 = _call(abi.mamba_selective_scan_fwd_noalloc, xd)
    y2 = torch.full_like(y1, float("nan"))
    h2 = torch.full_like(h1, float("nan"))
    _call(abi.mamba_selective_scan_fwd_noalloc, xd, y=y2, h=h2)
    torch.cuda.synchronize()
    assert abi.mamba_device_status() == 0
    for y, h in ((y1, h1), (y2, h2)):
        assert torch.equal(y, y_ref) and torch.equal(h, h_ref)
    chains = sample_chains(batch, dim, 6, seed=31)
    bi = torch.tensor([c[0] for c in chains])
    di = torch.tensor([c[1] for c in chains])
    yr, hr = oracle_scan(x, chains)
    assert rel_err(y1[bi, di].float().cpu().numpy(), yr) <= TOL[io]
    assert rel_err(h1[bi, di].cpu().numpy(), hr) <= TOL[io]


def test_noalloc_unsplit_scan_matches(cuda):
    """Many chains: no split, no scratch; still the same result."""
    x = workloads.make_scan_inputs(2, 300, 512, 16, "bf16", seed=32, d_mode="normal")
    xd = to_device(x, cuda)
    y_ref, h_ref = _call(abi.mamba_selective_scan_fwd, xd)
    y1, h1 = _call(abi.mamba_selective_scan_fwd_noalloc, xd)
    torch.cuda.synchronize()
    assert torch.equal(y1, y_ref) and torch.equal(h1, h_ref)


def test_noalloc_rejects_a_split_larger_than_its_scratch(cuda, monkeypatch):
    """Forcing more segments than the planner would choose needs more than the
    4 MiB buffer (4096 chains x 31 carried states x 17 floats); the call must
    fail with MAMBA_ERR_SCRATCH before launching anything, and leave the
    output untouched."""
    x = workloads.make_scan_inputs(1, 4096, 1024, 16, "bf16", seed=33)
    xd = to_device(x, cuda)
    y = torch.full_like(xd["u"], 7.0)
    monkeypatch.setenv("MAMBA_SCAN_SEGMENTS", "32")
    with pytest.raises(abi.MambaError, match="SCRATCH") as e:
        _call(abi.mamba_selective_scan_fwd_noalloc, xd, y=y)
    assert e.value.status == 9
    torch.cuda.synchronize()
    assert torch.all(y == 7.0)
    # The allocating entry point takes stream-ordered scratch for the same split.
    y_ref, _ = _call(abi.mamba_selective_scan_fwd, xd)
    monkeypatch.delenv("MAMBA_SCAN_SEGMENTS")
    y_one, _ = _call(abi.mamba_selective_scan_fwd, xd)
    torch.cuda.synchronize()
    assert rel_err(y_ref.float().cpu().numpy(), y_one.float().cpu().numpy()) <= TOL["bf16"]

