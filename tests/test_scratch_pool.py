"""The library's scratch memory pool (carried states of a split scan, the
backward's checkpoints).

The pool's release threshold is read once per process, when the pool is
created, so the case where it returns everything to the driver at each
synchronisation (MAMBA_SCRATCH_RETAIN_MB=0) runs in a child process: a split
forward scan and a backward must give, bit for bit, what they give with the
default pool in this process.
"""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from parity_util import to_device
from selective_state_space_140_b300 import abi, workloads

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys, numpy as np, torch
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
from parity_util import to_device
from selective_state_space_140_b300 import abi, workloads
dev = torch.device("cuda:0")
x = workloads.make_scan_inputs(1, 70, 2048, 16, "bf16", seed=91, d_mode="normal")
xd = to_device(x, dev)
outs = []
for _ in range(2):
    y, h = abi.mamba_selective_scan_fwd(xd["u"], xd["delta"], xd["A_log"], xd["B"], xd["C"],
                                        D=xd["D"], z=xd["z"], delta_bias=xd["delta_bias"])
    g = torch.Generator(device=dev).manual_seed(5)
    dout = torch.randn(xd["u"].shape, generator=g, device=dev).to(xd["u"].dtype)
    gr = abi.mamba_selective_scan_bwd(xd["u"], xd["delta"], xd["A_log"], xd["B"], xd["C"], dout,
                                      D=xd["D"], z=xd["z"], delta_bias=xd["delta_bias"])
    torch.cuda.synchronize()
    outs.append([y.float().cpu().numpy(), h.cpu().numpy(), gr["du"].float().cpu().numpy()])
assert all(np.array_equal(a, b) for a, b in zip(outs[0], outs[1]))
np.savez({out!r}, y=outs[0][0], h=outs[0][1], du=outs[0][2])
print("ok")
"""


def test_a_pool_that_keeps_nothing_gives_the_same_results(cuda, tmp_path, monkeypatch):
    monkeypatch.setenv("MAMBA_SCAN_SEGMENTS", "4")  # force the split (scratch for its carries)
    out = str(tmp_path / "child.npz")
    env = dict(os.environ, MAMBA_SCRATCH_RETAIN_MB="0", MAMBA_SCAN_SEGMENTS="4")
    code = CHILD.format(root=ROOT, tests=os.path.join(ROOT, "tests"), out=out)
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0 and "ok" in r.stdout, r.stderr[-2000:]
    child = np.load(out)
    x = workloads.make_scan_inputs(1, 70, 2048, 16, "bf16", seed=91, d_mode="normal")
    xd = to_device(x, cuda)
    y, h = abi.mamba_selective_scan_fwd(xd["u"], xd["delta"], xd["A_log"], xd["B"], xd["C"],
                                        D=xd["D"], z=xd["z"], delta_bias=xd["delta_bias"])
    g = torch.Generator(device=cuda).manual_seed(5)
    dout = torch.randn(xd["u"].shape, generator=g, device=cuda).to(xd["u"].dtype)
    gr = abi.mamba_selective_scan_bwd(xd["u"], xd["delta"], xd["A_log"], xd["B"], xd["C"], dout,
                                      D=xd["D"], z=xd["z"], delta_bias=xd["delta_bias"])
    torch.cuda.synchronize()
    assert np.array_equal(child["y"], y.float().cpu().numpy())
    assert np.array_equal(child["h"], h.cpu().numpy())
    assert np.array_equal(child["du"], gr["du"].float().cpu().numpy())
    assert abi.mamba_device_status() == 0
