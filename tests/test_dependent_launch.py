"""Programmatic dependent launch of the decode step and the conv1d.

Both kernels are launched so that their CTAs may start while the kernel
before them on the stream drains; they wait for that kernel to complete
before touching global memory.  Chains in which every launch reads what the
previous one wrote (the decode state updated in place step after step; a
conv1d fed its own output) must therefore give exactly what the same chain
gives launched the plain way (MAMBA_DECODE_PDL=0 / MAMBA_CONV_PDL=0), and the
decode chain must follow the fp64 oracle step by step.
"""
import numpy as np
import pytest
import torch

import oracle
from parity_util import TOL, rel_err, to_device
from selective_state_space_140_b300 import abi, workloads

pytestmark = pytest.mark.gpu


def _decode_chain(xs, state0, cuda):
    st = state0.clone()
    outs = []
    for xd in xs:
        outs.append(abi.mamba_selective_state_update(
            st, xd["x"], xd["dt"], xd["A_log"], xd["B"], xd["C"], D=xd["D"], z=xd["z"],
            dt_bias=xd["dt_bias"], softplus=xd["softplus"]))
    torch.cuda.synchronize()
    return [o.float().cpu().numpy() for o in outs], st.cpu().numpy()


@pytest.mark.parametrize("io,N,batch,dim", [("bf16", 16, 4, 1024), ("f32", 16, 2, 512),
                                            ("bf16", 64, 2, 256)])
def test_decode_chain_in_place_with_and_without_dependent_launch(cuda, io, N, batch, dim,
                                                                 monkeypatch):
    steps = 12
    xs_cpu = [workloads.make_decode_inputs(batch, dim, N, io, seed=300 + i) for i in range(steps)]
    xs = [to_device(x, cuda) for x in xs_cpu]
    state0 = xs[0]["state"]
    monkeypatch.delenv("MAMBA_DECODE_PDL", raising=False)
    outs_on, st_on = _decode_chain(xs, state0, cuda)
    monkeypatch.setenv("MAMBA_DECODE_PDL", "0")
    outs_off, st_off = _decode_chain(xs, state0, cuda)
    assert np.array_equal(st_on, st_off)
    for a, b in zip(outs_on, outs_off):
        assert np.array_equal(a, b)
    # the oracle, step by step from the same state
    f = workloads.to_f64
    h = f(xs_cpu[0]["state"])
    for i, x in enumerate(xs_cpu):
        y, h = oracle.selective_state_update(h, f(x["x"]), f(x["dt"]), f(x["A_log"]), f(x["B"]),
                                             f(x["C"]), D=f(x["D"]), z=f(x["z"]),
                                             dt_bias=f(x["dt_bias"]), softplus=x["softplus"])
        assert rel_err(outs_on[i], y) <= TOL[io], f"step {i}"
    assert rel_err(st_on, h) <= TOL[io]
    assert abi.mamba_device_status() == 0


def _conv_chain(x0, w, bias, n):
    x = x0
    for _ in range(n):
        x, _ = abi.mamba_causal_conv1d_fwd(x, w, bias=bias, silu=True, want_final_state=False)
    torch.cuda.synchronize()
    return x.float().cpu().numpy()


@pytest.mark.parametrize("io", ["bf16", "f32"])
def test_conv_chain_with_and_without_dependent_launch(cuda, io, monkeypatch):
    x = workloads.make_conv_inputs(2, 256, 4096, 4, io, seed=31)
    xd = to_device(x, cuda)
    monkeypatch.delenv("MAMBA_CONV_PDL", raising=False)
    on = _conv_chain(xd["x"], xd["weight"], xd["bias"], 6)
    monkeypatch.setenv("MAMBA_CONV_PDL", "0")
    off = _conv_chain(xd["x"], xd["weight"], xd["bias"], 6)
    assert np.array_equal(on, off)
    # and one step against the oracle
    monkeypatch.delenv("MAMBA_CONV_PDL", raising=False)
    one = _conv_chain(xd["x"], xd["weight"], xd["bias"], 1)
    f = workloads.to_f64
    ref, _ = oracle.causal_conv1d(f(x["x"]), f(x["weight"]), bias=f(x["bias"]), silu=True)
    assert rel_err(one, ref) <= (1e-5 if io == "f32" else 1e-2)


def test_decode_and_conv_captured_in_a_cuda_graph(cuda):
    """A decode loop captured into a CUDA graph (as a serving loop runs it) with
    the dependent launches inside: replaying the graph equals running the same
    calls eagerly, bit for bit."""
    batch, dim, N, io = 4, 1024, 16, "bf16"
    xs = [to_device(workloads.make_decode_inputs(batch, dim, N, io, seed=400 + i), cuda)
          for i in range(6)]
    cx = to_device(workloads.make_conv_inputs(batch, dim, 64, 4, io, seed=33), cuda)
    state0 = xs[0]["state"].clone()

    def run(st, outs, conv_out):
        for i, xd in enumerate(xs):
            abi.mamba_selective_state_update(
                st, xd["x"], xd["dt"], xd["A_log"], xd["B"], xd["C"], D=xd["D"], z=xd["z"],
                dt_bias=xd["dt_bias"], softplus=xd["softplus"], out=outs[i],
                stream=torch.cuda.current_stream())
        abi.mamba_causal_conv1d_fwd(cx["x"], cx["weight"], bias=cx["bias"], silu=True,
                                    out=conv_out, want_final_state=False,
                                    stream=torch.cuda.current_stream())

    st_e = state0.clone()
    outs_e = [torch.empty_like(xs[0]["x"]) for _ in xs]
    conv_e = torch.empty_like(cx["x"])
    run(st_e, outs_e, conv_e)
    torch.cuda.synchronize()

    st_g = state0.clone()
    outs_g = [torch.empty_like(xs[0]["x"]) for _ in xs]
    conv_g = torch.empty_like(cx["x"])
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        st_g.copy_(state0)
        torch.cuda.synchronize()
        with torch.cuda.graph(graph, stream=side):
            run(st_g, outs_g, conv_g)
    st_g.copy_(state0)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(st_g, st_e)
    for a, b in zip(outs_g, outs_e):
        assert torch.equal(a, b)
    assert torch.equal(conv_g, conv_e)
    # a second replay continues from the state the first one left
    graph.replay()
    run(st_e, outs_e, conv_e)
    torch.cuda.synchronize()
    assert torch.equal(st_g, st_e)
    assert abi.mamba_device_status() == 0
