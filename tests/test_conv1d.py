"""GPU causal depthwise conv1d (+ SiLU) vs the fp64 oracle, through the C ABI.

Error metric as for the scan (``parity_util.rel_err``).  Tolerances: fp32 io
1e-5 -- each output is width products and a bias summed in fp32 plus the SFU
form of SiLU (relative error about 2^-21); bf16 io 1e-2 -- the output is
rounded to bf16 (relative 2^-9, up to 2^-8 against the 0.1 rms floor).  The
states are copies of inputs and must match exactly.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from parity_util import blockwise_rel_err, channel_blocks, rel_err, to_device
from selective_state_space_140_b300 import abi, workloads

pytestmark = pytest.mark.gpu

CTOL = {"f32": 1e-5, "bf16": 1e-2}


def _gpu(x, device, silu=True, want_final=True, **kw):
    xd = to_device(x, device)
    out, fin = abi.mamba_causal_conv1d_fwd(xd["x"], xd["weight"], bias=xd["bias"],
                                           initial_state=xd["initial_state"], silu=silu,
                                           want_final_state=want_final, **kw)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), (None if fin is None else fin.float().cpu().numpy())


def _ref(x, silu=True):
    f = workloads.to_f64
    return oracle.causal_conv1d(f(x["x"]), f(x["weight"]), bias=f(x["bias"]),
                                initial_state=f(x["initial_state"]), silu=silu)


def _check(x, got, want, what=""):
    (og, fg), (orf, frf) = got, want
    err = rel_err(og, orf)
    assert err <= CTOL[x["io_dtype"]], f"{what}: out err {err:.2e}"
    if fg is not None:
        assert np.array_equal(fg, frf), f"{what}: final state differs"


SHAPES = [
    # batch, dim, L, width, io  -- L % 8 == 0 takes the vector path for bf16, % 4 for fp32
    (1, 1, 8, 4, "bf16"), (2, 3, 64, 4, "bf16"), (2, 5, 64, 4, "f32"), (1, 7, 13, 4, "bf16"),
    (1, 4, 3, 4, "f32"), (2, 6, 100, 4, "f32"), (1, 3, 256, 1, "bf16"), (1, 3, 256, 2, "f32"),
    (1, 3, 256, 3, "bf16"), (1, 3, 256, 5, "f32"), (1, 3, 256, 6, "f32"), (1, 3, 256, 8, "bf16"),
    (1, 3, 256, 8, "f32"), (2, 37, 1000, 4, "bf16"), (3, 64, 4096, 4, "bf16"),
    (1, 9, 4104, 4, "f32"), (1, 2, 1, 4, "bf16"), (1, 2, 2, 8, "bf16"),
]


@pytest.mark.parametrize("batch,dim,L,width,io", SHAPES, ids=lambda v: str(v))
@pytest.mark.parametrize("with_state", [False, True])
def test_shapes_match_oracle(cuda, batch, dim, L, width, io, with_state):
    x = workloads.make_conv_inputs(batch, dim, L, width, io, seed=batch + dim + L + width,
                                   with_state=with_state)
    _check(x, _gpu(x, cuda), _ref(x), what=str((batch, dim, L, width, io, with_state)))


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("silu,with_bias", [(False, True), (True, False), (False, False)])
def test_activation_and_bias_options(cuda, io, silu, with_bias):
    x = workloads.make_conv_inputs(2, 10, 96, 4, io, seed=21, with_bias=with_bias,
                                   with_state=True)
    _check(x, _gpu(x, cuda, silu=silu), _ref(x, silu=silu), what=f"silu={silu} bias={with_bias}")


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_scalar_and_vector_paths_agree_bitwise(cuda, monkeypatch, io):
    x = workloads.make_conv_inputs(2, 11, 512, 4, io, seed=22, with_state=True)
    o1, f1 = _gpu(x, cuda)
    monkeypatch.setenv("MAMBA_CONV_PATH", "scalar")
    o2, f2 = _gpu(x, cuda)
    assert np.array_equal(o1, o2) and np.array_equal(f1, f2)


def test_misaligned_rows_take_the_scalar_path(cuda):
    """x and out one element off a 16-byte boundary (views into larger buffers)."""
    x = workloads.make_conv_inputs(1, 6, 64, 4, "bf16", seed=23, with_state=True)
    xd = to_device(x, cuda)
    big = torch.zeros(6 * 64 + 1, dtype=torch.bfloat16, device=cuda)
    big[1:] = xd["x"].reshape(-1)
    xv = big[1:].view(1, 6, 64)
    obig = torch.empty(6 * 64 + 1, dtype=torch.bfloat16, device=cuda)
    ov = obig[1:].view(1, 6, 64)
    abi.mamba_causal_conv1d_fwd(xv, xd["weight"], bias=xd["bias"],
                                initial_state=xd["initial_state"], out=ov)
    torch.cuda.synchronize()
    orf, _ = _ref(x)
    assert rel_err(ov.float().cpu().numpy(), orf) <= CTOL["bf16"]


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_blocks_chained_through_the_state_equal_one_pass(cuda, io):
    """Block-by-block processing with final -> initial state gives the same
    outputs (bit for bit) as one pass over the whole sequence."""
    x = workloads.make_conv_inputs(2, 9, 160, 4, io, seed=24, with_state=True)
    xd = to_device(x, cuda)
    full, fin = abi.mamba_causal_conv1d_fwd(xd["x"], xd["weight"], bias=xd["bias"],
                                            initial_state=xd["initial_state"],
                                            want_final_state=True)
    st, outs = xd["initial_state"], []
    for lo, hi in ((0, 8), (8, 11), (11, 96), (96, 160)):
        o, st = abi.mamba_causal_conv1d_fwd(xd["x"][:, :, lo:hi].contiguous(), xd["weight"],
                                            bias=xd["bias"], initial_state=st,
                                            want_final_state=True)
        outs.append(o)
    torch.cuda.synchronize()
    assert torch.equal(torch.cat(outs, dim=2), full) and torch.equal(st, fin)


def test_empty_sequence_copies_the_state(cuda):
    x = workloads.make_conv_inputs(2, 3, 0, 4, "bf16", seed=25, with_state=True)
    out, fin = _gpu(x, cuda)
    assert out.shape == (2, 3, 0)
    assert np.array_equal(fin, x["initial_state"].float().numpy())
    x["initial_state"] = None
    _, fin = _gpu(x, cuda)
    assert not np.any(fin)


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("width", [1, 2, 4, 8])
def test_decode_steps_match_oracle_and_the_full_pass(cuda, io, width):
    """T decode steps from a conv state equal the oracle's conv over those T
    tokens with that initial state, and (bitwise) the GPU's one-pass conv."""
    T = 7
    x = workloads.make_conv_inputs(3, 20, T, width, io, seed=26 + width, with_state=True)
    xd = to_device(x, cuda)
    state = xd["initial_state"].clone()
    outs = []
    for t in range(T):
        outs.append(abi.mamba_causal_conv1d_update(state, xd["x"][:, :, t].contiguous(),
                                                   xd["weight"], bias=xd["bias"]))
    dec = torch.stack(outs, dim=2)
    full, fin = abi.mamba_causal_conv1d_fwd(xd["x"], xd["weight"], bias=xd["bias"],
                                            initial_state=xd["initial_state"],
                                            want_final_state=True)
    torch.cuda.synchronize()
    orf, frf = _ref(x)
    assert rel_err(dec.float().cpu().numpy(), orf) <= CTOL[io]
    assert np.array_equal(state.float().cpu().numpy(), frf)
    assert torch.equal(dec, full) and torch.equal(state, fin)


def test_full_size_layer_every_row(cuda):
    """The conv in front of the Mamba-1.4B-style layer (batch 4, d_inner 4096,
    L = 4096, width 4, bf16), launched as the bench times it; every row
    against the oracle, and every final state exactly."""
    x = workloads.make_conv_inputs(4, 4096, 4096, 4, "bf16", seed=27)
    out, fin = _gpu(x, cuda)
    f = workloads.to_f64

    def pair(blk):
        b, d0, d1 = blk
        o, s = oracle.causal_conv1d(f(x["x"][b:b + 1, d0:d1]), f(x["weight"][d0:d1]),
                                    bias=f(x["bias"][d0:d1]))
        assert np.array_equal(fin[b:b + 1, d0:d1], s), (b, d0)
        return {"out": (out[b:b + 1, d0:d1], o)}

    (e,) = blockwise_rel_err(channel_blocks(4, 4096, 512), pair, floors=(0.1,),
                             workers=os.cpu_count() or 1)["out"]
    assert e <= CTOL["bf16"], e
