"""GPU backward scan vs the fp64 oracle's adjoint, through the C ABI.

Every gradient is compared element by element with the metric of the forward
parity tests (``parity_util.rel_err``: max |gpu - ref| / max(|ref|, 0.1 rms)).
Tolerances, per io dtype, shared by the per-element gradients (du, ddelta,
dz) and the sums: fp32 io 3e-4 -- the backward is three fp32 evaluations in
a row, each held to the forward's 1e-4: the recomputed forward states, the
adjoint recurrence (a second length-L recurrence with the same decays, hence
the same error growth), and the parameter sums (dA_log, dD and the bias
gradient add one fp32 term per step and batch row).  bf16 io 1e-2 -- du,
ddelta and dz are rounded to bf16 (relative 2^-8) on top of the fp32 bound
of the bf16-input arithmetic (the bf16 forward's 2e-2 covers one pass; the
gradients read inputs that carry no extra rounding).
"""
import os

import numpy as np
import pytest
import torch

import oracle
from parity_util import blockwise_rel_err, rel_err, to_device
from selective_state_space_140_b300 import abi, workloads

pytestmark = pytest.mark.gpu

GTOL = {"f32": 3e-4, "bf16": 1e-2}
PER_ELEMENT = ("du", "ddelta", "dz")


def _dout(x, seed):
    gen = torch.Generator().manual_seed(int(seed) + 99)
    return torch.randn(x["u"].shape, generator=gen, dtype=torch.float32).to(x["u"].dtype)


def _gpu_bwd(x, dout, device, **kw):
    xd = to_device(x, device)
    g = abi.mamba_selective_scan_bwd(xd["u"], xd["delta"], xd["A_log"], xd["B"], xd["C"],
                                     dout.to(device), D=xd["D"], z=xd["z"],
                                     delta_bias=xd["delta_bias"], softplus=xd["softplus"], **kw)
    torch.cuda.synchronize()
    return {k: v.float().cpu().numpy() for k, v in g.items()}


def _oracle_bwd(x, dout):
    f = workloads.to_f64
    return oracle.selective_scan_bwd(f(x["u"]), f(x["delta"]), f(x["A_log"]), f(x["B"]),
                                     f(x["C"]), f(dout), D=f(x["D"]), z=f(x["z"]),
                                     delta_bias=f(x["delta_bias"]), softplus=x["softplus"])


def _assert_grads(x, gg, gr, what="", tol=None):
    tol = GTOL[x["io_dtype"]] if tol is None else tol
    assert set(gg) == set(gr), (sorted(gg), sorted(gr))
    errs = {k: rel_err(gg[k], gr[k]) for k in sorted(gr)}
    bad = {k: e for k, e in errs.items() if e > tol}
    shown = ", ".join(f"{k} {e:.2e}" for k, e in errs.items())
    assert not bad, f"{what}: {shown} (tol {tol})"
    return errs


SHAPES = [
    # batch, dim, L, N, io
    (1, 1, 1, 16, "f32"), (1, 3, 15, 4, "f32"), (1, 5, 16, 16, "f32"), (2, 7, 17, 16, "bf16"),
    (1, 33, 33, 16, "f32"), (2, 37, 100, 16, "bf16"), (1, 9, 63, 1, "f32"), (1, 6, 65, 3, "f32"),
    (2, 10, 70, 8, "f32"), (1, 5, 70, 17, "f32"), (1, 6, 50, 32, "bf16"), (1, 6, 50, 64, "f32"),
    (1, 4, 40, 100, "f32"), (1, 3, 30, 256, "f32"), (1, 130, 40, 8, "bf16"),
    (2, 70, 1000, 16, "f32"), (2, 70, 1000, 16, "bf16"), (1, 16, 2049, 16, "f32"),
]


@pytest.mark.parametrize("batch,dim,L,N,io", SHAPES, ids=lambda v: str(v))
def test_shapes_match_oracle(cuda, batch, dim, L, N, io):
    seed = batch * 1000 + dim + L + N
    x = workloads.make_scan_inputs(batch, dim, L, N, io, seed=seed, d_mode="normal")
    dout = _dout(x, seed)
    _assert_grads(x, _gpu_bwd(x, dout, cuda), _oracle_bwd(x, dout), what=str((batch, dim, L, N, io)))


@pytest.mark.parametrize("with_z,with_D,with_bias", [(False, True, True), (True, False, True),
                                                      (True, True, False), (False, False, False)])
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_optional_inputs(cuda, with_z, with_D, with_bias, io):
    x = workloads.make_scan_inputs(2, 21, 150, 16, io, seed=7, d_mode="normal", with_z=with_z,
                                   with_D=with_D, with_bias=with_bias)
    dout = _dout(x, 7)
    gg = _gpu_bwd(x, dout, cuda)
    gr = _oracle_bwd(x, dout)
    assert ("dz" in gg) == with_z and ("dD" in gr) == with_D
    # the wrapper returns dD / ddelta_bias even without D / bias: they are still
    # gradients (of the parameter at zero), which the oracle gives only when the
    # input exists; compare the ones it gives
    gg = {k: v for k, v in gg.items() if k in gr}
    _assert_grads(x, gg, gr, what=f"z={with_z} D={with_D} bias={with_bias}")


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_softplus_off(cuda, io):
    x = workloads.make_scan_inputs(1, 12, 200, 16, io, seed=8, d_mode="normal", with_bias=False)
    x["delta"] = (x["delta"].float().abs() * 0.05).to(x["delta"].dtype)
    x["softplus"] = False
    dout = _dout(x, 8)
    _assert_grads(x, _gpu_bwd(x, dout, cuda, want_ddelta_bias=False), _oracle_bwd(x, dout),
                  what="softplus off")


def test_large_and_very_negative_steps(cuda):
    """Biases from -30 (dt ~ 1e-13, softplus' ~ 0) to +25 (dt ~ 25: Abar
    underflows to zero, softplus' = 1)."""
    x = workloads.make_scan_inputs(1, 8, 64, 16, "f32", seed=9, d_mode="normal")
    x["delta_bias"] = torch.linspace(-30.0, 25.0, 8)
    dout = _dout(x, 9)
    _assert_grads(x, _gpu_bwd(x, dout, cuda), _oracle_bwd(x, dout), what="extreme steps")


def test_zero_output_gradient_gives_zero_gradients(cuda):
    x = workloads.make_scan_inputs(2, 40, 77, 16, "bf16", seed=10)
    g = _gpu_bwd(x, torch.zeros_like(x["u"]), cuda)
    for k, v in g.items():
        assert not np.any(v), k


def test_per_element_gradients_are_deterministic(cuda):
    x = workloads.make_scan_inputs(2, 70, 300, 16, "bf16", seed=11, d_mode="normal")
    dout = _dout(x, 11)
    g1 = _gpu_bwd(x, dout, cuda)
    g2 = _gpu_bwd(x, dout, cuda)
    for k in PER_ELEMENT:
        assert np.array_equal(g1[k], g2[k]), k
    for k in ("dA_log", "dB", "dC", "dD", "ddelta_bias"):
        assert rel_err(g2[k], g1[k]) < 1e-5, k


def test_preallocated_outputs_are_overwritten(cuda):
    """Outputs given by the caller start as garbage; the sums are zeroed by the call."""
    x = workloads.make_scan_inputs(1, 20, 90, 16, "f32", seed=12, d_mode="normal")
    dout = _dout(x, 12)
    gr = _oracle_bwd(x, dout)
    pre = {k: torch.full(v.shape, 7.0, device=cuda, dtype=torch.float32) for k, v in gr.items()}
    _assert_grads(x, _gpu_bwd(x, dout, cuda, grads=pre), gr, what="preallocated")


def test_empty_sizes(cuda):
    x = workloads.make_scan_inputs(1, 6, 0, 16, "f32", seed=13)
    g = _gpu_bwd(x, _dout(x, 13), cuda)
    assert g["du"].shape == (1, 6, 0) and g["dB"].shape == (1, 0, 16)
    assert not np.any(g["dA_log"]) and not np.any(g["dD"]) and not np.any(g["ddelta_bias"])


def test_gradient_check_against_forward_kernel(cuda):
    """The backward is the derivative of the CUDA forward: a central difference
    of sum(dout * y) along a random direction, both ends through the forward
    kernel at fp32, matches <gradient, direction> from the backward kernel."""
    x = workloads.make_scan_inputs(1, 16, 64, 16, "f32", seed=14, d_mode="normal")
    dout = _dout(x, 14)
    xd = to_device(x, cuda)
    g = abi.mamba_selective_scan_bwd(xd["u"], xd["delta"], xd["A_log"], xd["B"], xd["C"],
                                     dout.to(cuda), D=xd["D"], z=xd["z"],
                                     delta_bias=xd["delta_bias"])
    gen = torch.Generator().manual_seed(15)
    for name in ("u", "delta", "B", "C", "z", "A_log"):
        v = torch.randn(x[name].shape, generator=gen).to(cuda)
        eps = 1e-3

        def loss(sign):
            xs = dict(xd)
            xs[name] = (xd[name].double() + sign * eps * v.double()).float().contiguous()
            y, _ = abi.mamba_selective_scan_fwd(xs["u"], xs["delta"], xs["A_log"], xs["B"],
                                                xs["C"], D=xs["D"], z=xs["z"],
                                                delta_bias=xs["delta_bias"])
            return float((y.double() * dout.to(cuda).double()).sum())

        fd = (loss(1) - loss(-1)) / (2 * eps)
        an = float((g["d" + name].double() * v.double()).sum())
        assert abs(fd - an) <= 2e-3 * max(1.0, abs(an)), (name, fd, an)


def test_full_size_layer_every_chain(cuda):
    """Mamba-1.4B-style layer (batch 4, d_inner 4096, L=4096, N=16, bf16):
    every per-element gradient of every chain, dA_log / dD / the bias gradient
    of every channel (each a sum over the 4 batch rows) and dB / dC (sums over
    all 4096 channels) against the oracle, run channel block by channel block
    on the host's cores."""
    cfg = workloads.SCAN_CONFIGS["mamba1p4b_bf16"]
    x = workloads.make_config_inputs(cfg)
    dout = _dout(x, cfg.seed)
    gg = _gpu_bwd(x, dout, cuda)
    f = workloads.to_f64
    block = 64
    blocks = [(d0, min(cfg.dim, d0 + block)) for d0 in range(0, cfg.dim, block)]
    sums = {}

    def pair(blk):
        d0, d1 = blk
        sl = lambda t: None if t is None else t[:, d0:d1]
        sd = lambda t: None if t is None else t[d0:d1]
        gr = oracle.selective_scan_bwd(f(sl(x["u"])), f(sl(x["delta"])), f(x["A_log"][d0:d1]),
                                       f(x["B"]), f(x["C"]), f(sl(dout)), D=f(sd(x["D"])),
                                       z=f(sl(x["z"])), delta_bias=f(sd(x["delta_bias"])))
        sums[blk] = (gr["dB"], gr["dC"])  # this block's share of the sums over channels
        out = {k: (gg[k][:, d0:d1], gr[k]) for k in PER_ELEMENT}
        out.update({"dA_log": (gg["dA_log"][d0:d1], gr["dA_log"]),
                    "dD": (gg["dD"][d0:d1], gr["dD"]),
                    "ddelta_bias": (gg["ddelta_bias"][d0:d1], gr["ddelta_bias"])})
        return out

    errs = {k: e[0] for k, e in blockwise_rel_err(blocks, pair, floors=(0.1,),
                                                  workers=os.cpu_count() or 1).items()}
    for i, k in enumerate(("dB", "dC")):
        total = sums[blocks[0]][i].copy()
        for blk in blocks[1:]:
            total += sums[blk][i]
        errs[k] = rel_err(gg[k], total)
    tol = GTOL["bf16"]
    bad = {k: e for k, e in errs.items() if e > tol}
    assert not bad, ", ".join(f"{k} {e:.2e}" for k, e in errs.items()) + f" (tol {tol})"


@pytest.mark.parametrize("tile", ["0", "1"])
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_selectable_dstate16_tiles(cuda, monkeypatch, tile, io):
    """Every tile the dstate <= 16 dispatch can take (MAMBA_BWD_TILE) matches
    the oracle on a ragged shape with a partial CTA."""
    monkeypatch.setenv("MAMBA_BWD_TILE", tile)
    x = workloads.make_scan_inputs(2, 37, 201, 16, io, seed=16, d_mode="normal")
    dout = _dout(x, 16)
    _assert_grads(x, _gpu_bwd(x, dout, cuda), _oracle_bwd(x, dout), what=f"tile {tile}")


@pytest.mark.parametrize("segments", ["2", "3", "7"])
@pytest.mark.parametrize("batch,dim,L,N,io", [(1, 5, 1000, 16, "f32"), (2, 3, 333, 3, "f32"),
                                              (1, 17, 700, 16, "bf16"), (1, 4, 520, 64, "f32")],
                         ids=lambda v: str(v))
def test_time_split_matches_oracle(cuda, monkeypatch, segments, batch, dim, L, N, io):
    """A backward split along time (summary pass, carry of states forwards and
    of adjoints backwards, then every segment in parallel) matches the oracle;
    forced segment counts, ragged last segments, padded states."""
    monkeypatch.setenv("MAMBA_BWD_SEGMENTS", segments)
    x = workloads.make_scan_inputs(batch, dim, L, N, io, seed=19 + L, d_mode="normal")
    dout = _dout(x, 19)
    _assert_grads(x, _gpu_bwd(x, dout, cuda), _oracle_bwd(x, dout), what=f"{segments} segments")


def test_planner_splits_few_long_chains(cuda):
    """One CTA's worth of chains over 4096 steps: the planner splits the
    sequence by itself; the result matches the oracle and the unsplit run."""
    x = workloads.make_scan_inputs(1, 16, 4096, 16, "f32", seed=20, d_mode="normal")
    dout = _dout(x, 20)
    g = _gpu_bwd(x, dout, cuda)
    _assert_grads(x, g, _oracle_bwd(x, dout), what="planner split")


def test_long_sequence_layer_on_sampled_channels(cuda):
    """Long-sequence DNA-like layer (batch 1, d_inner 1536, L = 131072, N 16,
    bf16), split along time by the planner: per-element gradients of sampled
    channels and their dA_log / dD / bias gradients against the oracle."""
    cfg = workloads.SCAN_CONFIGS["dna_long_bf16"]
    x = workloads.make_config_inputs(cfg)
    dout = _dout(x, cfg.seed)
    gg = _gpu_bwd(x, dout, cuda)
    f = workloads.to_f64
    for d in (0, 777, 1535):
        sl = lambda t: None if t is None else t[:, d:d + 1]
        sd = lambda t: None if t is None else t[d:d + 1]
        gr = oracle.selective_scan_bwd(f(sl(x["u"])), f(sl(x["delta"])), f(x["A_log"][d:d + 1]),
                                       f(x["B"]), f(x["C"]), f(sl(dout)), D=f(sd(x["D"])),
                                       z=f(sl(x["z"])), delta_bias=f(sd(x["delta_bias"])))
        part = {k: gg[k][:, d:d + 1] for k in PER_ELEMENT}
        part.update({"dA_log": gg["dA_log"][d:d + 1], "dD": gg["dD"][d:d + 1],
                     "ddelta_bias": gg["ddelta_bias"][d:d + 1]})
        _assert_grads(x, part, {k: gr[k] for k in part}, what=f"channel {d}")


@pytest.mark.parametrize("N", [24, 32, 40, 64])
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_eight_state_tiles_for_wide_states(cuda, monkeypatch, N, io):
    """The selectable 8-state tiles for dstate 17..64 (8 x 4 and 8 x 8 lanes
    per chain, MAMBA_BWD_TILE=3) match the oracle, with a partial CTA and
    padded states (the default 4-state tiles are covered by every other test)."""
    monkeypatch.setenv("MAMBA_BWD_TILE", "3")
    x = workloads.make_scan_inputs(2, 11, 150, N, io, seed=21 + N, d_mode="normal")
    dout = _dout(x, 21)
    _assert_grads(x, _gpu_bwd(x, dout, cuda), _oracle_bwd(x, dout), what=f"N={N} tile 3")


def _bwd_ex(x, dout, device, h0, reset, **kw):
    xd = to_device(x, device)
    g = abi.mamba_selective_scan_bwd(xd["u"], xd["delta"], xd["A_log"], xd["B"], xd["C"],
                                     dout.to(device), D=xd["D"], z=xd["z"],
                                     delta_bias=xd["delta_bias"], softplus=xd["softplus"],
                                     h0=None if h0 is None else h0.to(device),
                                     reset=None if reset is None else reset.to(device), **kw)
    torch.cuda.synchronize()
    return {k: v.float().cpu().numpy() for k, v in g.items()}


def _oracle_bwd_ex(x, dout, h0, reset):
    f = workloads.to_f64
    return oracle.selective_scan_bwd(f(x["u"]), f(x["delta"]), f(x["A_log"]), f(x["B"]),
                                     f(x["C"]), f(dout), D=f(x["D"]), z=f(x["z"]),
                                     delta_bias=f(x["delta_bias"]), softplus=x["softplus"],
                                     h0=f(h0), reset=None if reset is None else reset.numpy())


def _doc_starts(batch, L, every, offset):
    r = torch.zeros((batch, L), dtype=torch.uint8)
    for b in range(batch):
        r[b, (offset + 29 * b) % every::every] = 1
    return r


@pytest.mark.parametrize("batch,dim,L,N,io", [(2, 37, 201, 16, "f32"), (2, 37, 201, 16, "bf16"),
                                              (1, 6, 130, 3, "f32"), (1, 5, 100, 64, "f32"),
                                              (2, 20, 64, 16, "f32")],
                         ids=lambda v: str(v))
def test_h0_and_document_resets_match_oracle(cuda, batch, dim, L, N, io):
    """The backward of the scan from h0 with document boundaries (every 37
    tokens, offset per row; the last case also at step 0, which must zero
    that row's dh0) against the oracle, dh0 included."""
    x = workloads.make_scan_inputs(batch, dim, L, N, io, seed=23 + L, d_mode="normal")
    dout = _dout(x, 23)
    h0 = torch.randn((batch, dim, N), generator=torch.Generator().manual_seed(24))
    reset = _doc_starts(batch, L, 37, 5)
    if L == 64:
        reset[0, 0] = 1
    g = _bwd_ex(x, dout, cuda, h0, reset)
    _assert_grads(x, g, _oracle_bwd_ex(x, dout, h0, reset), what=str((batch, dim, L, N, io)))
    if L == 64:
        assert not np.any(g["dh0"][0])


@pytest.mark.parametrize("segments", ["3", "7"])
def test_h0_and_resets_with_a_time_split(cuda, monkeypatch, segments):
    """Forced segments with h0 and document starts, one of them on a segment
    boundary (step 336 starts the second of 3 segments of 21 chunks)."""
    monkeypatch.setenv("MAMBA_BWD_SEGMENTS", segments)
    x = workloads.make_scan_inputs(1, 5, 1000, 16, "f32", seed=25, d_mode="normal")
    dout = _dout(x, 25)
    h0 = torch.randn((1, 5, 16), generator=torch.Generator().manual_seed(26))
    reset = _doc_starts(1, 1000, 97, 11)
    reset[0, 336] = 1
    g = _bwd_ex(x, dout, cuda, h0, reset)
    _assert_grads(x, g, _oracle_bwd_ex(x, dout, h0, reset), what=f"{segments} segments")


def test_ex_without_h0_or_resets_is_the_plain_backward(cuda):
    """No h0 and no resets: the per-element gradients equal the plain
    backward's bit for bit, and dh0 is the gradient of a zero start."""
    x = workloads.make_scan_inputs(2, 40, 300, 16, "bf16", seed=27, d_mode="normal")
    dout = _dout(x, 27)
    g_plain = _gpu_bwd(x, dout, cuda)
    g_ex = _bwd_ex(x, dout, cuda, None, None, want_dh0=True)
    for k in PER_ELEMENT:
        assert np.array_equal(g_plain[k], g_ex[k]), k
    zero = torch.zeros((2, 40, 16))
    gr = _oracle_bwd_ex(x, dout, zero, None)
    assert rel_err(g_ex["dh0"], gr["dh0"]) <= GTOL["bf16"]


def _oracle_bwd_dlast(x, dout, h0, reset, dlast):
    f = workloads.to_f64
    return oracle.selective_scan_bwd(f(x["u"]), f(x["delta"]), f(x["A_log"]), f(x["B"]),
                                     f(x["C"]), f(dout), D=f(x["D"]), z=f(x["z"]),
                                     delta_bias=f(x["delta_bias"]), softplus=x["softplus"],
                                     h0=f(h0), reset=None if reset is None else reset.numpy(),
                                     dlast_state=f(dlast))


@pytest.mark.parametrize("segments", [None, "3"])
@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("with_reset", [False, True])
def test_final_state_gradient_matches_oracle(cuda, monkeypatch, segments, io, with_reset):
    """A loss on the final state as well as on y (dlast_state, the gradient of
    last_state): every gradient and dh0 against the oracle, unsplit and with a
    forced time split (the carry pass starts its reverse sweep from it), with
    and without document starts (it must stop at the last one of a row)."""
    if segments:
        monkeypatch.setenv("MAMBA_BWD_SEGMENTS", segments)
    x = workloads.make_scan_inputs(2, 21, 700, 16, io, seed=81, d_mode="normal")
    dout = _dout(x, 81)
    gen = torch.Generator().manual_seed(82)
    h0 = torch.randn((2, 21, 16), generator=gen)
    dlast = torch.randn((2, 21, 16), generator=gen)
    reset = _doc_starts(2, 700, 173, 7) if with_reset else None
    g = _bwd_ex(x, dout, cuda, h0, reset, dlast_state=dlast.to(cuda))
    _assert_grads(x, g, _oracle_bwd_dlast(x, dout, h0, reset, dlast),
                  what=f"dlast, {segments} segments, reset {with_reset}")


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_two_blocks_train_as_one_sequence(cuda, io):
    """Block-by-block training of one long sequence: the forward runs block 1
    from zero and block 2 from block 1's final state; the backward runs block 2
    from that state, and block 1 with block 2's dh0 as its final-state
    gradient.  Together they must give the oracle's backward of the whole
    sequence: per-element gradients and dB / dC block by block, dA_log, dD and
    the bias gradient as the sum of the two blocks."""
    L1, L2 = 320, 208
    x = workloads.make_scan_inputs(2, 19, L1 + L2, 16, io, seed=83, d_mode="normal")
    dout = _dout(x, 83)
    whole = _oracle_bwd(x, dout)
    part = lambda t, lo, hi: None if t is None else t[..., lo:hi].contiguous()
    rows = lambda t, lo, hi: t[:, lo:hi].contiguous()
    x1 = dict(x, u=part(x["u"], 0, L1), delta=part(x["delta"], 0, L1), z=part(x["z"], 0, L1),
              B=rows(x["B"], 0, L1), C=rows(x["C"], 0, L1))
    x2 = dict(x, u=part(x["u"], L1, None), delta=part(x["delta"], L1, None),
              z=part(x["z"], L1, None), B=rows(x["B"], L1, None), C=rows(x["C"], L1, None))
    xd1 = to_device(x1, cuda)
    _, h1 = abi.mamba_selective_scan_fwd(xd1["u"], xd1["delta"], xd1["A_log"], xd1["B"],
                                         xd1["C"], D=xd1["D"], z=xd1["z"],
                                         delta_bias=xd1["delta_bias"])
    torch.cuda.synchronize()
    h1 = h1.cpu()
    g2 = _bwd_ex(x2, part(dout, L1, None), cuda, h1, None)
    g1 = _bwd_ex(x1, part(dout, 0, L1), cuda, None, None,
                 dlast_state=torch.from_numpy(g2["dh0"]).to(cuda))
    got = {k: np.concatenate([g1[k], g2[k]], axis=-1) for k in PER_ELEMENT}
    got.update({k: np.concatenate([g1[k], g2[k]], axis=1) for k in ("dB", "dC")})
    got.update({k: g1[k] + g2[k] for k in ("dA_log", "dD", "ddelta_bias")})
    _assert_grads(x, got, {k: whole[k] for k in got}, what="two blocks")


def test_final_state_gradient_of_an_empty_sequence_is_dh0(cuda):
    """No steps: the final state is h0, so dh0 equals the final-state gradient."""
    x = workloads.make_scan_inputs(2, 5, 0, 16, "f32", seed=84)
    dlast = torch.randn((2, 5, 16), generator=torch.Generator().manual_seed(84))
    g = _bwd_ex(x, torch.zeros(x["u"].shape), cuda, torch.zeros((2, 5, 16)), None,
                dlast_state=dlast.to(cuda))
    assert np.array_equal(g["dh0"], dlast.numpy())
