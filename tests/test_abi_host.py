"""Host-side checks of the C ABI (no GPU needed, no CUDA call is reached).

The library must load, export every function include/mamba_scan.h declares,
and reject bad arguments with the documented status before touching CUDA.
"""
import os
import re

import pytest

from selective_state_space_140_b300 import abi, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mamba_scan.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return abi.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(mamba_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_abi():
    assert declared_functions() == sorted(abi.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} is declared but not exported"


def test_version_and_status_strings(lib):
    assert abi.abi_version() == 10200
    for code, name in abi.STATUS.items():
        assert abi.status_string(code).startswith(name)
    assert abi.status_string(12345) == "unknown mamba_status_t"


# Fake, never-dereferenced device addresses (16-byte aligned, far apart).
P = [0x7f0000000000 + i * 0x100000000 for i in range(12)]
GOOD = dict(u=P[0], delta=P[1], A_log=P[2], B=P[3], C=P[4], D=P[5], z=P[6], delta_bias=P[7],
            softplus_flag=1, y=P[8], last_state=P[9], batch=2, dim=8, seqlen=16, dstate=16,
            io_dtype=abi.MAMBA_BF16, stream=None)


def scan(**over):
    kw = dict(GOOD)
    kw.update(over)
    return abi.raw_scan_fwd(**kw)


@pytest.mark.parametrize("name", ["u", "delta", "A_log", "B", "C", "y"])
def test_scan_rejects_null_required_pointer(lib, name):
    assert scan(**{name: None}) == 1  # MAMBA_ERR_NULL


@pytest.mark.parametrize("field,value", [("batch", -1), ("dim", -3), ("seqlen", -1),
                                         ("batch", 1 << 40), ("seqlen", 1 << 45)])
def test_scan_rejects_bad_sizes(lib, field, value):
    assert scan(**{field: value}) == 2  # MAMBA_ERR_SIZE


@pytest.mark.parametrize("dstate", [0, -1, 257, 1 << 20])
def test_scan_rejects_bad_dstate(lib, dstate):
    assert scan(dstate=dstate) == 3  # MAMBA_ERR_DSTATE


@pytest.mark.parametrize("io", [-1, 2, 7])
def test_scan_rejects_bad_dtype(lib, io):
    assert scan(io_dtype=io) == 5  # MAMBA_ERR_DTYPE


@pytest.mark.parametrize("name,io", [("u", abi.MAMBA_BF16), ("y", abi.MAMBA_F32),
                                     ("A_log", abi.MAMBA_BF16), ("last_state", abi.MAMBA_BF16),
                                     ("B", abi.MAMBA_F32)])
def test_scan_rejects_misaligned(lib, name, io):
    assert scan(**{name: GOOD[name] + 1, "io_dtype": io}) == 4  # MAMBA_ERR_ALIGN


def test_scan_rejects_aliasing(lib):
    assert scan(y=P[0]) == 8                 # y == u
    assert scan(y=P[3] + 32) == 8            # y starts inside B
    assert scan(last_state=P[2]) == 8        # state over A_log
    assert scan(last_state=P[8] + 64) == 8   # state inside y


def test_scan_empty_problems_return_ok_without_launch(lib):
    # Nothing to compute: returns before any CUDA call, so this is safe on CPU.
    assert scan(batch=0) == 0
    assert scan(dim=0) == 0


DGOOD = dict(state=P[0], x=P[1], dt=P[2], A_log=P[3], B=P[4], C=P[5], D=P[6], z=P[7], dt_bias=P[8],
             softplus_flag=1, out=P[9], batch=4, dim=8, dstate=16, io_dtype=abi.MAMBA_BF16,
             stream=None)


def upd(**over):
    kw = dict(DGOOD)
    kw.update(over)
    return abi.raw_state_update(**kw)


def test_state_update_validation(lib):
    for name in ("state", "x", "dt", "A_log", "B", "C", "out"):
        assert upd(**{name: None}) == 1
    assert upd(batch=-1) == 2
    assert upd(dstate=0) == 3 and upd(dstate=300) == 3
    assert upd(io_dtype=3) == 5
    assert upd(state=P[0] + 2) == 4
    assert upd(x=P[1] + 1) == 4
    assert upd(out=P[0]) == 8
    assert upd(batch=0) == 0


def test_binding_refuses_missing_library(tmp_path):
    with pytest.raises(RuntimeError, match="missing"):
        old, abi._lib = abi._lib, None
        try:
            abi.load(str(tmp_path / "nope.so"))
        finally:
            abi._lib = old


def test_noalloc_entry_validates_like_the_allocating_one(lib):
    """The no-allocation entry point shares the argument checks; every bad
    call returns before any CUDA call, with the same status."""
    cases = [dict(u=None), dict(B=None), dict(batch=-1), dict(dstate=0), dict(dstate=257),
             dict(io_dtype=9), dict(u=P[0] + 1), dict(y=P[0]), dict(last_state=P[2]),
             dict(batch=0), dict(dim=0)]
    for over in cases:
        kw = dict(GOOD)
        kw.update(over)
        assert abi.raw_scan_fwd_noalloc(**kw) == abi.raw_scan_fwd(**kw), over
    assert abi.status_string(9).startswith("MAMBA_ERR_SCRATCH")


def test_testing_header_symbols_are_exported(lib):
    text = open(os.path.join(ROOT, "include", "mamba_scan_testing.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    declared = sorted(set(re.findall(r"^\s*\w+\s*\*?\s*(mamba_\w+)\s*\(", text, flags=re.M)))
    assert declared == sorted(abi.TESTING_EXPORTED)
    for name in declared:
        assert hasattr(lib, name)


@pytest.mark.parametrize("polls", [0, -5, (1 << 20) + 1])
def test_bounded_wait_hook_rejects_bad_poll_counts(lib, polls):
    assert lib.mamba_test_bounded_wait(polls, None) == 2  # MAMBA_ERR_SIZE, nothing launched


def test_ex_entry_validates_like_the_plain_one_and_checks_h0_and_reset(lib):
    """mamba_selective_scan_fwd_ex shares the plain entry's argument checks
    (same status for every bad call) and adds its own: h0 aligned to 4 bytes,
    h0 overlapping y (or part of last_state) and a reset mask overlapping an
    output are MAMBA_ERR_ALIAS.  All return before any CUDA call."""
    cases = [dict(u=None), dict(B=None), dict(batch=-1), dict(dstate=0), dict(io_dtype=9),
             dict(u=P[0] + 1), dict(y=P[0]), dict(last_state=P[2]), dict(batch=0), dict(dim=0)]
    for over in cases:
        kw = dict(GOOD)
        kw.update(over)
        assert abi.raw_scan_fwd_ex(h0=None, reset=None, **kw) == abi.raw_scan_fwd(**kw), over
    ex = lambda **o: abi.raw_scan_fwd_ex(**{**GOOD, "h0": P[10], "reset": P[11], **o})
    assert ex(h0=P[10] + 2) == 4            # misaligned h0
    assert ex(h0=P[8] + 64) == 8            # h0 inside y
    assert ex(h0=P[9] + 16) == 8            # h0 straddles last_state
    assert ex(reset=P[8] + 3) == 8          # reset mask inside y
    assert ex(reset=P[9]) == 8              # reset mask over last_state


Q = [0x7e0000000000 + i * 0x100000000 for i in range(20)]
BGOOD = dict(u=Q[0], delta=Q[1], A_log=Q[2], B=Q[3], C=Q[4], D=Q[5], z=Q[6], delta_bias=Q[7],
             softplus_flag=1, dout=Q[8], du=Q[9], ddelta=Q[10], dz=Q[11], dA_log=Q[12], dB=Q[13],
             dC=Q[14], dD=Q[15], ddelta_bias=Q[16], batch=2, dim=8, seqlen=16, dstate=16,
             io_dtype=abi.MAMBA_BF16, stream=None)


def bwd(**over):
    return abi.raw_scan_bwd(**{**BGOOD, **over})


def test_bwd_entry_validation(lib):
    """mamba_selective_scan_bwd: required pointers, dz iff z, sizes, dstate,
    dtype, alignment, and no output overlapping an input or another output.
    Every case returns before any CUDA call."""
    for name in ("u", "delta", "A_log", "B", "C", "dout", "du", "ddelta", "dA_log", "dB", "dC"):
        assert bwd(**{name: None}) == 1, name                    # MAMBA_ERR_NULL
    assert bwd(dz=None) == 1                                     # z given, dz missing
    assert bwd(batch=-1) == 2 and bwd(seqlen=1 << 45) == 2       # MAMBA_ERR_SIZE
    assert bwd(dstate=0) == 3 and bwd(dstate=257) == 3           # MAMBA_ERR_DSTATE
    assert bwd(io_dtype=4) == 5                                  # MAMBA_ERR_DTYPE
    assert bwd(du=Q[9] + 1) == 4 and bwd(dB=Q[13] + 2) == 4      # MAMBA_ERR_ALIGN
    assert bwd(dout=Q[8] + 2, io_dtype=abi.MAMBA_F32) == 4
    assert bwd(du=Q[0]) == 8                                     # du over u
    assert bwd(ddelta=Q[8] + 64) == 8                            # ddelta inside dout
    assert bwd(dB=Q[3]) == 8                                     # dB over B
    assert bwd(dC=Q[13] + 256) == 8                              # dC inside dB
    assert bwd(dD=Q[12]) == 8                                    # dD over dA_log
    assert bwd(dz=Q[9]) == 8                                     # dz over du
    # optional outputs and a missing z
    assert bwd(dim=0, dD=None, ddelta_bias=None) == 0
    assert bwd(dim=0, z=None, dz=None) == 0
    assert bwd(dim=0, z=None, dz=Q[9]) == 0                      # dz ignored without z


CGOOD = dict(x=Q[0], weight=Q[1], bias=Q[2], initial_state=Q[3], silu_flag=1, out=Q[4],
             final_state=Q[5], batch=2, dim=8, seqlen=16, width=4, io_dtype=abi.MAMBA_BF16,
             stream=None)


def test_conv1d_entry_validation(lib):
    """mamba_causal_conv1d_fwd / _update: every bad call returns before any CUDA call."""
    conv = lambda **o: abi.raw_conv1d_fwd(**{**CGOOD, **o})
    for name in ("x", "weight", "out"):
        assert conv(**{name: None}) == 1, name                       # MAMBA_ERR_NULL
    assert conv(width=0) == 2 and conv(width=9) == 2                 # MAMBA_ERR_SIZE
    assert conv(batch=-1) == 2 and conv(seqlen=1 << 50) == 2
    assert conv(io_dtype=3) == 5                                     # MAMBA_ERR_DTYPE
    assert conv(x=Q[0] + 1) == 4 and conv(weight=Q[1] + 2) == 4      # MAMBA_ERR_ALIGN
    assert conv(out=Q[0]) == 8                                       # out over x
    assert conv(final_state=Q[3]) == 8                               # final over initial state
    assert conv(final_state=Q[4] + 8) == 8                           # final state inside out
    assert conv(dim=0) == 0 and conv(batch=0) == 0                   # nothing to do
    upd_ = lambda **o: abi.raw_conv1d_update(**{**dict(conv_state=Q[6], x=Q[0], weight=Q[1],
                                                       bias=Q[2], silu_flag=1, out=Q[4], batch=2,
                                                       dim=8, width=4, io_dtype=abi.MAMBA_BF16,
                                                       stream=None), **o})
    assert upd_(conv_state=None) == 1 and upd_(x=None) == 1
    assert upd_(width=9) == 2 and upd_(io_dtype=7) == 5
    assert upd_(out=Q[6]) == 8 and upd_(conv_state=Q[0]) == 8
    assert upd_(batch=0) == 0


def test_complex_scan_entry_validation(lib):
    kw = dict(u=Q[0], delta=Q[1], A_log_re=Q[2], A_im=Q[3], B=Q[4], C=Q[5], D=Q[6], z=Q[7],
              delta_bias=Q[8], softplus_flag=1, y=Q[9], last_state=Q[10], batch=2, dim=8,
              seqlen=16, dstate=16, io_dtype=abi.MAMBA_BF16, stream=None)
    cx = lambda **o: abi.raw_scan_complex_fwd(**{**kw, **o})
    for name in ("u", "delta", "A_log_re", "A_im", "B", "C", "y"):
        assert cx(**{name: None}) == 1, name                         # MAMBA_ERR_NULL
    assert cx(batch=-1) == 2 and cx(dstate=0) == 3 and cx(dstate=300) == 3
    assert cx(io_dtype=2) == 5
    assert cx(u=Q[0] + 1) == 4 and cx(last_state=Q[10] + 4) == 4    # state needs 8 bytes
    assert cx(y=Q[0]) == 8 and cx(last_state=Q[4] + 64) == 8         # y over u, state in B
    assert cx(dim=0) == 0 and cx(batch=0) == 0


def test_bwd_ex_entry_validation(lib):
    """mamba_selective_scan_bwd_ex validates like mamba_selective_scan_bwd and
    adds h0 / dh0 alignment and the aliasing of h0, the reset mask and dh0."""
    kw = {**BGOOD, "h0": Q[17], "reset": Q[18], "dh0": Q[19]}
    bx = lambda **o: abi.raw_scan_bwd_ex(**{**kw, **o})
    for over in (dict(u=None), dict(dz=None), dict(dstate=0), dict(io_dtype=4),
                 dict(du=Q[9] + 1), dict(du=Q[0]), dict(dC=Q[13] + 256), dict(dim=0)):
        plain = {k: v for k, v in {**BGOOD, **over}.items()}
        assert bx(**over) == abi.raw_scan_bwd(**plain), over
    assert bx(h0=Q[17] + 2) == 4 and bx(dh0=Q[19] + 2) == 4      # MAMBA_ERR_ALIGN
    assert bx(dh0=Q[17]) == 8                                    # dh0 over h0
    assert bx(dh0=Q[12]) == 8                                    # dh0 over dA_log
    assert bx(du=Q[18]) == 8                                     # du over the reset mask
    assert bx(dlast_state=Q[17] + 2) == 4                        # MAMBA_ERR_ALIGN
    assert bx(dlast_state=Q[19]) == 8                            # dh0 over dlast_state
    assert bx(dlast_state=Q[12]) == 8                            # dlast_state under dA_log
    assert bx(dim=0, h0=None, reset=None, dh0=None) == 0
