"""The algorithmic counts behind bench.py's roofline figures (CPU only).

The byte and exponential counts per launch are fixed by the shapes: every
input read once and every output written once, one exponential per state
update plus the per-element softplus and gate.  These pin the counts for the
benchmark workloads to values worked out by hand from those definitions.
"""
import bench
from selective_state_space_140_b300 import workloads


def test_forward_counts_of_the_benchmark_layer():
    c = bench.scan_counts(workloads.SCAN_CONFIGS["mamba1p4b_bf16"])
    B, D, L, N = 4, 4096, 4096, 16
    elems = B * D * L
    assert c["updates"] == elems * N == 1_073_741_824
    # u, delta, z read and y written (2 bytes each); B, C read once; the fp32
    # final state written; A_log read; D and the bias read
    assert c["bytes"] == 8 * elems + 2 * 2 * B * L * N + 4 * B * D * N + 4 * D * N + 8 * D
    assert c["bytes"] == 539_262_976
    assert c["exps"] == elems * (N + 2) == 1_207_959_552


def test_forward_counts_of_the_other_layers():
    assert bench.scan_counts(workloads.SCAN_CONFIGS["mamba130m_bf16"])["bytes"] == 203_272_192
    assert bench.scan_counts(workloads.SCAN_CONFIGS["dna_long_bf16"])["bytes"] == 1_619_210_240
    assert bench.scan_counts(workloads.SCAN_CONFIGS["large_state_f32"])["bytes"] == 546_848_768


def test_backward_counts_of_the_benchmark_layer():
    c = bench.bwd_counts(workloads.SCAN_CONFIGS["mamba1p4b_bf16"])
    B, D, L, N = 4, 4096, 4096, 16
    elems = B * D * L
    # u, delta, z, dout read and du, ddelta, dz written (bf16); B, C read
    # (bf16) and dB, dC written (fp32); A_log read and its gradient written;
    # D and bias read and their gradients written
    assert c["bytes"] == 14 * elems + 2 * 2 * B * L * N + 2 * 4 * B * L * N + 8 * D * N + 16 * D
    assert c["bytes"] == 943_259_648
    assert c["exps"] == elems * (3 * N + 3)


def test_decode_counts():
    c = bench.decode_counts(workloads.DECODE_CONFIGS["decode_bf16"])
    B, D, N = 256, 4096, 16
    # the fp32 state read and written, x, dt, z read and out written (bf16),
    # B and C read, A_log, D and the bias read
    assert c["bytes"] == 8 * B * D * N + 4 * B * D * 2 + 2 * B * N * 2 + 4 * D * N + 8 * D
    assert c["bytes"] == 142_917_632
    assert c["updates"] == B * D * N


def test_launch_count_mirrors_the_split_planner():
    """One kernel per step when the grid fills the GPU; summary, carry and full
    pass (3) for few chains and a long sequence, on a 148-SM B300."""
    cfgs = workloads.SCAN_CONFIGS
    assert bench.launches_per_step(cfgs["mamba1p4b_bf16"], 148) == 1
    assert bench.launches_per_step(cfgs["mamba130m_bf16"], 148) == 1
    assert bench.launches_per_step(cfgs["dna_long_bf16"], 148) == 3
    assert bench.launches_per_step(cfgs["large_state_f32"], 148) == 1
