"""Write the stored expected outputs under tests/golden/ from the fp64 oracle.

Only the oracle and the seeded input generator are used; nothing here touches
the CUDA library.  Run from the repository root:

    python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from selective_state_space_140_b300 import workloads  # noqa: E402


def tiny_f32():
    cfg = workloads.SCAN_CONFIGS["tiny_f32"]
    x = workloads.make_config_inputs(cfg)
    f = workloads.to_f64
    y, hL, _ = oracle.selective_scan(f(x["u"]), f(x["delta"]), f(x["A_log"]), f(x["B"]), f(x["C"]),
                                     D=f(x["D"]), z=f(x["z"]), delta_bias=f(x["delta_bias"]),
                                     softplus=True, nthreads=1)
    path = os.path.join(HERE, "tiny_f32.txt")
    with open(path, "w") as fh:
        fh.write("# fp64 oracle outputs for the tiny fp32 scan (batch 1, 16 channels, L=64, N=4,\n")
        fh.write("# seed 0, inputs from selective_state_space_140_b300.workloads).  Written by\n")
        fh.write("# tests/golden/make_golden.py; the pages print no worked example, so this\n")
        fh.write("# fixture is the oracle's, not the pages'.\n")
        fh.write(f"# y {y.size}\n")
        np.savetxt(fh, y.reshape(-1), fmt="%.17g")
        fh.write(f"# last_state {hL.size}\n")
        np.savetxt(fh, hL.reshape(-1), fmt="%.17g")
    return path


if __name__ == "__main__":
    print(tiny_f32())
