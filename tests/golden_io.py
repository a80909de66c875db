"""Read the stored expected values under tests/golden/."""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load_tiny_f32():
    """Return (y [1,16,64], last_state [1,16,4]) from tests/golden/tiny_f32.txt."""
    sections, cur = {}, None
    with open(os.path.join(GOLDEN, "tiny_f32.txt")) as fh:
        for line in fh:
            if line.startswith("# y ") or line.startswith("# last_state "):
                cur = line.split()[1]
                sections[cur] = []
            elif line.startswith("#") or not line.strip():
                continue
            else:
                sections[cur].append(float(line))
    return (np.array(sections["y"]).reshape(1, 16, 64),
            np.array(sections["last_state"]).reshape(1, 16, 4))
