"""Writes the stored expected values under tests/golden/ by calling the oracle only.

Run from the repository root: ``python tests/golden/make_golden.py``.
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

from oracle import mla_oracle as O  # noqa: E402


def rope_worked_example():
    # Partial interleaved RoPE ("glm52-mla.ts", partialInterleavedRopeMlx): d = 4 of a
    # width-6 feature axis, theta = 1e4, one token at position 1.  The pair angles are
    # 1 rad and f32(0.01) rad; the last two features are the kept tail.
    x = [0.5, -1.25, 2.0, 0.75, 3.0, -4.0]
    y = O.rope_partial_interleaved(np.array(x).reshape(1, 1, 1, 6), 1, 4, 10000.0)
    return {
        "source": "glm52-mla.ts (mlx-bun 0.0.11 -> 0.0.13), partialInterleavedRopeMlx",
        "input": x, "position": 1, "rotary_dims": 4, "theta": 10000.0,
        "expected": [float(v) for v in y.reshape(-1)],
    }


if __name__ == "__main__":
    with open(os.path.join(HERE, "rope_worked_example.json"), "w") as f:
        json.dump(rope_worked_example(), f, indent=1)
        f.write("\n")
