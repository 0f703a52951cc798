"""Write the stored oracle values under tests/golden/ (calls only oracle/ and the
seeded input generators; run from the repository root:
``python tests/golden/make_golden.py``)."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import oracle  # noqa: E402
from workloads import TINY, make_inputs  # noqa: E402

ROWS = [0, 1, 17, 128, 200, 255]
COLS = [0, 1, 31, 63]


def tiny_forward_sample():
    q, k, v, _, _ = make_inputs(TINY)
    o, lse = oracle.forward(q, k, v, TINY.scale, rows=np.array(ROWS))
    return {
        "workload": TINY.describe(),
        "source": "oracle.forward on workloads.make_inputs(TINY) (seed 0)",
        "rows": ROWS,
        "cols": COLS,
        "o": [[[float(o[0, h, r, c]) for c in COLS] for r in range(len(ROWS))]
              for h in range(TINY.Hq)],
        "lse": [[float(lse[0, h, r]) for r in range(len(ROWS))] for h in range(TINY.Hq)],
    }


if __name__ == "__main__":
    out = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_forward_sample.json")
    with open(out, "w") as f:
        json.dump(tiny_forward_sample(), f, indent=1)
    print("wrote", out)
