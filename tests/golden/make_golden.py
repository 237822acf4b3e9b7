"""Writes tests/golden/tile_counts.json by calling only the oracle.

Run from the repository root:  python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)
from oracle import FULL, PARTIAL, SKIP, tile_classes  # noqa: E402

CASES = [
    # prefill of a 32,768-token sequence, 100-token prefix, 4,096 window
    dict(name="prefill_32768_P100_W4096", S=32768, P=100, W=4096, BM=128, BN=128),
    # truncated-backprop forward: 8,192 tokens, 256-token prefix, 2,048 window
    dict(name="train_8192_P256_W2048", S=8192, P=256, W=2048, BM=128, BN=128),
    # ragged tail and odd shapes
    dict(name="ragged_1000_P37_W300", S=1000, P=37, W=300, BM=128, BN=128),
]


def main():
    out = []
    for c in CASES:
        pos = np.arange(c["S"])
        cls = tile_classes(pos, pos, c["P"], c["W"], c["BM"], c["BN"])
        counts = [int((cls == k).sum()) for k in (SKIP, PARTIAL, FULL)]
        out.append(dict(c, skip_partial_full=counts))
        print(c["name"], counts)
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tile_counts.json")
    with open(path, "w") as f:
        json.dump({"written_by": "tests/golden/make_golden.py (oracle.tile_classes)",
                   "cases": out}, f, indent=1)


if __name__ == "__main__":
    main()
