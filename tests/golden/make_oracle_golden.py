"""Write tests/golden/tiny_oracle.json: oracle outputs for the seeded tiny workload.

These are regression values for the oracle itself (produced only by calling ``oracle``), so a
later change to the oracle's arithmetic shows up as a diff of this file.  They are not pins:
the pins are the closed forms, brute force and library checks in tests/test_oracle.py.

Run from the repository root:  python tests/golden/make_oracle_golden.py
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from context_math_non_b300.inputs import WORKLOADS, draw_qkv  # noqa: E402

ROWS = [0, 1, 63, 64, 127, 128, 200, 255]


def main():
    q, k, v = draw_qkv(WORKLOADS["tiny"])
    o, lse = oracle.attention(q, k, v)
    op, lp = oracle.attention_chunked(q, k, v, 4)
    out = {
        "workload": "tiny: B=1 H=2 S=256 D=64, bf16-rounded N(0,1) draws, seed 1000",
        "rows": ROWS,
        "o_head0_cols0to3": [[float(x) for x in o[0, 0, r, :4]] for r in ROWS],
        "lse": [[float(lse[0, h, r]) for r in ROWS] for h in range(2)],
        "lse_parts_P4_head1": [[float(lp[c, 0, 1, r]) for r in ROWS] for c in range(4)],
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_oracle.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
