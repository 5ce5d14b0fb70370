"""Write the oracle's outputs for a few tiny seeded workloads to ``oracle_tiny.json``.

The attention pages print no numeric worked example of O or LSE, so the stored
values here come from the fp64 oracle (and only from it): they freeze its
results so that any later change to its arithmetic shows up as a test failure
and has to be justified.  Inputs follow ``attn_inputs.make_qkv`` on the CPU.

Run from the repository root:  python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import attn_inputs  # noqa: E402
import oracle  # noqa: E402

CASES = [
    # B, H, Nq, Nk, d, dtype, causal, seed
    (1, 1, 5, 5, 4, "f16", True, 11),
    (1, 2, 3, 7, 8, "bf16", False, 12),
    (1, 1, 6, 3, 4, "bf16", True, 13),  # Nq > Nk: three fully masked rows
    (2, 1, 1, 9, 16, "bf16", False, 14),  # one query row (decode shape)
]


def compute(case):
    B, H, Nq, Nk, d, dt, causal, seed = case
    q, k, v = attn_inputs.make_qkv(B, H, Nq, Nk, d, dt, seed, "cpu")
    o, lse = oracle.attention(q, k, v, causal, 1.0 / d ** 0.5)
    return o, lse


def main():
    out = []
    for case in CASES:
        o, lse = compute(case)
        out.append({"case": list(case), "o": [repr(float(x)) for x in o.ravel()],
                    "lse": [repr(float(x)) for x in lse.ravel()]})
    with open(os.path.join(HERE, "oracle_tiny.json"), "w") as f:
        json.dump({"source": "tests/golden/make_golden.py (fp64 oracle)", "cases": out}, f, indent=1)


if __name__ == "__main__":
    main()
