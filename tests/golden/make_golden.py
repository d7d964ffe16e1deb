"""Writes the oracle regression fixture ``oracle_regression.json``.

The pages that describe the method print no worked attention values, so
nothing in this folder comes from them.  This fixture only freezes the
oracle's own fp64 output for one tiny seeded input (stored with it as bf16
bit patterns), so that a later change to the oracle, or a different host
compiler or C library, that moves any result by more than rounding is
noticed.  It calls the oracle and nothing else.

Run from the repository root:  python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402


def main():
    rng = np.random.default_rng(2024)
    B, H, N, D = 1, 2, 9, 8
    # bf16 bit patterns of small dyadic values: exact, and independent of any
    # floating-point rounding in the generator
    def draw():
        vals = rng.integers(-24, 25, size=(B, H, N, D)).astype(np.float32) / 8.0
        return (vals.view(np.uint32) >> 16).astype(np.uint16)
    q, k, v = draw(), draw(), draw()
    cases = []
    for causal in (False, True):
        O, L = oracle.attn_fwd(q, k, v, causal, 0.35)
        cases.append({"causal": causal, "scale": 0.35,
                      "O": [repr(float(x)) for x in O.ravel()],
                      "LSE": [repr(float(x)) for x in L.ravel()]})
    doc = {"shape": [B, H, N, D],
           "q_bits": [int(x) for x in q.ravel()],
           "k_bits": [int(x) for x in k.ravel()],
           "v_bits": [int(x) for x in v.ravel()],
           "cases": cases}
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_regression.json")
    with open(path, "w") as f:
        json.dump(doc, f, indent=0)
        f.write("\n")
    print("wrote", path)


if __name__ == "__main__":
    main()
