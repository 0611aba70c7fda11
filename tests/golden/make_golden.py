"""Writes tests/golden/codebooks.json from the oracle alone (Lloyd-Max codebooks, fp64).

Run from the repository root:  python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from oracle import lloyd_max_codebook  # noqa: E402


def main():
    out = {"source": "oracle.lloyd_max_codebook (fp64, closed-form cell integrals)", "codebooks": {}}
    for d in (64, 128, 256):
        for b in (1, 2, 3, 4):
            c, t = lloyd_max_codebook(d, b)
            out["codebooks"][f"d{d}_b{b}"] = {"centroids": [float(x) for x in c], "boundaries": [float(x) for x in t]}
    with open(os.path.join(HERE, "codebooks.json"), "w") as f:
        json.dump(out, f, indent=1)


if __name__ == "__main__":
    main()
