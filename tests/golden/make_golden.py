"""Writes tests/golden/tiny_oracle_digest.txt from the oracle alone.

The pages print no worked example of the KDA layer, so the only stored
values here are the oracle's own outputs on the seeded tiny workload
(1 sequence, T=64, H=2, dk=dv=32, conv 4, fp32, safe gate lb=-5, zero
states), kept as a regression guard: a later change to the oracle's
arithmetic must say which passage justifies it and regenerate this file.

    python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from linear_attention_serving_kda_gb300 import workloads  # noqa: E402

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_oracle_digest.txt")


def digest():
    wl = workloads.tiny_oracle_case()
    res = oracle.forward(wl, threads=1)
    lines = ["# oracle digest of the seeded tiny workload; written by make_golden.py"]
    for key in ("out", "rec_state", "conv_state"):
        a = res[key].ravel()
        lines.append(f"{key} sum {float(a.sum())!r} l2 {float(np.linalg.norm(a))!r}")
        idx = np.linspace(0, a.size - 1, 8).astype(int)
        lines.append(f"{key} samples " + " ".join(f"{i}:{float(a[i])!r}" for i in idx))
    return "\n".join(lines) + "\n"


if __name__ == "__main__":
    with open(OUT, "w") as fh:
        fh.write(digest())
    print(OUT)
