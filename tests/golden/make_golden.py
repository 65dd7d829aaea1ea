"""Write tiny_fp32_oracle.txt: sampled oracle outputs of the tiny fp32 workload.

Calls only the CPU oracle and the seeded input generator.  The file is a
regression anchor: a later change to the oracle's arithmetic shows up as a
mismatch and has to be justified by the definition it follows.

    python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from linear_attention_speculative_gb300 import workloads as wk  # noqa: E402


def main():
    out = oracle.verify(wk.make_inputs(wk.TINY), wk.TINY.gate)
    rng = np.random.default_rng(2024)
    lines = ["# oracle outputs of the tiny fp32 workload (N=2 T=2 H=HV=2 K=V=32, softplus, seed 0)",
             "# written by tests/golden/make_golden.py; key  index  value"]
    for key in ("o", "inter_ssm", "conv_snapshots", "conv_state"):
        arr = out[key]
        for _ in range(12):
            idx = tuple(int(rng.integers(0, d)) for d in arr.shape)
            lines.append(f"{key} {','.join(map(str, idx))} {float(arr[idx])!r}")
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_fp32_oracle.txt")
    with open(path, "w") as f:
        f.write("\n".join(lines) + "\n")
    print("wrote", path)


if __name__ == "__main__":
    main()
