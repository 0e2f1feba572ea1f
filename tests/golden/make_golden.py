"""Writes the oracle regression fixtures in this folder.

Calls only ``oracle/`` (on inputs from ``workloads/``). The fixtures are not
pins: they record what the oracle computed when it was last checked against
its pins, so that a later change to its arithmetic shows up as a diff that
must name its reason. Run from the repository root:

    python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
import workloads as W  # noqa: E402

CASES = {
    "decode_b1_l1_t1": W.WORKLOADS["decode_b1_l1_t1"],
    "verify_b2_l1_t3_ragged": W.WORKLOADS["verify_b16_l36_t8_ragged"].scaled(B=2, L=1, T=3),
}
# Fixed sample points: (t, flat y index) and (head, i, j).
Y_POINTS = [(0, 0), (0, 127), (0, 128), (0, 3071), (0, 6143)]
S_POINTS = [(0, 0, 0), (5, 17, 99), (23, 127, 0), (47, 127, 127)]


def digest(case):
    h = W.host_inputs(case, threads=4)
    y, st, cs = oracle.gdn_decode(h["qkv"], h["z"], h["alpha"], h["beta"], h["dt"], h["ssm_a"], h["conv_w"],
                                  h["ssm_norm"], h["conv_state"], h["state"], seq_len=h["seq_len"])
    lines = []
    for b in range(case.B):
        yv = np.nan_to_num(y[b, 0], nan=0.0)
        lines.append(f"b{b} y_sum {yv.sum():.17g}")
        lines.append(f"b{b} y_sumsq {(yv * yv).sum():.17g}")
        lines.append(f"b{b} state_sum {st[b, 0].sum():.17g}")
        lines.append(f"b{b} state_sumsq {(st[b, 0] ** 2).sum():.17g}")
        lines.append(f"b{b} conv_state_sum {cs[b, 0].astype(np.float64).sum():.17g}")
        for t, i in Y_POINTS:
            lines.append(f"b{b} y[{t}][{i}] {y[b, 0, t, i]:.17g}")
        for hh, i, j in S_POINTS:
            lines.append(f"b{b} state[{hh}][{i}][{j}] {st[b, 0, hh, i, j]:.17g}")
    return lines


def main():
    for name, case in CASES.items():
        path = os.path.join(HERE, f"oracle_{name}.txt")
        with open(path, "w") as f:
            f.write(f"# oracle regression digest for {name} (written by tests/golden/make_golden.py)\n")
            f.write("\n".join(digest(case)) + "\n")
        print("wrote", path)


if __name__ == "__main__":
    main()
