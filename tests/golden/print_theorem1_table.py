"""Prints the Theorem 1 diagnostic table: the distribution of
RMS_exact * inv_rms (oracle, c = 1) on the first 16,384 rows of each
synthetic workload.  Calls only the oracle and the seeded input generator.

    python tests/golden/print_theorem1_table.py
"""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

from mx_scale_reusing_gb300 import synth  # noqa: E402  (seeded inputs only)
from oracle import theorem1  # noqa: E402

ROWS_CAP = 16384


def main():
    print("| workload | fmt | p | rows | mean | std | cv | min | max |")
    print("|---|---|---|---|---|---|---|---|---|")
    for name, w in synth.WORKLOADS.items():
        x = synth.make_activations(w, rows=min(w.T, ROWS_CAP))
        for p in (1, 2):
            s = theorem1.summary(x, p, w.fmt)
            print(f"| {name} | {w.fmt} | {p} | {s['rows']} | {s['mean']:.2f} | {s['std']:.2f} | {s['cv']:.4f} | "
                  f"{s['min']:.2f} | {s['max']:.2f} |")


if __name__ == "__main__":
    main()
