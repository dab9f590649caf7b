"""Write tests/golden/workload_digests.txt: the sha256 of each seeded
synthetic workload's bf16 bit patterns (little-endian uint16, row-major) --
the whole tiny workload, and the first 1024 rows of each other one.  Calls
only the input generator (mx_scale_reusing_gb300.synth); the oracle and the
CUDA path play no part.  The CPU test test_synth_digests.py recomputes these
so that a change of the generator, or of numpy's random streams, shows up.

    python tests/golden/write_workload_digests.py
"""
import hashlib
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

from mx_scale_reusing_gb300 import synth  # noqa: E402

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "workload_digests.txt")
ROWS = 1024


def digest_rows(name: str):
    w = synth.WORKLOADS[name]
    rows = w.T if w.T <= ROWS else ROWS
    xb = synth.make_activations(w, rows=rows)
    return rows, hashlib.sha256(xb.astype("<u2").tobytes()).hexdigest()


def main():
    lines = ["# workload  rows_hashed  sha256 of the bf16 bits (uint16 little-endian, row-major)"]
    for name in synth.WORKLOADS:
        rows, h = digest_rows(name)
        lines.append(f"{name} {rows} {h}")
    with open(OUT, "w") as f:
        f.write("\n".join(lines) + "\n")
    print(OUT)


if __name__ == "__main__":
    main()
