"""The seeded synthetic workloads are what they were: the sha256 of each
one's bf16 bits (the tiny workload whole, the first 1024 rows of the
others) against tests/golden/workload_digests.txt, which
tests/golden/write_workload_digests.py wrote from the generator alone.  A
change of the generator or of numpy's random streams fails here, not as a
silent change of every parity and benchmark input."""
import hashlib
import os

import numpy as np
import pytest

from mx_scale_reusing_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "workload_digests.txt")


def stored():
    out = {}
    for line in open(GOLDEN):
        if line.strip() and not line.startswith("#"):
            name, rows, h = line.split()
            out[name] = (int(rows), h)
    return out


def test_every_workload_has_a_digest():
    assert set(stored()) == set(synth.WORKLOADS)


@pytest.mark.parametrize("name", sorted(synth.WORKLOADS))
def test_workload_digest(name):
    rows, h = stored()[name]
    w = synth.WORKLOADS[name]
    assert rows == min(w.T, 1024)
    xb = synth.make_activations(w, rows=rows)
    assert hashlib.sha256(xb.astype("<u2").tobytes()).hexdigest() == h


def test_prefix_is_independent_of_rows_requested():
    """The first rows do not depend on how many rows are asked for, so the
    stored prefix digests describe the full-size inputs too."""
    w = synth.WORKLOADS["llama3_1b_32768x2048"]
    a = synth.make_activations(w, rows=1500)
    b = synth.make_activations(w, rows=1024)
    assert np.array_equal(a[:1024], b)
