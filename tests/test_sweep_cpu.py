"""Host logic of the D = 4096 sparsity x batch sweep (bench.py --sweep).

The sweep builds each gate's weight sets once and sets a sparsity by
rewriting the bias column with -Phi^{-1}(s).  That must give exactly the
weights the generator produces for that sparsity, bit for bit, for both
gates, so that every point of the sweep runs the workload it names.
"""
import os
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from activation_sparse_gated_gb300 import synthetic as syn  # noqa: E402

NAME = "sweep-bf16-D4096-H14336"


@pytest.mark.parametrize("gate", ["standard", "lopa"])
def test_bias_rewrite_equals_generating_at_that_sparsity(gate):
    base = syn.workload_layers(NAME, sets=1, gate=gate, s=0.9)[0]
    for s in (0.5, 0.75, 0.95):
        want = syn.workload_layers(NAME, sets=1, gate=gate, s=s)[0]
        got = bench.set_sparsity(base, s)
        for k in ("W1", "U", "V", "W3", "W2"):
            a, b = getattr(got, k), getattr(want, k)
            assert (a is None) == (b is None), k
            if a is not None:
                assert torch.equal(a.view(torch.int16), b.view(torch.int16)), (gate, s, k)


def test_sweep_grid_is_the_stated_one():
    w = syn.WORKLOADS[NAME]
    assert w["s"] == (0.5, 0.75, 0.9, 0.95) and w["B"] == (1, 8, 32, 128)
    assert (w["D"], w["H"], w["r"], w["Hp"]) == (4096, 14336, 640, 19649)
    # H' = D (3H - r) / (r + 2D) rounded to the nearest integer (iso-parameter width)
    assert w["Hp"] == round(4096 * (3 * 14336 - 640) / (640 + 2 * 4096))
