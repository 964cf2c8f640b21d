"""Pins of the oracle's smooth gate with a live threshold.

"Model casting: compute the gate, then skip most of the FFN" (sections on
SiLU and on thresholding small values): SiLU(z) = z sigmoid(z) is never
exactly zero, so a unit is treated as dead when |A(z)| <= epsilon, which turns
the exact skip into an approximation with an error budget.  The oracle keeps
unit i iff |A(z_i)| > thr.  Pins: thr = 0 is the dense SwiGLU product computed
with torch's SiLU; a threshold above every |A| gives y = 0; the error against
thr = 0 stays within the closed-form bound thr * sum_i |W2[m,i]| |u_i|; the
live count falls monotonically with thr; gate-first equals dense; for ReLU and
R-S+ thr = 0 is the plain definition.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from activation_sparse_gated_gb300 import synthetic as syn

F32, BF16, RELU, RSP, SILU = oracle.F32, oracle.BF16, oracle.RELU, oracle.RSP, oracle.SILU


def layer(D, H, B, seed):
    rng = np.random.default_rng(seed)
    W1 = (rng.standard_normal((H, D)) / math.sqrt(D)).astype(np.float32)
    W3 = (rng.standard_normal((H, D)) / math.sqrt(D)).astype(np.float32)
    W2 = (rng.standard_normal((D, H)) / math.sqrt(H)).astype(np.float32)
    x = rng.standard_normal((B, D)).astype(np.float32)
    return W1, W3, W2, x


def swiglu_torch(W1, W3, W2, x):
    d = [torch.from_numpy(a.astype(np.float64)) for a in (W1, W3, W2, x)]
    return ((torch.nn.functional.silu(d[3] @ d[0].T) * (d[3] @ d[1].T)) @ d[2].T).numpy()


def test_silu_hand_worked():
    """D = 2, H = 3: z = (1, -1, 0) exactly; SiLU(0) = 0 is the only dead unit."""
    W1 = np.array([[1.0, 0.0], [-1.0, 0.0], [0.0, 0.0]], dtype=np.float32)
    W3 = np.array([[2.0, 0.0], [0.0, 3.0], [5.0, 5.0]], dtype=np.float32)
    W2 = np.array([[1.0, 1.0, 7.0], [0.0, -1.0, 7.0]], dtype=np.float32)
    x = np.array([[1.0, 1.0]], dtype=np.float32)
    y, z, n = oracle.ffn_dense_ex(2, 3, 0, SILU, F32, 0, W1, None, None, W3, W2, x)
    s1 = 1.0 / (1.0 + math.exp(-1.0))
    a0, a1 = s1, -(1.0 - s1)  # SiLU(1) = sigmoid(1); SiLU(-1) = -sigmoid(-1)
    np.testing.assert_allclose(y[0], [a0 * 2 + a1 * 3, -a1 * 3], rtol=1e-15)
    assert n[0] == 2


@pytest.mark.parametrize("dtype", [F32, BF16])
def test_threshold_zero_is_dense_swiglu(dtype):
    D, H, B = 48, 130, 4
    W1, W3, W2, x = layer(D, H, B, 1)
    if dtype == BF16:  # the values the oracle sees: bf16-rounded
        rt = lambda a: torch.from_numpy(a).bfloat16().float().numpy()  # noqa: E731
        W1, W3, W2, x = rt(W1), rt(W3), rt(W2), rt(x)
        view = lambda a: syn.oracle_view(torch.from_numpy(a).bfloat16())  # noqa: E731
    else:
        view = lambda a: a  # noqa: E731
    y, _, n = oracle.ffn_dense_ex(D, H, 0, SILU, dtype, 0, view(W1), None, None, view(W3), view(W2), view(x))
    np.testing.assert_allclose(y, swiglu_torch(W1, W3, W2, x), rtol=1e-12, atol=1e-12)
    assert (n == H).all()


def test_threshold_above_every_activation_gives_zero():
    D, H, B = 32, 90, 3
    W1, W3, W2, x = layer(D, H, B, 2)
    y, _, n = oracle.ffn_dense_ex(D, H, 0, SILU, F32, 0, W1, None, None, W3, W2, x, thr=1e6)
    assert (y == 0).all() and (n == 0).all()


def test_threshold_error_bound_and_monotone_count():
    D, H, B = 40, 200, 5
    W1, W3, W2, x = layer(D, H, B, 3)
    y0, _, _ = oracle.ffn_dense_ex(D, H, 0, SILU, F32, 0, W1, None, None, W3, W2, x)
    u = x.astype(np.float64) @ W3.astype(np.float64).T
    absW2 = np.abs(W2.astype(np.float64))
    prev = None
    for thr in (0.01, 0.05, 0.1, 0.2, 0.4):
        y, _, n = oracle.ffn_dense_ex(D, H, 0, SILU, F32, 0, W1, None, None, W3, W2, x, thr=thr)
        assert (np.abs(y - y0) <= thr * (np.abs(u) @ absW2.T) + 1e-12).all()
        if prev is not None:
            assert (n <= prev).all()
        prev = n
    assert prev.max() < H  # the thresholds really drop units


@pytest.mark.parametrize("act", [RELU, RSP])
def test_zero_threshold_is_the_plain_definition(act):
    D, H, B = 24, 60, 3
    W1, W3, W2, x = layer(D, H, B, 4)
    y1, z1, n1 = oracle.ffn_dense(D, H, 0, act, F32, W1, None, None, W3, W2, x)
    y2, z2, n2 = oracle.ffn_dense_ex(D, H, 0, act, F32, 0, W1, None, None, W3, W2, x, thr=0.0)
    assert np.array_equal(y1, y2) and np.array_equal(z1, z2) and np.array_equal(n1, n2)


@pytest.mark.parametrize("act", [SILU, RSP, RELU])
@pytest.mark.parametrize("thr", [0.0, 0.05, 0.3])
def test_gate_first_equals_dense_with_threshold(act, thr):
    D, H, r, B = 32, 96, 8, 3
    rng = np.random.default_rng(5)
    U = (rng.standard_normal((H, r)) / math.sqrt(r)).astype(np.float32)
    V = (rng.standard_normal((r, D)) / math.sqrt(D)).astype(np.float32)
    _, W3, W2, x = layer(D, H, B, 6)
    for flags, gate in ((0, (layer(D, H, B, 7)[0], None, None, 0)), (oracle.FLAG_DOUBLE_ACT, (None, U, V, r))):
        W1, Ug, Vg, rr = gate
        y_d, z, n_d = oracle.ffn_dense_ex(D, H, rr, act, F32, flags, W1, Ug, Vg, W3, W2, x, thr=thr)
        y_g, idx, n_g = oracle.ffn_gate_first_ex(D, H, rr, act, F32, flags, W1, Ug, Vg, W3, W2, x, thr=thr)
        np.testing.assert_allclose(y_g, y_d, rtol=1e-12, atol=1e-13)
        assert np.array_equal(n_d, n_g)
