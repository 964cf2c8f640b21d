"""Pins of the oracle's full low-rank gate ("LoPA Gating: moving the ceiling").

The pages' full form is W1(x) = Gx + U RMSNorm(Vx) with G the tiled identity
((Gx)_i = x_{i mod D}, appendix Figure 6 (c)) and the activation applied to
both W1x and W3x ("double activation").  Each pin ties the flagged oracle to
something it does not compute itself: the already-pinned standard-gate oracle
on a materialised gate matrix, an exact identity of ReLU, an invariance of
RMSNorm, or a hand-worked value.
"""
import math

import numpy as np
import pytest

import oracle

F32, RELU, RSP = oracle.F32, oracle.RELU, oracle.RSP
TG, RN, DA = oracle.FLAG_TILED_G, oracle.FLAG_RMSNORM, oracle.FLAG_DOUBLE_ACT


def f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def tiled_identity(H, D):
    T = np.zeros((H, D), dtype=np.float32)
    T[np.arange(H), np.arange(H) % D] = 1.0
    return T


def small_int_lowrank(D, H, r, seed):
    """U, V with small integer entries: U V + T is exact in fp32 (and bf16)."""
    rng = np.random.default_rng(seed)
    U = rng.integers(-2, 3, size=(H, r)).astype(np.float32)
    V = rng.integers(-1, 2, size=(r, D)).astype(np.float32)
    return U, V


def dense_parts(D, H, seed):
    rng = np.random.default_rng(seed)
    W3 = f32(rng.standard_normal((H, D)) / math.sqrt(D))
    W2 = f32(rng.standard_normal((D, H)) / math.sqrt(H))
    return W3, W2


@pytest.mark.parametrize("act", [RELU, RSP])
@pytest.mark.parametrize("extra", [0, DA])
def test_tiled_g_equals_materialised_gate(act, extra):
    """Gx + U(Vx) with exact integer U V is the standard gate with W1 = T + U V."""
    D, H, r, B = 8, 21, 4, 5
    U, V = small_int_lowrank(D, H, r, 1)
    W3, W2 = dense_parts(D, H, 2)
    x = f32(np.random.default_rng(3).standard_normal((B, D)))
    W1 = f32(tiled_identity(H, D) + U @ V)
    y_lr, z_lr, n_lr = oracle.ffn_dense_ex(D, H, r, act, F32, TG | extra, None, f32(U), f32(V), W3, W2, x)
    if extra:
        y_st, z_st, n_st = oracle.ffn_dense_ex(D, H, 0, act, F32, extra, W1, None, None, W3, W2, x)
    else:
        y_st, z_st, n_st = oracle.ffn_dense(D, H, 0, act, F32, W1, None, None, W3, W2, x)
    np.testing.assert_allclose(z_lr, z_st, rtol=0, atol=1e-12)
    np.testing.assert_allclose(y_lr, y_st, rtol=1e-12, atol=1e-12)
    assert np.array_equal(n_lr, n_st)


def test_tiled_g_alone_when_v_is_zero():
    """V = 0: RMSNorm(0) = 0 (eps keeps it finite), so z_i = x_{i mod D} exactly."""
    D, H, r = 6, 20, 3
    U, _ = small_int_lowrank(D, H, r, 4)
    V = np.zeros((r, D), dtype=np.float32)
    W3, W2 = dense_parts(D, H, 5)
    x = f32(np.random.default_rng(6).standard_normal((2, D)))
    _, z, _ = oracle.ffn_dense_ex(D, H, r, RELU, F32, TG | RN, None, f32(U), V, W3, W2, x)
    assert np.array_equal(z, x[:, np.arange(H) % D].astype(np.float64))


def test_rmsnorm_hand_worked():
    """t = V x = (3, 4): RMS = sqrt(12.5 + eps); z = U t / RMS."""
    D, H, r = 2, 4, 2
    V = f32([[3.0, 0.0], [0.0, 4.0]])
    U = f32([[1.0, 0.0], [0.0, 1.0], [1.0, 1.0], [-1.0, 0.0]])
    x = f32([[1.0, 1.0]])
    W3, W2 = dense_parts(D, H, 7)
    _, z, n = oracle.ffn_dense_ex(D, H, r, RELU, F32, RN, None, U, V, W3, W2, x, eps=1e-6)
    s = math.sqrt(12.5 + 1e-6)
    np.testing.assert_allclose(z[0], [3 / s, 4 / s, 7 / s, -3 / s], rtol=1e-14)
    assert n[0] == 3


def test_rmsnorm_scale_invariances():
    """RMSNorm(c v) = RMSNorm(v): scaling V leaves y unchanged; scaling x (G off)
    leaves z unchanged, so y -- linear in W3 x -- scales by the same factor."""
    D, H, r, B = 16, 40, 8, 3
    rng = np.random.default_rng(8)
    U = f32(rng.standard_normal((H, r)))
    V = f32(rng.standard_normal((r, D)))
    W3, W2 = dense_parts(D, H, 9)
    x = f32(rng.standard_normal((B, D)))
    y1, z1, _ = oracle.ffn_dense_ex(D, H, r, RELU, F32, RN, None, U, V, W3, W2, x, eps=0.0)
    y2, z2, _ = oracle.ffn_dense_ex(D, H, r, RELU, F32, RN, None, U, f32(4 * V), W3, W2, x, eps=0.0)
    np.testing.assert_allclose(y2, y1, rtol=1e-12, atol=1e-14)
    y3, z3, _ = oracle.ffn_dense_ex(D, H, r, RELU, F32, RN, None, U, V, W3, W2, f32(2 * x), eps=0.0)
    np.testing.assert_allclose(z3, z1, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(y3, 2 * y1, rtol=1e-12, atol=1e-14)
    # without RMSNorm the gate scales with x as well, so y scales by 4 under ReLU
    y4, _, _ = oracle.ffn_dense_ex(D, H, r, RELU, F32, 0, None, U, V, W3, W2, x)
    y5, _, _ = oracle.ffn_dense_ex(D, H, r, RELU, F32, 0, None, U, V, W3, W2, f32(2 * x))
    np.testing.assert_allclose(y5, 4 * y4, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("r", [0, 6])
def test_double_activation_relu_identity(r):
    """relu(u) - relu(-u) = u: y(W3) - y(-W3) under the double activation is the
    single-activation y, which the standard pins already fix."""
    D, H, B = 12, 30, 4
    rng = np.random.default_rng(10)
    W1 = f32(rng.standard_normal((H, D)))
    U = f32(rng.standard_normal((H, max(r, 1))))[:, :r] if r else None
    V = f32(rng.standard_normal((r, D))) if r else None
    W3, W2 = dense_parts(D, H, 11)
    x = f32(rng.standard_normal((B, D)))
    gate = (None, f32(U), V) if r else (W1, None, None)
    y_pos, _, _ = oracle.ffn_dense_ex(D, H, r, RELU, F32, DA, *gate, W3, W2, x)
    y_neg, _, _ = oracle.ffn_dense_ex(D, H, r, RELU, F32, DA, *gate, f32(-W3), W2, x)
    y_one, _, _ = oracle.ffn_dense(D, H, r, RELU, F32, *gate, W3, W2, x)
    np.testing.assert_allclose(y_pos - y_neg, y_one, rtol=1e-12, atol=1e-13)
    # and the double activation really drops the negative part
    assert not np.allclose(y_pos, y_one)


@pytest.mark.parametrize("flags", [TG, RN, DA, TG | RN, TG | RN | DA])
@pytest.mark.parametrize("act", [RELU, RSP])
def test_gate_first_ex_equals_dense_ex(flags, act):
    """Skipping the dead units leaves y unchanged for every flag combination."""
    D, H, r, B = 24, 70, 8, 3
    rng = np.random.default_rng(12)
    U = f32(rng.standard_normal((H, r)) / math.sqrt(r))
    V = f32(rng.standard_normal((r, D)) / math.sqrt(D))
    W3, W2 = dense_parts(D, H, 13)
    x = f32(rng.standard_normal((B, D)))
    y_d, z, n_d = oracle.ffn_dense_ex(D, H, r, act, F32, flags, None, U, V, W3, W2, x)
    y_g, idx, n_g = oracle.ffn_gate_first_ex(D, H, r, act, F32, flags, None, U, V, W3, W2, x)
    np.testing.assert_allclose(y_g, y_d, rtol=1e-12, atol=1e-13)
    assert np.array_equal(n_d, n_g)
    for b in range(B):
        assert np.array_equal(idx[b, :n_g[b]], np.nonzero(z[b] > 0)[0])


def test_bad_flags_rejected():
    D, H = 4, 8
    W1 = f32(np.ones((H, D)))
    W3, W2 = dense_parts(D, H, 14)
    x = f32(np.ones((1, D)))
    with pytest.raises(RuntimeError):  # the tiled identity belongs to the low-rank gate
        oracle.ffn_dense_ex(D, H, 0, RELU, F32, TG, W1, None, None, W3, W2, x)
    with pytest.raises(RuntimeError):
        oracle.ffn_dense_ex(D, H, 0, RELU, F32, 8, W1, None, None, W3, W2, x)
