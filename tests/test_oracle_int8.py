"""Pins of the oracle's weight-only int8 path.

"Model Casting and Low-Parameter Gating", appendix Table 17: the cast models
are quantised weight-only to int8.  The oracle reads this as symmetric
per-output-channel quantisation (s = max|w| / 127, codes rounded half to even
in binary32, clamped to [-127, 127]) and evaluates the FFN definition on the
dequantised weights q * s.  Pins: hand-worked codes (the rounding rule and the
scale), invariants that hold for any matrix, weights whose dequantised value
is exactly representable (then the int8 oracle must equal the already-pinned
float32 oracle), and a hand-worked forward.
"""
import numpy as np
import pytest
import torch

import oracle

F32, RELU, RSP, SILU = oracle.F32, oracle.RELU, oracle.RSP, oracle.SILU


def bf16_bits(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).bfloat16().view(torch.int16).numpy().view(
        np.uint16)


def test_quantize_hand_worked():
    W = np.array([[127.0, -63.5, 2.5, -3.5, 0.4, 0.0],      # s = 1: ties go to the even code
                  [0.0, 0.0, 0.0, 0.0, 0.0, 0.0],            # an all-zero row: s = 0, codes 0
                  [254.0, 1.0, 3.0, -5.0, 127.0, -128.0]],   # s = 2: 0.5 -> 0, 1.5 -> 2, -2.5 -> -2
                 dtype=np.float32)
    q, s = oracle.quantize_rows(W)
    assert s.tolist() == [1.0, 0.0, 2.0]
    assert q.tolist() == [[127, -64, 2, -4, 0, 0], [0] * 6, [127, 0, 2, -2, 64, -64]]


def test_quantize_invariants():
    rng = np.random.default_rng(1)
    W = (rng.standard_normal((64, 300)) * rng.uniform(0.01, 10.0, size=(64, 1))).astype(np.float32)
    q, s = oracle.quantize_rows(W)
    assert q.dtype == np.int8 and (np.abs(q.astype(np.int32)) <= 127).all()
    # the largest magnitude of every row maps to +-127 and keeps its sign
    j = np.abs(W).argmax(axis=1)
    assert (np.abs(q[np.arange(64), j].astype(np.int32)) == 127).all()
    assert (np.sign(q[np.arange(64), j]) == np.sign(W[np.arange(64), j])).all()
    # round to nearest: at most half a step away (plus binary32 rounding of w / s)
    err = np.abs(W.astype(np.float64) - q.astype(np.float64) * s[:, None].astype(np.float64))
    assert (err <= s[:, None].astype(np.float64) * (0.5 + 1e-5)).all()
    # no sign flips
    assert (q.astype(np.int32) * np.sign(W) >= 0).all()


def exact_layer(D, H, seed):
    """Codes with a +-127 in every row and power-of-two scales: q * s is exact in binary32."""
    rng = np.random.default_rng(seed)

    def mat(rows, cols):
        q = rng.integers(-127, 128, size=(rows, cols)).astype(np.int8)
        q[np.arange(rows), rng.integers(0, cols, size=rows)] = rng.choice([-127, 127], size=rows)
        s = np.ldexp(1.0, -rng.integers(3, 9, size=rows)).astype(np.float32)
        return q, s, (q.astype(np.float32) * s[:, None]).astype(np.float32)

    return mat(H, D), mat(H, D), mat(D, H)


@pytest.mark.parametrize("act", [RELU, RSP, SILU])
@pytest.mark.parametrize("flags", [0, oracle.FLAG_DOUBLE_ACT])
def test_q8_equals_float_oracle_on_exact_weights(act, flags):
    D, H, B = 48, 130, 4
    (q1, s1, W1), (q3, s3, W3), (q2, s2, W2) = exact_layer(D, H, 2)
    # quantising the exact weights gives back the same codes and scales
    for q, s, W in ((q1, s1, W1), (q3, s3, W3), (q2, s2, W2)):
        qq, ss = oracle.quantize_rows(W)
        assert np.array_equal(qq, q) and np.array_equal(ss, s)
    x = torch.from_numpy(np.random.default_rng(3).standard_normal((B, D)).astype(np.float32)).bfloat16()
    xf = x.float().numpy()
    thr = 0.05 if act == SILU else 0.0
    y8, z8, n8 = oracle.ffn_dense_q8(D, H, act, flags, q1, s1, q3, s3, q2, s2, bf16_bits(xf), thr=thr)
    yf, zf, nf = oracle.ffn_dense_ex(D, H, 0, act, F32, flags, W1, None, None, W3, W2, xf, thr=thr)
    np.testing.assert_allclose(z8, zf, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(y8, yf, rtol=1e-12, atol=1e-12)
    assert np.array_equal(n8, nf)


def test_q8_hand_worked():
    """D = 2, H = 2: z = (s1 q1) x, u = (s3 q3) x, y = (s2 q2) (relu(z) u) by hand."""
    q1 = np.array([[2, -1], [-3, 1]], dtype=np.int8); s1 = np.array([0.5, 0.25], dtype=np.float32)
    q3 = np.array([[1, 1], [4, 0]], dtype=np.int8); s3 = np.array([2.0, 1.0], dtype=np.float32)
    q2 = np.array([[1, 5], [-2, 7]], dtype=np.int8); s2 = np.array([0.125, 4.0], dtype=np.float32)
    x = np.array([[3.0, 1.0]], dtype=np.float32)
    # z = (0.5 * (6 - 1), 0.25 * (-9 + 1)) = (2.5, -2); u = (2 * 4, 12); h = (20, 0)
    y, z, n = oracle.ffn_dense_q8(2, 2, RELU, 0, q1, s1, q3, s3, q2, s2, bf16_bits(x))
    assert z.tolist() == [[2.5, -2.0]] and n.tolist() == [1]
    assert y.tolist() == [[0.125 * 20.0, 4.0 * -2.0 * 20.0]]


def test_q8_rejects_low_rank_flags():
    q = np.zeros((4, 8), dtype=np.int8)
    s = np.ones(4, dtype=np.float32)
    x = bf16_bits(np.ones((1, 8), dtype=np.float32))
    with pytest.raises(RuntimeError):
        oracle.ffn_dense_q8(8, 4, RELU, oracle.FLAG_TILED_G, q, s, q, s, q.T.copy(), np.ones(8, np.float32), x)


# Weight-only int4 ("Model Casting and Low-Parameter Gating", appendix Table 17, quantises the cast
# models to int4 too): the same convention with 7 in place of 127, codes in [-7, 7].

def test_quantize_int4_hand_worked():
    W = np.array([[7.0, -3.5, 2.5, 0.5, -1.5, 0.0],       # s = 1: ties go to the even code
                  [0.0, 0.0, 0.0, 0.0, 0.0, 0.0],         # all zero: s = 0, codes 0
                  [-14.0, 3.0, 5.0, 1.0, 13.0, -9.0]],    # s = 2: 1.5 -> 2, 2.5 -> 2, 0.5 -> 0, 6.5 -> 6, -4.5 -> -4
                 dtype=np.float32)
    q, s = oracle.quantize_rows(W, qmax=7)
    assert s.tolist() == [1.0, 0.0, 2.0]
    assert q.tolist() == [[7, -4, 2, 0, -2, 0], [0] * 6, [-7, 2, 2, 0, 6, -4]]


def test_quantize_int4_invariants():
    rng = np.random.default_rng(4)
    W = (rng.standard_normal((48, 256)) * rng.uniform(0.01, 10.0, size=(48, 1))).astype(np.float32)
    q, s = oracle.quantize_rows(W, qmax=7)
    assert (np.abs(q.astype(np.int32)) <= 7).all()
    j = np.abs(W).argmax(axis=1)
    assert (np.abs(q[np.arange(48), j].astype(np.int32)) == 7).all()
    err = np.abs(W.astype(np.float64) - q.astype(np.float64) * s[:, None].astype(np.float64))
    assert (err <= s[:, None].astype(np.float64) * (0.5 + 1e-5)).all()
    assert (q.astype(np.int32) * np.sign(W) >= 0).all()
    # an int8 grid is 127 / 7 times finer: the int4 error bound is the looser one
    q8, s8 = oracle.quantize_rows(W)
    np.testing.assert_allclose(s, s8 * (127.0 / 7.0), rtol=1e-6)


def test_quantize_rejects_a_code_range_outside_int8():
    W = np.ones((2, 4), dtype=np.float32)
    for qmax in (0, 128):
        with pytest.raises(RuntimeError):
            oracle.quantize_rows(W, qmax=qmax)


@pytest.mark.parametrize("act", [RELU, SILU])
def test_int4_codes_through_the_q8_forward_equal_the_float_oracle(act):
    """int4 codes are small integers; with power-of-two scales q * s is exact, so the _q8 forward on
    them must equal the pinned float32 oracle on the dequantised weights."""
    D, H, B = 32, 70, 3
    rng = np.random.default_rng(5)

    def mat(rows, cols):
        q = rng.integers(-7, 8, size=(rows, cols)).astype(np.int8)
        q[np.arange(rows), rng.integers(0, cols, size=rows)] = rng.choice([-7, 7], size=rows)
        s = np.ldexp(1.0, -rng.integers(1, 5, size=rows)).astype(np.float32)
        return q, s, (q.astype(np.float32) * s[:, None]).astype(np.float32)

    (q1, s1, W1), (q3, s3, W3), (q2, s2, W2) = mat(H, D), mat(H, D), mat(D, H)
    for q, s, W in ((q1, s1, W1), (q3, s3, W3), (q2, s2, W2)):
        qq, ss = oracle.quantize_rows(W, qmax=7)
        assert np.array_equal(qq, q) and np.array_equal(ss, s)
    xf = torch.from_numpy(rng.standard_normal((B, D)).astype(np.float32)).bfloat16().float().numpy()
    thr = 0.05 if act == SILU else 0.0
    y4, z4, n4 = oracle.ffn_dense_q8(D, H, act, 0, q1, s1, q3, s3, q2, s2, bf16_bits(xf), thr=thr)
    yf, zf, nf = oracle.ffn_dense_ex(D, H, 0, act, F32, 0, W1, None, None, W3, W2, xf, thr=thr)
    np.testing.assert_allclose(z4, zf, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(y4, yf, rtol=1e-12, atol=1e-12)
    assert np.array_equal(n4, nf)


# int4 for W1 and W3 takes one scale per group of oracle.INT4_GROUP columns (see the C file: with one
# scale per row, a single large entry rounds every ordinary entry of the row to 0).

def test_quantize_grouped_hand_worked():
    W = np.array([[7.0, 1.0, -3.5, 0.5, 14.0, 2.0, -5.0, 3.0],    # groups of 4: s = 1, then s = 2
                  [0.0, 0.0, 0.0, 0.0, -0.5, 0.25, 0.0, 0.0]],   # an all-zero group: s = 0; s = 1/14
                 dtype=np.float32)
    q, s = oracle.quantize_rows(W, 7, group=4)
    assert s.shape == (2, 2)
    assert s[0].tolist() == [1.0, 2.0] and s[1, 0] == 0.0
    assert s[1, 1] == np.float32(np.float32(0.5) / np.float32(7.0))
    assert q[0].tolist() == [7, 1, -4, 0, 7, 1, -2, 2]            # -3.5 -> -4, 0.5 -> 0, -2.5 -> -2, 1.5 -> 2
    # binary32: fl(0.5 / 7) lies above 0.5 / 7, so 0.25 / s = 3.4999998 and the code is 3, not 4
    assert q[1].tolist() == [0, 0, 0, 0, -7, 3, 0, 0]


def test_quantize_grouped_with_one_group_is_per_row():
    rng = np.random.default_rng(6)
    W = rng.standard_normal((9, 192)).astype(np.float32)
    for qmax in (7, 127):
        qg, sg = oracle.quantize_rows(W, qmax, group=192)
        q, s = oracle.quantize_rows(W, qmax)
        assert np.array_equal(qg, q) and np.array_equal(sg[:, 0], s)


def test_grouped_int4_keeps_a_row_with_one_large_entry():
    """A row of N(0, 1/D) entries with one entry of -1.28 (a gate bias carried as a column): one int4
    scale per row rounds almost every other entry to 0; one per 64-column group keeps the other groups."""
    rng = np.random.default_rng(7)
    D = 512
    W = (rng.standard_normal((4, D)) / np.sqrt(D)).astype(np.float32)
    W[:, D - 1] = -1.28
    q_row, _ = oracle.quantize_rows(W, 7)
    assert (q_row[:, :D - 1] != 0).mean() < 0.06                  # a step of 1.28 / 7: ~2 sigma, ~95 % zeros
    q_g, s_g = oracle.quantize_rows(W, 7, group=oracle.INT4_GROUP)
    assert (q_g[:, :D - 64] != 0).mean() > 0.6
    assert (np.abs(q_g[:, :D - 64]).max(axis=1) == 7).all()      # every other group uses the full range
    err = np.abs(W.astype(np.float64) - q_g * np.repeat(s_g, oracle.INT4_GROUP, axis=1).astype(np.float64))
    assert (err <= np.repeat(s_g, oracle.INT4_GROUP, axis=1) * (0.5 + 1e-5)).all()


@pytest.mark.parametrize("act,flags", [(RELU, 0), (SILU, 0), (RELU, oracle.FLAG_DOUBLE_ACT)])
def test_grouped_forward_equals_float_oracle_on_exact_weights(act, flags):
    """Codes with power-of-two scales per 16-column group: q * s is exact, so the grouped forward must
    equal the pinned float32 oracle on the dequantised weights."""
    D, H, B, G = 64, 90, 3, 16
    rng = np.random.default_rng(8)

    def grouped(rows, cols, g):
        q = rng.integers(-7, 8, size=(rows, cols)).astype(np.int8)
        q.reshape(rows, cols // g, g)[:, :, 0] = rng.choice([-7, 7], size=(rows, cols // g))
        s = np.ldexp(1.0, -rng.integers(1, 6, size=(rows, cols // g))).astype(np.float32)
        return q, s, (q.astype(np.float32) * np.repeat(s, g, axis=1)).astype(np.float32)

    (q1, s1, W1), (q3, s3, W3) = grouped(H, D, G), grouped(H, D, G)
    q2, s2, W2 = grouped(D, H, H)
    s2 = s2[:, 0]
    for q, s, W in ((q1, s1, W1), (q3, s3, W3)):
        qq, ss = oracle.quantize_rows(W, 7, group=G)
        assert np.array_equal(qq, q) and np.array_equal(ss, s)
    xf = torch.from_numpy(rng.standard_normal((B, D)).astype(np.float32)).bfloat16().float().numpy()
    thr = 0.05 if act == SILU else 0.0
    yg, zg, ng = oracle.ffn_dense_q8(D, H, act, flags, q1, s1, q3, s3, q2, s2, bf16_bits(xf), thr=thr, group=G)
    yf, zf, nf = oracle.ffn_dense_ex(D, H, 0, act, F32, flags, W1, None, None, W3, W2, xf, thr=thr)
    np.testing.assert_allclose(zg, zf, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(yg, yf, rtol=1e-12, atol=1e-12)
    assert np.array_equal(ng, nf)


def test_grouped_forward_hand_worked():
    """D = 4, groups of 2, H = 1: z = 0.5 (2 - 1) + 2 (3 + 1) = 8.5 for x = (1, 1, 1, 1)."""
    q1 = np.array([[2, -1, 3, 1]], dtype=np.int8); s1 = np.array([[0.5, 2.0]], dtype=np.float32)
    q3 = np.array([[1, 1, 0, 1]], dtype=np.int8); s3 = np.array([[1.0, 0.25]], dtype=np.float32)
    q2 = np.array([[1], [2], [-1], [4]], dtype=np.int8); s2 = np.array([1.0, 0.5, 2.0, 0.125], dtype=np.float32)
    x = bf16_bits(np.ones((1, 4), dtype=np.float32))
    y, z, n = oracle.ffn_dense_q8(4, 1, RELU, 0, q1, s1, q3, s3, q2, s2, x, group=2)
    # u = 1 (1 + 1) + 0.25 (0 + 1) = 2.25; h = 8.5 * 2.25 = 19.125
    assert z.tolist() == [[8.5]] and n.tolist() == [1]
    assert y.tolist() == [[19.125, 19.125, -38.25, 9.5625]]


# The low-rank gate ("LoPA Gating: moving the ceiling", z = U (V x)) with int8 weights, one scale per
# row of U, V, W3 and W2.

@pytest.mark.parametrize("act,flags", [(RELU, 0), (RSP, oracle.FLAG_DOUBLE_ACT), (SILU, 0)])
def test_lopa_q8_equals_float_oracle_on_exact_weights(act, flags):
    """Codes with power-of-two scales: q * s is exact in binary32, so the int8 low-rank forward must equal
    the pinned float32 low-rank oracle on the dequantised weights."""
    D, H, r, B = 40, 70, 16, 3
    rng = np.random.default_rng(9)

    def mat(rows, cols):
        q = rng.integers(-127, 128, size=(rows, cols)).astype(np.int8)
        q[np.arange(rows), rng.integers(0, cols, size=rows)] = rng.choice([-127, 127], size=rows)
        s = np.ldexp(1.0, -rng.integers(4, 9, size=rows)).astype(np.float32)
        return q, s, (q.astype(np.float32) * s[:, None]).astype(np.float32)

    (qU, sU, U), (qV, sV, V), (q3, s3, W3), (q2, s2, W2) = mat(H, r), mat(r, D), mat(H, D), mat(D, H)
    for q, s, W in ((qU, sU, U), (qV, sV, V)):
        qq, ss = oracle.quantize_rows(W)
        assert np.array_equal(qq, q) and np.array_equal(ss, s)
    xf = torch.from_numpy(rng.standard_normal((B, D)).astype(np.float32)).bfloat16().float().numpy()
    thr = 0.05 if act == SILU else 0.0
    y8, z8, n8 = oracle.ffn_lopa_q8(D, H, r, act, flags, qU, sU, qV, sV, q3, s3, q2, s2, bf16_bits(xf), thr=thr)
    yf, zf, nf = oracle.ffn_dense_ex(D, H, r, act, F32, flags, None, U, V, W3, W2, xf, thr=thr)
    np.testing.assert_allclose(z8, zf, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(y8, yf, rtol=1e-12, atol=1e-12)
    assert np.array_equal(n8, nf)


def test_lopa_q8_hand_worked():
    """D = 2, H = 2, r = 1: t = 0.5 (2 * 3 - 1 * 1) = 2.5; z = (0.25 * 4, 0.25 * -2) t = (2.5, -1.25)."""
    qV = np.array([[2, -1]], np.int8); sV = np.array([0.5], np.float32)
    qU = np.array([[4], [-2]], np.int8); sU = np.array([0.25, 0.25], np.float32)
    q3 = np.array([[1, 0], [0, 1]], np.int8); s3 = np.array([1.0, 1.0], np.float32)
    q2 = np.array([[2, 1], [1, 1]], np.int8); s2 = np.array([0.5, 1.0], np.float32)
    x = bf16_bits(np.array([[3.0, 1.0]], dtype=np.float32))
    y, z, n = oracle.ffn_lopa_q8(2, 2, 1, RELU, 0, qU, sU, qV, sV, q3, s3, q2, s2, x)
    # u = (3, 1); h = (2.5 * 3, 0) = (7.5, 0); y = (0.5 * 2 * 7.5, 1 * 1 * 7.5)
    assert z.tolist() == [[2.5, -1.25]] and n.tolist() == [1]
    assert y.tolist() == [[7.5, 7.5]]


def test_lopa_q8_rejects_bad_arguments():
    q = np.zeros((4, 8), dtype=np.int8)
    s = np.ones(4, dtype=np.float32)
    x = bf16_bits(np.ones((1, 8), dtype=np.float32))
    with pytest.raises(RuntimeError):   # the tiled identity is not part of this form
        oracle.ffn_lopa_q8(8, 4, 8, RELU, oracle.FLAG_TILED_G, np.zeros((4, 8), np.int8), s,
                           np.zeros((8, 8), np.int8), np.ones(8, np.float32), q, s, q.T.copy(),
                           np.ones(8, np.float32), x)
