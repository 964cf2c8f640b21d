"""Pins of the fp64 oracle against facts that do not come from the oracle itself.

Each test fixes the oracle to something independent: a value the pages print,
a hand-worked case, a closed form, an invariant of the formula, or a special
case that reduces to a library routine.  Together they are chosen so that a
plausible slip in the oracle (a dropped term, a wrong sign, a transposed W2, a
wrong row index, a wrong bf16 widening) fails at least one of them.

Formula: y = W2 (A(W1 x) .* (W3 x)), "Model casting: compute the gate, then skip
most of the FFN", section "What an FFN actually computes".
"""
import math
import os

import numpy as np
import pytest

import oracle
from oracle import flops
from activation_sparse_gated_gb300 import synthetic as syn

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def run(W1, W3, W2, x, act=oracle.RELU, U=None, V=None, r=0, dtype=oracle.F32, fn=oracle.ffn_dense):
    H, D = W3.shape
    if dtype == oracle.F32:
        cast = lambda a: None if a is None else np.ascontiguousarray(a, dtype=np.float32)  # noqa: E731
    else:
        cast = lambda a: None if a is None else syn.oracle_view(  # noqa: E731
            __import__("torch").from_numpy(np.ascontiguousarray(a, dtype=np.float32)).bfloat16())
    return fn(D, H, r, act, dtype, cast(W1), cast(U), cast(V), cast(W3), cast(W2), cast(x))


# --------------------------------------------------------------------------- hand-worked case
# D = 3, H = 4, x = (1, -2, 1)   (channel D-1 = 1 is the bias channel)
HAND_X = np.array([[1.0, -2.0, 1.0]])
HAND_W1 = np.array([[1.0, 0.0, -0.5],    # z0 = 1 - 0.5          =  0.5   live
                    [0.0, 1.0, 0.0],     # z1 = -2                        dead
                    [-1.0, -1.0, 0.25],  # z2 = -1 + 2 + 0.25    =  1.25  live
                    [2.0, 1.0, 0.0]])    # z3 = 2 - 2            =  0     dead (z = 0 exactly)
HAND_W3 = np.array([[1.0, 1.0, 3.0],     # u0 = 1 - 2 + 3 = 2
                    [5.0, 0.0, 0.0],     # u1 = 5  (dead unit: must not contribute)
                    [0.0, -1.0, 1.0],    # u2 = 2 + 1     = 3
                    [7.0, 0.0, 0.0]])    # u3 = 7  (dead)
HAND_W2 = np.array([[1.0, 100.0, 2.0, 100.0],    # dead columns hold 100 so a
                    [-1.0, 100.0, 0.5, 100.0],   # leak of a dead unit is visible
                    [0.0, 100.0, -4.0, 100.0]])


def test_hand_case_relu():
    # ReLU: a = (0.5, 0, 1.25, 0); h = a*u = (1, 0, 3.75, 0)
    # y0 = 1*1 + 2*3.75 = 8.5 ; y1 = -1*1 + 0.5*3.75 = 0.875 ; y2 = 0*1 - 4*3.75 = -15
    for dtype in (oracle.F32, oracle.BF16):
        y, z, n = run(HAND_W1, HAND_W3, HAND_W2, HAND_X, dtype=dtype)
        assert y.tolist() == [[8.5, 0.875, -15.0]]
        assert z.tolist() == [[0.5, -2.0, 1.25, 0.0]]
        assert n.tolist() == [2]


def test_hand_case_rsp_closed_form():
    # R-S+: a = z * sigmoid(z) for z >= 0, 0 below; dead units identical to ReLU.
    # sigmoid(0.5) = 1/(1+e^-0.5), sigmoid(1.25) = 1/(1+e^-1.25)
    s05 = 1.0 / (1.0 + math.exp(-0.5))
    s125 = 1.0 / (1.0 + math.exp(-1.25))
    h0, h2 = 0.5 * s05 * 2.0, 1.25 * s125 * 3.0
    want = [h0 * 1 + h2 * 2, -h0 + h2 * 0.5, -4.0 * h2]
    y, _, n = run(HAND_W1, HAND_W3, HAND_W2, HAND_X, act=oracle.RSP)
    np.testing.assert_allclose(y[0], want, rtol=1e-15, atol=1e-15)
    assert n.tolist() == [2]


def test_rsp_at_log3_uses_sigmoid_three_quarters():
    # sigmoid(ln 3) = 1/(1 + 1/3) = 3/4, so R-S+(ln 3) = 0.75 ln 3 (closed form,
    # independent of how the oracle evaluates the sigmoid).  One live unit, x = e_0.
    D, H = 2, 3
    W1 = np.array([[math.log(3.0), 0.0], [-1.0, 0.0], [-2.0, 0.0]])
    W3 = np.array([[1.0, 0.0], [1.0, 0.0], [1.0, 0.0]])
    W2 = np.array([[1.0, 9.0, 9.0], [2.0, 9.0, 9.0]])
    x = np.array([[1.0, 0.0]])
    y, _, _ = run(W1, W3, W2, x, act=oracle.RSP)
    z = float(np.float32(math.log(3.0)))           # stored value of ln 3
    a = z * 0.75                                   # sigmoid(z) = 3/4 up to |z - ln 3| ~ 1e-8
    np.testing.assert_allclose(y[0], [a, 2 * a], rtol=1e-7)
    # sigmoid(-z) would give 1/4, plain ReLU would give z: both are far outside 1e-7


# --------------------------------------------------------------------------- closed forms
def _dyadic(rng, shape, lo=-8, hi=8, scale=8.0):
    """Values k/8: exact in bf16, fp32 and fp64, so sums of a few stay exact."""
    return rng.integers(lo, hi + 1, size=shape).astype(np.float64) / scale


@pytest.mark.parametrize("dtype", [oracle.F32, oracle.BF16])
def test_one_live_unit_closed_form(dtype):
    # x = e_k, so z_i = W1[i,k] and u_i = W3[i,k]; make only unit i live:
    # y = W1[i,k] * W3[i,k] * W2[:, i]   (the skip argument with |S| = 1)
    rng = np.random.default_rng(1)
    D, H, i, k = 6, 10, 7, 2
    W1 = _dyadic(rng, (H, D))
    W1[:, k] = -np.abs(W1[:, k]) - 0.125
    W1[i, k] = 0.75
    W3 = _dyadic(rng, (H, D))
    W3[i, k] = -1.25
    W2 = _dyadic(rng, (D, H))
    x = np.zeros((1, D)); x[0, k] = 1.0
    y, z, n = run(W1, W3, W2, x, dtype=dtype)
    assert n.tolist() == [1]
    assert y[0].tolist() == (0.75 * -1.25 * W2[:, i]).tolist()
    _, idx, _ = run(W1, W3, W2, x, dtype=dtype, fn=oracle.ffn_gate_first)
    assert idx[0, 0] == i and idx[0, 1] == -1


@pytest.mark.parametrize("act", [oracle.RELU, oracle.RSP])
def test_no_live_unit_gives_zero(act):
    rng = np.random.default_rng(2)
    D, H = 8, 12
    W1 = _dyadic(rng, (H, D)); W1[:, D - 1] = -20.0     # bias column far below any gate
    W3, W2 = _dyadic(rng, (H, D)), _dyadic(rng, (D, H))
    x = _dyadic(rng, (3, D), -4, 4, 4.0); x[:, D - 1] = 1.0
    y, z, n = run(W1, W3, W2, x, act=act)
    assert n.tolist() == [0, 0, 0]
    assert (y == 0).all()
    assert (z < 0).all()


def test_all_live_reduces_to_bilinear_map_library():
    # With every gate unit live, ReLU is the identity on z and the FFN is the
    # bilinear map y = W2 diag(W3 x) W1 x; numpy's matmul (a library routine the
    # oracle does not use) evaluates it.
    rng = np.random.default_rng(3)
    D, H, B = 24, 40, 3
    W1 = rng.standard_normal((H, D)).astype(np.float32) / np.float32(5)
    W1[:, D - 1] = 10.0                                # all units live
    W3 = rng.standard_normal((H, D)).astype(np.float32)
    W2 = rng.standard_normal((D, H)).astype(np.float32)
    x = rng.standard_normal((B, D)).astype(np.float32); x[:, D - 1] = 1.0
    y, z, n = run(W1, W3, W2, x)
    assert n.tolist() == [H] * B
    W1d, W3d, W2d, xd = (a.astype(np.float64) for a in (W1, W3, W2, x))
    want = ((xd @ W1d.T) * (xd @ W3d.T)) @ W2d.T
    np.testing.assert_allclose(y, want, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(z, xd @ W1d.T, rtol=1e-13, atol=1e-13)


# --------------------------------------------------------------------------- invariants
def _random_layer(rng, D, H, B, dyadic=True):
    if dyadic:
        W1, W3, W2 = _dyadic(rng, (H, D)), _dyadic(rng, (H, D)), _dyadic(rng, (D, H))
        x = _dyadic(rng, (B, D), -4, 4, 4.0)
    else:
        W1 = rng.standard_normal((H, D)) / math.sqrt(D)
        W3 = rng.standard_normal((H, D)) / math.sqrt(D)
        W2 = rng.standard_normal((D, H)) / math.sqrt(H)
        x = rng.standard_normal((B, D))
    x[:, D - 1] = 1.0
    W1[:, D - 1] = -0.5
    return W1, W3, W2, x


def test_permuting_hidden_units_permutes_live_set_only():
    rng = np.random.default_rng(4)
    D, H, B = 16, 48, 4
    W1, W3, W2, x = _random_layer(rng, D, H, B)
    p = rng.permutation(H)
    y, z, n = run(W1, W3, W2, x)
    yp, zp, np_ = run(W1[p], W3[p], W2[:, p], x)
    assert np.array_equal(y, yp)          # dyadic data: every partial sum is exact
    assert np.array_equal(zp, z[:, p])
    assert np.array_equal(n, np_)
    assert 0 < n.min() and n.max() < H


def test_homogeneity():
    # ReLU is positively homogeneous, the FFN is linear in W3 and in W2, and of
    # degree 2 in x:  y(2 W1) = y(2 W3) = y(2 W2) = 2 y,  y(2 x) = 4 y  (all exact).
    rng = np.random.default_rng(5)
    D, H, B = 12, 30, 2
    W1, W3, W2, x = _random_layer(rng, D, H, B, dyadic=False)
    y, _, _ = run(W1, W3, W2, x)
    for args in ((2 * W1, W3, W2, x), (W1, 2 * W3, W2, x), (W1, W3, 2 * W2, x)):
        assert np.array_equal(run(*args)[0], 2 * y)
    assert np.array_equal(run(W1, W3, W2, 2 * x)[0], 4 * y)
    # W3 negated flips y; W1 negated changes the live set (not a symmetry)
    assert np.array_equal(run(W1, -W3, W2, x)[0], -y)


def test_relu_and_rsp_share_the_zero_set():
    rng = np.random.default_rng(6)
    D, H, B = 32, 64, 5
    W1, W3, W2, x = _random_layer(rng, D, H, B, dyadic=False)
    _, zr, nr = run(W1, W3, W2, x, act=oracle.RELU)
    _, zs, ns = run(W1, W3, W2, x, act=oracle.RSP)
    assert np.array_equal(zr, zs) and np.array_equal(nr, ns)


def test_tokens_are_independent():
    rng = np.random.default_rng(7)
    D, H, B = 16, 40, 5
    W1, W3, W2, x = _random_layer(rng, D, H, B, dyadic=False)
    y, z, n = run(W1, W3, W2, x)
    for b in range(B):
        yb, zb, nb = run(W1, W3, W2, x[b:b + 1])
        assert np.array_equal(yb[0], y[b]) and np.array_equal(zb[0], z[b]) and nb[0] == n[b]


def test_bf16_widening_matches_f32_on_representable_values():
    # The same bf16-representable values given as fp32 and as bf16 bit patterns
    # must give identical outputs (pins the exact widening of the bf16 bits).
    rng = np.random.default_rng(8)
    D, H, B = 16, 24, 3
    W1, W3, W2, x = _random_layer(rng, D, H, B)
    a = run(W1, W3, W2, x, dtype=oracle.F32)
    b = run(W1, W3, W2, x, dtype=oracle.BF16)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)
    # and a few known bit patterns: 0x3F80 = 1.0, 0xC000 = -2.0, 0x3EAB = 0.333984375
    D, H = 3, 1
    bits = lambda vals: np.array(vals, dtype=np.uint16)  # noqa: E731
    y, z, n = oracle.ffn_dense(D, H, 0, oracle.RELU, oracle.BF16,
                               bits([0x3F80, 0x3F80, 0x3F80]), None, None,
                               bits([0x3F80, 0x0000, 0x0000]), bits([0x3F80, 0x3F80, 0x3F80]),
                               bits([0x3EAB, 0xC000, 0x3F80]))
    assert z[0, 0] == 0.333984375 - 2.0 + 1.0 < 0 and n[0] == 0
    y, z, n = oracle.ffn_dense(D, H, 0, oracle.RELU, oracle.BF16,
                               bits([0x3F80, 0x0000, 0x0000]), None, None,
                               bits([0xC000, 0x0000, 0x0000]), bits([0x3F80, 0xC000, 0x3EAB]),
                               bits([0x3EAB, 0x3F80, 0x3F80]))
    # z = u-scale: z = 0.333984375, u = -2 * 0.333984375, h = z*u
    h = 0.333984375 * (-2.0 * 0.333984375)
    assert y[0].tolist() == [h, -2.0 * h, 0.333984375 * h]


# --------------------------------------------------------------------------- method facts
@pytest.mark.parametrize("act", [oracle.RELU, oracle.RSP])
def test_gate_first_equals_dense_exactly(act):
    # Skipping dead units changes nothing: the dead terms are exact zeros
    # (the skip argument of "What an FFN actually computes").
    lw = syn.standard_layer(256, 640, dtype="bf16", seed=11)
    x = syn.tokens(4, 256, dtype="bf16", seed=12)
    v = {k: syn.oracle_view(t) for k, t in lw.tensors().items()}
    xs = syn.oracle_view(x)
    yd, z, nd = oracle.ffn_dense(256, 640, 0, act, oracle.BF16, v["W1"], None, None, v["W3"], v["W2"], xs)
    yg, idx, ng = oracle.ffn_gate_first(256, 640, 0, act, oracle.BF16, v["W1"], None, None, v["W3"], v["W2"], xs)
    assert np.array_equal(yd, yg) and np.array_equal(nd, ng)
    for b in range(4):
        assert idx[b, :ng[b]].tolist() == np.nonzero(z[b] > 0)[0].tolist()
    assert 0 < nd.min() and nd.max() < 640


def test_lopa_materialised_equals_standard_gate():
    # W1 := U V turns the low-rank gate into the standard gate.  Integer data
    # keeps every product and sum exact, so the two must agree bit for bit.
    rng = np.random.default_rng(13)
    D, H, r, B = 16, 40, 4, 3
    U = rng.integers(-3, 4, size=(H, r)).astype(np.float64)
    V = rng.integers(-3, 4, size=(r, D)).astype(np.float64)
    W3 = rng.integers(-3, 4, size=(H, D)).astype(np.float64)
    W2 = rng.integers(-3, 4, size=(D, H)).astype(np.float64)
    x = rng.integers(-3, 4, size=(B, D)).astype(np.float64)
    yl, zl, nl = run(None, W3, W2, x, U=U, V=V, r=r)
    ys, zs, ns = run(U @ V, W3, W2, x)
    assert np.array_equal(yl, ys) and np.array_equal(zl, zs) and np.array_equal(nl, ns)
    assert 0 < nl.min() and nl.max() < H


def test_lopa_materialised_random_floats():
    # Random low-rank factors: the oracle's low-rank gate equals x W1^T with the
    # materialised W1 = U V formed by numpy's matmul (fp64), up to rounding order.
    lw = syn.lopa_layer(64, 150, 16, dtype="f32", seed=14)
    x = syn.tokens(3, 64, dtype="f32", seed=15)
    yl, zl, nl = oracle.ffn_dense(64, 150, 16, oracle.RELU, oracle.F32, None, lw.U.numpy(),
                                  lw.V.numpy(), lw.W3.numpy(), lw.W2.numpy(), x.numpy())
    W1 = lw.U.double().numpy() @ lw.V.double().numpy()
    np.testing.assert_allclose(zl, x.double().numpy() @ W1.T, rtol=1e-12, atol=1e-12)
    assert (nl == (zl > 0).sum(axis=1)).all()


# --------------------------------------------------------------------------- FLOP counter vs printed values
def _golden_rows():
    rows = []
    with open(os.path.join(GOLDEN, "paper_counts.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, value, how, params, cite = [c.strip() for c in line.split("|")]
            rows.append((name, float(value), how, params, cite))
    return rows


def _interval(pct):
    """A sparsity printed as a percentage with d decimals covers +-0.5 units of the last digit."""
    d = len(pct.split(".")[1]) if "." in pct else 0
    half = 0.5 * 10 ** (-d)
    v = float(pct)
    return (v - half) / 100.0, (v + half) / 100.0


def _printed_interval(value, how):
    if how.startswith("round"):
        d = int(how[5:])
        h = 0.5 * 10 ** (-d)
        return value - h, value + h
    if how == "trunc1":
        return value, value + 0.1
    if how == "about":
        return value - 0.15, value + 0.15
    if how.startswith("pct"):
        d = int(how[3:])
        h = 0.5 * 10 ** (-d)
        return value - h, value + h
    raise ValueError(how)


def _computed(name):
    D, H, r = 2560, 7168, 400
    Hp = 9787
    # the explainer's ideal shapes: H = 8D/3, r = D/8 (any D; ratios are scale free)
    Di = 3 * 8 * 100
    Hi, ri = 8 * Di / 3, Di / 8
    table = {
        "fig2_dense_matrix_M": lambda: flops.dense_macs(D, H) / 3 / 1e6,
        "fig2_sparse_w3_M": lambda: (flops.sparse_macs(D, H, 0.1 * H) - H * D) / 2 / 1e6,
        "fig2_lopa_gate_M": lambda: flops.lopa_gate_macs(D, Hp, r) / 1e6,
        "fig2_lopa_w3_M": lambda: (flops.lopa_macs(D, Hp, r, 0.1 * Hp) - flops.lopa_gate_macs(D, Hp, r)) / 2 / 1e6,
        "fig2_iso_width": lambda: flops.iso_width(D, H, r),
        "eq2_s090": lambda: flops.ratio_standard(0.90),
        "eq2_s095": lambda: flops.ratio_standard(0.95),
        "eq4_s090": lambda: flops.ratio_lopa(0.90, Di, Hi, ri),
        "eq4_limit": lambda: flops.ratio_lopa(1.0, Di, Hi, ri),
        "widget_gate_share": lambda: 100 * flops.shares_lopa(0.9, Di, Hi, ri)[0],
        "widget_w3_share": lambda: 100 * flops.shares_lopa(0.9, Di, Hi, ri)[1],
        "widget_total_share": lambda: 100 * flops.shares_lopa(0.9, Di, Hi, ri)[3],
        "widget_saved": lambda: 100 * (1 - flops.shares_lopa(0.9, Di, Hi, ri)[3]),
        "table6_std_s75": lambda: flops.ratio_standard(0.75),
    }
    intervals = {   # printed sparsity -> ratio over the whole rounding interval of s
        "table1_rsp_s69": ("69", lambda s: flops.ratio_standard(s)),
        "table1_rsp_l1_s89": ("89", lambda s: flops.ratio_standard(s)),
        "table3_s896": ("89.6", lambda s: flops.ratio_standard(s)),
        "table3_s895": ("89.5", lambda s: flops.ratio_standard(s)),
        "fig1_lopa_s89": ("89", lambda s: flops.ratio_lopa(s, Di, Hi, ri)),
    }
    if name in table:
        v = table[name]()
        return v, v
    pct, f = intervals[name]
    lo, hi = _interval(pct)
    return f(lo), f(hi)   # both ratios increase with s


@pytest.mark.parametrize("row", _golden_rows(), ids=lambda r: r[0])
def test_flop_counter_matches_printed_values(row):
    name, value, how, params, cite = row
    clo, chi = _computed(name)
    plo, phi = _printed_interval(value, how)
    # the computed value (or the interval the printed sparsity allows) must reach
    # the interval the printed figure stands for
    assert clo < phi and chi >= plo, (name, clo, chi, plo, phi, cite)


def test_flop_counter_structure():
    # Eq. 2 is the ratio of the two counters; 3x is its limit, 1x its value at s = 0
    D, H = 2560, 7168
    for s in (0.0, 0.5, 0.9, 0.95):
        assert flops.dense_macs(D, H) / flops.sparse_macs(D, H, (1 - s) * H) == pytest.approx(flops.ratio_standard(s))
    assert flops.ratio_standard(0.0) == 1.0
    assert flops.ratio_standard(1.0) == pytest.approx(3.0)
    # the iso-parameter width keeps the parameter count: r(D+H') + 2H'D == 3HD
    r = 400
    Hp = flops.iso_width(D, H, r)
    assert r * (D + Hp) + 2 * Hp * D == pytest.approx(3 * H * D)
    # LoPA with s -> 1 is limited by the gate alone: 136/10 = 13.6 at H=8D/3, r=D/8
    assert flops.ratio_lopa(1.0, 2400, 6400, 300) == pytest.approx(13.6)


# --------------------------------------------------------------------------- generator statistics
def test_generator_gives_about_ten_percent_live():
    lw = syn.standard_layer(2560, 7168, dtype="bf16", seed=1000)
    x = syn.tokens(8, 2560, dtype="bf16", seed=1500)
    v = {k: syn.oracle_view(t) for k, t in lw.tensors().items()}
    _, z, n = oracle.ffn_dense(2560, 7168, 0, oracle.RELU, oracle.BF16, v["W1"], None, None,
                               v["W3"], v["W2"], syn.oracle_view(x))
    frac = n.sum() / (8 * 7168)
    assert 0.09 < frac < 0.11, frac


def test_lopa_generator_bias_channel_and_live_fraction():
    D, Hp, r = 512, 2000, 64
    lw = syn.lopa_layer(D, Hp, r, dtype="bf16", seed=2000)
    Vf = lw.V.float().numpy()
    assert Vf[r - 1, D - 1] == 1.0 and (Vf[r - 1, :D - 1] == 0).all() and (Vf[:r - 1, D - 1] == 0).all()
    x = syn.tokens(8, D, dtype="bf16", seed=2500)
    v = {k: syn.oracle_view(t) for k, t in lw.tensors().items()}
    _, z, n = oracle.ffn_dense(D, Hp, r, oracle.RELU, oracle.BF16, None, v["U"], v["V"],
                               v["W3"], v["W2"], syn.oracle_view(x))
    frac = n.sum() / (8 * Hp)
    assert 0.07 < frac < 0.13, frac
