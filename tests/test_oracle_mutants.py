"""The oracle's pins have teeth: plant plausible mistakes in copies of the C
source, build each copy, and check that at least one pin rejects it.

Every mistake is planted in the oracle (CPU only); nothing here touches the GPU.
"""
import math
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle

SRC = os.path.join(os.path.dirname(oracle.__file__), "sffn_oracle.c")

MUTANTS = {
    "w2_transposed": ("widen_row(W2, dtype, (size_t)m * H, H, row);",
                      "for (int i2 = 0; i2 < H; ++i2) row[i2] = elem(W2, dtype, (size_t)i2 * D + m);"),
    "w3_dropped": ("g[i] = gate_value(act, thr, zb[i]) * up_value(act, flags, u);",
                   "g[i] = gate_value(act, thr, zb[i]);"),
    "gate_row_off_by_one": ("widen_row(W1, dtype, (size_t)i * D, D, row);",
                            "widen_row(W1, dtype, (size_t)((i + 1) % H) * D, D, row);"),
    "live_count_ge": ("cnt += (fabs(activation(act, zb[i])) > thr);", "cnt += (fabs(activation(act, zb[i])) >= thr);"),
    "activation_wrong_side": ("if (!(z > 0.0)) return 0.0;", "if (!(z < 0.0)) return 0.0;"),
    "rsp_sigmoid_sign": ("return z / (1.0 + exp(-z));", "return z / (1.0 + exp(z));"),
    "rsp_missing_z": ("return z / (1.0 + exp(-z));", "return 1.0 / (1.0 + exp(-z));"),
    "bf16_widen_shift": ("<< 16;", "<< 15;"),
    "dot_drops_last_term": ("for (int j = 0; j < n; ++j) s += a[j] * b[j];",
                            "for (int j = 0; j + 1 < n; ++j) s += a[j] * b[j];"),
    "u_transposed": ("widen_row(U, dtype, (size_t)i * r, r, row);",
                     "for (int k2 = 0; k2 < r; ++k2) row[k2] = elem(U, dtype, (size_t)k2 * H + i);"),
    "gate_first_skips_first_live": ("for (int q = 0; q < k; ++q) {\n        if (!row) continue;",
                                    "for (int q = 1; q < k; ++q) {\n        if (!row) continue;"),
    # the full low-rank gate
    "tiled_g_index_shift": ("z[i] += xd[i % D];", "z[i] += xd[(i + 1) % D];"),
    "rmsnorm_sum_not_mean": ("sqrt(ss / (double)r + eps)", "sqrt(ss + eps)"),
    "rmsnorm_eps_outside_root": ("1.0 / sqrt(ss / (double)r + eps)", "1.0 / (sqrt(ss / (double)r) + eps)"),
    "double_act_dropped": ("return (flags & OR_FLAG_DOUBLE_ACT) ? activation(act, u) : u;", "return u;"),
    # SiLU and the live threshold
    "silu_negative_side_zeroed": ("if (act == OR_SILU) return z / (1.0 + exp(-z));", ""),
    "threshold_not_absolute": ("return fabs(a) > thr ? a : 0.0;", "return a > thr ? a : 0.0;"),
    "threshold_ignored_in_dense": ("g[i] = gate_value(act, thr, zb[i]) * up_value(act, flags, u);",
                                   "g[i] = activation(act, zb[i]) * up_value(act, flags, u);"),
    # weight-only int8
    "q8_truncate": ("v = rintf(w[j] / sc);", "v = truncf(w[j] / sc);"),
    "q8_round_half_away": ("v = rintf(w[j] / sc);", "v = roundf(w[j] / sc);"),
    "q8_amax_signed": ("const float a = fabsf(w[j]);", "const float a = w[j];"),
    "q8_one_scale": ("(double)s[i * ng + (size_t)(j / group)];", "(double)s[0];"),
    "q8_down_uses_gate_scales": ("dequant_row(q2, s2, (size_t)m, H, row);", "dequant_row(q2, s1, (size_t)m, H, row);"),
    "q8_up_uses_gate_codes": ("dequant_row_g(q3, s3, (size_t)i, D, group, row);",
                              "dequant_row_g(q1, s3, (size_t)i, D, group, row);"),
    # int4 groups of columns
    "group_scale_index_mod": ("(double)s[i * ng + (size_t)(j / group)];", "(double)s[i * ng + (size_t)(j % ng)];"),
    "group_amax_of_first_group": ("const float* w = W + (size_t)i * cols + (size_t)g * group;",
                                  "const float* w = W + (size_t)i * cols;"),
    "group_scale_of_row": ("s[(size_t)i * ng + g] = sc;", "s[(size_t)i * ng] = sc;"),
    # the low-rank gate with int8 weights
    "lopa_q8_gate_on_x": ("zb[i] = dot(row, t, r);", "zb[i] = dot(row, xd, r);"),
    "lopa_q8_v_scaled_by_u": ("dequant_row(qV, sV, (size_t)k, D, row);", "dequant_row(qV, sU, (size_t)k, D, row);"),
}


def _bf16_bits(a):
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).bfloat16()
    return t.view(torch.int16).numpy().view(np.uint16)


def _cast(a, dtype):
    if a is None:
        return None
    return np.ascontiguousarray(a, dtype=np.float32) if dtype == oracle.F32 else _bf16_bits(a)


def _pins(mod):
    """Run a compact set of the pins against `mod`; return the names that fail."""
    failed = []

    def run(W1, W3, W2, x, act=oracle.RELU, U=None, V=None, r=0, dtype=oracle.F32, fn="ffn_dense"):
        H, D = W3.shape
        c = lambda a: _cast(a, dtype)  # noqa: E731
        return getattr(mod, fn)(D, H, r, act, dtype, c(W1), c(U), c(V), c(W3), c(W2), c(x))

    def check(name, cond):
        if not cond:
            failed.append(name)

    # hand-worked case (values derived in test_oracle_pins)
    X = np.array([[1.0, -2.0, 1.0]])
    W1 = np.array([[1.0, 0.0, -0.5], [0.0, 1.0, 0.0], [-1.0, -1.0, 0.25], [2.0, 1.0, 0.0]])
    W3 = np.array([[1.0, 1.0, 3.0], [5.0, 0.0, 0.0], [0.0, -1.0, 1.0], [7.0, 0.0, 0.0]])
    W2 = np.array([[1.0, 100.0, 2.0, 100.0], [-1.0, 100.0, 0.5, 100.0], [0.0, 100.0, -4.0, 100.0]])
    for dt in (oracle.F32, oracle.BF16):
        y, z, n = run(W1, W3, W2, X, dtype=dt)
        check("hand_relu", y.tolist() == [[8.5, 0.875, -15.0]] and n.tolist() == [2])
        yg, idx, ng = run(W1, W3, W2, X, dtype=dt, fn="ffn_gate_first")
        check("hand_gate_first", yg.tolist() == [[8.5, 0.875, -15.0]] and ng.tolist() == [2])
    s05, s125 = 1 / (1 + math.exp(-0.5)), 1 / (1 + math.exp(-1.25))
    h0, h2 = 0.5 * s05 * 2.0, 1.25 * s125 * 3.0
    y, _, _ = run(W1, W3, W2, X, act=oracle.RSP)
    check("hand_rsp", np.allclose(y[0], [h0 + 2 * h2, -h0 + 0.5 * h2, -4 * h2], rtol=1e-15, atol=1e-15))
    # all-live bilinear map through numpy
    rng = np.random.default_rng(3)
    D, H, B = 24, 40, 3
    A1 = rng.standard_normal((H, D)).astype(np.float32) / np.float32(5); A1[:, D - 1] = 10.0
    A3 = rng.standard_normal((H, D)).astype(np.float32)
    A2 = rng.standard_normal((D, H)).astype(np.float32)
    xa = rng.standard_normal((B, D)).astype(np.float32); xa[:, D - 1] = 1.0
    y, z, n = run(A1, A3, A2, xa)
    d = [a.astype(np.float64) for a in (A1, A3, A2, xa)]
    want = ((d[3] @ d[0].T) * (d[3] @ d[1].T)) @ d[2].T
    check("all_live_library", np.allclose(y, want, rtol=1e-12, atol=1e-12))
    # low-rank gate with integer factors == standard gate with W1 = U V (numpy)
    rng = np.random.default_rng(13)
    D, H, r, B = 16, 40, 4, 3
    U = rng.integers(-3, 4, size=(H, r)).astype(np.float64)
    V = rng.integers(-3, 4, size=(r, D)).astype(np.float64)
    L3 = rng.integers(-3, 4, size=(H, D)).astype(np.float64)
    L2 = rng.integers(-3, 4, size=(D, H)).astype(np.float64)
    xl = rng.integers(-3, 4, size=(B, D)).astype(np.float64)
    yl, zl, _ = run(None, L3, L2, xl, U=U, V=V, r=r)
    check("lopa_materialised", np.array_equal(zl, xl @ (U @ V).T))
    # bf16 bit patterns 0x3F80 = 1, 0xC000 = -2, 0x3EAB = 0.333984375
    bits = lambda v: np.array(v, dtype=np.uint16)  # noqa: E731
    y, z, n = mod.ffn_dense(3, 1, 0, oracle.RELU, oracle.BF16, bits([0x3F80, 0, 0]), None, None,
                            bits([0xC000, 0, 0]), bits([0x3F80, 0xC000, 0x3EAB]),
                            bits([0x3EAB, 0x3F80, 0x3F80]))
    h = 0.333984375 * (-2.0 * 0.333984375)
    check("bf16_bits", y[0].tolist() == [h, -2.0 * h, 0.333984375 * h])
    # full low-rank gate (values derived in test_oracle_lopa_full)
    f = lambda a: np.ascontiguousarray(a, dtype=np.float32)  # noqa: E731
    rng = np.random.default_rng(21)
    D, H, r, B = 8, 21, 4, 3
    Ui = rng.integers(-2, 3, size=(H, r)).astype(np.float32)
    Vi = rng.integers(-1, 2, size=(r, D)).astype(np.float32)
    T = np.zeros((H, D), dtype=np.float32)
    T[np.arange(H), np.arange(H) % D] = 1.0
    G3 = f(rng.standard_normal((H, D)) / 3)
    G2 = f(rng.standard_normal((D, H)) / 5)
    xg = f(rng.standard_normal((B, D)))
    yg, zg, _ = mod.ffn_dense_ex(D, H, r, oracle.RELU, oracle.F32, oracle.FLAG_TILED_G, None, f(Ui), f(Vi),
                                 G3, G2, xg)
    ys, zs, _ = mod.ffn_dense(D, H, 0, oracle.RELU, oracle.F32, f(T + Ui @ Vi), None, None, G3, G2, xg)
    check("tiled_g_materialised", np.allclose(zg, zs, rtol=0, atol=1e-12) and np.allclose(yg, ys, rtol=1e-12))
    Vh, Uh = f([[3.0, 0.0], [0.0, 4.0]]), f([[1.0, 0.0], [0.0, 1.0], [1.0, 1.0], [-1.0, 0.0]])
    _, zh, _ = mod.ffn_dense_ex(2, 4, 2, oracle.RELU, oracle.F32, oracle.FLAG_RMSNORM, None, Uh, Vh,
                                f(np.ones((4, 2))), f(np.ones((2, 4))), f([[1.0, 1.0]]), 1e-6)
    sh = math.sqrt(12.5 + 1e-6)
    check("rmsnorm_hand", np.allclose(zh[0], [3 / sh, 4 / sh, 7 / sh, -3 / sh], rtol=1e-14, atol=0))
    yp, _, _ = mod.ffn_dense_ex(D, H, 0, oracle.RELU, oracle.F32, oracle.FLAG_DOUBLE_ACT, f(T + Ui @ Vi), None,
                                None, G3, G2, xg)
    yn, _, _ = mod.ffn_dense_ex(D, H, 0, oracle.RELU, oracle.F32, oracle.FLAG_DOUBLE_ACT, f(T + Ui @ Vi), None,
                                None, f(-G3), G2, xg)
    check("double_act_relu_identity", np.allclose(yp - yn, ys, rtol=1e-12, atol=1e-13) and
          not np.allclose(yp, ys))
    # SiLU at threshold 0 is the dense SwiGLU product (torch's silu in fp64)
    D, H, B = 10, 26, 3
    S1, S3 = f(rng.standard_normal((H, D))), f(rng.standard_normal((H, D)))
    S2, xs = f(rng.standard_normal((D, H))), f(rng.standard_normal((B, D)))
    y0, _, n0 = mod.ffn_dense_ex(D, H, 0, oracle.SILU, oracle.F32, 0, S1, None, None, S3, S2, xs, 1e-6, 0.0)
    d = [torch.from_numpy(a.astype(np.float64)) for a in (S1, S3, S2, xs)]
    want = (torch.nn.functional.silu(d[3] @ d[0].T) * (d[3] @ d[1].T)) @ d[2].T
    check("silu_swiglu_library", np.allclose(y0, want.numpy(), rtol=1e-12, atol=1e-12) and (n0 == H).all())
    # a threshold keeps |A(z)| > thr: the error is at most thr * sum_i |W2[m,i]| |u_i|
    thr = 0.3
    yt, zt, nt = mod.ffn_dense_ex(D, H, 0, oracle.SILU, oracle.F32, 0, S1, None, None, S3, S2, xs, 1e-6, thr)
    u = (d[3] @ d[1].T).numpy()
    bound = thr * (np.abs(u) @ np.abs(d[2].numpy()).T)
    a = torch.nn.functional.silu(torch.from_numpy(zt)).numpy()
    check("threshold_error_bound", (np.abs(yt - y0) <= bound + 1e-12).all() and
          (nt == (np.abs(a) > thr).sum(axis=1)).all() and (nt < H).all() and not np.allclose(yt, y0))
    # weight-only int8 (values derived in test_oracle_int8)
    q, sc = mod.quantize_rows(f([[127.0, -63.5, 2.5, -3.5, 0.4, 0.0], [254.0, 1.0, 3.0, -5.0, 127.0, -128.0]]))
    check("q8_hand_codes", q.tolist() == [[127, -64, 2, -4, 0, 0], [127, 0, 2, -2, 64, -64]] and
          sc.tolist() == [1.0, 2.0])
    Wr = f(rng.standard_normal((16, 40)) * 3)
    q, sc = mod.quantize_rows(Wr)
    err = np.abs(Wr.astype(np.float64) - q.astype(np.float64) * sc[:, None])
    check("q8_round_trip", (err <= sc[:, None].astype(np.float64) * (0.5 + 1e-5)).all())
    D, H, B = 12, 30, 3
    mats = []
    for rows, cols in ((H, D), (H, D), (D, H)):
        qq = rng.integers(-127, 128, size=(rows, cols)).astype(np.int8)
        qq[:, 0] = 127
        ss = np.ldexp(1.0, -rng.integers(3, 9, size=rows)).astype(np.float32)
        mats.append((qq, ss, f(qq.astype(np.float32) * ss[:, None])))
    (q1, s1, E1), (q3, s3, E3), (q2, s2, E2) = mats
    xq = f(torch.from_numpy(f(rng.standard_normal((B, D)))).bfloat16().float().numpy())
    y8, _, n8 = mod.ffn_dense_q8(D, H, oracle.RELU, 0, q1, s1, q3, s3, q2, s2, _bf16_bits(xq))
    yf, _, nf = mod.ffn_dense(D, H, 0, oracle.RELU, oracle.F32, E1, None, None, E3, E2, xq)
    check("q8_exact_weights", np.allclose(y8, yf, rtol=1e-12, atol=1e-12) and np.array_equal(n8, nf))
    # int4 groups (values derived in test_oracle_int8)
    q, sc = mod.quantize_rows(f([[7.0, 1.0, -3.5, 0.5, 14.0, 2.0, -5.0, 3.0]]), 7, 4)
    check("q4g_hand_codes", q.tolist() == [[7, 1, -4, 0, 7, 1, -2, 2]] and sc.tolist() == [[1.0, 2.0]])
    yg, zg, ng = mod.ffn_dense_q8(4, 1, oracle.RELU, 0, np.array([[2, -1, 3, 1]], np.int8), f([[0.5, 2.0]]),
                                  np.array([[1, 1, 0, 1]], np.int8), f([[1.0, 0.25]]),
                                  np.array([[1], [2], [-1], [4]], np.int8), f([1.0, 0.5, 2.0, 0.125]),
                                  _bf16_bits(f(np.ones((1, 4)))), 0.0, 2)
    check("q4g_hand_forward", zg.tolist() == [[8.5]] and yg.tolist() == [[19.125, 19.125, -38.25, 9.5625]])
    # the low-rank gate with int8 weights (values derived in test_oracle_int8)
    yl, zl, nl = mod.ffn_lopa_q8(2, 2, 1, oracle.RELU, 0, np.array([[4], [-2]], np.int8), f([0.25, 0.25]),
                                 np.array([[2, -1]], np.int8), f([0.5]), np.array([[1, 0], [0, 1]], np.int8),
                                 f([1.0, 1.0]), np.array([[2, 1], [1, 1]], np.int8), f([0.5, 1.0]),
                                 _bf16_bits(f([[3.0, 1.0]])))
    check("lopa_q8_hand", zl.tolist() == [[2.5, -1.25]] and yl.tolist() == [[7.5, 7.5]])
    return failed


def test_pins_pass_on_the_oracle():
    assert _pins(oracle) == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-std=c99", "-fopenmp", "-fPIC", "-shared", "-o", str(so),
                    str(mutated), "-lm"], check=True)
    failed = _pins(oracle.Variant(str(so)))
    assert failed, f"mutant {name} passed every pin"
