"""GPU parity of the weight-only int8 and int4 paths (dtypes SFFN_I8W, SFFN_I4W) against the oracle.

* The device quantiser must give the oracle's codes and scales bit for bit
  (an integer result decided in binary32 on both sides).
* The forward must match the oracle's int8 definition (dequantised weights
  q * s, fp64) within the bf16 output bar, with the live set identical outside
  the 1e-2 band, for every activation, the live threshold, the double
  activation and batches (one streaming pass per token).
* int4 is the same convention with codes in [-7, 7] (held two per byte on the
  device); every forward case runs for both.
"""
import numpy as np
import pytest
import torch

import oracle
import activation_sparse_gated_gb300 as sffn
from activation_sparse_gated_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu

TOL = 2e-2
BAND = 1e-2
K_ELEM = 1.0  # element-wise bar: max |y - y*| <= K_ELEM * TOL * rms(y*) (derivation in test_gpu_parity.py)
ACTS = {"relu": oracle.RELU, "rsp": oracle.RSP, "silu": oracle.SILU}
QMAX = {"int8": 127, "int4": 7}
DTYPES = ["int8", "int4"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from activation_sparse_gated_gb300 import build
    build.build()
    sffn.load()
    torch.cuda.set_device(0)


def floats(lw):
    t = lw.tensors()
    return [t[k].float().numpy() for k in ("W1", "W3", "W2")]


def oracle_codes(lw, dtype="int8"):
    W1, W3, W2 = floats(lw)
    if dtype == "int4":  # W1, W3 one scale per group of 64 columns, W2 one per row
        return oracle.quantize_int4(W1, W3, W2)
    return oracle.quantize_rows(W1) + oracle.quantize_rows(W3) + oracle.quantize_rows(W2)


def make_int8(lw, act="relu", flags=0, thr=0.0, dtype="int8"):
    ffn = sffn.SparseFFN(lw.D, lw.H, 0, act, dtype, flags=flags)
    t = lw.tensors()
    ffn.set_weights(t["W1"].cuda(), None, t["W3"].cuda(), t["W2"].cuda())
    if thr:
        ffn.set_live_threshold(thr)
    return ffn


def run(ffn, x, B=1):
    xd = x.cuda()
    ys, counts, masks = [], [], []
    for s in range(0, x.shape[0], B):
        xb = xd[s:s + B].contiguous()
        y = ffn(xb)
        counts += ffn.active_counts(xb.shape[0])
        masks.append(ffn.active_mask(xb.shape[0]))
        ys.append(y.float().cpu().numpy().astype(np.float64))
    return np.concatenate(ys), np.array(counts), np.concatenate(masks)


def act_val(act, z):
    if act == "silu":
        return z / (1.0 + np.exp(-z))
    return np.maximum(z, 0.0) if act == "relu" else np.where(z > 0, z / (1.0 + np.exp(-z)), 0.0)


def flip_adjusted(yref, z, gpu_live, ref_live, W3, W2, xb, act, flags):
    """y* moved to the GPU's live set (units inside the decision band may go either
    way; each flip moves a few elements of y by its whole term).  W3, W2 are the
    dequantised weights."""
    flips = np.nonzero(gpu_live != ref_live)[0]
    if flips.size == 0:
        return yref
    u = W3[flips] @ xb
    h = act_val(act, z[flips]) * (act_val(act, u) if flags & sffn.SFFN_DOUBLE_ACT else u)
    return yref + W2[:, flips] @ (np.where(gpu_live[flips], 1.0, -1.0) * h)


def act_abs(act, z):
    if act == "silu":
        return np.abs(z / (1.0 + np.exp(-z)))
    zp = np.maximum(z, 0.0)
    return zp if act == "relu" else np.where(z > 0, z / (1.0 + np.exp(-z)), 0.0)


def check(lw, x, y, counts, masks, act="relu", flags=0, thr=0.0, codes=None, dtype="int8"):
    q1, s1, q3, s3, q2, s2 = codes if codes is not None else oracle_codes(lw, dtype)
    group = oracle.INT4_GROUP if dtype == "int4" else None
    yref, z, n = oracle.ffn_dense_q8(lw.D, lw.H, ACTS[act], flags, q1, s1, q3, s3, q2, s2,
                                     syn.oracle_view(x), thr=thr, group=group)
    A = act_abs(act, z)
    s3v = np.asarray(s3, np.float64)
    W3 = q3.astype(np.float64) * (np.repeat(s3v, group, axis=1) if group else s3v[:, None])
    W2 = q2.astype(np.float64) * np.asarray(s2, np.float64)[:, None]
    xv = x.double().numpy()
    for b in range(x.shape[0]):
        den = np.linalg.norm(yref[b])
        live = A[b] > thr
        if den == 0:
            assert (y[b] == 0).all(), f"token {b}: no live unit but y != 0"
        else:
            err = np.linalg.norm(y[b] - yref[b]) / den
            assert err <= TOL, f"token {b}: relative L2 {err:.3e} > {TOL}"
            # element by element too: max |y - y*| <= K_ELEM * TOL * rms(y*), as in the bf16 parity tests
            ya = flip_adjusted(yref[b], z[b], masks[b].astype(bool), live, W3, W2, xv[b], act, flags)
            rms = np.sqrt(np.mean(yref[b] ** 2))
            worst = np.abs(y[b] - ya).max()
            assert worst <= K_ELEM * TOL * rms, f"token {b}: element error {worst:.3e} > {K_ELEM * TOL * rms:.3e}"
        sure = (np.abs(z[b]) > BAND) if thr == 0 else (np.abs(A[b] - thr) > 1e-3)
        bad = np.nonzero(sure & (masks[b].astype(bool) != live))[0]
        assert bad.size == 0, f"token {b}: live set differs at units {bad[:10]}"
        assert counts[b] == masks[b].sum()
    return yref, z, n


def crafted_rows(W):
    """Put the hand-worked quantisation rows (ties, an all-zero row) into W."""
    W = W.copy()
    W[0, :6] = [127.0, -63.5, 2.5, -3.5, 0.5, 0.0]
    W[0, 6:] = 0.0
    W[1, :] = 0.0
    W[2, :6] = [254.0, 1.0, 3.0, -5.0, 127.0, -128.0]
    W[2, 6:] = 0.0
    return W


@pytest.mark.parametrize("D,H", [(512, 1500), (2560, 7168)])
def test_device_quantiser_is_bitexact(D, H):
    lw = syn.standard_layer(D, H, dtype="bf16", seed=81)
    t = lw.tensors()
    W1 = crafted_rows(t["W1"].float().numpy())
    W1b = torch.from_numpy(W1).bfloat16()
    assert np.array_equal(W1b.float().numpy(), W1)  # the crafted values are bf16 numbers
    ffn = sffn.SparseFFN(D, H, 0, "relu", "int8")
    ffn.set_weights(W1b.cuda(), None, t["W3"].cuda(), t["W2"].cuda())
    got = [a.cpu().numpy() for a in ffn.int8_weights()]
    want = oracle.quantize_rows(W1) + oracle.quantize_rows(t["W3"].float().numpy()) + \
        oracle.quantize_rows(t["W2"].float().numpy())
    for g, w, name in zip(got, want, ("W1q", "s1", "W3q", "s3", "W2q", "s2")):
        assert g.shape == w.shape, name
        assert np.array_equal(g.view(np.uint8) if g.dtype == np.int8 else g.view(np.uint32),
                              w.view(np.uint8) if w.dtype == np.int8 else w.view(np.uint32)), name
    assert got[0][0, :6].tolist() == [127, -64, 2, -4, 0, 0] and got[1][0] == 1.0
    assert (got[0][1] == 0).all() and got[1][1] == 0.0
    assert got[0][2, :6].tolist() == [127, 0, 2, -2, 64, -64] and got[1][2] == 2.0


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("act,flags,thr", [("relu", 0, 0.0), ("rsp", 0, 0.0), ("relu", sffn.SFFN_DOUBLE_ACT, 0.0),
                                           ("silu", 0, 0.3), ("relu", 0, 0.05)])
@pytest.mark.parametrize("B", [1, 3])
def test_forward_matches_oracle(act, flags, thr, B, dtype):
    kw = {"shift": 0.0} if act == "silu" else {}
    lw = syn.standard_layer(512, 1500, dtype="bf16", seed=82, **kw)
    x = syn.tokens(2 * B, 512, dtype="bf16", seed=83)
    ffn = make_int8(lw, act, flags, thr, dtype)
    y, c, m = run(ffn, x, B=B)
    check(lw, x, y, c, m, act, flags, thr, dtype=dtype)


@pytest.mark.parametrize("dtype", DTYPES)
def test_full_size_workload(dtype):
    name = "std-bf16-D2560-H7168-B1"
    lw = syn.workload_layers(name, sets=1)[0]
    x = syn.workload_tokens(name, 6)
    ffn = make_int8(lw, dtype=dtype)
    y, c, m = run(ffn, x)
    _, _, n = check(lw, x, y, c, m, dtype=dtype)
    assert 0.02 < n.mean() / lw.H < 0.3


@pytest.mark.parametrize("dtype", DTYPES)
def test_d4096_shape(dtype):
    lw = syn.workload_layers("sweep-bf16-D4096-H14336", sets=1, s=0.75)[0]
    x = syn.workload_tokens("sweep-bf16-D4096-H14336", 2)
    ffn = make_int8(lw, dtype=dtype)
    y, c, m = run(ffn, x)
    check(lw, x, y, c, m, dtype=dtype)


@pytest.mark.parametrize("dtype,D,H", [("int8", 16, 1), ("int8", 16, 37), ("int8", 64, 151), ("int8", 64, 153),
                                       ("int8", 48, 300), ("int4", 64, 1), ("int4", 64, 37), ("int4", 64, 151),
                                       ("int4", 192, 300), ("int4", 4096, 40)])
def test_ragged_shapes(dtype, D, H):
    lw = syn.standard_layer(D, H, dtype="bf16", seed=84)
    x = syn.tokens(3, D, dtype="bf16", seed=85)
    ffn = make_int8(lw, dtype=dtype)
    y, c, m = run(ffn, x)
    check(lw, x, y, c, m, dtype=dtype)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("shift", [+20.0, -20.0])
def test_all_live_and_none_live(shift, dtype):
    lw = syn.standard_layer(256, 700, dtype="bf16", seed=86, shift=shift)
    x = syn.tokens(2, 256, dtype="bf16", seed=87)
    ffn = make_int8(lw, dtype=dtype)
    y, c, m = run(ffn, x)
    check(lw, x, y, c, m, dtype=dtype)
    if shift < 0:
        assert (c == 0).all() and (y == 0).all()
    else:
        assert (c == lw.H).all()


@pytest.mark.parametrize("dtype", DTYPES)
def test_external_codes_and_round_trip(dtype):
    """Codes and scales quantised by the oracle, loaded with sffn_set_weights_int8, give the
    same layer as the device quantiser, and read back unchanged (int4: packed two per byte on
    the device and unpacked on the way out)."""
    lw = syn.standard_layer(384, 1200, dtype="bf16", seed=88)
    x = syn.tokens(4, 384, dtype="bf16", seed=89)
    codes = oracle_codes(lw, dtype)
    ext = sffn.SparseFFN(384, 1200, 0, "relu", dtype)
    ext.set_weights_int8(*[torch.from_numpy(a).cuda() for a in codes])
    back = [a.cpu().numpy() for a in ext.int8_weights()]
    for g, w in zip(back, codes):
        assert np.array_equal(g, w)
    y1, c1, m1 = run(ext, x)
    y2, c2, m2 = run(make_int8(lw, dtype=dtype), x)
    check(lw, x, y1, c1, m1, codes=codes, dtype=dtype)
    assert np.array_equal(m1, m2) and np.array_equal(c1, c2)
    np.testing.assert_allclose(y1, y2, rtol=1e-2, atol=1e-6)


def test_int8_argument_errors():
    with pytest.raises(sffn.SffnError):
        sffn.SparseFFN(256, 512, 40, "relu", "int8")          # low-rank gate with r % 16 != 0
    with pytest.raises(sffn.SffnError):
        sffn.SparseFFN(40, 512, 0, "relu", "int8")            # D % 16 != 0
    bf = sffn.SparseFFN(256, 512, 0, "relu", "bf16")
    q = torch.zeros(512, 256, dtype=torch.int8, device="cuda")
    s = torch.ones(512, device="cuda")
    with pytest.raises(sffn.SffnError) as e:
        bf.set_weights_int8(q, s, q, s, torch.zeros(256, 512, dtype=torch.int8, device="cuda"),
                            torch.ones(256, device="cuda"))
    assert e.value.code == sffn.SFFN_ERR_STATE


def crafted_rows_int4(W):
    """The int4 hand-worked rows of the oracle pins (ties, an all-zero row, a scale of 2)."""
    W = W.copy()
    W[0, :6] = [7.0, -3.5, 2.5, 0.5, -1.5, 0.0]
    W[0, 6:] = 0.0
    W[1, :] = 0.0
    W[2, :6] = [-14.0, 3.0, 5.0, 1.0, 13.0, -9.0]
    W[2, 6:] = 0.0
    return W


@pytest.mark.parametrize("D,H", [(512, 1500), (2560, 7168)])
def test_device_quantiser_is_bitexact_int4(D, H):
    lw = syn.standard_layer(D, H, dtype="bf16", seed=91)
    t = lw.tensors()
    W1 = crafted_rows_int4(t["W1"].float().numpy())
    W1b = torch.from_numpy(W1).bfloat16()
    assert np.array_equal(W1b.float().numpy(), W1)
    ffn = sffn.SparseFFN(D, H, 0, "relu", "int4")
    ffn.set_weights(W1b.cuda(), None, t["W3"].cuda(), t["W2"].cuda())
    got = [a.cpu().numpy() for a in ffn.int8_weights()]
    want = oracle.quantize_int4(W1, t["W3"].float().numpy(), t["W2"].float().numpy())
    for g, w, name in zip(got, want, ("W1q", "s1", "W3q", "s3", "W2q", "s2")):
        assert g.shape == w.shape, name
        assert np.array_equal(g.view(np.uint8) if g.dtype == np.int8 else g.view(np.uint32),
                              w.view(np.uint8) if w.dtype == np.int8 else w.view(np.uint32)), name
    # the crafted rows fill the first group of 64 columns (the rest of it zero)
    assert got[0][0, :6].tolist() == [7, -4, 2, 0, -2, 0] and got[1][0, 0] == 1.0
    assert (got[0][1] == 0).all() and (got[1][1] == 0.0).all()
    assert got[0][2, :6].tolist() == [-7, 2, 2, 0, 6, -4] and got[1][2, 0] == 2.0


def test_int4_argument_errors():
    with pytest.raises(sffn.SffnError):
        sffn.SparseFFN(256, 512, 32, "relu", "int4")          # low-rank gate
    with pytest.raises(sffn.SffnError):
        sffn.SparseFFN(96, 512, 0, "relu", "int4")            # D % 64 != 0
    h = sffn.SparseFFN(256, 512, 0, "relu", "int4")
    q = torch.zeros(512, 256, dtype=torch.int8, device="cuda")
    q[3, 7] = 8                                                # outside [-7, 7]
    s = torch.ones(512, 4, device="cuda")
    with pytest.raises(sffn.SffnError) as e:
        h.set_weights_int8(q, s, torch.zeros_like(q), s, torch.zeros(256, 512, dtype=torch.int8, device="cuda"),
                           torch.ones(256, device="cuda"))
    assert e.value.code == sffn.SFFN_ERR_ARG
    with pytest.raises(sffn.SffnError) as e:                   # and the handle has no weights
        h(torch.zeros(1, 256, dtype=torch.bfloat16, device="cuda"))
    assert e.value.code == sffn.SFFN_ERR_STATE


# The low-rank gate with int8 weights: z = sU (qU t), t = sV (qV x), one scale per row of U, V, W3, W2.

def oracle_codes_lowrank(lw):
    t = lw.tensors()
    U, V, W3, W2 = (t[k].float().numpy() for k in ("U", "V", "W3", "W2"))
    return oracle.quantize_rows(U) + oracle.quantize_rows(V) + oracle.quantize_rows(W3) + oracle.quantize_rows(W2)


def make_lowrank_int8(lw, act="relu", flags=0, thr=0.0):
    ffn = sffn.SparseFFN(lw.D, lw.H, lw.r, act, "int8", flags=flags)
    t = lw.tensors()
    ffn.set_weights(t["U"].cuda(), t["V"].cuda(), t["W3"].cuda(), t["W2"].cuda())
    if thr:
        ffn.set_live_threshold(thr)
    return ffn


def check_lowrank(lw, x, y, counts, masks, act="relu", flags=0, thr=0.0):
    qU, sU, qV, sV, q3, s3, q2, s2 = oracle_codes_lowrank(lw)
    yref, z, n = oracle.ffn_lopa_q8(lw.D, lw.H, lw.r, ACTS[act], flags, qU, sU, qV, sV, q3, s3, q2, s2,
                                    syn.oracle_view(x), thr=thr)
    A = act_abs(act, z)
    W3 = q3.astype(np.float64) * np.asarray(s3, np.float64)[:, None]
    W2 = q2.astype(np.float64) * np.asarray(s2, np.float64)[:, None]
    xv = x.double().numpy()
    for b in range(x.shape[0]):
        den = np.linalg.norm(yref[b])
        live = A[b] > thr
        if den == 0:
            assert (y[b] == 0).all(), f"token {b}: no live unit but y != 0"
        else:
            err = np.linalg.norm(y[b] - yref[b]) / den
            assert err <= TOL, f"token {b}: relative L2 {err:.3e} > {TOL}"
            ya = flip_adjusted(yref[b], z[b], masks[b].astype(bool), live, W3, W2, xv[b], act, flags)
            rms = np.sqrt(np.mean(yref[b] ** 2))
            worst = np.abs(y[b] - ya).max()
            assert worst <= K_ELEM * TOL * rms, f"token {b}: element error {worst:.3e} > {K_ELEM * TOL * rms:.3e}"
        sure = (np.abs(z[b]) > BAND) if thr == 0 else (np.abs(A[b] - thr) > 1e-3)
        bad = np.nonzero(sure & (masks[b].astype(bool) != live))[0]
        assert bad.size == 0, f"token {b}: live set differs at units {bad[:10]}"
        assert counts[b] == masks[b].sum()
    return yref, z, n


@pytest.mark.parametrize("act,flags,thr", [("relu", 0, 0.0), ("rsp", 0, 0.0), ("relu", sffn.SFFN_DOUBLE_ACT, 0.0),
                                           ("silu", 0, 0.3)])
@pytest.mark.parametrize("B", [1, 3])
def test_lowrank_int8_matches_oracle(act, flags, thr, B):
    kw = {"shift": 0.0} if act == "silu" else {}
    lw = syn.lopa_layer(512, 1500, 64, dtype="bf16", seed=92, **kw)
    x = syn.tokens(2 * B, 512, dtype="bf16", seed=93)
    ffn = make_lowrank_int8(lw, act, flags, thr)
    y, c, m = run(ffn, x, B=B)
    check_lowrank(lw, x, y, c, m, act, flags, thr)


@pytest.mark.parametrize("D,H,r", [(64, 151, 16), (256, 700, 48), (2560, 9787, 400)])
def test_lowrank_int8_shapes_and_codes(D, H, r):
    """Ragged and full-size shapes; U's codes and scales read back bit-exact with the oracle's."""
    lw = syn.lopa_layer(D, H, r, dtype="bf16", seed=94)
    x = syn.tokens(3, D, dtype="bf16", seed=95)
    ffn = make_lowrank_int8(lw)
    y, c, m = run(ffn, x)
    _, _, n = check_lowrank(lw, x, y, c, m)
    qU, sU = oracle.quantize_rows(lw.tensors()["U"].float().numpy())
    got = ffn.int8_weights()
    assert np.array_equal(got[0].cpu().numpy(), qU) and np.array_equal(got[1].cpu().numpy(), sU)
    if D == 2560:
        assert 0.02 < n.mean() / H < 0.3


def test_lowrank_int8_takes_bf16_weights_only():
    lw = syn.lopa_layer(256, 700, 48, dtype="bf16", seed=96)
    ffn = sffn.SparseFFN(256, 700, 48, "relu", "int8")
    q = torch.zeros(700, 256, dtype=torch.int8, device="cuda")
    s = torch.ones(700, device="cuda")
    with pytest.raises(sffn.SffnError) as e:
        ffn.set_weights_int8(q, s, q, s, torch.zeros(256, 700, dtype=torch.int8, device="cuda"),
                             torch.ones(256, device="cuda"))
    assert e.value.code == sffn.SFFN_ERR_STATE
    with pytest.raises(sffn.SffnError):
        sffn.SparseFFN(256, 700, 48, "relu", "int4")          # int4 is the standard gate only
