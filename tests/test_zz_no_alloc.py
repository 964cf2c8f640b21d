"""The allocation-free forward agrees with the fp64 oracle and with the handle's forward.

Some callers cannot call cudaMalloc: a serving runtime that gives all device
memory to its own arena at start-up, or code on a latency-critical path where
an allocation would stall the device.  They use sffn_forward_noalloc, which
keeps its scratch in a fixed static array inside the library and takes the
weights (W2 transposed) from the caller.  These tests call it through the C ABI
twice in a row (the second call reuses the scratch the first one left) and
compare each result with the oracle, within the parity tests' tolerances, and
with sffn_forward on a handle holding the same weights.

This file is collected last on purpose, so that a run stopping at its first
failure has already run every other test.
"""
import numpy as np
import pytest
import torch

import oracle
import activation_sparse_gated_gb300 as sffn
from activation_sparse_gated_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu

TOL = {"bf16": 2e-2, "f32": 1e-5}
BAND = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from activation_sparse_gated_gb300 import build
    build.build()
    sffn.load()
    torch.cuda.set_device(0)


def _rel_l2(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return np.linalg.norm(a - b, axis=-1) / np.linalg.norm(b, axis=-1)


def _oracle(lw, x, act):
    v = {k: syn.oracle_view(t) for k, t in lw.tensors().items()}
    a = oracle.RELU if act == "relu" else oracle.RSP
    dt = oracle.F32 if lw.dtype == "f32" else oracle.BF16
    return oracle.ffn_dense(lw.D, lw.H, 0, a, dt, v["W1"], v["U"], v["V"], v["W3"], v["W2"],
                            syn.oracle_view(x))


@pytest.mark.parametrize("dtype,D,H,B,act", [("bf16", 2560, 7168, 2, "relu"), ("f32", 384, 1024, 3, "relu"),
                                             ("bf16", 512, 2048, 2, "rsp"), ("f32", 256, 640, 2, "rsp"),
                                             ("bf16", 4096, 1000, 2, "relu")])
def test_noalloc_matches_oracle_and_handle_twice(dtype, D, H, B, act):
    lw = syn.standard_layer(D, H, dtype=dtype, seed=77)
    ffn = sffn.SparseFFN(D, H, 0, act, dtype)
    W1, W3, W2 = lw.W1.cuda(), lw.W3.cuda(), lw.W2.cuda()
    ffn.set_weights(W1, None, W3, W2)
    W2t = W2.t().contiguous()
    dt = sffn.SFFN_BF16 if dtype == "bf16" else sffn.SFFN_F32
    a = sffn.SFFN_ACT_RELU if act == "relu" else sffn.SFFN_ACT_RSP
    x = syn.tokens(2 * B, D, dtype=dtype, seed=78)
    yref, z, n = _oracle(lw, x, act)
    xd = x.cuda()
    for call in range(2):                      # two calls in a row share the static scratch
        sl = slice(call * B, (call + 1) * B)
        xb = xd[sl].contiguous()
        y = torch.empty_like(xb)
        counts = torch.full((B,), -1, dtype=torch.int32, device="cuda")
        sffn.sffn_forward_noalloc(W1, W3, W2t, xb, y, counts, D, H, B, a, dt)
        torch.cuda.synchronize()
        yn = y.float().cpu().numpy()
        err = _rel_l2(yn, yref[sl])
        assert (err <= TOL[dtype]).all(), ("oracle", call, err)
        rms = np.sqrt(np.mean(yref[sl] ** 2, axis=-1))
        assert (np.abs(yn - yref[sl]).max(axis=-1) <= TOL[dtype] * rms).all(), ("oracle, element-wise", call)
        c = counts.cpu().numpy()
        band = (np.abs(z[sl]) <= BAND).sum(axis=1)
        assert (np.abs(c - n[sl]) <= band).all(), ("counts vs oracle", call, c, n[sl])
        y_ref = ffn(xb)
        assert (_rel_l2(yn, y_ref.float().cpu().numpy()) <= TOL[dtype]).all(), ("handle", call)
        assert c.tolist() == ffn.active_counts(B), ("counts vs handle", call)
        assert all(0 < k < H for k in c)


def test_noalloc_without_counts_buffer_and_counts_at_an_int_offset():
    D, H = 512, 2048
    lw = syn.standard_layer(D, H, dtype="bf16", seed=79)
    W1, W3, W2 = lw.W1.cuda(), lw.W3.cuda(), lw.W2.cuda()
    W2t = W2.t().contiguous()
    x = syn.tokens(2, D, dtype="bf16", seed=80)
    yref, z, n = _oracle(lw, x, "relu")
    xd = x.cuda()
    y = torch.empty_like(xd)
    sffn.sffn_forward_noalloc(W1, W3, W2t, xd, y, None, D, H, 2, sffn.SFFN_ACT_RELU, sffn.SFFN_BF16)
    torch.cuda.synchronize()
    assert (_rel_l2(y.float().cpu().numpy(), yref) <= TOL["bf16"]).all()
    # a counts buffer one int into an allocation: 4-byte aligned, accepted
    buf = torch.full((3,), -1, dtype=torch.int32, device="cuda")
    sffn.sffn_forward_noalloc(W1, W3, W2t, xd, y, buf[1:], D, H, 2, sffn.SFFN_ACT_RELU, sffn.SFFN_BF16)
    torch.cuda.synchronize()
    c = buf.cpu().numpy()
    assert c[0] == -1 and (np.abs(c[1:] - n) <= (np.abs(z) <= BAND).sum(axis=1)).all()


def test_noalloc_rejects_sizes_beyond_its_scratch_and_misaligned_pointers():
    W = torch.zeros(8, 8192, dtype=torch.bfloat16, device="cuda")
    x = torch.zeros(1, 8192, dtype=torch.bfloat16, device="cuda")
    y = torch.zeros_like(x)
    with pytest.raises(sffn.SffnError) as e:
        sffn.sffn_forward_noalloc(W, W, W, x, y, None, 8192, 8, 1, sffn.SFFN_ACT_RELU, sffn.SFFN_BF16)
    assert e.value.code == sffn.SFFN_ERR_ARG and "scratch" in str(e.value)
    W = torch.zeros(8, 72, dtype=torch.bfloat16, device="cuda")
    x = torch.zeros(2, 72, dtype=torch.bfloat16, device="cuda")
    y = torch.zeros(2, 72, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(sffn.SffnError) as e:     # x one element (2 bytes) into its buffer
        sffn.sffn_forward_noalloc(W, W, W, x.view(-1)[1:65], y, None, 64, 8, 1, sffn.SFFN_ACT_RELU,
                                  sffn.SFFN_BF16)
    assert e.value.code == sffn.SFFN_ERR_ALIGN
