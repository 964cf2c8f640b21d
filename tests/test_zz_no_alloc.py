"""The allocation-free forward agrees with the handle's forward.

Some callers cannot call cudaMalloc: a serving runtime that gives all device
memory to its own arena at start-up, or code on a latency-critical path where
an allocation would stall the device.  They use sffn_forward_noalloc, which
keeps its scratch in a fixed static array inside the library and takes the
weights (W2 transposed) from the caller.  These tests call it through the C ABI
twice in a row and compare each result with sffn_forward on a handle holding
the same weights, within the tolerances of the parity tests.

This file is collected last on purpose, so that a run stopping at its first
failure has already run every other test.
"""
import numpy as np
import pytest
import torch

import activation_sparse_gated_gb300 as sffn
from activation_sparse_gated_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu

TOL = {"bf16": 2e-2, "f32": 1e-5}


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from activation_sparse_gated_gb300 import build
    build.build()
    sffn.load()
    torch.cuda.set_device(0)


def _rel_l2(a, b):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    return np.linalg.norm(a - b, axis=-1) / np.linalg.norm(b, axis=-1)


@pytest.mark.parametrize("dtype,D,H,B", [("bf16", 2560, 7168, 2), ("f32", 384, 1024, 3)])
def test_noalloc_matches_handle_forward_twice(dtype, D, H, B):
    lw = syn.standard_layer(D, H, dtype=dtype, seed=77)
    ffn = sffn.SparseFFN(D, H, 0, "relu", dtype)
    W1, W3, W2 = lw.W1.cuda(), lw.W3.cuda(), lw.W2.cuda()
    ffn.set_weights(W1, None, W3, W2)
    W2t = W2.t().contiguous()
    dt = sffn.SFFN_BF16 if dtype == "bf16" else sffn.SFFN_F32
    x = syn.tokens(2 * B, D, dtype=dtype, seed=78).cuda()
    for call in range(2):                      # two calls in a row share the static scratch
        xb = x[call * B:(call + 1) * B].contiguous()
        y = torch.empty_like(xb)
        counts = torch.full((B,), -1, dtype=torch.int32, device="cuda")
        sffn.sffn_forward_noalloc(W1, W3, W2t, xb, y, counts, D, H, B, sffn.SFFN_ACT_RELU, dt)
        torch.cuda.synchronize()
        y_ref = ffn(xb)
        c_ref = ffn.active_counts(B)
        err = _rel_l2(y.float(), y_ref.float())
        assert (err <= TOL[dtype]).all(), (call, err)
        assert counts.cpu().tolist() == c_ref, (call, counts.cpu().tolist(), c_ref)
        assert all(0 < c < H for c in c_ref)


def test_noalloc_without_counts_buffer():
    D, H = 512, 2048
    lw = syn.standard_layer(D, H, dtype="bf16", seed=79)
    ffn = sffn.SparseFFN(D, H, 0, "relu", "bf16")
    W1, W3, W2 = lw.W1.cuda(), lw.W3.cuda(), lw.W2.cuda()
    ffn.set_weights(W1, None, W3, W2)
    x = syn.tokens(1, D, dtype="bf16", seed=80).cuda()
    y = torch.empty_like(x)
    sffn.sffn_forward_noalloc(W1, W3, W2.t().contiguous(), x, y, None, D, H, 1, sffn.SFFN_ACT_RELU,
                              sffn.SFFN_BF16)
    torch.cuda.synchronize()
    assert (_rel_l2(y.float(), ffn(x).float()) <= TOL["bf16"]).all()


def test_noalloc_rejects_sizes_beyond_its_scratch():
    W = torch.zeros(8, 8192, dtype=torch.bfloat16, device="cuda")
    x = torch.zeros(1, 8192, dtype=torch.bfloat16, device="cuda")
    y = torch.zeros_like(x)
    with pytest.raises(sffn.SffnError) as e:
        sffn.sffn_forward_noalloc(W, W, W, x, y, None, 8192, 8, 1, sffn.SFFN_ACT_RELU, sffn.SFFN_BF16)
    assert e.value.code == sffn.SFFN_ERR_ARG and "scratch" in str(e.value)
