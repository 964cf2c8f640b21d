"""fp64 CPU oracle of the gate-first sparse gated FFN.

TEST INFRASTRUCTURE ONLY: imported by the test suite, the smoke check and the
benchmark's CPU-baseline leg, never by the library.  It shares no code with the
CUDA path.  The arithmetic lives in ``sffn_oracle.c`` (plain C99 + OpenMP, fp64)
and in ``flops.py`` (operation counts); this module only compiles and loads the
C file and marshals numpy arrays into it.

Formulas followed: "Model casting: compute the gate, then skip most of the FFN"
(ai.thesatyajit.com), sections "What an FFN actually computes" (y = W2(A(W1x) .*
W3x)), "Model casting: make sparsity a target" (R-S+), "LoPA Gating: moving the
ceiling" (W1 = G + UV; the UV part only).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

from . import flops  # noqa: F401  (re-exported)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sffn_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

F32, BF16 = 0, 1
RELU, RSP, SILU = 0, 1, 2

_lib = None


def build(force: bool = False) -> str:
    """Compile sffn_oracle.c into liboracle.so next to it (gcc, OpenMP, -O2)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c99", "-fopenmp", "-fPIC", "-shared",
               "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _bind(path):
    lib = ctypes.CDLL(path)
    vp, ip = ctypes.c_void_p, ctypes.c_int
    for name in ("oracle_ffn_dense", "oracle_ffn_gate_first"):
        f = getattr(lib, name)
        f.restype = ip
        f.argtypes = [ip] * 6 + [vp] * 9
    for name in ("oracle_ffn_dense_ex", "oracle_ffn_gate_first_ex"):
        f = getattr(lib, name)
        f.restype = ip
        f.argtypes = [ip] * 7 + [ctypes.c_double] * 2 + [vp] * 9
    lib.oracle_num_threads.restype = ip
    lib.oracle_num_threads.argtypes = []
    lib.oracle_quantize_rows.restype = ip
    lib.oracle_quantize_rows.argtypes = [ip, ip, vp, vp, vp]
    lib.oracle_quantize_rows_q.restype = ip
    lib.oracle_quantize_rows_q.argtypes = [ip, ip, ip, vp, vp, vp]
    lib.oracle_quantize_rows_g.restype = ip
    lib.oracle_quantize_rows_g.argtypes = [ip, ip, ip, ip, vp, vp, vp]
    lib.oracle_ffn_dense_q8.restype = ip
    lib.oracle_ffn_dense_q8.argtypes = [ip] * 5 + [ctypes.c_double] + [vp] * 10
    lib.oracle_ffn_dense_qg.restype = ip
    lib.oracle_ffn_dense_qg.argtypes = [ip] * 5 + [ctypes.c_double, ip] + [vp] * 10
    lib.oracle_ffn_lopa_q8.restype = ip
    lib.oracle_ffn_lopa_q8.argtypes = [ip] * 6 + [ctypes.c_double] + [vp] * 12
    return lib


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = _bind(_LIB)
    return _lib


class Variant:
    """The oracle's entry points bound to another build of the C source.

    Used only by the test that plants mistakes in a copy of the source to check
    that the pins catch them.
    """

    def __init__(self, so_path):
        self._lib = _bind(so_path)

    def ffn_dense(self, *a):
        return _call("oracle_ffn_dense", *a[:5], *a[5:11],
                     lambda B: np.zeros((B, a[1]), dtype=np.float64), lib=self._lib)

    def ffn_gate_first(self, *a):
        return _call("oracle_ffn_gate_first", *a[:5], *a[5:11],
                     lambda B: np.full((B, a[1]), -1, dtype=np.int32), lib=self._lib)

    def ffn_dense_ex(self, D, H, r, act, dtype, flags, W1, U, V, W3, W2, x, eps=1e-6, thr=0.0):
        return _call("oracle_ffn_dense_ex", D, H, r, act, dtype, W1, U, V, W3, W2, x,
                     lambda B: np.zeros((B, H), dtype=np.float64), lib=self._lib, flags=flags, eps=eps,
                     thr=thr)

    def quantize_rows(self, W, qmax=127, group=None):
        return _quantize_rows(W, self._lib, qmax, group)

    def ffn_lopa_q8(self, D, H, r, act, flags, qU, sU, qV, sV, q3, s3, q2, s2, x, thr=0.0):
        return _ffn_lopa_q8(D, H, r, act, flags, qU, sU, qV, sV, q3, s3, q2, s2, x, thr, self._lib)

    def ffn_dense_q8(self, D, H, act, flags, q1, s1, q3, s3, q2, s2, x, thr=0.0, group=None):
        return _ffn_dense_q8(D, H, act, flags, q1, s1, q3, s3, q2, s2, x, thr, self._lib, group)


def num_threads() -> int:
    """OpenMP threads the oracle uses (OMP_NUM_THREADS, else all cores)."""
    return int(_load().oracle_num_threads())


def _as_input(a, dtype):
    """Check an input array against the stored dtype: float32, or uint16 bf16 bits."""
    if a is None:
        return None
    want = np.float32 if dtype == F32 else np.uint16
    a = np.ascontiguousarray(a)
    if a.dtype != want:
        raise TypeError(f"oracle input must be {np.dtype(want).name}, got {a.dtype}")
    return a


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _call(name, D, H, r, act, dtype, W1, U, V, W3, W2, x, extra, lib=None, flags=None, eps=0.0, thr=0.0):
    x = _as_input(x, dtype)
    B = x.size // D
    if x.size != B * D:
        raise ValueError("x size is not a multiple of D")
    arrs = [_as_input(a, dtype) for a in (W1, U, V, W3, W2)]
    W1, U, V, W3, W2 = arrs
    if r == 0:
        assert W1 is not None and W1.size == H * D
    else:
        assert U is not None and U.size == H * r and V is not None and V.size == r * D
    assert W3.size == H * D and W2.size == D * H
    y = np.zeros((B, D), dtype=np.float64)
    n_live = np.zeros(B, dtype=np.int32)
    out = extra(B)
    head = (D, H, r, act, dtype, B) if flags is None else (D, H, r, act, dtype, B, flags, float(eps), float(thr))
    rc = getattr(lib or _load(), name)(*head, _ptr(W1), _ptr(U), _ptr(V),
                                       _ptr(W3), _ptr(W2), _ptr(x), _ptr(y), _ptr(out), _ptr(n_live))
    if rc != 0:
        raise RuntimeError(f"{name} failed with code {rc}")
    return y, out, n_live


def ffn_dense(D, H, r, act, dtype, W1, U, V, W3, W2, x):
    """Dense definition.  Returns (y[B,D] f64, z[B,H] f64 pre-activations, n_live[B])."""
    return _call("oracle_ffn_dense", D, H, r, act, dtype, W1, U, V, W3, W2, x,
                 lambda B: np.zeros((B, H), dtype=np.float64))


def ffn_gate_first(D, H, r, act, dtype, W1, U, V, W3, W2, x):
    """Gate-first evaluation.  Returns (y[B,D] f64, idx[B,H] live set padded with -1, n_live[B])."""
    return _call("oracle_ffn_gate_first", D, H, r, act, dtype, W1, U, V, W3, W2, x,
                 lambda B: np.full((B, H), -1, dtype=np.int32))


# Full low-rank gate of the pages ("LoPA Gating: moving the ceiling"): flags of the "_ex" forms.
FLAG_TILED_G = 1      # z_i += x_{i mod D}  (G = tiled identity)
FLAG_RMSNORM = 2      # t = RMSNorm(V x) = V x / sqrt(mean((V x)^2) + eps), no gain
FLAG_DOUBLE_ACT = 4   # u = A(W3 x) instead of W3 x (either gate)
RMSNORM_EPS = 1e-6


def ffn_dense_ex(D, H, r, act, dtype, flags, W1, U, V, W3, W2, x, eps=RMSNORM_EPS, thr=0.0):
    """Dense definition with the full low-rank gate options and a live threshold
    (unit i is live iff |A(z_i)| > thr).  Returns (y, z, n_live)."""
    return _call("oracle_ffn_dense_ex", D, H, r, act, dtype, W1, U, V, W3, W2, x,
                 lambda B: np.zeros((B, H), dtype=np.float64), flags=flags, eps=eps, thr=thr)


def ffn_gate_first_ex(D, H, r, act, dtype, flags, W1, U, V, W3, W2, x, eps=RMSNORM_EPS, thr=0.0):
    """Gate-first evaluation with the same options.  Returns (y, idx, n_live)."""
    return _call("oracle_ffn_gate_first_ex", D, H, r, act, dtype, W1, U, V, W3, W2, x,
                 lambda B: np.full((B, H), -1, dtype=np.int32), flags=flags, eps=eps, thr=thr)



# Weight-only int8 ("Model Casting and Low-Parameter Gating", appendix Table 17):
# symmetric per-output-channel scales, codes decided in binary32 (see the C file).
def _quantize_rows(W, lib=None, qmax=127, group=None):
    W = np.ascontiguousarray(W, dtype=np.float32)
    rows, cols = W.shape
    q = np.zeros((rows, cols), dtype=np.int8)
    if group is None:
        s = np.zeros(rows, dtype=np.float32)
        rc = (lib or _load()).oracle_quantize_rows_q(rows, cols, int(qmax), _ptr(W), _ptr(q), _ptr(s))
    else:
        s = np.zeros((rows, cols // group if group > 0 else 0), dtype=np.float32)
        rc = (lib or _load()).oracle_quantize_rows_g(rows, cols, int(qmax), int(group), _ptr(W), _ptr(q),
                                                     _ptr(s))
    if rc != 0:
        raise RuntimeError(f"oracle quantisation failed with code {rc}")
    return q, s


def quantize_rows(W, qmax=127, group=None):
    """Codes in [-qmax, qmax] (127: int8 weights, 7: int4) and fp32 scales of a float32 matrix:
    (q[rows, cols] int8, s[rows] f32) with one scale per row, or s[rows, cols // group] with one
    per group of `group` consecutive columns."""
    return _quantize_rows(W, qmax=qmax, group=group)


def quantize_int4(W1, W3, W2):
    """The int4 convention: W1, W3 [H, D] with a scale per group of INT4_GROUP columns, W2 [D, H]
    with a scale per row.  Returns (q1, s1, q3, s3, q2, s2)."""
    return (quantize_rows(W1, 7, INT4_GROUP) + quantize_rows(W3, 7, INT4_GROUP) + quantize_rows(W2, 7))


INT4_GROUP = 64


def _ffn_dense_q8(D, H, act, flags, q1, s1, q3, s3, q2, s2, x, thr=0.0, lib=None, group=None):
    g = D if group is None else int(group)
    if g < 1 or D % g:
        raise RuntimeError(f"group {g} does not divide D={D}")
    i8 = lambda a, n: np.ascontiguousarray(a, dtype=np.int8).reshape(n)  # noqa: E731
    f32 = lambda a, n: np.ascontiguousarray(a, dtype=np.float32).reshape(n)  # noqa: E731
    q1, q3, q2 = i8(q1, H * D), i8(q3, H * D), i8(q2, D * H)
    s1, s3, s2 = f32(s1, H * (D // g)), f32(s3, H * (D // g)), f32(s2, D)
    x = _as_input(x, BF16)
    B = x.size // D
    y = np.zeros((B, D), dtype=np.float64)
    z = np.zeros((B, H), dtype=np.float64)
    n_live = np.zeros(B, dtype=np.int32)
    rc = (lib or _load()).oracle_ffn_dense_qg(D, H, act, B, flags, float(thr), g, _ptr(q1), _ptr(s1), _ptr(q3),
                                              _ptr(s3), _ptr(q2), _ptr(s2), _ptr(x), _ptr(y), _ptr(z),
                                              _ptr(n_live))
    if rc != 0:
        raise RuntimeError(f"oracle_ffn_dense_qg failed with code {rc}")
    return y, z, n_live


def _ffn_lopa_q8(D, H, r, act, flags, qU, sU, qV, sV, q3, s3, q2, s2, x, thr=0.0, lib=None):
    i8 = lambda a, n: np.ascontiguousarray(a, dtype=np.int8).reshape(n)  # noqa: E731
    f32 = lambda a, n: np.ascontiguousarray(a, dtype=np.float32).reshape(n)  # noqa: E731
    qU, qV, q3, q2 = i8(qU, H * r), i8(qV, r * D), i8(q3, H * D), i8(q2, D * H)
    sU, sV, s3, s2 = f32(sU, H), f32(sV, r), f32(s3, H), f32(s2, D)
    x = _as_input(x, BF16)
    B = x.size // D
    y = np.zeros((B, D), dtype=np.float64)
    z = np.zeros((B, H), dtype=np.float64)
    n_live = np.zeros(B, dtype=np.int32)
    rc = (lib or _load()).oracle_ffn_lopa_q8(D, H, r, act, B, flags, float(thr), _ptr(qU), _ptr(sU), _ptr(qV),
                                             _ptr(sV), _ptr(q3), _ptr(s3), _ptr(q2), _ptr(s2), _ptr(x), _ptr(y),
                                             _ptr(z), _ptr(n_live))
    if rc != 0:
        raise RuntimeError(f"oracle_ffn_lopa_q8 failed with code {rc}")
    return y, z, n_live


def ffn_lopa_q8(D, H, r, act, flags, qU, sU, qV, sV, q3, s3, q2, s2, x, thr=0.0):
    """The low-rank gate z = U (V x) with int8 weights, one scale per row of each matrix (qU [H, r],
    qV [r, D], q3 [H, D], q2 [D, H]); bf16 x.  flags: 0 or FLAG_DOUBLE_ACT.  Returns (y, z, n_live)."""
    return _ffn_lopa_q8(D, H, r, act, flags, qU, sU, qV, sV, q3, s3, q2, s2, x, thr)


def ffn_dense_q8(D, H, act, flags, q1, s1, q3, s3, q2, s2, x, thr=0.0, group=None):
    """Dense definition with quantised weights (q1, q3 [H, D] with scales [H], or [H, D // group]
    with one per group of columns; q2 [D, H], scales [D]) and bf16 x (uint16 bits).  flags: 0 or
    FLAG_DOUBLE_ACT.  Returns (y, z, n_live)."""
    return _ffn_dense_q8(D, H, act, flags, q1, s1, q3, s3, q2, s2, x, thr, group=group)
