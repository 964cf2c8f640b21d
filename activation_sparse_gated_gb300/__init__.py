"""Gate-first sparse gated-FFN forward for GB300: Python binding of include/sffn.h.

Argument marshalling only: every step of the forward pass runs in the CUDA
kernels of ``libsffn.so`` (built in-tree by ``build.py``).  PyTorch supplies
device memory and streams.  There is no CPU fallback: if the library is missing
or fails to load, every entry point raises.

The functions mirror the C ABI one to one (``sffn_create``, ``sffn_set_live_fraction_hint``, ``sffn_set_weights``,
``sffn_forward``, ``sffn_active_counts``, ``sffn_active_mask``,
``sffn_synchronize``, ``sffn_destroy``, ``sffn_strerror``, ``sffn_last_error``,
``sffn_version``, ``sffn_debug_timeout_probe``, ``sffn_forward_noalloc``,
``sffn_set_weights_int8``, ``sffn_get_weights_int8``).  Tensor arguments are passed by
their data pointer; ``stream`` defaults to the current torch stream.
``SparseFFN`` wraps one handle.
"""
from __future__ import annotations

import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libsffn.so")

SFFN_F32, SFFN_BF16, SFFN_I8W, SFFN_I4W = 0, 1, 2, 3
INT4_GROUP = 64  # int4 W1, W3: columns per scale
SFFN_ACT_RELU, SFFN_ACT_RSP, SFFN_ACT_SILU = 0, 1, 2
SFFN_OK = 0
SFFN_ERR_ARG, SFFN_ERR_ALIGN, SFFN_ERR_DTYPE, SFFN_ERR_CUDA = -1, -2, -3, -4
SFFN_ERR_TIMEOUT, SFFN_ERR_STATE, SFFN_ERR_NOMEM, SFFN_ERR_DEVICE = -5, -6, -7, -8
SFFN_MAX_BATCH = 128
SFFN_GATE_TILED_G, SFFN_GATE_RMSNORM, SFFN_DOUBLE_ACT, SFFN_DETERMINISTIC = 1, 2, 4, 8

#: every symbol include/sffn.h declares
EXPORTS = ("sffn_create", "sffn_create_ex", "sffn_set_live_threshold", "sffn_set_live_fraction_hint", "sffn_set_weights", "sffn_forward", "sffn_active_counts",
           "sffn_active_mask", "sffn_synchronize", "sffn_destroy", "sffn_strerror",
           "sffn_last_error", "sffn_version", "sffn_debug_timeout_probe", "sffn_forward_noalloc",
           "sffn_set_weights_int8", "sffn_get_weights_int8")

_lib = None


class SffnError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"{message} (status {code})")
        self.code = code


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libsffn.so and declare its signatures.  Raises if it is not built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with activation_sparse_gated_gb300/build.py "
                          "(there is no CPU fallback)")
    lib = ctypes.CDLL(path)
    vp, ip, cp = ctypes.c_void_p, ctypes.c_int, ctypes.c_char_p
    sig = {
        "sffn_create": (vp, [ip, ip, ip, ip, ip]),
        "sffn_create_ex": (vp, [ip, ip, ip, ip, ip, ip]),
        "sffn_set_live_threshold": (ip, [vp, ctypes.c_float]),
        "sffn_set_live_fraction_hint": (ip, [vp, ctypes.c_float]),
        "sffn_set_weights": (ip, [vp, vp, vp, vp, vp, vp]),
        "sffn_forward": (ip, [vp, vp, vp, ip, vp]),
        "sffn_active_counts": (ip, [vp, vp, ip]),
        "sffn_active_mask": (ip, [vp, vp, ip]),
        "sffn_synchronize": (ip, [vp]),
        "sffn_destroy": (None, [vp]),
        "sffn_strerror": (cp, [ip]),
        "sffn_last_error": (cp, []),
        "sffn_version": (ip, []),
        "sffn_debug_timeout_probe": (ip, [vp, ip, vp]),
        "sffn_forward_noalloc": (ip, [vp, vp, vp, vp, vp, vp, ip, ip, ip, ip, ip, vp]),
        "sffn_set_weights_int8": (ip, [vp] * 8),
        "sffn_get_weights_int8": (ip, [vp] * 8),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def _ptr(a):
    """Data pointer of a tensor / ndarray / int / None."""
    if a is None:
        return None
    if isinstance(a, int):
        return a
    if hasattr(a, "data_ptr"):
        return a.data_ptr()
    if hasattr(a, "ctypes"):
        return a.ctypes.data
    raise TypeError(f"cannot take a pointer of {type(a)}")


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc: int):
    if rc != SFFN_OK:
        raise SffnError(rc, sffn_last_error() or sffn_strerror(rc))
    return rc


def sffn_version() -> int:
    return load().sffn_version()


def sffn_strerror(code: int) -> str:
    return load().sffn_strerror(code).decode()


def sffn_last_error() -> str:
    return load().sffn_last_error().decode()


def sffn_create(D: int, H: int, r: int, act: int, dtype: int) -> int:
    h = load().sffn_create(D, H, r, act, dtype)
    if not h:
        raise SffnError(SFFN_ERR_ARG, sffn_last_error())
    return h


def sffn_create_ex(D: int, H: int, r: int, act: int, dtype: int, flags: int) -> int:
    h = load().sffn_create_ex(D, H, r, act, dtype, flags)
    if not h:
        raise SffnError(SFFN_ERR_ARG, sffn_last_error())
    return h


def sffn_set_live_threshold(h, thr: float):
    return _check(load().sffn_set_live_threshold(h, float(thr)))


def sffn_set_live_fraction_hint(h, rho: float):
    return _check(load().sffn_set_live_fraction_hint(h, float(rho)))


def sffn_set_weights(h, W1_or_U, V, W3, W2, stream=None):
    return _check(load().sffn_set_weights(h, _ptr(W1_or_U), _ptr(V), _ptr(W3), _ptr(W2), _stream(stream)))


def sffn_forward(h, x, y, B: int, stream=None):
    return _check(load().sffn_forward(h, _ptr(x), _ptr(y), B, _stream(stream)))


def sffn_active_counts(h, B: int):
    counts = (ctypes.c_int * B)()
    _check(load().sffn_active_counts(h, counts, B))
    return list(counts)


def sffn_active_mask(h, B: int, H: int):
    import numpy as np
    out = np.zeros((B, H), dtype=np.uint8)
    _check(load().sffn_active_mask(h, out.ctypes.data, B))
    return out


def sffn_synchronize(h):
    return _check(load().sffn_synchronize(h))


def sffn_destroy(h):
    if h:
        load().sffn_destroy(h)


def sffn_debug_timeout_probe(h, limit_us: int, stream=None):
    return _check(load().sffn_debug_timeout_probe(h, limit_us, _stream(stream)))


def sffn_forward_noalloc(W1, W3, W2t, x, y, counts, D: int, H: int, B: int, act: int, dtype: int,
                         stream=None):
    """Forward that allocates no device memory (see include/sffn.h); W2t is W2 transposed, [H, D]."""
    return _check(load().sffn_forward_noalloc(_ptr(W1), _ptr(W3), _ptr(W2t), _ptr(x), _ptr(y),
                                               _ptr(counts), D, H, B, act, dtype, _stream(stream)))


def sffn_set_weights_int8(h, W1q, s1, W3q, s3, W2q, s2, stream=None):
    """Load int8 codes and fp32 scales (W1q, W3q [H, D] with s1, s3 [H]; W2q [D, H] with s2 [D])."""
    return _check(load().sffn_set_weights_int8(h, _ptr(W1q), _ptr(s1), _ptr(W3q), _ptr(s3), _ptr(W2q),
                                                _ptr(s2), _stream(stream)))


def sffn_get_weights_int8(h, W1q, s1, W3q, s3, W2q, s2, stream=None):
    """Copy the handle's int8 codes and scales out (same layout as sffn_set_weights_int8; None skips)."""
    return _check(load().sffn_get_weights_int8(h, _ptr(W1q), _ptr(s1), _ptr(W3q), _ptr(s3), _ptr(W2q),
                                                _ptr(s2), _stream(stream)))


class SparseFFN:
    """One FFN layer held by the library (a wrapper around one handle).

    ``SparseFFN(D, H, r=0, act="relu", dtype="bf16", flags=0)`` (flags: the
    SFFN_GATE_TILED_G | SFFN_GATE_RMSNORM | SFFN_DOUBLE_ACT options); ``set_weights(W1_or_U, V,
    W3, W2)`` with torch tensors in the layer's dtype (W2 as [D, H]);
    ``forward(x, y=None)`` with x [B, D] on the handle's device.  dtype "int8" / "int4":
    weight-only int8 / int4 (bf16 weights given to ``set_weights`` are quantised on the device;
    x and y bf16).
    """

    def __init__(self, D: int, H: int, r: int = 0, act: str = "relu", dtype: str = "bf16", flags: int = 0):
        self.D, self.H, self.r = D, H, r
        self.dtype = dtype
        self.flags = flags
        self._act = {"relu": SFFN_ACT_RELU, "rsp": SFFN_ACT_RSP, "silu": SFFN_ACT_SILU}[act]
        self._dt = {"f32": SFFN_F32, "bf16": SFFN_BF16, "int8": SFFN_I8W, "int4": SFFN_I4W}[dtype]
        self.h = sffn_create_ex(D, H, r, self._act, self._dt, flags)

    def set_weights(self, W1_or_U, V, W3, W2, stream=None):
        for t in (W1_or_U, V, W3, W2):
            if t is not None and hasattr(t, "is_contiguous") and not t.is_contiguous():
                raise ValueError("weights must be contiguous")
        sffn_set_weights(self.h, W1_or_U, V, W3, W2, stream)

    def forward(self, x, y=None, stream=None):
        import torch
        if x.dim() == 1:
            x = x.unsqueeze(0)
        if not x.is_contiguous():
            raise ValueError("x must be contiguous")
        if y is None:
            y = torch.empty_like(x)
        sffn_forward(self.h, x, y, x.shape[0], stream)
        return y

    __call__ = forward

    def active_counts(self, B: int = 1):
        return sffn_active_counts(self.h, B)

    def active_mask(self, B: int = 1):
        return sffn_active_mask(self.h, B, self.H)

    def synchronize(self):
        sffn_synchronize(self.h)

    def set_weights_int8(self, W1q, s1, W3q, s3, W2q, s2, stream=None):
        """Codes and scales quantised elsewhere (int8 [H, D], [H, D], [D, H]; fp32 [H], [H], [D]); on an
        int4 handle one code per byte in [-7, 7] and s1, s3 [H, D // 64] (one per group of 64 columns)."""
        sffn_set_weights_int8(self.h, W1q, s1, W3q, s3, W2q, s2, stream)

    def int8_weights(self, device="cuda"):
        """The handle's codes (one per byte, also for int4) and scales as tensors: (W1q, s1, W3q, s3,
        W2q, s2), W2q as [D, H]; s1, s3 [H], or [H, D // 64] on an int4 handle; with the low-rank gate
        (int8) W1q holds U's codes [H, r] and s1 its scales."""
        import torch
        D, H = self.D, self.H
        ss = (H,) if self.dtype != "int4" else (H, D // INT4_GROUP)
        gk = self.r if self.r > 0 else D  # the low-rank gate: U's codes [H, r]
        out = (torch.empty(H, gk, dtype=torch.int8, device=device), torch.empty(ss, device=device),
               torch.empty(H, D, dtype=torch.int8, device=device), torch.empty(ss, device=device),
               torch.empty(D, H, dtype=torch.int8, device=device), torch.empty(D, device=device))
        sffn_get_weights_int8(self.h, *out)
        return out

    def set_live_threshold(self, thr: float):
        """Units with |A(z)| <= thr are skipped (0: the exact skip of ReLU / R-S+)."""
        sffn_set_live_threshold(self.h, thr)

    def set_live_fraction_hint(self, rho: float):
        """Expected live fraction per token (negative: unknown); picks the kernels of 3..16-token batches."""
        sffn_set_live_fraction_hint(self.h, rho)

    def close(self):
        if getattr(self, "h", None):
            sffn_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
