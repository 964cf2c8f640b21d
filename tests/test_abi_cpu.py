"""The C-ABI library builds, loads without a GPU and exports every declared symbol."""
import ctypes
import os
import re
import subprocess

import pytest

import activation_sparse_gated_gb300 as sffn
from activation_sparse_gated_gb300 import build as libbuild

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "sffn.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sffn_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return sffn.load()


def test_header_declares_the_binding_exports():
    assert declared_functions() == sorted(sffn.EXPORTS)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", sffn.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (sffn_\w+)", out))
    assert set(declared_functions()) <= exported


def test_constants_match_header():
    text = open(HEADER).read()
    for name in ("SFFN_F32", "SFFN_BF16", "SFFN_ACT_RELU", "SFFN_ACT_RSP", "SFFN_OK", "SFFN_ERR_ARG",
                 "SFFN_ERR_ALIGN", "SFFN_ERR_DTYPE", "SFFN_ERR_CUDA", "SFFN_ERR_TIMEOUT",
                 "SFFN_ERR_STATE", "SFFN_ERR_NOMEM", "SFFN_ERR_DEVICE", "SFFN_GATE_TILED_G", "SFFN_GATE_RMSNORM",
                 "SFFN_DOUBLE_ACT", "SFFN_DETERMINISTIC", "SFFN_ACT_SILU", "SFFN_I8W", "SFFN_I4W"):
        m = re.search(rf"\b{name}\s*=\s*(-?\d+)", text)
        assert m and int(m.group(1)) == getattr(sffn, name), name
    assert int(re.search(r"#define SFFN_MAX_BATCH (\d+)", text).group(1)) == sffn.SFFN_MAX_BATCH


def test_host_only_calls(lib):
    assert sffn.sffn_version() == 100
    assert sffn.sffn_strerror(0) == "success"
    assert "timed out" in sffn.sffn_strerror(sffn.SFFN_ERR_TIMEOUT)
    assert "check failed" in sffn.sffn_strerror(sffn.SFFN_ERR_DEVICE)
    assert sffn.sffn_strerror(12345) == "unknown status"


def test_null_handle_is_rejected_on_host(lib):
    # argument checks happen before any CUDA call
    assert lib.sffn_forward(None, None, None, 1, None) == sffn.SFFN_ERR_ARG
    assert lib.sffn_set_weights(None, None, None, None, None, None) == sffn.SFFN_ERR_ARG
    assert lib.sffn_active_counts(None, None, 1) == sffn.SFFN_ERR_ARG
    assert lib.sffn_synchronize(None) == sffn.SFFN_ERR_ARG
    assert lib.sffn_set_weights_int8(None, None, None, None, None, None, None, None) == sffn.SFFN_ERR_ARG
    assert lib.sffn_get_weights_int8(None, None, None, None, None, None, None, None) == sffn.SFFN_ERR_ARG
    lib.sffn_destroy(None)


@pytest.mark.parametrize("args", [(0, 64, 0, 0, 1), (12, 64, 0, 0, 1), (8192, 64, 0, 0, 1),
                                  (4096, 64, 0, 0, 0), (64, 0, 0, 0, 1), (64, 64, 12, 0, 1),
                                  (64, 64, 128, 0, 1), (64, 64, 0, 3, 1), (64, 64, 0, 0, 7),
                                  (64, 64, 8, 0, 2), (24, 64, 0, 0, 2), (8192, 64, 0, 0, 2)])
def test_create_rejects_bad_shapes_before_touching_the_device(lib, args):
    h = lib.sffn_create(*args)
    assert not h
    assert sffn.sffn_last_error()


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    monkeypatch.setattr(sffn, "_lib", None)
    with pytest.raises(ImportError):
        sffn.load(str(tmp_path / "nope.so"))


def test_noalloc_rejects_bad_sizes_on_host(lib):
    # size checks come before any CUDA call, so they work without a GPU
    for D, H, B, dt in ((8192, 8, 1, 1), (4096, 8, 1, 0), (12, 8, 1, 1), (64, 0, 1, 1), (64, 8, 0, 1),
                        (64, 8, 129, 1)):
        rc = lib.sffn_forward_noalloc(16, 16, 16, 16, 4096, None, D, H, B, 0, dt, None)
        assert rc == sffn.SFFN_ERR_ARG, (D, H, B, dt)
        assert "sffn_forward_noalloc" in sffn.sffn_last_error()


@pytest.mark.parametrize("r,flags", [(64, 16), (64, -1), (0, sffn.SFFN_GATE_TILED_G), (0, sffn.SFFN_GATE_RMSNORM)])
def test_create_ex_rejects_bad_options_before_touching_the_device(lib, r, flags):
    """Unknown option bits, or a low-rank option without a low-rank gate."""
    h = lib.sffn_create_ex(512, 1024, r, sffn.SFFN_ACT_RELU, sffn.SFFN_BF16, flags)
    assert not h
    assert "flags" in sffn.sffn_last_error() or "low-rank" in sffn.sffn_last_error()


@pytest.mark.parametrize("dtype", [sffn.SFFN_F32, sffn.SFFN_I8W, sffn.SFFN_I4W])
def test_deterministic_option_is_bf16_only_checked_on_host(lib, dtype):
    h = lib.sffn_create_ex(512, 1024, 0, sffn.SFFN_ACT_RELU, dtype, sffn.SFFN_DETERMINISTIC)
    assert not h
    msg = sffn.sffn_last_error()
    assert "deterministic" in msg or (dtype in (sffn.SFFN_I8W, sffn.SFFN_I4W) and "int" in msg), msg


def test_live_threshold_rejects_bad_values_on_host(lib):
    import ctypes
    assert lib.sffn_set_live_threshold(None, ctypes.c_float(0.1)) == sffn.SFFN_ERR_ARG


def test_live_fraction_hint_rejects_a_null_handle_on_host(lib):
    import ctypes
    assert lib.sffn_set_live_fraction_hint(None, ctypes.c_float(0.1)) == sffn.SFFN_ERR_ARG


@pytest.mark.parametrize("args", [(96, 64, 0, 0), (64, 64, 8, 0), (64, 64, 0, 8)])
def test_int4_handle_shape_rules_checked_on_host(lib, args):
    """int4 weights: standard gate only, D a multiple of 64 (the scale groups), no low-rank option."""
    D, H, r, flags = args
    h = lib.sffn_create_ex(D, H, r, sffn.SFFN_ACT_RELU, sffn.SFFN_I4W, flags)
    assert not h
    assert "int4" in sffn.sffn_last_error()


@pytest.mark.parametrize("args", [(512, 64, 24, 0), (512, 64, 64, sffn.SFFN_GATE_TILED_G),
                                  (512, 64, 64, sffn.SFFN_GATE_RMSNORM), (520, 64, 0, 0)])
def test_int8_handle_shape_rules_checked_on_host(lib, args):
    """int8 weights: D and r multiples of 16 (16-code pieces), the low-rank gate in its plain form only."""
    D, H, r, flags = args
    h = lib.sffn_create_ex(D, H, r, sffn.SFFN_ACT_RELU, sffn.SFFN_I8W, flags)
    assert not h
    assert "int8" in sffn.sffn_last_error()
