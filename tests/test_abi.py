"""The C ABI library loads and exports every function include/mars.h declares
(CPU only: no kernel is launched)."""
import ctypes
import os
import re

import pytest

from token_decoding_gb300 import build as mars_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mars.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mars_[a-z_0-9]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    path = mars_build.build()
    return ctypes.CDLL(path)


def test_header_declares_the_boundary():
    assert declared_functions() == sorted([
        "mars_accept", "mars_accept_ex", "mars_accept_margin", "mars_accept_noalloc", "mars_accept_workspace_size",
        "mars_decode_attn", "mars_decode_attn_deferred", "mars_decode_attn_workspace_size", "mars_last_cuda_error", "mars_lm_head_accept",
        "mars_lm_head_accept_workspace_size", "mars_selftest_wait_timeout",
        "mars_train_attn_bwd", "mars_train_attn_bwd_workspace_size", "mars_status_string", "mars_train_attn", "mars_version"])


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings_and_version(lib):
    lib.mars_status_string.restype = ctypes.c_char_p
    for code in range(7):
        assert lib.mars_status_string(code)
    assert b"unknown" in lib.mars_status_string(99)
    assert lib.mars_version() == 100


def test_workspace_size_is_host_only(lib):
    lib.mars_decode_attn_workspace_size.restype = ctypes.c_size_t
    assert lib.mars_decode_attn_workspace_size(64, 8, 28, 128, 4096) == 0  # the merge never leaves the cluster
    lib.mars_accept_workspace_size.restype = ctypes.c_size_t
    assert lib.mars_accept_workspace_size(0, 4, 10) == 0
    n = lib.mars_accept_workspace_size(64, 8, 152064)
    assert 0 < n < 8 * 1024 * 1024 and n % 256 == 0


def test_invalid_arguments_are_rejected_before_any_cuda_call(lib):
    """Null pointers and unsupported shapes return MARS_ERR_INVALID_ARG on the host."""
    P = ctypes.c_void_p
    f = lib.mars_train_attn
    f.argtypes = [P, P, P, P, P] + [ctypes.c_int] * 6 + [ctypes.c_float, P, P]
    assert f(None, None, None, None, None, 1, 64, 4, 1, 1, 64, 0.125, None, None) == 1
    fake = P(4096)
    assert f(fake, fake, fake, fake, None, 1, 64, 4, 1, 1, 96, 0.125, None, None) == 1    # D = 96
    assert f(fake, fake, fake, fake, None, 1, 64, 4, 3, 2, 64, 0.125, None, None) == 1    # Hq % Hkv
    assert f(P(4097), fake, fake, fake, None, 1, 64, 4, 1, 1, 64, 0.125, None, None) == 1  # misaligned
    d = lib.mars_decode_attn
    d.argtypes = [P] * 6 + [ctypes.c_int] * 7 + [ctypes.c_float, P, P, P]
    assert d(fake, fake, fake, fake, fake, fake, 1, 17, 4, 1, 64, 100, 50, 0.1, fake, None, None) == 1  # B > 16
    assert d(fake, fake, fake, fake, fake, fake, 1, 4, 4, 1, 64, 100, 101, 0.1, fake, None, None) == 1  # max_len > cap
    a = lib.mars_accept
    a.argtypes = ([P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_float] + [P] * 5 +
                  [ctypes.c_int] * 3 + [P] * 5 + [ctypes.c_size_t, P])
    assert a(fake, 1, 4, 100, 0.5, fake, fake, fake, fake, fake, 1, 64, 10,
             fake, fake, fake, None, fake, 16, None) == 2  # workspace too small
    assert a(fake, 1, 0, 100, 0.5, fake, fake, fake, fake, fake, 1, 64, 10,
             fake, fake, fake, None, fake, 1 << 20, None) == 1  # B = 0


def test_python_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    import token_decoding_gb300._lib as L

    monkeypatch.setattr(L, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(L, "_lib", None)
    monkeypatch.setattr(L, "_fns", {})
    with pytest.raises(RuntimeError, match="no fallback"):
        L.version()
