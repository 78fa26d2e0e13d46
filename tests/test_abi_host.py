"""The C-ABI library on the host: it loads, exports every symbol that
include/fa.h declares, and rejects bad arguments before any CUDA work.
No call here reaches a kernel, so no GPU is needed."""

import ctypes
import os
import re

import pytest

from exact_attention_84_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))
           if f.endswith(".h")]


def declared_functions():
    names = []
    for h in HEADERS:
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(fa_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    return _lib.load()


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert "fa_forward" in names and "fa_decode" in names and "fa_backward" in names
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(_lib.SIGNATURES) == names


FAKE = 0x10000          # aligned, never dereferenced: validation fails first
MIS = 0x10001


def test_forward_validation(lib):
    E = _lib
    assert E.fa_forward(None, FAKE, FAKE, FAKE, None, 1, 1, 8, 128, 0.1, 0, None) == E.FA_ERR_INVALID_ARG
    assert "null" in E.fa_last_error()
    assert E.fa_forward(FAKE, FAKE, FAKE, FAKE, None, 1, 1, 8, 64, 0.1, 0, None) == E.FA_ERR_UNSUPPORTED
    assert E.fa_forward(FAKE, FAKE, FAKE, FAKE, None, 0, 1, 8, 128, 0.1, 0, None) == E.FA_ERR_INVALID_ARG
    assert E.fa_forward(FAKE, FAKE, FAKE, FAKE, None, 1, 1, 8, 128, -1.0, 0, None) == E.FA_ERR_INVALID_ARG
    assert E.fa_forward(FAKE, FAKE, FAKE, FAKE, None, 1, 1, 8, 128, float("nan"), 0, None) == E.FA_ERR_INVALID_ARG
    assert E.fa_forward(FAKE, FAKE, FAKE, FAKE, None, 1, 1, 8, 128, 0.1, 2, None) == E.FA_ERR_INVALID_ARG
    assert E.fa_forward(FAKE, MIS, FAKE, FAKE, None, 1, 1, 8, 128, 0.1, 0, None) == E.FA_ERR_INVALID_ARG
    assert "aligned" in E.fa_last_error()
    assert E.fa_forward_fp32(FAKE, FAKE, FAKE, FAKE, None, 1, 1, 8, 48, 0.1, 0, None) == E.FA_ERR_UNSUPPORTED
    assert E.fa_forward_fp32(FAKE, FAKE, None, FAKE, None, 1, 1, 8, 64, 0.1, 0, None) == E.FA_ERR_INVALID_ARG


def test_backward_validation(lib):
    E = _lib
    args = [FAKE] * 9
    assert E.fa_backward(*args[:4], None, *args[5:], 1, 1, 8, 128, 0.1, 0, None) == E.FA_ERR_INVALID_ARG
    assert E.fa_backward(*args, 1, 1, 8, 96, 0.1, 0, None) == E.FA_ERR_UNSUPPORTED
    # caller workspace too small / misaligned
    assert E.fa_backward_ex(*args, 1, 1, 8, 128, 0.1, 0, FAKE, 16, None) == E.FA_ERR_INVALID_ARG
    assert "workspace" in E.fa_last_error()
    need = E.fa_workspace_size(E.FA_OP_BACKWARD, 1, 1, 8, 128, 0)
    assert E.fa_backward_ex(*args, 1, 1, 8, 128, 0.1, 0, FAKE + 16, need, None) == E.FA_ERR_INVALID_ARG


def test_decode_validation(lib):
    E = _lib
    assert E.fa_decode(FAKE, FAKE, FAKE, FAKE, 1, 1, 100, 128, 0, None) == E.FA_ERR_INVALID_ARG
    assert E.fa_decode(FAKE, FAKE, FAKE, FAKE, 1, 1, 100, 128, 101, None) == E.FA_ERR_INVALID_ARG
    assert E.fa_decode(FAKE, FAKE, FAKE, FAKE, 1, 1, 5000, 128, 1025, None) == E.FA_ERR_INVALID_ARG
    assert "num_splits" in E.fa_last_error()
    assert E.fa_decode(FAKE, FAKE, FAKE, FAKE, 1, 1, 100, 64, 4, None) == E.FA_ERR_UNSUPPORTED
    assert E.fa_decode(FAKE, None, FAKE, FAKE, 1, 1, 100, 128, 4, None) == E.FA_ERR_INVALID_ARG
    assert E.fa_decode_ex(FAKE, FAKE, FAKE, FAKE, None, 1, 1, 100, 128, 4, 0.1, FAKE, 8, None) == E.FA_ERR_INVALID_ARG


def test_gqa_window_validation(lib):
    E = _lib
    f = E.fa_forward_gqa
    # Hq must be a multiple of Hkv
    assert f(FAKE, FAKE, FAKE, FAKE, None, 1, 6, 4, 8, 128, 0.1, 1, 0, None, None) == E.FA_ERR_INVALID_ARG
    assert "multiple" in E.fa_last_error()
    assert f(FAKE, FAKE, FAKE, FAKE, None, 1, 4, 0, 8, 128, 0.1, 1, 0, None, None) == E.FA_ERR_INVALID_ARG
    # a window needs the causal mask; negative windows are invalid
    assert f(FAKE, FAKE, FAKE, FAKE, None, 1, 4, 2, 8, 128, 0.1, 0, 4, None, None) == E.FA_ERR_UNSUPPORTED
    assert "causal" in E.fa_last_error()
    assert f(FAKE, FAKE, FAKE, FAKE, None, 1, 4, 2, 8, 128, 0.1, 1, -1, None, None) == E.FA_ERR_INVALID_ARG
    assert f(FAKE, FAKE, FAKE, FAKE, None, 1, 4, 2, 8, 64, 0.1, 1, 4, None, None) == E.FA_ERR_UNSUPPORTED
    args = [FAKE] * 9
    b = E.fa_backward_gqa
    assert b(*args, 1, 4, 3, 8, 128, 0.1, 1, 0, None, 0, None, 0, None) == E.FA_ERR_INVALID_ARG
    assert b(*args, 1, 4, 2, 8, 128, 0.1, 0, 2, None, 0, None, 0, None) == E.FA_ERR_UNSUPPORTED
    assert b(*args, 1, 4, 2, 8, 128, 0.1, 1, 2, None, 0, FAKE, 16, None) == E.FA_ERR_INVALID_ARG
    assert "workspace" in E.fa_last_error()
    # misaligned slopes
    assert f(FAKE, FAKE, FAKE, FAKE, None, 1, 4, 2, 8, 128, 0.1, 1, 0, MIS, None) == E.FA_ERR_INVALID_ARG
    p8 = E.fa_forward_fp8
    assert p8(FAKE, FAKE, FAKE, FAKE, None, 1, 2, 2, 8, 128, 0.1, 1.0, 0.0, 1.0, 1, 0, None, None, 0,
              None) == E.FA_ERR_INVALID_ARG
    assert "descale" in E.fa_last_error()
    assert p8(FAKE, FAKE, FAKE, FAKE, None, 1, 2, 2, 8, 128, 0.1, 1.0, 1.0, 1.0, 0, 3, None, None, 0,
              None) == E.FA_ERR_UNSUPPORTED
    assert p8(FAKE, FAKE, FAKE, FAKE, None, 1, 2, 2, 8, 128, 0.1, 1.0, 1.0, 1.0, 1, 0, None, FAKE, 8,
              None) == E.FA_ERR_INVALID_ARG
    d = E.fa_decode_gqa
    assert d(FAKE, FAKE, FAKE, FAKE, None, 1, 8, 3, 100, 128, 2, 0.1, None, None, 0, None) == E.FA_ERR_INVALID_ARG
    assert d(FAKE, FAKE, FAKE, FAKE, None, 1, 8, 2, 100, 128, -1, 0.1, None, None, 0, None) == E.FA_ERR_INVALID_ARG
    assert d(FAKE, FAKE, FAKE, FAKE, None, 1, 8, 2, 100, 128, 2, 0.1, None, FAKE, 8, None) == E.FA_ERR_INVALID_ARG
    assert d(FAKE, None, FAKE, FAKE, None, 1, 8, 2, 100, 128, 2, 0.1, None, None, 0, None) == E.FA_ERR_INVALID_ARG


def test_size_limits(lib):
    """Sizes past what the kernels index are refused before any launch."""
    E = _lib
    assert E.fa_forward(FAKE, FAKE, FAKE, FAKE, None, 1, 1, (1 << 30) + 1, 128, 0.1, 0, None) == E.FA_ERR_UNSUPPORTED
    assert E.fa_forward(FAKE, FAKE, FAKE, FAKE, None, 1 << 16, 1 << 15, 8, 128, 0.1, 0, None) == E.FA_ERR_UNSUPPORTED
    assert E.fa_decode(FAKE, FAKE, FAKE, FAKE, 256, 256, 100, 128, 1, None) == E.FA_ERR_UNSUPPORTED
    assert E.fa_forward_fp32(FAKE, FAKE, FAKE, FAKE, None, 256, 256, 8, 64, 0.1, 0, None) == E.FA_ERR_UNSUPPORTED
    # per-dimension limits pass, the thread-block count does not
    assert E.fa_forward(FAKE, FAKE, FAKE, FAKE, None, 1 << 10, 1 << 10, 1 << 20, 128, 0.1, 0, None) == E.FA_ERR_UNSUPPORTED
    assert "2^31" in E.fa_last_error()
    args9 = [FAKE] * 9
    assert E.fa_backward(*args9, 1 << 10, 1 << 10, 1 << 20, 128, 0.1, 1, None) == E.FA_ERR_UNSUPPORTED
    assert E.fa_decode_noalloc(FAKE, FAKE, FAKE, FAKE, None, 64, 32, 32768, 128, 16, 0.1, None) == E.FA_ERR_UNSUPPORTED
    assert "scratch" in E.fa_last_error()


def test_decode_splits_choice(lib):
    E = _lib
    assert E.fa_decode_splits(0, 8, 2, 100) == 0 and E.fa_decode_splits(1, 8, 3, 100) == 0
    for B, Hq, Hkv, L in ((64, 32, 32, 32768), (64, 32, 8, 32768), (1, 1, 1, 10), (1, 64, 1, 300000)):
        s = E.fa_decode_splits(B, Hq, Hkv, L)
        assert 1 <= s <= min(L, 1024) and (s == 1 or L // s >= 512)


def test_selftest_validation(lib):
    E = _lib
    assert E.fa_selftest_timeout(0, None) == E.FA_ERR_INVALID_ARG
    assert E.fa_selftest_timeout(20000, None) == E.FA_ERR_INVALID_ARG


def test_workspace_sizes(lib):
    E = _lib
    assert E.fa_workspace_size(E.FA_OP_FORWARD, 1, 1, 8, 128, 0) == 0
    bwd = E.fa_workspace_size(E.FA_OP_BACKWARD, 8, 32, 4096, 128, 0)
    rows = 8 * 32 * 4096
    assert bwd >= rows * 128 * 4 + rows * 4 and bwd % 256 == 0
    dec = E.fa_workspace_size(E.FA_OP_DECODE, 64, 32, 32768, 128, 16)
    assert dec >= 64 * 32 * 16 * (128 + 1) * 4
    assert E.fa_workspace_size(E.FA_OP_DECODE, 64, 32, 32768, 128, 0) == 0
    assert E.fa_workspace_size(7, 1, 1, 8, 128, 1) == 0


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        _lib.load()
