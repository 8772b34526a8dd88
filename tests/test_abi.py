"""The C ABI: the library loads, exports what include/qk.h declares, and rejects
bad arguments with status codes before touching the GPU (no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    src = open(os.path.join(ROOT, "include", "qk.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(qk_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_entry_points():
    names = header_functions()
    for n in ("qk_dequant_q4k", "qk_dequant_q6k", "qk_matmul_q4k", "qk_matmul_q6k", "qk_gateup_swiglu_q4k",
              "qk_get_device_status", "qk_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(qk_lib):
    L = qk_lib.lib()
    for name in header_functions():
        assert hasattr(L, name), name
    assert set(qk_lib.SYMBOLS) <= set(header_functions())


def test_status_strings(qk_lib):
    L = qk_lib.lib()
    for code in range(-8, 1):
        s = L.qk_status_string(code).decode()
        assert s.startswith("QK_") and "unknown" not in s
    assert "unknown" in L.qk_status_string(-99).decode()
    assert L.qk_version() >= 100


# Fake, never-dereferenced addresses: validation must reject the call first.
A16, A8 = 0x10000, 0x10008


@pytest.mark.parametrize("fn", ["qk_matmul_q4k", "qk_matmul_q6k"])
def test_matmul_rejects_bad_arguments_on_the_host(qk_lib, fn):
    f = getattr(qk_lib.lib(), fn)
    assert f(A16, A16, A16, 4, 8, 300, None) == -3        # K % 256
    assert f(A16, A16, A16, 4, 8, 0, None) == -3          # K = 0
    assert f(A16, A16, A16, -1, 8, 256, None) == -3       # negative M
    assert f(A16, A16, A16, 4, -8, 256, None) == -3       # negative N
    assert f(A16, A16, A16, 1 << 31, 8, 256, None) == -3  # too large
    assert f(None, A16, A16, 4, 8, 256, None) == -1       # NULL weights
    assert f(A16, None, A16, 4, 8, 256, None) == -1
    assert f(A16, A16, None, 4, 8, 256, None) == -1
    assert f(A8, A16, A16, 4, 8, 256, None) == -2         # misaligned
    assert f(A16, A8, A16, 4, 8, 256, None) == -2
    assert f(A16, A16, A8, 4, 8, 256, None) == -2
    assert f(None, None, None, 0, 8, 256, None) == 0      # M = 0: no-op
    assert f(None, None, None, 4, 0, 256, None) == 0      # N = 0: no-op


def test_gateup_and_dequant_reject_bad_arguments_on_the_host(qk_lib):
    L = qk_lib.lib()
    assert L.qk_gateup_swiglu_q4k(A16, None, A16, A16, 4, 8, 256, None) == -1
    assert L.qk_gateup_swiglu_q4k(A16, A8, A16, A16, 4, 8, 256, None) == -2
    assert L.qk_gateup_swiglu_q4k(A16, A16, A16, A16, 4, 8, 100, None) == -3
    assert L.qk_gateup_swiglu_q4k(None, None, None, None, 0, 8, 256, None) == 0
    for f in (L.qk_dequant_q4k, L.qk_dequant_q6k):
        assert f(None, 0, None, None) == 0
        assert f(None, 4, A16, None) == -1
        assert f(A16, 4, None, None) == -1
        assert f(A8, 4, A16, None) == -2
        assert f(A16, -1, A16, None) == -3
        assert f(A16, 1 << 61, A16, None) == -3


def test_binding_raises_with_the_status(qk_lib):
    with pytest.raises(qk_lib.QKError) as e:
        qk_lib.qk_matmul_q4k(A16, A16, A16, 4, 8, 300, stream=0)
    assert e.value.status == -3


def test_batch_rejects_bad_arguments_on_the_host(qk_lib):
    L = qk_lib.lib()
    D = qk_lib.qk_matmul_desc
    assert L.qk_matmul_batch(None, 0, None) == 0
    assert L.qk_matmul_batch(None, 2, None) == -1
    assert L.qk_matmul_batch(None, -1, None) == -3
    arr = (D * 2)(D(0, A16, None, A16, A16, 1, 8, 256), D(7, A16, None, A16, A16, 1, 8, 256))
    assert L.qk_matmul_batch(arr, 2, None) == -3                       # unknown qtype
    arr = (D * 1)(D(1, A16, A16, A16, A16, 1, 8, 256))
    assert L.qk_matmul_batch(arr, 1, None) == -3                       # gate/up must be Q4_K
    arr = (D * 1)(D(0, A16, None, A16, A8, 1, 8, 256))
    assert L.qk_matmul_batch(arr, 1, None) == -2
    arr = (D * 1)(D(0, A16, None, A16, A16, 1, 8, 300))
    assert L.qk_matmul_batch(arr, 1, None) == -3
