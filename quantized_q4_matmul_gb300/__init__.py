"""Python binding of libqk, the GB300 (sm_103a) quantized Q4_K / Q6_K matmul library.

This module only marshals arguments: every step of the computation runs in the
CUDA kernels behind the C ABI declared in ``include/qk.h``.  Functions take
torch tensors (device memory) or raw integer addresses, plus an optional CUDA
stream (default: torch's current stream), and raise ``QKError`` on any non-zero
status.  There is no CPU fallback: if ``libqk.so`` is missing or cannot be
loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "QKError", "lib", "lib_path", "qk_dequant_q4k", "qk_dequant_q6k", "qk_matmul_q4k", "qk_matmul_q6k",
    "qk_gateup_swiglu_q4k", "qk_matmul_batch", "qk_get_device_status", "qk_debug_wait_timeout",
    "qk_status_string", "qk_version", "QK_BLOCK_BYTES", "qk_matmul_desc",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
QK_BLOCK_BYTES = {"q4k": 144, "q6k": 210}

SYMBOLS = ("qk_dequant_q4k", "qk_dequant_q6k", "qk_matmul_q4k", "qk_matmul_q6k", "qk_gateup_swiglu_q4k",
           "qk_matmul_batch", "qk_get_device_status", "qk_debug_wait_timeout", "qk_status_string", "qk_version")

QK_Q4_K, QK_Q6_K = 0, 1


class qk_matmul_desc(ctypes.Structure):
    """Mirror of ``qk_matmul_desc`` in include/qk.h."""
    _fields_ = [("qtype", ctypes.c_int), ("blocks", ctypes.c_void_p), ("up_blocks", ctypes.c_void_p),
                ("x_f16", ctypes.c_void_p), ("y", ctypes.c_void_p), ("M", ctypes.c_int64),
                ("N", ctypes.c_int64), ("K", ctypes.c_int64)]


class QKError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s failed: %s (%d)" % (where, qk_status_string(status), status))


def lib_path() -> str:
    return os.environ.get("QK_LIB", os.path.join(_HERE, "libqk.so"))


_lib = None


def lib():
    """The loaded libqk (raises if it has not been built)."""
    global _lib
    if _lib is None:
        path = lib_path()
        if not os.path.exists(path):
            raise RuntimeError("libqk.so not found at %s: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`" % path)
        L = ctypes.CDLL(path)
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        for name in ("qk_dequant_q4k", "qk_dequant_q6k"):
            f = getattr(L, name)
            f.restype, f.argtypes = i32, [vp, i64, vp, vp]
        for name in ("qk_matmul_q4k", "qk_matmul_q6k"):
            f = getattr(L, name)
            f.restype, f.argtypes = i32, [vp, vp, vp, i64, i64, i64, vp]
        L.qk_gateup_swiglu_q4k.restype = i32
        L.qk_gateup_swiglu_q4k.argtypes = [vp, vp, vp, vp, i64, i64, i64, vp]
        L.qk_matmul_batch.restype = i32
        L.qk_matmul_batch.argtypes = [ctypes.POINTER(qk_matmul_desc), i32, vp]
        L.qk_get_device_status.restype, L.qk_get_device_status.argtypes = i32, [vp]
        L.qk_debug_wait_timeout.restype, L.qk_debug_wait_timeout.argtypes = i32, [i64, vp]
        L.qk_status_string.restype, L.qk_status_string.argtypes = ctypes.c_char_p, [i32]
        L.qk_version.restype, L.qk_version.argtypes = i32, []
        _lib = L
    return _lib


def _addr(t) -> int:
    if t is None:
        return 0
    if isinstance(t, int):
        return t
    return int(t.data_ptr())


def _stream(stream) -> int:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def _check(status: int, where: str) -> None:
    if status != 0:
        raise QKError(status, where)


def qk_status_string(status: int) -> str:
    return lib().qk_status_string(int(status)).decode()


def qk_version() -> int:
    return int(lib().qk_version())


def qk_dequant_q4k(blocks, n_blocks: int, out, stream=None) -> None:
    _check(lib().qk_dequant_q4k(_addr(blocks), int(n_blocks), _addr(out), _stream(stream)), "qk_dequant_q4k")


def qk_dequant_q6k(blocks, n_blocks: int, out, stream=None) -> None:
    _check(lib().qk_dequant_q6k(_addr(blocks), int(n_blocks), _addr(out), _stream(stream)), "qk_dequant_q6k")


def qk_matmul_q4k(blocks, x_f16, y, M: int, N: int, K: int, stream=None) -> None:
    _check(lib().qk_matmul_q4k(_addr(blocks), _addr(x_f16), _addr(y), int(M), int(N), int(K), _stream(stream)),
           "qk_matmul_q4k")


def qk_matmul_q6k(blocks, x_f16, y, M: int, N: int, K: int, stream=None) -> None:
    _check(lib().qk_matmul_q6k(_addr(blocks), _addr(x_f16), _addr(y), int(M), int(N), int(K), _stream(stream)),
           "qk_matmul_q6k")


def qk_gateup_swiglu_q4k(gate_blocks, up_blocks, x_f16, y_f16, M: int, N_ff: int, K: int, stream=None) -> None:
    _check(lib().qk_gateup_swiglu_q4k(_addr(gate_blocks), _addr(up_blocks), _addr(x_f16), _addr(y_f16), int(M),
                                      int(N_ff), int(K), _stream(stream)), "qk_gateup_swiglu_q4k")


def qk_matmul_batch(problems, stream=None) -> None:
    """Run independent problems in as few launches as possible.  Each problem is
    a dict with keys qtype ("q4k"/"q6k" or 0/1), blocks, x_f16, y, M, N, K and
    optionally up_blocks (fused gate/up + SwiGLU, fp16 y)."""
    arr = (qk_matmul_desc * max(1, len(problems)))()
    for i, p in enumerate(problems):
        qt = p["qtype"]
        qt = {"q4k": QK_Q4_K, "q6k": QK_Q6_K}.get(qt, qt)
        arr[i] = qk_matmul_desc(int(qt), _addr(p["blocks"]), _addr(p.get("up_blocks")), _addr(p["x_f16"]),
                                _addr(p["y"]), int(p["M"]), int(p["N"]), int(p["K"]))
    _check(lib().qk_matmul_batch(arr, len(problems), _stream(stream)), "qk_matmul_batch")


def qk_get_device_status(stream=None) -> None:
    _check(lib().qk_get_device_status(_stream(stream)), "qk_get_device_status")


def qk_debug_wait_timeout(limit_ns: int, stream=None) -> None:
    """Enqueue a kernel whose only wait times out after ``limit_ns`` (see include/qk.h)."""
    _check(lib().qk_debug_wait_timeout(int(limit_ns), _stream(stream)), "qk_debug_wait_timeout")
