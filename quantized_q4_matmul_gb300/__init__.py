"""Python binding of libqk, the GB300 (sm_103a) quantized Q4_K / Q6_K matmul library.

This module only marshals arguments: every step of the computation runs in the
CUDA kernels behind the C ABI declared in ``include/qk.h``.  Functions take
torch tensors (device memory) or raw integer addresses, plus an optional CUDA
stream (default: torch's current stream), and raise ``QKError`` on any non-zero
status.  A tensor argument must be contiguous and large enough for the call
(x and fp16 outputs fp16, or its bits as int16 / uint16; fp32 outputs
float32), else ``ValueError`` is raised before the library is called; raw
addresses are the caller's responsibility.  There is no CPU fallback: if ``libqk.so`` is missing or cannot be
loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "QKError", "lib", "lib_path", "qk_dequant_q4k", "qk_dequant_q6k", "qk_matmul_q4k", "qk_matmul_q6k",
    "qk_gateup_swiglu_q4k", "qk_matmul_batch", "qk_matmul_batch_q8x", "qk_matmul_q8x_q4k", "qk_matmul_q8x_q6k",
    "qk_get_device_status", "qk_debug_wait_timeout",
    "qk_decode_uses_gemv", "qk_uses_gemv", "qk_gemm_plan", "qk_rmsnorm_matmul_batch", "qk_rmsnorm_matmul_q4k",
    "qk_rmsnorm_matmul_q6k", "qk_rmsnorm_gateup_swiglu_q4k", "qk_rmsnorm_scratch_bytes",
    "qk_rmsnorm_matmul_batch_static", "qk_status_string", "qk_version", "QK_BLOCK_BYTES", "qk_matmul_desc",
    "qk_gemm_plan_info", "qk_gqa_attention",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
QK_BLOCK_BYTES = {"q4k": 144, "q6k": 210}

SYMBOLS = ("qk_dequant_q4k", "qk_dequant_q6k", "qk_matmul_q4k", "qk_matmul_q6k", "qk_gateup_swiglu_q4k",
           "qk_matmul_batch", "qk_matmul_batch_q8x", "qk_matmul_q8x_q4k", "qk_matmul_q8x_q6k",
           "qk_get_device_status", "qk_debug_wait_timeout", "qk_decode_uses_gemv",
           "qk_uses_gemv", "qk_gemm_plan", "qk_rmsnorm_matmul_batch", "qk_rmsnorm_matmul_q4k",
           "qk_rmsnorm_matmul_q6k", "qk_rmsnorm_gateup_swiglu_q4k", "qk_rmsnorm_scratch_bytes",
    "qk_rmsnorm_matmul_batch_static", "qk_status_string",
           "qk_version", "qk_gqa_attention")

QK_Q4_K, QK_Q6_K = 0, 1


class qk_matmul_desc(ctypes.Structure):
    """Mirror of ``qk_matmul_desc`` in include/qk.h."""
    _fields_ = [("qtype", ctypes.c_int), ("blocks", ctypes.c_void_p), ("up_blocks", ctypes.c_void_p),
                ("x_f16", ctypes.c_void_p), ("y", ctypes.c_void_p), ("M", ctypes.c_int64),
                ("N", ctypes.c_int64), ("K", ctypes.c_int64)]


class qk_gemm_plan_info(ctypes.Structure):
    """Mirror of ``qk_gemm_plan_info`` in include/qk.h."""
    _fields_ = [(n, ctypes.c_int) for n in ("token_tile", "x_stages", "a_stages", "packed_stages", "a_in_tmem",
                                             "tmem_cols", "smem_bytes", "max_ctas_per_sm")]


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
        L.qk_matmul_batch_q8x.restype = i32
        L.qk_matmul_batch_q8x.argtypes = [ctypes.POINTER(qk_matmul_desc), i32, vp]
        for f in (L.qk_matmul_q8x_q4k, L.qk_matmul_q8x_q6k):
            f.restype, f.argtypes = i32, [vp, vp, vp, i64, i64, i64, vp]
        L.qk_get_device_status.restype, L.qk_get_device_status.argtypes = i32, [vp]
        L.qk_debug_wait_timeout.restype, L.qk_debug_wait_timeout.argtypes = i32, [i64, vp]
        L.qk_decode_uses_gemv.restype, L.qk_decode_uses_gemv.argtypes = i32, [i32, i32, i64]
        L.qk_uses_gemv.restype, L.qk_uses_gemv.argtypes = i32, [i32, i32, i64, i64]
        f32 = ctypes.c_float
        L.qk_rmsnorm_matmul_batch.restype = i32
        L.qk_rmsnorm_matmul_batch.argtypes = [ctypes.POINTER(qk_matmul_desc), i32, vp, f32, vp, vp]
        for name in ("qk_rmsnorm_matmul_q4k", "qk_rmsnorm_matmul_q6k"):
            f = getattr(L, name)
            f.restype, f.argtypes = i32, [vp, vp, vp, f32, vp, vp, i64, i64, i64, vp]
        L.qk_rmsnorm_gateup_swiglu_q4k.restype = i32
        L.qk_rmsnorm_gateup_swiglu_q4k.argtypes = [vp, vp, vp, vp, f32, vp, vp, i64, i64, i64, vp]
        L.qk_rmsnorm_scratch_bytes.restype, L.qk_rmsnorm_scratch_bytes.argtypes = i64, [i32, i32, i64, i64]
        L.qk_rmsnorm_matmul_batch_static.restype = i32
        L.qk_rmsnorm_matmul_batch_static.argtypes = [ctypes.POINTER(qk_matmul_desc), i32, vp, f32, vp]
        L.qk_gemm_plan.restype = i32
        L.qk_gemm_plan.argtypes = [i32, i32, i64, i64, i64, ctypes.POINTER(qk_gemm_plan_info)]
        L.qk_gqa_attention.restype = i32
        L.qk_gqa_attention.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, f32, vp]
        L.qk_status_string.restype, L.qk_status_string.argtypes = ctypes.c_char_p, [i32]
        L.qk_version.restype, L.qk_version.argtypes = i32, []
        _lib = L
    return _lib


# dtypes accepted for fp16 buffers (x, the SwiGLU output): fp16 itself or its bits
_F16 = ("torch.float16", "torch.uint16", "torch.int16")
_F32 = ("torch.float32",)


def _buf(t, nbytes: int, what: str, dtypes=None) -> int:
    """The address of a buffer argument.  A raw integer address (or None) is
    passed through unchecked.  A tensor must be contiguous, of one of `dtypes`
    (any dtype if None), and hold at least `nbytes` bytes: the C ABI takes
    plain pointers and cannot see how large a buffer is."""
    if t is None:
        return 0
    if isinstance(t, int):
        return t
    if dtypes is not None and str(t.dtype) not in dtypes:
        raise ValueError("%s: dtype %s, expected one of %s" % (what, t.dtype, ", ".join(dtypes)))
    if not t.is_contiguous():
        raise ValueError("%s: the tensor is not contiguous" % what)
    have = t.numel() * t.element_size()
    if have < nbytes:
        raise ValueError("%s: holds %d bytes, the call needs %d" % (what, have, nbytes))
    return int(t.data_ptr())


def _n(v) -> int:
    return max(int(v), 0)


def _weight_bytes(qtype, N, K) -> int:
    """Bytes of N rows of K/256 super-blocks (0 for shapes the library rejects)."""
    bb = {QK_Q4_K: 144, QK_Q6_K: 210}.get(qtype, 0)
    return _n(N) * (_n(K) // 256) * bb


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


def _dequant(name, qtype, blocks, n_blocks, out, stream):
    nb = _n(n_blocks)
    w = _buf(blocks, nb * (144 if qtype == QK_Q4_K else 210), name + ": blocks")
    o = _buf(out, nb * 256 * 4, name + ": out", _F32)
    _check(getattr(lib(), name)(w, int(n_blocks), o, _stream(stream)), name)


def qk_dequant_q4k(blocks, n_blocks: int, out, stream=None) -> None:
    _dequant("qk_dequant_q4k", QK_Q4_K, blocks, n_blocks, out, stream)


def qk_dequant_q6k(blocks, n_blocks: int, out, stream=None) -> None:
    _dequant("qk_dequant_q6k", QK_Q6_K, blocks, n_blocks, out, stream)


def _matmul(name, qtype, blocks, x_f16, y, M, N, K, stream):
    w = _buf(blocks, _weight_bytes(qtype, N, K), name + ": blocks")
    x = _buf(x_f16, _n(M) * _n(K) * 2, name + ": x_f16", _F16)
    o = _buf(y, _n(M) * _n(N) * 4, name + ": y", _F32)
    _check(getattr(lib(), name)(w, x, o, int(M), int(N), int(K), _stream(stream)), name)


def qk_matmul_q4k(blocks, x_f16, y, M: int, N: int, K: int, stream=None) -> None:
    _matmul("qk_matmul_q4k", QK_Q4_K, blocks, x_f16, y, M, N, K, stream)


def qk_matmul_q6k(blocks, x_f16, y, M: int, N: int, K: int, stream=None) -> None:
    _matmul("qk_matmul_q6k", QK_Q6_K, blocks, x_f16, y, M, N, K, stream)


def qk_gateup_swiglu_q4k(gate_blocks, up_blocks, x_f16, y_f16, M: int, N_ff: int, K: int, stream=None) -> None:
    name = "qk_gateup_swiglu_q4k"
    wb = _weight_bytes(QK_Q4_K, N_ff, K)
    g = _buf(gate_blocks, wb, name + ": gate_blocks")
    u = _buf(up_blocks, wb, name + ": up_blocks")
    x = _buf(x_f16, _n(M) * _n(K) * 2, name + ": x_f16", _F16)
    o = _buf(y_f16, _n(M) * _n(N_ff) * 2, name + ": y_f16", _F16)
    _check(lib().qk_gateup_swiglu_q4k(g, u, x, o, int(M), int(N_ff), int(K), _stream(stream)), name)


def _descs(problems):
    arr = (qk_matmul_desc * max(1, len(problems)))()
    for i, p in enumerate(problems):
        qt = p["qtype"]
        qt = int({"q4k": QK_Q4_K, "q6k": QK_Q6_K}.get(qt, qt))
        M, N, K = int(p["M"]), int(p["N"]), int(p["K"])
        what = "qk_matmul_batch[%d]" % i
        gu = p.get("up_blocks") is not None
        wb = _weight_bytes(qt, N, K)
        arr[i] = qk_matmul_desc(qt, _buf(p["blocks"], wb, what + ": blocks"),
                                _buf(p.get("up_blocks"), wb, what + ": up_blocks"),
                                _buf(p["x_f16"], _n(M) * _n(K) * 2, what + ": x_f16", _F16),
                                _buf(p["y"], _n(M) * _n(N) * (2 if gu else 4), what + ": y", _F16 if gu else _F32),
                                M, N, K)
    return arr


def qk_matmul_batch(problems, stream=None) -> None:
    """Run independent problems in as few launches as possible.  Each problem is
    a dict with keys qtype ("q4k"/"q6k" or 0/1), blocks, x_f16, y, M, N, K and
    optionally up_blocks (fused gate/up + SwiGLU, fp16 y)."""
    arr = _descs(problems)
    _check(lib().qk_matmul_batch(arr, len(problems), _stream(stream)), "qk_matmul_batch")


def qk_matmul_batch_q8x(problems, stream=None) -> None:
    """qk_matmul_batch with int8 activations (decode only; see include/qk.h)."""
    arr = _descs(problems)
    _check(lib().qk_matmul_batch_q8x(arr, len(problems), _stream(stream)), "qk_matmul_batch_q8x")


def qk_matmul_q8x_q4k(blocks, x_f16, y, M: int, N: int, K: int, stream=None) -> None:
    """y = int8(x) . W^T for Q4_K W, M <= 1 (see include/qk.h)."""
    qk_matmul_batch_q8x([dict(qtype=QK_Q4_K, blocks=blocks, x_f16=x_f16, y=y, M=M, N=N, K=K)], stream)


def qk_matmul_q8x_q6k(blocks, x_f16, y, M: int, N: int, K: int, stream=None) -> None:
    """y = int8(x) . W^T for Q6_K W, M <= 1 (see include/qk.h)."""
    qk_matmul_batch_q8x([dict(qtype=QK_Q6_K, blocks=blocks, x_f16=x_f16, y=y, M=M, N=N, K=K)], stream)


def qk_rmsnorm_scratch_bytes(qtype, M: int, K: int, gateup: bool = False) -> int:
    """Scratch bytes an M-token problem needs under the RMSNorm entry points
    (0 when the GEMV fuses the norm); host only."""
    qt = {"q4k": QK_Q4_K, "q6k": QK_Q6_K}.get(qtype, qtype)
    r = int(lib().qk_rmsnorm_scratch_bytes(int(qt), int(bool(gateup)), int(M), int(K)))
    if r < 0:
        raise ValueError("qk_rmsnorm_scratch_bytes: invalid qtype %r, M %d or K %d" % (qtype, M, K))
    return r


def _scratch(problems, scratch, what):
    need = 0
    for p in problems:
        qt = {"q4k": QK_Q4_K, "q6k": QK_Q6_K}.get(p["qtype"], p["qtype"])
        if int(p["M"]) > 0 and int(p["N"]) > 0:
            need = max(need, qk_rmsnorm_scratch_bytes(qt, p["M"], p["K"], p.get("up_blocks") is not None))
    return _buf(scratch, need, what + ": scratch", _F16 + ("torch.uint8",))


def qk_rmsnorm_matmul_batch(problems, gamma_f16, eps: float, scratch=None, stream=None) -> None:
    """qk_matmul_batch over RMSNorm(x) * gamma (see include/qk.h); `scratch` is
    needed for problems the tensor-core GEMM runs (qk_rmsnorm_scratch_bytes)."""
    what = "qk_rmsnorm_matmul_batch"
    arr = _descs(problems)
    K = max([int(p["K"]) for p in problems] or [0])
    g = _buf(gamma_f16, 2 * K, what + ": gamma_f16", _F16)
    sc = _scratch(problems, scratch, what)
    _check(lib().qk_rmsnorm_matmul_batch(arr, len(problems), g, float(eps), sc, _stream(stream)), what)


def qk_rmsnorm_matmul_batch_static(problems, gamma_f16, eps: float, stream=None) -> None:
    """qk_rmsnorm_matmul_batch for callers that cannot allocate device memory
    (a CUDA graph being captured, a framework whose pool owns the GPU, a loop
    that must not block in cudaMalloc): the scratch is a fixed 8 MiB array in
    the library, shared by every call, so calls that may overlap on the GPU
    race on it.  Problems needing more scratch raise QKError (QK_ERR_SCRATCH)."""
    what = "qk_rmsnorm_matmul_batch_static"
    arr = _descs(problems)
    K = max([int(p["K"]) for p in problems] or [0])
    g = _buf(gamma_f16, 2 * K, what + ": gamma_f16", _F16)
    _check(lib().qk_rmsnorm_matmul_batch_static(arr, len(problems), g, float(eps), _stream(stream)), what)


def _rms_single(name, qtype, blocks, up_blocks, x_f16, gamma_f16, eps, scratch, y, M, N, K, stream):
    gu = up_blocks is not None
    wb = _weight_bytes(qtype, N, K)
    w = _buf(blocks, wb, name + ": blocks")
    x = _buf(x_f16, _n(M) * _n(K) * 2, name + ": x_f16", _F16)
    g = _buf(gamma_f16, 2 * _n(K), name + ": gamma_f16", _F16)
    need = qk_rmsnorm_scratch_bytes(qtype, max(0, int(M)), K, gu) if int(K) > 0 and int(K) % 256 == 0 else 0
    sc = _buf(scratch, need, name + ": scratch", _F16 + ("torch.uint8",))
    if gu:
        u = _buf(up_blocks, wb, name + ": up_blocks")
        o = _buf(y, _n(M) * _n(N) * 2, name + ": y_f16", _F16)
        rc = lib().qk_rmsnorm_gateup_swiglu_q4k(w, u, x, g, float(eps), sc, o, int(M), int(N), int(K), _stream(stream))
    else:
        o = _buf(y, _n(M) * _n(N) * 4, name + ": y", _F32)
        rc = getattr(lib(), name)(w, x, g, float(eps), sc, o, int(M), int(N), int(K), _stream(stream))
    _check(rc, name)


def qk_rmsnorm_matmul_q4k(blocks, x_f16, gamma_f16, eps, y, M, N, K, scratch=None, stream=None) -> None:
    _rms_single("qk_rmsnorm_matmul_q4k", QK_Q4_K, blocks, None, x_f16, gamma_f16, eps, scratch, y, M, N, K, stream)


def qk_rmsnorm_matmul_q6k(blocks, x_f16, gamma_f16, eps, y, M, N, K, scratch=None, stream=None) -> None:
    _rms_single("qk_rmsnorm_matmul_q6k", QK_Q6_K, blocks, None, x_f16, gamma_f16, eps, scratch, y, M, N, K, stream)


def qk_rmsnorm_gateup_swiglu_q4k(gate_blocks, up_blocks, x_f16, gamma_f16, eps, y_f16, M, N_ff, K, scratch=None,
                                 stream=None) -> None:
    _rms_single("qk_rmsnorm_gateup_swiglu_q4k", QK_Q4_K, gate_blocks, up_blocks, x_f16, gamma_f16, eps, scratch,
                y_f16, M, N_ff, K, stream)


def qk_decode_uses_gemv(qtype, K: int, gateup: bool = False) -> bool:
    """Whether an M = 1 problem of this format and K runs on the decode GEMV
    (True) or on the tensor-core GEMM (False); host only."""
    qt = {"q4k": QK_Q4_K, "q6k": QK_Q6_K}.get(qtype, qtype)
    r = int(lib().qk_decode_uses_gemv(int(qt), int(bool(gateup)), int(K)))
    if r < 0:
        raise ValueError("qk_decode_uses_gemv: invalid qtype %r or K %d" % (qtype, K))
    return bool(r)


def qk_uses_gemv(qtype, M: int, K: int, gateup: bool = False) -> bool:
    """Whether an M-token problem of this format and K runs on the GEMV (True)
    or on the tensor-core GEMM (False); host only."""
    qt = {"q4k": QK_Q4_K, "q6k": QK_Q6_K}.get(qtype, qtype)
    r = int(lib().qk_uses_gemv(int(qt), int(bool(gateup)), int(M), int(K)))
    if r < 0:
        raise ValueError("qk_uses_gemv: invalid qtype %r, M %d or K %d" % (qtype, M, K))
    return bool(r)


def qk_gemm_plan(qtype, M: int, N: int, K: int, gateup: bool = False) -> dict:
    """The tensor-core GEMM's launch plan for an M x N x K problem (host only)."""
    qt = {"q4k": QK_Q4_K, "q6k": QK_Q6_K}.get(qtype, qtype)
    info = qk_gemm_plan_info()
    _check(lib().qk_gemm_plan(int(qt), int(bool(gateup)), int(M), int(N), int(K), ctypes.byref(info)),
           "qk_gemm_plan")
    return {n: getattr(info, n) for n, _ in qk_gemm_plan_info._fields_}


def qk_gqa_attention(q_f16, k_cache, v_cache, out, M: int, H: int, H_kv: int, D: int, pos0: int, L_max: int,
                     scale: float, stream=None) -> None:
    """GQA attention over a KV cache (see include/qk.h): q [M][H][D] fp16,
    caches [H_kv][L_max][D] fp16, out [M][H][D] fp32."""
    what = "qk_gqa_attention"
    qn = _n(M) * _n(H) * _n(D)
    cn = _n(H_kv) * _n(L_max) * _n(D)
    _check(lib().qk_gqa_attention(_buf(q_f16, 2 * qn, what + ": q_f16", _F16),
                                  _buf(k_cache, 2 * cn, what + ": k_cache", _F16),
                                  _buf(v_cache, 2 * cn, what + ": v_cache", _F16),
                                  _buf(out, 4 * qn, what + ": out", _F32), int(M), int(H), int(H_kv), int(D),
                                  int(pos0), int(L_max), float(scale), _stream(stream)), what)


def qk_get_device_status(stream=None) -> None:
    _check(lib().qk_get_device_status(_stream(stream)), "qk_get_device_status")


def qk_debug_wait_timeout(limit_ns: int, stream=None) -> None:
    """Enqueue a kernel whose only wait times out after ``limit_ns`` (see include/qk.h)."""
    _check(lib().qk_debug_wait_timeout(int(limit_ns), _stream(stream)), "qk_debug_wait_timeout")
