"""CPU oracle for the quantized Q4_K / Q6_K matmul path.

TEST INFRASTRUCTURE, NOT PRODUCT CODE: only the test suite, the smoke check and
the benchmark's CPU-baseline leg may import this package.  The CUDA library and
its Python binding never import it.

``qk_oracle.c`` holds the arithmetic (GGUF Q4_K / Q6_K block decoding in fp32,
fp64-accumulated matmul, fp64 SwiGLU, fp64 RMSNorm in front of a linear, int8
activations per block of 32, fp64 GQA attention over a KV cache); this module
only builds it with gcc and marshals numpy arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qk_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

Q4K, Q6K = 0, 1
BLOCK_BYTES = {Q4K: 144, Q6K: 210}
QK = 256


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile the oracle into a shared library (plain C, fp contraction off)."""
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        tmp = out + ".tmp%d" % os.getpid()
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
               "-fPIC", "-shared", src, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, out)
    return out


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _rows(N, rows):
    if rows is None:
        rows = np.arange(N, dtype=np.int64)
    return np.ascontiguousarray(rows, dtype=np.int64)


class Oracle:
    """ctypes view of one compiled copy of ``qk_oracle.c``."""

    def __init__(self, path: str):
        L = ctypes.CDLL(path)
        L.oracle_half_to_float.restype = ctypes.c_float
        L.oracle_half_to_float.argtypes = [ctypes.c_uint16]
        L.oracle_dequant.restype = ctypes.c_int
        L.oracle_dequant.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]
        L.oracle_matmul_rows.restype = ctypes.c_int
        L.oracle_matmul_rows.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                         ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]
        L.oracle_gateup_swiglu_rows.restype = ctypes.c_int
        L.oracle_gateup_swiglu_rows.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                                ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
                                                ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                                                ctypes.c_void_p]
        L.oracle_rmsnorm.restype = ctypes.c_int
        L.oracle_rmsnorm.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                     ctypes.c_double, ctypes.c_void_p]
        L.oracle_rmsnorm_matmul_rows.restype = ctypes.c_int
        L.oracle_rmsnorm_matmul_rows.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                                 ctypes.c_double, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
                                                 ctypes.c_int64, ctypes.c_void_p]
        L.oracle_rmsnorm_gateup_swiglu_rows.restype = ctypes.c_int
        L.oracle_rmsnorm_gateup_swiglu_rows.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                                        ctypes.c_void_p, ctypes.c_double, ctypes.c_int64,
                                                        ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64,
                                                        ctypes.c_void_p]
        L.oracle_quantize_q8.restype = ctypes.c_int
        L.oracle_quantize_q8.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
                                         ctypes.c_void_p]
        L.oracle_q8_matmul_rows.restype = ctypes.c_int
        L.oracle_q8_matmul_rows.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                            ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]
        L.oracle_q8_gateup_swiglu_rows.restype = ctypes.c_int
        L.oracle_q8_gateup_swiglu_rows.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                                   ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]
        L.oracle_gqa_attention.restype = ctypes.c_int
        L.oracle_gqa_attention.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                           ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                           ctypes.c_int64, ctypes.c_double, ctypes.c_void_p, ctypes.c_int64,
                                           ctypes.c_void_p]
        L.oracle_num_threads.restype = ctypes.c_int
        L.oracle_set_num_threads.argtypes = [ctypes.c_int]
        self.L = L

    def half_to_float(self, bits: int) -> float:
        return float(self.L.oracle_half_to_float(int(bits) & 0xFFFF))

    def dequant(self, qtype: int, blocks: np.ndarray) -> np.ndarray:
        """fp32 weights of ``blocks`` (uint8, whole blocks), flattened."""
        b = np.ascontiguousarray(blocks, dtype=np.uint8).reshape(-1)
        nb = b.size // BLOCK_BYTES[qtype]
        assert nb * BLOCK_BYTES[qtype] == b.size
        out = np.empty(nb * QK, dtype=np.float32)
        rc = self.L.oracle_dequant(qtype, _ptr(b), nb, _ptr(out))
        assert rc == 0, rc
        return out

    def matmul(self, qtype: int, W: np.ndarray, x: np.ndarray, N: int, K: int, rows=None) -> np.ndarray:
        """fp64 y[M][len(rows)] = x . W[rows]^T, W = N rows of K/256 blocks, x fp16 [M][K]."""
        W = np.ascontiguousarray(W, dtype=np.uint8).reshape(-1)
        assert W.size == N * (K // QK) * BLOCK_BYTES[qtype]
        x = np.ascontiguousarray(x, dtype=np.float16).reshape(-1, K)
        M = x.shape[0]
        r = _rows(N, rows)
        assert r.size == 0 or (r.min() >= 0 and r.max() < N)
        y = np.empty((M, r.size), dtype=np.float64)
        rc = self.L.oracle_matmul_rows(qtype, _ptr(W), _ptr(x.view(np.uint16)), M, K, _ptr(r), r.size,
                                       _ptr(y))
        assert rc == 0, rc
        return y

    def gateup_swiglu(self, Wg, Wu, x, N_ff: int, K: int, rows=None, return_gu: bool = False):
        """fp64 silu(x.Wg^T) * (x.Wu^T) for Q4_K gate / up weights of N_ff rows each."""
        Wg = np.ascontiguousarray(Wg, dtype=np.uint8).reshape(-1)
        Wu = np.ascontiguousarray(Wu, dtype=np.uint8).reshape(-1)
        assert Wg.size == Wu.size == N_ff * (K // QK) * BLOCK_BYTES[Q4K]
        x = np.ascontiguousarray(x, dtype=np.float16).reshape(-1, K)
        M = x.shape[0]
        r = _rows(N_ff, rows)
        assert r.size == 0 or (r.min() >= 0 and r.max() < N_ff)
        out = np.empty((M, r.size), dtype=np.float64)
        g = np.empty_like(out) if return_gu else None
        u = np.empty_like(out) if return_gu else None
        rc = self.L.oracle_gateup_swiglu_rows(_ptr(Wg), _ptr(Wu), _ptr(x.view(np.uint16)), M, K, _ptr(r),
                                              r.size, _ptr(out), _ptr(g), _ptr(u))
        assert rc == 0, rc
        return (out, g, u) if return_gu else out

    def rmsnorm(self, x, gamma, eps: float) -> np.ndarray:
        """fp64 x / sqrt(mean(x^2) + eps) * gamma per row; x fp16 [M][K], gamma fp16 [K]."""
        g = np.ascontiguousarray(gamma, dtype=np.float16).reshape(-1)
        x = np.ascontiguousarray(x, dtype=np.float16).reshape(-1, g.size)
        out = np.empty(x.shape, dtype=np.float64)
        rc = self.L.oracle_rmsnorm(_ptr(x.view(np.uint16)), _ptr(g.view(np.uint16)), x.shape[0], g.size,
                                   float(eps), _ptr(out))
        assert rc == 0, rc
        return out

    def rmsnorm_matmul(self, qtype: int, W, x, gamma, eps: float, N: int, K: int, rows=None) -> np.ndarray:
        """fp64 y[M][len(rows)] = (RMSNorm(x) * gamma) . W[rows]^T."""
        W = np.ascontiguousarray(W, dtype=np.uint8).reshape(-1)
        assert W.size == N * (K // QK) * BLOCK_BYTES[qtype]
        g = np.ascontiguousarray(gamma, dtype=np.float16).reshape(-1)
        assert g.size == K
        x = np.ascontiguousarray(x, dtype=np.float16).reshape(-1, K)
        r = _rows(N, rows)
        y = np.empty((x.shape[0], r.size), dtype=np.float64)
        rc = self.L.oracle_rmsnorm_matmul_rows(qtype, _ptr(W), _ptr(x.view(np.uint16)), _ptr(g.view(np.uint16)),
                                               float(eps), x.shape[0], K, _ptr(r), r.size, _ptr(y))
        assert rc == 0, rc
        return y

    def rmsnorm_gateup_swiglu(self, Wg, Wu, x, gamma, eps: float, N_ff: int, K: int, rows=None) -> np.ndarray:
        """fp64 silu(xhat.Wg^T) * (xhat.Wu^T) with xhat = RMSNorm(x) * gamma."""
        Wg = np.ascontiguousarray(Wg, dtype=np.uint8).reshape(-1)
        Wu = np.ascontiguousarray(Wu, dtype=np.uint8).reshape(-1)
        assert Wg.size == Wu.size == N_ff * (K // QK) * BLOCK_BYTES[Q4K]
        g = np.ascontiguousarray(gamma, dtype=np.float16).reshape(-1)
        assert g.size == K
        x = np.ascontiguousarray(x, dtype=np.float16).reshape(-1, K)
        r = _rows(N_ff, rows)
        out = np.empty((x.shape[0], r.size), dtype=np.float64)
        rc = self.L.oracle_rmsnorm_gateup_swiglu_rows(_ptr(Wg), _ptr(Wu), _ptr(x.view(np.uint16)),
                                                      _ptr(g.view(np.uint16)), float(eps), x.shape[0], K, _ptr(r),
                                                      r.size, _ptr(out))
        assert rc == 0, rc
        return out

    def num_threads(self) -> int:
        return int(self.L.oracle_num_threads())

    def set_num_threads(self, n: int) -> None:
        self.L.oracle_set_num_threads(int(n))

    def quantize_q8(self, x):
        """(q int8 [M][K], d fp32 [M][K/32]): x per block of 32 as int8 with one scale."""
        x = np.ascontiguousarray(x, dtype=np.float16)
        x = x.reshape(-1, x.shape[-1])
        M, K = x.shape
        q = np.empty((M, K), dtype=np.int8)
        d = np.empty((M, K // 32), dtype=np.float32)
        rc = self.L.oracle_quantize_q8(_ptr(x.view(np.uint16)), M, K, _ptr(q), _ptr(d))
        assert rc == 0, rc
        return q, d

    def q8_matmul(self, qtype: int, W, x, N: int, K: int, rows=None) -> np.ndarray:
        """fp64 y[M][len(rows)] = (d * q)(x) . W[rows]^T with x quantized as in quantize_q8."""
        W = np.ascontiguousarray(W, dtype=np.uint8).reshape(-1)
        assert W.size == N * (K // QK) * BLOCK_BYTES[qtype]
        x = np.ascontiguousarray(x, dtype=np.float16).reshape(-1, K)
        r = _rows(N, rows)
        y = np.empty((x.shape[0], r.size), dtype=np.float64)
        rc = self.L.oracle_q8_matmul_rows(qtype, _ptr(W), _ptr(x.view(np.uint16)), x.shape[0], K, _ptr(r), r.size,
                                          _ptr(y))
        assert rc == 0, rc
        return y

    def q8_gateup_swiglu(self, Wg, Wu, x, N_ff: int, K: int, rows=None) -> np.ndarray:
        """fp64 silu(x~.Wg^T) * (x~.Wu^T) with x~ the int8 activations of quantize_q8."""
        Wg = np.ascontiguousarray(Wg, dtype=np.uint8).reshape(-1)
        Wu = np.ascontiguousarray(Wu, dtype=np.uint8).reshape(-1)
        assert Wg.size == Wu.size == N_ff * (K // QK) * BLOCK_BYTES[Q4K]
        x = np.ascontiguousarray(x, dtype=np.float16).reshape(-1, K)
        r = _rows(N_ff, rows)
        out = np.empty((x.shape[0], r.size), dtype=np.float64)
        rc = self.L.oracle_q8_gateup_swiglu_rows(_ptr(Wg), _ptr(Wu), _ptr(x.view(np.uint16)), x.shape[0], K, _ptr(r),
                                                 r.size, _ptr(out))
        assert rc == 0, rc
        return out

    def gqa_attention(self, q, k_cache, v_cache, H: int, Hkv: int, pos0: int, scale: float, qrows=None):
        """fp64 GQA attention: q fp16 [M][H][D] (query i at position pos0 + i,
        causal), caches fp16 [Hkv][L_max][D]; out [len(qrows)][H][D]."""
        kc = np.ascontiguousarray(k_cache, dtype=np.float16)
        vc = np.ascontiguousarray(v_cache, dtype=np.float16)
        assert kc.shape == vc.shape and kc.ndim == 3 and kc.shape[0] == Hkv
        Lmax, D = kc.shape[1], kc.shape[2]
        q = np.ascontiguousarray(q, dtype=np.float16).reshape(-1, H, D)
        M = q.shape[0]
        r = _rows(M, qrows)
        out = np.empty((r.size, H, D), dtype=np.float64)
        rc = self.L.oracle_gqa_attention(_ptr(q.view(np.uint16)), _ptr(kc.view(np.uint16)), _ptr(vc.view(np.uint16)),
                                         M, H, Hkv, D, int(pos0), Lmax, float(scale),
                                         _ptr(r) if qrows is not None else None, r.size, _ptr(out))
        assert rc == 0, rc
        return out


_default = None


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default


def half_to_float(bits):
    return default().half_to_float(bits)


def dequant(qtype, blocks):
    return default().dequant(qtype, blocks)


def matmul(qtype, W, x, N, K, rows=None):
    return default().matmul(qtype, W, x, N, K, rows)


def gateup_swiglu(Wg, Wu, x, N_ff, K, rows=None, return_gu=False):
    return default().gateup_swiglu(Wg, Wu, x, N_ff, K, rows, return_gu)


def rmsnorm(x, gamma, eps):
    return default().rmsnorm(x, gamma, eps)


def rmsnorm_matmul(qtype, W, x, gamma, eps, N, K, rows=None):
    return default().rmsnorm_matmul(qtype, W, x, gamma, eps, N, K, rows)


def rmsnorm_gateup_swiglu(Wg, Wu, x, gamma, eps, N_ff, K, rows=None):
    return default().rmsnorm_gateup_swiglu(Wg, Wu, x, gamma, eps, N_ff, K, rows)


def num_threads():
    return default().num_threads()


def set_num_threads(n):
    default().set_num_threads(n)


def quantize_q8(x):
    return default().quantize_q8(x)


def q8_matmul(qtype, W, x, N, K, rows=None):
    return default().q8_matmul(qtype, W, x, N, K, rows)


def q8_gateup_swiglu(Wg, Wu, x, N_ff, K, rows=None):
    return default().q8_gateup_swiglu(Wg, Wu, x, N_ff, K, rows)


def gqa_attention(q, k_cache, v_cache, H, Hkv, pos0, scale, qrows=None):
    return default().gqa_attention(q, k_cache, v_cache, H, Hkv, pos0, scale, qrows)
