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
    for code in range(-10, 1):
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
    assert f(A16, A16, A16, 65535 * 128 + 1, 8, 256, None) == -3  # more token tiles than the grid holds
    assert f(A16, A16, A16, 4, 1 << 31, 256, None) == -3
    assert f(A16, A16, A16, 4, 8, 1 << 31, None) == -3
    # the largest M passes the host checks (then the fake pointers are refused)
    assert f(A16, A16, A16, 65535 * 128, 8, 256, None) in (-4, -6, -8)
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


def test_binding_checks_tensor_buffers_before_the_call(qk_lib):
    """Tensor arguments are checked for dtype, contiguity and size in the
    binding (the C ABI sees only pointers), before the library is called."""
    torch = pytest.importorskip("torch")
    M, N, K = 4, 8, 256
    W = torch.zeros(N * 144, dtype=torch.uint8)
    x = torch.zeros(M, K, dtype=torch.float16)
    y = torch.zeros(M, N, dtype=torch.float32)
    bad = [
        lambda: qk_lib.qk_matmul_q4k(W, x.float(), y, M, N, K, stream=0),             # x not fp16
        lambda: qk_lib.qk_matmul_q4k(W, x.t().contiguous().t(), y, M, N, K, stream=0),  # x not contiguous
        lambda: qk_lib.qk_matmul_q4k(W, x, y[:, :4], M, N, K, stream=0),               # y not contiguous
        lambda: qk_lib.qk_matmul_q4k(W, x, y.half(), M, N, K, stream=0),               # y not fp32
        lambda: qk_lib.qk_matmul_q4k(W, x, y[:3], M, N, K, stream=0),                  # y too small
        lambda: qk_lib.qk_matmul_q4k(W[:-1], x, y, M, N, K, stream=0),                 # weights too small
        lambda: qk_lib.qk_matmul_q6k(W, x, y, M, N, K, stream=0),                      # 144 B < 210 B blocks
        lambda: qk_lib.qk_matmul_q4k(W, x[:, :128], y, M, N, K, stream=0),             # x not contiguous
        lambda: qk_lib.qk_gateup_swiglu_q4k(W, W, x, y, M, N, K, stream=0),            # SwiGLU output is fp16
        lambda: qk_lib.qk_gateup_swiglu_q4k(W, W[:10], x, y.half(), M, N, K, stream=0),  # up too small
        lambda: qk_lib.qk_dequant_q4k(W, N, torch.zeros(N * 256, dtype=torch.float16), stream=0),
        lambda: qk_lib.qk_dequant_q6k(W, N, torch.zeros(N * 256), stream=0),          # 8 x 210 B > W
        lambda: qk_lib.qk_matmul_batch([dict(qtype="q4k", blocks=W, x_f16=x, y=y[:2], M=M, N=N, K=K)], stream=0),
        lambda: qk_lib.qk_matmul_batch([dict(qtype="q4k", blocks=W, up_blocks=W, x_f16=x, y=y, M=M, N=N, K=K)],
                                       stream=0),                                       # gate/up y is fp16
    ]
    for i, call in enumerate(bad):
        with pytest.raises(ValueError):
            call()
    # Well-formed host tensors pass the binding and reach the library, which
    # rejects them (no device here, or host memory on a GPU machine).
    for call in (lambda: qk_lib.qk_matmul_q4k(W, x, y, M, N, K, stream=0),
                 lambda: qk_lib.qk_matmul_q4k(W, x.view(torch.int16), y, M, N, K, stream=0),
                 lambda: qk_lib.qk_gateup_swiglu_q4k(W, W, x, y.half(), M, N, K, stream=0),
                 lambda: qk_lib.qk_matmul_batch([dict(qtype="q4k", blocks=W, up_blocks=W, x_f16=x, y=y.half(), M=M,
                                                      N=N, K=K)], stream=0)):
        with pytest.raises(qk_lib.QKError) as e:
            call()
        assert e.value.status in (-4, -6, -8)  # CUDA error, unsupported device, inaccessible pointer


def test_decode_kernel_choice_on_the_host(qk_lib):
    """Which kernel an M = 1 problem runs on is decided on the host from the
    decode GEMV's shared-memory plan: the x table and its sums (1088 bytes per
    Q4_K block, 1152 per Q6_K block), x itself, and at least two stages of 16
    rows, either whole rows (one bulk copy per tensor) or a chunk of cb blocks
    per row whose copies start on 16-byte boundaries, in 227 KB.  Q4_K rows
    chunk at any block count: K <= 35840 (gate/up 35072 with 8 compute warps).  Q6_K blocks are 210
    bytes, so a Q6_K row chunks only when its block count is a multiple of 8;
    other Q6_K rows run on the GEMV while two whole 16-row tiles fit (up to
    K = 6912) and on the GEMM beyond."""
    use = qk_lib.qk_decode_uses_gemv
    for qt, gu, kmax in (("q4k", False, 35840), ("q4k", True, 35072)):
        for K in list(range(256, 8192 + 1, 256)) + [kmax - 256, kmax]:
            assert use(qt, K, gu), (qt, gu, K)
        for K in (kmax + 256, kmax + 512, 65536):
            assert not use(qt, K, gu), (qt, gu, K)
    for K in list(range(256, 6912 + 1, 256)) + [8192, 16384, 26624]:
        assert use("q6k", K), K
    for K in (7168, 8448, 9472, 16640, 28672, 65536):
        assert not use("q6k", K), K
    L = qk_lib.lib()
    # several tokens (2 <= M <= 8) run on the GEMV too while the x table of M
    # tokens fits: the model's K = 3072 and K = 8192; from M = 9 on the GEMM
    uses = qk_lib.qk_uses_gemv
    for qt, gu in (("q4k", False), ("q6k", False), ("q4k", True)):
        for M in (1, 2, 5, 8):
            assert uses(qt, M, 3072, gu), (qt, M)
        for M in (2, 8):
            assert uses(qt, M, 8192, gu), (qt, M)
        for M in (9, 16, 17):
            assert not uses(qt, M, 3072, gu) and not uses(qt, M, 8192, gu), (qt, M)
        assert uses(qt, 1, 8192, gu) == use(qt, 8192, gu)
    assert L.qk_uses_gemv(0, 0, 0, 3072) == -1 and L.qk_uses_gemv(0, 0, 4, 300) == -1
    assert L.qk_decode_uses_gemv(2, 0, 3072) == -1      # unknown format
    assert L.qk_decode_uses_gemv(1, 1, 3072) == -1      # gate/up is Q4_K only
    assert L.qk_decode_uses_gemv(0, 0, 300) == -1       # K % 256
    assert L.qk_decode_uses_gemv(0, 0, 0) == -1


def test_rmsnorm_rejects_bad_arguments_on_the_host(qk_lib):
    L = qk_lib.lib()
    f = L.qk_rmsnorm_matmul_q4k
    assert f(A16, A16, None, 1e-5, A16, A16, 4, 8, 256, None) == -1          # gamma NULL
    assert f(A16, A16, A16, -1.0, A16, A16, 4, 8, 256, None) == -3           # eps < 0
    assert f(A16, A16, A16, float("inf"), A16, A16, 4, 8, 256, None) == -3   # eps not finite
    assert f(A16, A16, A8, 1e-5, A16, A16, 4, 8, 256, None) == -2            # gamma misaligned
    assert f(A16, A16, A16, 1e-5, A16, A16, 4, 8, 300, None) == -3           # K % 256
    assert f(None, None, A16, 1e-5, None, None, 0, 8, 256, None) == 0        # M = 0: no-op
    D = qk_lib.qk_matmul_desc
    arr = (D * 2)(D(0, A16, None, A16, A16, 1, 8, 256), D(0, A16, None, A16, A16, 1, 8, 512))
    assert L.qk_rmsnorm_matmul_batch(arr, 2, A16, 1e-5, None, None) in (-3, -4, -6, -8)
    assert L.qk_rmsnorm_gateup_swiglu_q4k(A16, None, A16, A16, 1e-5, A16, A16, 4, 8, 256, None) == -1
    # the scratch an M-token problem needs: none where the GEMV fuses the norm
    sb = qk_lib.qk_rmsnorm_scratch_bytes
    assert sb("q4k", 1, 3072) == 0 and sb("q6k", 8, 3072) == 0 and sb("q4k", 8, 8192, True) == 0
    assert sb("q6k", 16, 3072) == 16 * 3072 * 2  # M > 8: the GEMM, through the scratch
    assert sb("q4k", 17, 3072) == 17 * 3072 * 2 and sb("q6k", 1024, 8192) == 1024 * 8192 * 2
    assert L.qk_rmsnorm_scratch_bytes(1, 1, 4, 256) == -1 and L.qk_rmsnorm_scratch_bytes(0, 0, 4, 300) == -1


def test_q8x_rejects_on_the_host(qk_lib):
    """int8 activations: several tokens and bad shapes are refused before any
    pointer is looked at."""
    L = qk_lib.lib()
    assert L.qk_matmul_q8x_q4k(A16, A16, A16, 2, 8, 256, None) == -3   # M > 1
    assert L.qk_matmul_q8x_q6k(A16, A16, A16, 1, 8, 300, None) == -3   # K % 256
    assert L.qk_matmul_q8x_q4k(None, None, None, 0, 8, 256, None) == 0  # nothing to do
    assert L.qk_matmul_batch_q8x(None, 0, None) == 0
    assert L.qk_matmul_batch_q8x(None, 1, None) == -1
