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
    GEMV's shared-memory plan (x of K plus two weight stages).  The model's
    inner sizes stay on the GEMV; K values it cannot stage go to the GEMM."""
    use = qk_lib.qk_decode_uses_gemv
    for qt, gu in (("q4k", False), ("q6k", False), ("q4k", True)):
        for K in range(256, 6144 + 1, 256):
            assert use(qt, K, gu), (qt, gu, K)
        assert use(qt, 8192, gu)
        # x alone (fp16 copy plus 16-wide sums, 2.25 bytes per k) exceeds 227 KB
        assert not use(qt, 131072, gu)
    # Q6_K rows of an odd number of 8-block groups cannot be chunked 16-byte
    # aligned, and whole 16-row tiles no longer fit three times
    assert not use("q6k", 8448)
    assert not use("q4k", 6400, True)   # gate/up: two tensors per stage
    assert not use("q4k", 11520)
    assert use("q6k", 16384) and use("q4k", 16384, True)  # 64 blocks: chunks of 8 fit
    L = qk_lib.lib()
    assert L.qk_decode_uses_gemv(2, 0, 3072) == -1      # unknown format
    assert L.qk_decode_uses_gemv(1, 1, 3072) == -1      # gate/up is Q4_K only
    assert L.qk_decode_uses_gemv(0, 0, 300) == -1       # K % 256
    assert L.qk_decode_uses_gemv(0, 0, 0) == -1


def test_gemm_plans_fit_tensor_memory_on_a_shared_sm(qk_lib):
    """tcgen05.alloc waits without a time limit for free tensor-memory columns,
    so the CTAs that can share an SM must fit in its 512 columns together.
    Checked on the host for every linear of the model at every swept M (and the
    small-M shapes that pick narrow token tiles), for both A-tile placements."""
    import subprocess
    import sys
    from tests import synth
    shapes = sorted({(lin.qtype, lin.N, lin.K) for _, lin in synth.model_linears()})
    Ms = sorted(set(synth.SWEEP_M) | {2, 17, 33, 48, 64, 100, 200, 300, 513, 4096})
    seen_tmem = set()
    for qt, N, K in shapes:
        for M in Ms:
            p = qk_lib.qk_gemm_plan(qt, M, N, K)
            assert p["max_ctas_per_sm"] >= 1
            assert p["max_ctas_per_sm"] * p["tmem_cols"] <= 512, (qt, N, K, M, p)
            assert p["smem_bytes"] <= 227 * 1024
            seen_tmem.add(p["a_in_tmem"])
    for M in Ms:
        p = qk_lib.qk_gemm_plan("q4k", M, synth.FFN, synth.HIDDEN, gateup=True)
        assert p["max_ctas_per_sm"] * p["tmem_cols"] <= 512, (M, p)
    assert seen_tmem == {0, 1}
    # A narrow token tile with A tiles in tensor memory needs 2*64 + 5*32 = 288
    # columns (allocated as 512) in ~70 KB of shared memory: padded to one CTA.
    p = qk_lib.qk_gemm_plan("q4k", 64, 4096, 4096)
    assert p["token_tile"] == 64 and p["a_in_tmem"] == 1 and p["tmem_cols"] == 512
    assert p["max_ctas_per_sm"] == 1
    # The shared-memory A path (QK_A_TMEM=0) in a child process: same rule.
    code = ("import sys; sys.path.insert(0, %r); import quantized_q4_matmul_gb300 as qk\n"
            "for M in (16, 64, 128, 1024):\n"
            "    p = qk.qk_gemm_plan('q6k', M, 3072, 8192)\n"
            "    assert p['a_in_tmem'] == 0 and p['max_ctas_per_sm'] * p['tmem_cols'] <= 512, p\n"
            "print('ok')" % ROOT)
    r = subprocess.run([sys.executable, "-c", code], env=dict(os.environ, QK_A_TMEM="0"), capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr


def test_gemm_plan_rejects_bad_arguments(qk_lib):
    L = qk_lib.lib()
    info = qk_lib.qk_gemm_plan_info()
    import ctypes as C
    assert L.qk_gemm_plan(0, 0, 16, 3072, 3072, None) == -1
    assert L.qk_gemm_plan(2, 0, 16, 3072, 3072, C.byref(info)) == -3
    assert L.qk_gemm_plan(1, 1, 16, 3072, 3072, C.byref(info)) == -3
    assert L.qk_gemm_plan(0, 0, 16, 3072, 300, C.byref(info)) == -3
    assert L.qk_gemm_plan(0, 0, 0, 3072, 3072, C.byref(info)) == -3
    assert L.qk_gemm_plan(0, 0, 16, 3072, 3072, C.byref(info)) == 0 and info.token_tile == 16
