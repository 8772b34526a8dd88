"""qk_rmsnorm_matmul_batch_static: the RMSNorm batch entry point that allocates
nothing.

Some callers cannot allocate device memory at the moment they run a layer: a
CUDA graph being captured (an allocation is not recorded into the graph), a
framework whose memory pool owns the GPU, or a real-time loop that allocates
nothing after start-up because cudaMalloc can block and synchronise the
device.  This entry point keeps its scratch (the normalized activations the
tensor-core GEMM reads) in a fixed array inside the library.

The GPU test compares it, on two calls in a row with different inputs and
sizes, with qk_rmsnorm_matmul_batch given a caller-allocated scratch, within
the parity bar of the other GPU tests (max |diff| <= 1e-2 * rms).  The file's
name puts it last in collection order.
"""
import numpy as np
import pytest

from tests import synth

TOL = 1e-2
EPS = 1e-5
QK_ERR_SCRATCH = -9
STATIC_SCRATCH_BYTES = 8 << 20


def _dev(a, cuda):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to(cuda)


def _f16_dev(a, cuda):
    return _dev(a.view(np.uint16), cuda)


def _close(got, ref, what):
    rms = float(np.sqrt(np.mean(ref ** 2)))
    err = float(np.max(np.abs(got - ref)))
    assert np.isfinite(got).all(), what
    assert err <= TOL * rms, "%s: max|diff| %.3e > %.0e * rms %.3e" % (what, err, TOL, rms)


def _problems(qk, rng, cuda, M, K, gu_M):
    """q, k, v linears (Q4_K, Q4_K, Q6_K) on one x of M tokens and a fused
    gate/up + SwiGLU on another x of gu_M tokens, all with the same K; each
    problem twice, once per entry point, with its own output."""
    import torch
    x = _f16_dev(synth.activations(rng, M, K), cuda)
    xg = _f16_dev(synth.activations(rng, gu_M, K), cuda)
    mine, theirs = [], []
    for qt, N in (("q4k", 256), ("q4k", 128), ("q6k", 160)):
        W = _dev(synth.weights(rng, qt, N, K), cuda)
        for out in (mine, theirs):
            out.append(dict(qtype=qt, blocks=W, x_f16=x, M=M, N=N, K=K,
                            y=torch.full((M, N), float("nan"), device=cuda)))
    N = 192
    Wg, Wu = _dev(synth.q4k_weights(rng, N, K), cuda), _dev(synth.q4k_weights(rng, N, K), cuda)
    for out in (mine, theirs):
        out.append(dict(qtype="q4k", blocks=Wg, up_blocks=Wu, x_f16=xg, M=gu_M, N=N, K=K,
                        y=torch.full((gu_M, N), float("nan"), dtype=torch.float16, device=cuda)))
    return mine, theirs


@pytest.mark.gpu
def test_static_scratch_matches_caller_scratch_on_two_calls(qk_lib, cuda):
    import torch
    # the first call writes more of the built-in scratch than the second reads,
    # so a second call that read stale rows would show
    for call, (M, gu_M, K, seed) in enumerate(((96, 200, 3072, 1), (40, 24, 3072, 2))):
        rng = synth.rng_for(4242, seed)
        mine, theirs = _problems(qk_lib, rng, cuda, M, K, gu_M)
        need = max(qk_lib.qk_rmsnorm_scratch_bytes(p["qtype"], p["M"], K, "up_blocks" in p) for p in mine)
        assert 0 < need <= STATIC_SCRATCH_BYTES  # these problems do use scratch
        g = _f16_dev((1.0 + 0.1 * rng.standard_normal(K)).astype(np.float16), cuda)
        qk_lib.qk_rmsnorm_matmul_batch_static(mine, g, EPS)
        sc = torch.empty(need // 2, dtype=torch.float16, device=cuda)
        qk_lib.qk_rmsnorm_matmul_batch(theirs, g, EPS, scratch=sc)
        qk_lib.qk_get_device_status()
        torch.cuda.synchronize()
        for a, b in zip(mine, theirs):
            what = "call %d %s M%d N%d%s" % (call + 1, a["qtype"], a["M"], a["N"], " gate/up" if "up_blocks" in a else "")
            _close(a["y"].float().cpu().numpy().astype(np.float64), b["y"].float().cpu().numpy().astype(np.float64),
                   what)


@pytest.mark.gpu
def test_static_scratch_rejects_too_large_and_enqueues_nothing(qk_lib, cuda):
    import torch
    M, N, K = 2048, 64, 4096  # M * K * 2 = 16 MiB of normalized activations
    assert qk_lib.qk_rmsnorm_scratch_bytes("q4k", M, K) > STATIC_SCRATCH_BYTES
    W = torch.zeros(N * (K // 256) * 144, dtype=torch.uint8, device=cuda)
    x = torch.zeros(M * K, dtype=torch.float16, device=cuda)
    g = torch.ones(K, dtype=torch.float16, device=cuda)
    y = torch.full((M, N), float("nan"), device=cuda)
    L = qk_lib.lib()
    arr = qk_lib._descs([dict(qtype="q4k", blocks=W, x_f16=x, y=y, M=M, N=N, K=K)])
    s = torch.cuda.current_stream().cuda_stream
    assert L.qk_rmsnorm_matmul_batch_static(arr, 1, g.data_ptr(), EPS, s) == QK_ERR_SCRATCH
    assert "scratch" in L.qk_status_string(QK_ERR_SCRATCH).decode()
    torch.cuda.synchronize()
    assert torch.isnan(y).all()
    with pytest.raises(qk_lib.QKError):
        qk_lib.qk_rmsnorm_matmul_batch_static([dict(qtype="q4k", blocks=W, x_f16=x, y=y, M=M, N=N, K=K)], g, EPS)
