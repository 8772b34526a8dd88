"""int8-activation decode path (qk_matmul_batch_q8x / qk_matmul_q8x_*) against
the oracle, through the C ABI.

Bars:
* against the oracle's int8-activation matmul (the same quantized x): the
  kernel decides every int8 value and scale in the same fp32 arithmetic, and
  its integer dot products are exact, so only the fp32 scaling and summation
  order differ: max |y - y_oracle| <= 2e-3 * rms(y_oracle);
* against the exact fp16 matmul: within the quantization bound
  sum over 32-blocks of (d / 2) * sum |w|, per output, plus that fp32 margin.
"""
import numpy as np
import pytest

import oracle
from tests import synth

pytestmark = pytest.mark.gpu

TOL_Q8 = 2e-3
QT = {"q4k": oracle.Q4K, "q6k": oracle.Q6K}


def _dev(a, cuda):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to(cuda)


def _q8(qk, qtype, W, x, N, K, cuda):
    import torch
    y = torch.full((1, N), float("nan"), device=cuda)
    fn = qk.qk_matmul_q8x_q4k if qtype == "q4k" else qk.qk_matmul_q8x_q6k
    fn(_dev(W, cuda), _dev(x.view(np.uint16), cuda), y, 1, N, K)
    qk.qk_get_device_status()
    return y.cpu().numpy().astype(np.float64)


def _close(got, ref, what, tol=TOL_Q8):
    rms = float(np.sqrt(np.mean(ref ** 2)))
    err = float(np.max(np.abs(got - ref)))
    assert np.isfinite(got).all(), what
    assert err <= tol * rms, "%s: max|err| %.3e > %.0e * rms %.3e" % (what, err, tol, rms)


@pytest.mark.parametrize("qtype", ["q4k", "q6k"])
@pytest.mark.parametrize("N,K", [(200, 3072), (64, 8192), (130, 1024), (1, 256), (33, 2304), (3072, 3072)])
def test_q8_matmul(qk_lib, cuda, qtype, N, K):
    rng = synth.rng_for(N + 5, K)
    W = synth.weights(rng, qtype, N, K)
    x = synth.activations(rng, 1, K)
    got = _q8(qk_lib, qtype, W, x, N, K, cuda)
    _close(got, oracle.q8_matmul(QT[qtype], W, x, N, K), "q8 %s N%d K%d" % (qtype, N, K))
    # and within the quantization bound of the exact fp16 product
    q, d = oracle.quantize_q8(x)
    w = oracle.dequant(QT[qtype], W).astype(np.float64).reshape(N, K)
    bound = (np.repeat(d.astype(np.float64), 32, axis=1) / 2) @ np.abs(w).T
    exact = oracle.matmul(QT[qtype], W, x, N, K)
    rms = float(np.sqrt(np.mean(exact ** 2)))
    assert np.all(np.abs(got - exact) <= bound + TOL_Q8 * rms)


def test_q8_grid_matches_fp16_path(qk_lib, cuda):
    """x already on its int8 grid: the int8 path and the fp16 oracle agree
    within the fp32 margin (the quantization is exact)."""
    rng = synth.rng_for(91, 0)
    N, K = 96, 3072
    q = rng.integers(-127, 128, size=(1, K))
    q[0, ::32] = 127
    x = (q * 2.0 ** -9).astype(np.float16)
    for qt in ("q4k", "q6k"):
        W = synth.weights(rng, qt, N, K)
        _close(_q8(qk_lib, qt, W, x, N, K, cuda), oracle.matmul(QT[qt], W, x, N, K), "q8 on grid " + qt)


def test_q8_gateup_and_batch(qk_lib, cuda):
    """A grouped launch with the fused gate/up + SwiGLU (fp16 output, with the
    output's own half ulp on top of the bar) and plain problems of both
    formats; each result equals its single call bit for bit."""
    import torch
    rng = synth.rng_for(92, 0)
    K, Nf = 3072, 320
    x = synth.activations(rng, 1, K)
    xd = _dev(x.view(np.uint16), cuda)
    Wg, Wu = synth.q4k_weights(rng, Nf, K), synth.q4k_weights(rng, Nf, K)
    yg = torch.full((1, Nf), float("nan"), dtype=torch.float16, device=cuda)
    probs = [dict(qtype="q4k", blocks=_dev(Wg, cuda), up_blocks=_dev(Wu, cuda), x_f16=xd, y=yg, M=1, N=Nf, K=K)]
    refs, singles = [], []
    for qt, N in (("q4k", 256), ("q6k", 128)):
        W = synth.weights(rng, qt, N, K)
        y = torch.full((1, N), float("nan"), device=cuda)
        probs.append(dict(qtype=qt, blocks=_dev(W, cuda), x_f16=xd, y=y, M=1, N=N, K=K))
        refs.append(oracle.q8_matmul(QT[qt], W, x, N, K))
        singles.append(_q8(qk_lib, qt, W, x, N, K, cuda))
    qk_lib.qk_matmul_batch_q8x(probs)
    qk_lib.qk_get_device_status()
    ref = oracle.q8_gateup_swiglu(Wg, Wu, x, Nf, K)
    got = yg.float().cpu().numpy().astype(np.float64)
    half_ulp = np.ldexp(0.5, np.floor(np.log2(np.maximum(np.abs(ref), 2.0 ** -14))).astype(np.int64) - 10)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    assert np.isfinite(got).all() and np.max(np.abs(got - ref) - half_ulp) <= TOL_Q8 * rms
    for p, r, single in zip(probs[1:], refs, singles):
        out = p["y"].cpu().numpy().astype(np.float64)
        assert np.array_equal(out, single)
        _close(out, r, "q8 batch " + p["qtype"])


def test_q8_rejects_what_it_cannot_run(qk_lib, cuda):
    """Several tokens, and a K the decode GEMV cannot stage, are refused."""
    import torch
    L = qk_lib.lib()
    W = torch.zeros(130 * 256 * 144, dtype=torch.uint8, device=cuda)
    x = torch.zeros(2 * 65536, dtype=torch.float16, device=cuda)
    y = torch.zeros(2 * 130, device=cuda)
    s = torch.cuda.current_stream().cuda_stream
    assert L.qk_matmul_q8x_q4k(W.data_ptr(), x.data_ptr(), y.data_ptr(), 2, 16, 256, s) == -3   # M > 1
    assert L.qk_matmul_q8x_q4k(W.data_ptr(), x.data_ptr(), y.data_ptr(), 1, 2, 65536, s) == -3  # K too large
    assert L.qk_matmul_q8x_q4k(W.data_ptr(), x.data_ptr(), y.data_ptr(), 0, 16, 256, s) == 0    # nothing to do
    assert L.qk_get_device_status(s) == 0
