"""GQA attention over a KV cache (qk_gqa_attention) against the oracle, through
the C ABI.

Bar, per call, relative to the largest |v| the queries can see: both kernels
score in fp32 (fp16 operands, fp32 accumulation) and round the softmax weights
to fp16 for the P.V product (relative error 2^-11 each) while their sum stays
in fp32, which bounds the error by about 2^-10 * max|v|: 2e-3 * max|v|.
Cache positions past the last query are filled with NaN: a kernel that read
one would return NaN.
"""
import numpy as np
import pytest

import oracle
from tests import synth

pytestmark = pytest.mark.gpu

D = 128
TOL_DECODE = TOL_PREFILL = 2e-3


def _inputs(seed, M, H, Hkv, pos0, Lmax):
    rng = synth.rng_for(seed, M * 1000 + pos0)
    q = rng.standard_normal((M, H, D)).astype(np.float16)
    k = np.full((Hkv, Lmax, D), np.nan, np.float16)
    v = np.full((Hkv, Lmax, D), np.nan, np.float16)
    n = pos0 + M
    k[:, :n] = rng.standard_normal((Hkv, n, D)).astype(np.float16)
    v[:, :n] = rng.standard_normal((Hkv, n, D)).astype(np.float16)
    return q, k, v


def _run(qk, cuda, q, k, v, M, H, Hkv, pos0, scale):
    import torch
    Lmax = k.shape[1]
    dq = torch.from_numpy(q.view(np.uint16)).to(cuda)
    dk = torch.from_numpy(k.view(np.uint16)).to(cuda)
    dv = torch.from_numpy(v.view(np.uint16)).to(cuda)
    out = torch.full((M, H, D), float("nan"), device=cuda)
    qk.qk_gqa_attention(dq, dk, dv, out, M, H, Hkv, D, pos0, Lmax, scale)
    qk.qk_get_device_status()
    return out.cpu().numpy().astype(np.float64)


def _check(got, ref, v, n, tol, what):
    vmax = float(np.abs(v[:, :n].astype(np.float64)).max())
    err = float(np.max(np.abs(got - ref)))
    assert np.isfinite(got).all(), what
    assert err <= tol * vmax, "%s: max|err| %.3e > %.0e * max|v| %.3e" % (what, err, tol, vmax)


@pytest.mark.parametrize("L", [1, 2, 63, 64, 65, 300, 1024, 4097])
def test_decode_llama_heads(qk_lib, cuda, L):
    """One decode step of Llama-3.2-3B's attention (24 query heads, 8 KV heads)."""
    H, Hkv, pos0 = 24, 8, L - 1
    q, k, v = _inputs(81, 1, H, Hkv, pos0, L + 7)
    scale = 1 / np.sqrt(D)
    got = _run(qk_lib, cuda, q, k, v, 1, H, Hkv, pos0, scale)
    _check(got, oracle.gqa_attention(q, k, v, H, Hkv, pos0, scale), v, L, TOL_DECODE, "decode L=%d" % L)


@pytest.mark.parametrize("H,Hkv,L", [(8, 8, 700), (32, 4, 2000), (6, 2, 129), (4, 1, 513)])
def test_decode_group_sizes(qk_lib, cuda, H, Hkv, L):
    q, k, v = _inputs(82, 1, H, Hkv, L - 1, L)
    scale = 0.09
    got = _run(qk_lib, cuda, q, k, v, 1, H, Hkv, L - 1, scale)
    _check(got, oracle.gqa_attention(q, k, v, H, Hkv, L - 1, scale), v, L, TOL_DECODE, "decode H%d/%d" % (H, Hkv))


@pytest.mark.parametrize("M,pos0", [(2, 0), (17, 0), (64, 0), (100, 0), (257, 0), (33, 37), (130, 200)])
def test_prefill_llama_heads(qk_lib, cuda, M, pos0):
    """Causal prefill (pos0 = 0) and a prefill chunk after pos0 cached positions."""
    H, Hkv = 24, 8
    q, k, v = _inputs(83, M, H, Hkv, pos0, pos0 + M + 9)
    scale = 1 / np.sqrt(D)
    got = _run(qk_lib, cuda, q, k, v, M, H, Hkv, pos0, scale)
    _check(got, oracle.gqa_attention(q, k, v, H, Hkv, pos0, scale), v, pos0 + M, TOL_PREFILL,
           "prefill M=%d pos0=%d" % (M, pos0))


@pytest.mark.parametrize("H,Hkv", [(8, 8), (32, 4), (4, 1)])
def test_prefill_group_sizes(qk_lib, cuda, H, Hkv):
    M, pos0 = 90, 11
    q, k, v = _inputs(84, M, H, Hkv, pos0, pos0 + M)
    got = _run(qk_lib, cuda, q, k, v, M, H, Hkv, pos0, 0.1)
    _check(got, oracle.gqa_attention(q, k, v, H, Hkv, pos0, 0.1), v, pos0 + M, TOL_PREFILL, "prefill H%d/%d" % (H, Hkv))


def test_prefill_m1024_sampled(qk_lib, cuda):
    """The benchmark's prefill shape (M = 1024, 24 / 8 heads), sampled query rows."""
    H, Hkv, M = 24, 8, 1024
    q, k, v = _inputs(85, M, H, Hkv, 0, M)
    scale = 1 / np.sqrt(D)
    got = _run(qk_lib, cuda, q, k, v, M, H, Hkv, 0, scale)
    rows = np.unique(np.concatenate([[0, 1, 63, 64, 511, M - 1], synth.rng_for(86, 0).choice(M, 40, replace=False)]))
    _check(got[rows], oracle.gqa_attention(q, k, v, H, Hkv, 0, scale, qrows=rows), v, M, TOL_PREFILL, "prefill M=1024")


def test_decode_step_matches_prefill_row(qk_lib, cuda):
    """The last row of a prefill equals a decode step at that position (two
    kernels, two precisions: within the prefill bar)."""
    H, Hkv, M = 24, 8, 300
    q, k, v = _inputs(87, M, H, Hkv, 0, M)
    scale = 1 / np.sqrt(D)
    pre = _run(qk_lib, cuda, q, k, v, M, H, Hkv, 0, scale)
    dec = _run(qk_lib, cuda, np.ascontiguousarray(q[M - 1:]), k, v, 1, H, Hkv, M - 1, scale)
    _check(pre[M - 1:], dec, v, M, TOL_PREFILL, "prefill row vs decode")


def test_attention_is_deterministic(qk_lib, cuda):
    H, Hkv = 24, 8
    for M, pos0 in ((1, 3000), (200, 0)):
        q, k, v = _inputs(88, M, H, Hkv, pos0, pos0 + M)
        a = _run(qk_lib, cuda, q, k, v, M, H, Hkv, pos0, 0.088)
        b = _run(qk_lib, cuda, q, k, v, M, H, Hkv, pos0, 0.088)
        assert np.array_equal(a, b)


def test_attention_rejects(qk_lib, cuda):
    import torch
    L = qk_lib.lib()
    s = torch.cuda.current_stream().cuda_stream
    qb = torch.zeros(4 * 32 * D, dtype=torch.float16, device=cuda)
    kb = torch.zeros(8 * 64 * D, dtype=torch.float16, device=cuda)
    vb = torch.zeros(8 * 64 * D, dtype=torch.float16, device=cuda)
    ob = torch.zeros(4 * 32 * D, dtype=torch.float32, device=cuda)
    q, k, v, o = qb.data_ptr(), kb.data_ptr(), vb.data_ptr(), ob.data_ptr()
    assert L.qk_gqa_attention(q, k, v, o, 1, 24, 8, 64, 0, 64, 0.1, s) == -3      # D != 128
    assert L.qk_gqa_attention(q, k, v, o, 1, 24, 7, 128, 0, 64, 0.1, s) == -3     # H % H_kv
    assert L.qk_gqa_attention(q, k, v, o, 1, 32, 2, 128, 0, 64, 0.1, s) == -3     # group of 16
    assert L.qk_gqa_attention(q, k, v, o, 4, 24, 8, 128, 61, 64, 0.1, s) == -3    # past L_max
    assert L.qk_gqa_attention(q, k, v, q, 1, 24, 8, 128, 0, 64, 0.1, s) == -7     # out over q
    assert L.qk_gqa_attention(q, k, v, o, 0, 24, 8, 128, 0, 64, 0.1, s) == 0      # nothing to do
    assert L.qk_gqa_attention(q + 8, k, v, o, 1, 24, 8, 128, 0, 64, 0.1, s) == -2  # misaligned
    assert L.qk_get_device_status(s) == 0
