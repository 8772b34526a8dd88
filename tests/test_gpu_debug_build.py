"""The checked build (-DQK_DEBUG): every bulk and tensor copy is tested for
alignment and shared-memory extent before it is issued, and a failed check is
reported as QK_ERR_BAD_COPY by qk_get_device_status.  The library is built into
a temporary directory and exercised in a child process over each kernel family
(dequant, decode GEMV, tensor-core GEMM with and without split K, fused
gate/up, int8-activation GEMV, RMSNorm batch, GQA attention decode and
prefill); every call must leave the status clean and match the oracle."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

_CHILD = r"""
import sys, numpy as np, torch
sys.path.insert(0, sys.argv[1])
import oracle, quantized_q4_matmul_gb300 as qk
from tests import synth
dev = torch.device("cuda", 0)
L = qk.lib()

def status():
    torch.cuda.synchronize()
    st = L.qk_get_device_status(None)
    assert st == 0, L.qk_status_string(st).decode()

def close(got, ref, what, tol=1e-2):
    err = np.max(np.abs(got - ref)) / max(np.sqrt(np.mean(ref ** 2)), 1e-30)
    assert err <= tol, (what, err)

QT = {"q4k": oracle.Q4K, "q6k": oracle.Q6K}
# dequant, bit-exact
for qt in ("q4k", "q6k"):
    rng = synth.rng_for(41, 7)
    W = synth.weights(rng, qt, 64, 1024)
    nb = 64 * 1024 // 256
    out = torch.empty(nb * 256, dtype=torch.float32, device=dev)
    (qk.qk_dequant_q4k if qt == "q4k" else qk.qk_dequant_q6k)(torch.from_numpy(W).to(dev), nb, out)
    status()
    assert np.array_equal(out.cpu().numpy().view(np.uint32),
                          np.asarray(oracle.dequant(QT[qt], W), np.float32).reshape(-1).view(np.uint32)), qt
# matmuls: GEMV (M <= 8), split-K GEMM, GEMM with a ragged tail
for qt, M, N, K in [("q4k", 1, 512, 3072), ("q6k", 4, 384, 3072), ("q4k", 48, 1024, 8192),
                    ("q6k", 16, 512, 4096), ("q4k", 200, 640, 2560), ("q6k", 300, 1024, 3072)]:
    rng = synth.rng_for(42, M * N)
    W = synth.weights(rng, qt, N, K)
    x = synth.activations(rng, M, K)
    y = torch.empty(M, N, dtype=torch.float32, device=dev)
    (qk.qk_matmul_q4k if qt == "q4k" else qk.qk_matmul_q6k)(
        torch.from_numpy(W).to(dev), torch.from_numpy(x.view(np.uint16)).to(dev), y, M, N, K)
    status()
    close(y.cpu().numpy().astype(np.float64), oracle.matmul(QT[qt], W, x, N, K), (qt, M, N, K))
# fused gate/up + SwiGLU: GEMV, split K, 3 x + 3 A stages
for M, N, K in [(1, 512, 3072), (16, 512, 4096), (192, 1024, 3072)]:
    rng = synth.rng_for(43, M)
    Wg, Wu = synth.q4k_weights(rng, N, K), synth.q4k_weights(rng, N, K)
    x = synth.activations(rng, M, K)
    y = torch.empty(M, N, dtype=torch.float16, device=dev)
    qk.qk_gateup_swiglu_q4k(torch.from_numpy(Wg).to(dev), torch.from_numpy(Wu).to(dev),
                            torch.from_numpy(x.view(np.uint16)).to(dev), y, M, N, K)
    status()
    close(y.float().cpu().numpy().astype(np.float64), oracle.gateup_swiglu(Wg, Wu, x, N, K), ("gate/up", M))
# int8 activations (decode)
rng = synth.rng_for(44, 1)
W = synth.q4k_weights(rng, 256, 3072)
x = synth.activations(rng, 1, 3072)
y = torch.empty(1, 256, dtype=torch.float32, device=dev)
qk.qk_matmul_q8x_q4k(torch.from_numpy(W).to(dev), torch.from_numpy(x.view(np.uint16)).to(dev), y, 1, 256, 3072)
status()
close(y.cpu().numpy().astype(np.float64), oracle.matmul(oracle.Q4K, W, x, 256, 3072), "q8x", tol=5e-2)
# RMSNorm in front of a grouped call (GEMV and GEMM problems)
for M in (1, 64):
    rng = synth.rng_for(45, M)
    K, N = 3072, 256
    W = synth.q4k_weights(rng, N, K)
    x = synth.activations(rng, M, K)
    gamma = (1.0 + 0.1 * rng.standard_normal(K)).astype(np.float16)
    y = torch.empty(M, N, dtype=torch.float32, device=dev)
    scratch = torch.empty(max(qk.qk_rmsnorm_scratch_bytes("q4k", M, K), 16), dtype=torch.uint8, device=dev)
    qk.qk_rmsnorm_matmul_batch([dict(qtype="q4k", blocks=torch.from_numpy(W).to(dev),
                                     x_f16=torch.from_numpy(x.view(np.uint16)).to(dev), y=y, M=M, N=N, K=K)],
                               torch.from_numpy(gamma.view(np.uint16)).to(dev), 1e-5, scratch)
    status()
    close(y.cpu().numpy().astype(np.float64), oracle.rmsnorm_matmul(oracle.Q4K, W, x, gamma, 1e-5, N, K),
          ("rmsnorm", M))
# GQA attention: decode over a cache, then a causal prefill chunk
H, Hkv, D, Lmax = 24, 8, 128, 512
for M, pos0 in [(1, 300), (160, 40)]:
    rng = synth.rng_for(46, M)
    q = rng.standard_normal((M, H, D)).astype(np.float16)
    k = np.zeros((Hkv, Lmax, D), np.float16)
    v = np.zeros((Hkv, Lmax, D), np.float16)
    n = pos0 + M
    k[:, :n] = rng.standard_normal((Hkv, n, D)).astype(np.float16)
    v[:, :n] = rng.standard_normal((Hkv, n, D)).astype(np.float16)
    out = torch.empty((M, H, D), dtype=torch.float32, device=dev)
    qk.qk_gqa_attention(torch.from_numpy(q.view(np.uint16)).to(dev), torch.from_numpy(k.view(np.uint16)).to(dev),
                        torch.from_numpy(v.view(np.uint16)).to(dev), out, M, H, Hkv, D, pos0, Lmax, D ** -0.5)
    status()
    ref = oracle.gqa_attention(q, k, v, H, Hkv, pos0, D ** -0.5)
    err = np.max(np.abs(out.cpu().numpy().astype(np.float64) - ref)) / np.abs(v[:, :n].astype(np.float64)).max()
    assert err <= 2e-3, ("attention", M, err)
print("ok")
"""


def test_checked_build_runs_clean(qk_lib, cuda, tmp_path):
    from quantized_q4_matmul_gb300 import build as qk_build
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    lib = qk_build.build(extra_flags=["-DQK_DEBUG"], out_dir=str(tmp_path))
    env = dict(os.environ, QK_LIB=lib)
    r = subprocess.run([sys.executable, "-c", _CHILD, root], env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout[-2000:] + r.stderr[-3000:]
