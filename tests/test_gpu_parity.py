"""GPU path against the oracle, through the C ABI.

Bars (stated by the workload definition):
* dequant: bit-exact fp32 (NaN matches NaN);
* matmul: max |y - y_oracle| <= 1e-2 * rms(y_oracle) per call;
* gate/up + SwiGLU, whose output format is fp16: the same bar on top of the
  output's own rounding, i.e. |y - y_oracle| - ulp16(y)/2 <= 1e-2 * rms(y_oracle)
  (the SwiGLU output is heavy-tailed, max ~ 25 x rms, so fp16 rounding of the
  largest outputs alone reaches ~0.7% of rms).
Inputs are the seeded synthetic weights / activations of ``tests/synth.py``.
Full-size workloads are checked on seeded samples of output rows (all tokens),
which the oracle computes one row at a time.
"""
import numpy as np
import pytest

import oracle
from tests import synth
from tests.oracle_pins import random_blocks, same_bits

pytestmark = pytest.mark.gpu

TOL = 1e-2
QT = {"q4k": oracle.Q4K, "q6k": oracle.Q6K}


def _dev(a, cuda):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to(cuda)


def _x_dev(x, cuda):
    return _dev(x.view(np.uint16), cuda)


def gpu_matmul(qk, qtype, W, x, N, K, cuda, rows=None):
    import torch
    M = x.shape[0]
    y = torch.empty(M, N, dtype=torch.float32, device=cuda)
    fn = qk.qk_matmul_q4k if qtype == "q4k" else qk.qk_matmul_q6k
    fn(_dev(W, cuda), _x_dev(x, cuda), y, M, N, K)
    qk.qk_get_device_status()
    y = y.cpu().numpy().astype(np.float64)
    return y if rows is None else y[:, rows]


# achieved max|err| / rms per check, printed at the end of the session (conftest)
MARGINS = []


def check_close(got, ref, what):
    rms = float(np.sqrt(np.mean(ref ** 2)))
    err = float(np.max(np.abs(got - ref))) if ref.size else 0.0
    assert np.isfinite(got).all(), what
    assert err <= TOL * rms, "%s: max|err| %.3e > %.0e * rms %.3e" % (what, err, TOL, rms)
    MARGINS.append((what, err / rms if rms else 0.0))
    return err / rms if rms else 0.0


def check_close_f16out(got, ref, what):
    """As check_close for an fp16 output, with two bars:
    * the output format's own rounding (half an fp16 ulp of the value) allowed on
      top of the 1e-2 * rms bar, against the exact (fp64) oracle;
    * against the oracle rounded to fp16 itself: each output within 1e-2 * rms
      or, where an fp16 ulp of the value is larger than that, within one ulp (an
      exact value next to a rounding midpoint may round either way after the
      kernel's fp32 sums).  A kernel arithmetic error such as a coarse sigmoid
      shows as several ulps at the large outputs and fails it."""
    rms = float(np.sqrt(np.mean(ref ** 2)))
    mag = np.maximum(np.abs(ref), np.abs(got))
    half_ulp = np.ldexp(0.5, np.floor(np.log2(np.maximum(mag, 2.0 ** -14))).astype(np.int64) - 10)
    err = np.abs(got - ref)
    assert np.isfinite(got).all(), what
    worst = float(np.max(err - half_ulp)) if ref.size else 0.0
    assert worst <= TOL * rms, "%s: max(|err| - half_ulp) %.3e > %.0e * rms %.3e" % (what, worst, TOL, rms)
    ref16 = ref.astype(np.float16).astype(np.float64)
    err16 = np.abs(got - ref16)
    bar16 = np.maximum(TOL * rms, 2.0 * half_ulp)
    over = float(np.max(err16 - bar16)) if ref.size else 0.0
    assert over <= 0.0, "%s: |err vs fp16(oracle)| above max(%.0e * rms, 1 ulp) by %.3e (rms %.3e)" % (
        what, TOL, over, rms)
    small = err16[bar16 <= TOL * rms]
    MARGINS.append((what + " (vs fp16 oracle)", float(np.max(small)) / rms if rms and small.size else 0.0))


def sample_rows(N, n, seed):
    rng = synth.rng_for(seed, 777)
    k = min(N, n)
    rows = rng.choice(N, size=k, replace=False)
    rows[0], rows[-1] = 0, N - 1
    return np.unique(rows)


# ---------------------------------------------------------------------------
# Dequant
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("qtype", ["q4k", "q6k"])
@pytest.mark.parametrize("nb", [1, 7, 33, 4099, 250_000])
def test_dequant_bit_exact(qk_lib, cuda, qtype, nb):
    import torch
    blocks = random_blocks(QT[qtype], nb, seed=nb)
    out = torch.empty(nb * 256, dtype=torch.float32, device=cuda)
    fn = qk_lib.qk_dequant_q4k if qtype == "q4k" else qk_lib.qk_dequant_q6k
    fn(_dev(blocks, cuda), nb, out)
    qk_lib.qk_get_device_status()
    assert same_bits(out.cpu().numpy(), oracle.dequant(QT[qtype], blocks))


def test_dequant_into_unaligned_tail_region(qk_lib, cuda):
    # Q6_K blocks are 210 bytes: an odd block count leaves the tensor end 2 mod 16.
    import torch
    blocks = random_blocks(oracle.Q6K, 3, seed=5)
    out = torch.empty(3 * 256, dtype=torch.float32, device=cuda)
    qk_lib.qk_dequant_q6k(_dev(blocks, cuda), 3, out)
    assert same_bits(out.cpu().numpy(), oracle.dequant(oracle.Q6K, blocks))


# ---------------------------------------------------------------------------
# Matmul: small shapes spanning several tiles with ragged tails
# ---------------------------------------------------------------------------
SHAPES = [
    (1, 128, 256), (1, 200, 768), (1, 1024, 3072), (1, 40, 8192),
    (2, 128, 256), (5, 300, 512), (16, 256, 768), (17, 130, 1024),
    (64, 384, 512), (100, 200, 1280), (256, 128, 2048), (300, 260, 512), (513, 128, 256),
]


@pytest.mark.parametrize("qtype", ["q4k", "q6k"])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_matmul_small(qk_lib, cuda, qtype, M, N, K):
    rng = synth.rng_for(M * 7 + N, K)
    W = synth.weights(rng, qtype, N, K)
    x = synth.activations(rng, M, K)
    ref = oracle.matmul(QT[qtype], W, x, N, K)
    check_close(gpu_matmul(qk_lib, qtype, W, x, N, K, cuda), ref, "%s M%d N%d K%d" % (qtype, M, N, K))


# Several tokens on the GEMV (tokens in the MMA columns) for M <= 8, ragged N,
# both K of the model; M = 9..16 on the tensor-core GEMM, next to them.
SMALL_M = [(M, N, K) for M in (2, 3, 7, 8, 9, 12, 16) for N, K in ((200, 3072), (48, 1024))] + \
          [(M, 80, 8192) for M in (2, 5, 8, 16)]


@pytest.mark.parametrize("qtype", ["q4k", "q6k"])
@pytest.mark.parametrize("M,N,K", SMALL_M)
def test_matmul_small_m_gemv(qk_lib, cuda, qtype, M, N, K):
    assert qk_lib.qk_uses_gemv(qtype, M, K) == (M <= 8)
    rng = synth.rng_for(M * 13 + N, K + 1)
    W = synth.weights(rng, qtype, N, K)
    x = synth.activations(rng, M, K)
    ref = oracle.matmul(QT[qtype], W, x, N, K)
    check_close(gpu_matmul(qk_lib, qtype, W, x, N, K, cuda), ref, "%s M%d N%d K%d" % (qtype, M, N, K))


@pytest.mark.parametrize("M", [2, 8, 16])
def test_gateup_small_m_gemv(qk_lib, cuda, M):
    import torch
    N, K = 144, 3072
    assert qk_lib.qk_uses_gemv("q4k", M, K, gateup=True) == (M <= 8)
    rng = synth.rng_for(M, 77)
    Wg, Wu = synth.q4k_weights(rng, N, K), synth.q4k_weights(rng, N, K)
    x = synth.activations(rng, M, K)
    y = torch.empty(M, N, dtype=torch.float16, device=cuda)
    qk_lib.qk_gateup_swiglu_q4k(_dev(Wg, cuda), _dev(Wu, cuda), _x_dev(x, cuda), y, M, N, K)
    qk_lib.qk_get_device_status()
    check_close_f16out(y.float().cpu().numpy().astype(np.float64), oracle.gateup_swiglu(Wg, Wu, x, N, K),
                       "gate/up M%d" % M)


def test_batch_small_m_matches_single_calls(qk_lib, cuda):
    """QKV-shaped problems at M = 8 in one grouped launch: bit-identical to the
    single calls (each keeps its own plan and split over warps)."""
    import torch
    probs, singles = [], []
    for i, (qt, N) in enumerate((("q4k", 3072), ("q4k", 1024), ("q6k", 1024))):
        rng = synth.rng_for(81, i)
        W = synth.weights(rng, qt, N, 3072)
        x = synth.activations(rng, 8, 3072)
        y = torch.full((8, N), float("nan"), device=cuda)
        probs.append(dict(qtype=qt, blocks=_dev(W, cuda), x_f16=_x_dev(x, cuda), y=y, M=8, N=N, K=3072))
        singles.append(gpu_matmul(qk_lib, qt, W, x, N, 3072, cuda))
    qk_lib.qk_matmul_batch(probs)
    qk_lib.qk_get_device_status()
    for p, single in zip(probs, singles):
        assert np.array_equal(p["y"].cpu().numpy().astype(np.float64), single)


@pytest.mark.parametrize("qtype", ["q4k", "q6k"])
def test_matmul_deterministic(qk_lib, cuda, qtype):
    rng = synth.rng_for(3, 3)
    W = synth.weights(rng, qtype, 256, 1024)
    for M in (1, 200):
        x = synth.activations(rng, M, 1024)
        a = gpu_matmul(qk_lib, qtype, W, x, 256, 1024, cuda)
        b = gpu_matmul(qk_lib, qtype, W, x, 256, 1024, cuda)
        assert np.array_equal(a, b)


@pytest.mark.parametrize("kind,N,K,M", [("gateup", 8192, 3072, 1024), ("q4k", 8192, 3072, 1024),
                                        ("q4k", 3072, 3072, 1024), ("q6k", 3072, 8192, 1024),
                                        ("q6k", 16384, 3072, 1024), ("gateup", 8192, 3072, 960),
                                        ("gateup", 8192, 3072, 192)])
def test_full_size_repeatable(qk_lib, cuda, kind, N, K, M):
    """Repeated launches give bit-identical outputs.  These shapes cover every
    pipeline configuration of the prefill GEMM (two-tensor split producer, one
    and two packed stages, gate/up with 3 x + 2 A and 3 x + 3 A stages); a
    missing ordering between the dequant threads' reads of a packed slot and its
    refill showed up as run-to-run differences."""
    import torch
    rng = synth.rng_for(11, N)
    x = _x_dev(synth.activations(rng, M, K), cuda)
    if kind == "gateup":
        Wg, Wu = _dev(synth.q4k_weights(rng, N, K), cuda), _dev(synth.q4k_weights(rng, N, K), cuda)
        y = torch.empty(M, N, dtype=torch.float16, device=cuda)
        call = lambda: qk_lib.qk_gateup_swiglu_q4k(Wg, Wu, x, y, M, N, K)
    else:
        W = _dev(synth.weights(rng, kind, N, K), cuda)
        y = torch.empty(M, N, dtype=torch.float32, device=cuda)
        fn = qk_lib.qk_matmul_q4k if kind == "q4k" else qk_lib.qk_matmul_q6k
        call = lambda: fn(W, x, y, M, N, K)
    call()
    first = y.clone()
    for _ in range(6):
        call()
        assert torch.equal(y, first)
    qk_lib.qk_get_device_status()


_SMEM_A_CHILD = """
import sys, numpy as np, torch
sys.path.insert(0, sys.argv[1])
import oracle, quantized_q4_matmul_gb300 as qk
from tests import synth
dev = torch.device("cuda", 0)
for qtype, M, N, K in [("q4k", 200, 384, 1024), ("q6k", 200, 384, 1024), ("q4k", 37, 200, 768),
                       ("q6k", 37, 200, 768), ("q6k", 300, 1024, 3072)]:
    rng = synth.rng_for(31, N)
    W = synth.weights(rng, qtype, N, K)
    x = synth.activations(rng, M, K)
    y = torch.empty(M, N, dtype=torch.float32, device=dev)
    fn = qk.qk_matmul_q4k if qtype == "q4k" else qk.qk_matmul_q6k
    fn(torch.from_numpy(W).to(dev), torch.from_numpy(x.view(np.uint16)).to(dev), y, M, N, K)
    qk.qk_get_device_status()
    ref = oracle.matmul(oracle.Q4K if qtype == "q4k" else oracle.Q6K, W, x, N, K)
    err = np.max(np.abs(y.cpu().numpy() - ref)) / np.sqrt(np.mean(ref ** 2))
    assert err <= 1e-2, (qtype, M, N, K, err)
print("ok")
"""


def test_shared_memory_a_tiles_path(qk_lib, cuda):
    """Single-tensor GEMMs keep A tiles in tensor memory by default; the
    shared-memory A path (QK_A_TMEM=0, read once per process) is checked
    against the oracle in a child process."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, QK_A_TMEM="0")
    r = subprocess.run([sys.executable, "-c", _SMEM_A_CHILD, root], env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout[-2000:] + r.stderr[-2000:]


@pytest.mark.parametrize("qtype", ["q4k", "q6k"])
def test_matmul_special_scales(qk_lib, cuda, qtype):
    """Zero, subnormal and large fp16 scale fields (finite)."""
    rng = synth.rng_for(9, 9)
    N, K = 128, 512
    W = synth.weights(rng, qtype, N, K).reshape(-1, 144 if qtype == "q4k" else 210).copy()
    vals = np.array([0.0, 6e-8, 3e-5, 1e-3, 0.25], np.float16).view(np.uint8).reshape(-1, 2)
    pick = rng.integers(0, len(vals), size=len(W))
    if qtype == "q4k":
        W[:, 0:2] = vals[pick]
        W[:, 2:4] = vals[rng.integers(0, len(vals), size=len(W))]
    else:
        W[:, 208:210] = vals[pick]
    for M in (1, 48):
        x = synth.activations(rng, M, K)
        ref = oracle.matmul(QT[qtype], W, x, N, K)
        check_close(gpu_matmul(qk_lib, qtype, W, x, N, K, cuda), ref, "special scales M%d" % M)


# ---------------------------------------------------------------------------
# The workloads at full size
# ---------------------------------------------------------------------------
def test_workload_attn_q_m16(qk_lib, cuda):
    """Single Q4_K matmul, M=16, K=3072, N=3072, seed 0 (checked in full)."""
    rng = synth.rng_for(0, 0)
    W = synth.q4k_weights(rng, 3072, 3072)
    x = synth.activations(rng, 16, 3072)
    ref = oracle.matmul(oracle.Q4K, W, x, 3072, 3072)
    check_close(gpu_matmul(qk_lib, "q4k", W, x, 3072, 3072, cuda), ref, "attn_q M16")


def test_workload_decode_layer_m1(qk_lib, cuda):
    """Decode GEMV, M=1, over the seven linears of one layer (checked in full)."""
    for tag, lin, M in synth.workloads()["decode_layer_m1"].linears:
        rng = synth.rng_for(1, tag)
        W = synth.weights(rng, lin.qtype, lin.N, lin.K)
        x = synth.activations(rng, M, lin.K)
        ref = oracle.matmul(QT[lin.qtype], W, x, lin.N, lin.K)
        check_close(gpu_matmul(qk_lib, lin.qtype, W, x, lin.N, lin.K, cuda), ref, lin.name)


def test_workload_prefill_gateup_swiglu_m1024(qk_lib, cuda):
    """Fused gate/up + SwiGLU, M=1024, K=3072, N_ff=8192 (sampled output features)."""
    import torch
    rng = synth.rng_for(2, 0)
    M, N, K = 1024, 8192, 3072
    Wg = synth.q4k_weights(rng, N, K)
    Wu = synth.q4k_weights(rng, N, K)
    x = synth.activations(rng, M, K)
    y = torch.empty(M, N, dtype=torch.float16, device=cuda)
    qk_lib.qk_gateup_swiglu_q4k(_dev(Wg, cuda), _dev(Wu, cuda), _x_dev(x, cuda), y, M, N, K)
    qk_lib.qk_get_device_status()
    rows = sample_rows(N, 96, 2)
    ref = oracle.gateup_swiglu(Wg, Wu, x, N, K, rows=rows)
    check_close_f16out(y.float().cpu().numpy().astype(np.float64)[:, rows], ref, "gate/up swiglu")


def test_workload_prefill_down_v_m1024(qk_lib, cuda):
    """Q6_K down 8192->3072 and attn_v 3072->1024 at M=1024 (sampled output features)."""
    for tag, lin, M in synth.workloads()["prefill_down_v_m1024"].linears:
        rng = synth.rng_for(3, tag)
        W = synth.weights(rng, lin.qtype, lin.N, lin.K)
        x = synth.swiglu_activations(rng, M, lin.K)
        rows = sample_rows(lin.N, 64, 3 + tag)
        ref = oracle.matmul(QT[lin.qtype], W, x, lin.N, lin.K, rows=rows)
        check_close(gpu_matmul(qk_lib, lin.qtype, W, x, lin.N, lin.K, cuda, rows=rows), ref, lin.name)


SWEEP_SHAPES = sorted({(lin.qtype, lin.N, lin.K) for _, lin in synth.model_linears()})


@pytest.mark.parametrize("qtype,N,K", SWEEP_SHAPES)
def test_workload_model_sweep(qk_lib, cuda, qtype, N, K):
    """Every distinct linear of the 3B model (incl. the tied LM head) at M in 1..2048, sampled rows."""
    rng = synth.rng_for(4, N + K + (qtype == "q6k"))
    W = synth.weights(rng, qtype, N, K)
    Wd = _dev(W, cuda)
    import torch
    for M in synth.SWEEP_M:
        x = synth.activations(rng, M, K)
        y = torch.empty(M, N, dtype=torch.float32, device=cuda)
        fn = qk_lib.qk_matmul_q4k if qtype == "q4k" else qk_lib.qk_matmul_q6k
        fn(Wd, _x_dev(x, cuda), y, M, N, K)
        qk_lib.qk_get_device_status()
        rows = sample_rows(N, 24 if M >= 512 else 64, M)
        ref = oracle.matmul(QT[qtype], W, x, N, K, rows=rows)
        check_close(y.cpu().numpy().astype(np.float64)[:, rows], ref, "%s N%d K%d M%d" % (qtype, N, K, M))
        del y


# ---------------------------------------------------------------------------
# Gate/up + SwiGLU small shapes
# ---------------------------------------------------------------------------
def test_gateup_model_sweep(qk_lib, cuda):
    """Fused gate/up + SwiGLU at the model's shape (N_ff = 8192, K = 3072) over the
    token counts whose launch configurations differ (split K at small M, token
    tile and pipeline depths at large M); sampled output features."""
    import torch
    rng = synth.rng_for(12, 0)
    N, K = 8192, 3072
    Wg, Wu = synth.q4k_weights(rng, N, K), synth.q4k_weights(rng, N, K)
    Wgd, Wud = _dev(Wg, cuda), _dev(Wu, cuda)
    for M in (16, 128, 192, 512, 960, 2048):
        x = synth.activations(rng, M, K)
        y = torch.empty(M, N, dtype=torch.float16, device=cuda)
        qk_lib.qk_gateup_swiglu_q4k(Wgd, Wud, _x_dev(x, cuda), y, M, N, K)
        qk_lib.qk_get_device_status()
        rows = sample_rows(N, 24, M)
        ref = oracle.gateup_swiglu(Wg, Wu, x, N, K, rows=rows)
        check_close_f16out(y.float().cpu().numpy().astype(np.float64)[:, rows], ref, "gate/up M%d" % M)
        del y


@pytest.mark.parametrize("M,N,K", [(1, 128, 256), (16, 256, 512), (37, 200, 768), (300, 384, 1024)])
def test_gateup_small(qk_lib, cuda, M, N, K):
    import torch
    rng = synth.rng_for(M, N + K)
    Wg = synth.q4k_weights(rng, N, K)
    Wu = synth.q4k_weights(rng, N, K)
    x = synth.activations(rng, M, K)
    y = torch.empty(M, N, dtype=torch.float16, device=cuda)
    qk_lib.qk_gateup_swiglu_q4k(_dev(Wg, cuda), _dev(Wu, cuda), _x_dev(x, cuda), y, M, N, K)
    qk_lib.qk_get_device_status()
    ref = oracle.gateup_swiglu(Wg, Wu, x, N, K)
    check_close_f16out(y.float().cpu().numpy().astype(np.float64), ref, "gateup M%d N%d K%d" % (M, N, K))


# Split K with the reduce-scatter exchange: few row tiles, so the planner splits
# K over up to 8 CTAs, at token tiles of 3, 5, 7 and 16 chunks of 16 -- ranks
# that own one slice, several, or none of the tile's columns.
SPLIT_SHAPES = [(48, 1024, 8192), (80, 512, 4096), (112, 256, 12288), (256, 1024, 3072), (200, 640, 2560)]


@pytest.mark.parametrize("qtype", ["q4k", "q6k"])
@pytest.mark.parametrize("M,N,K", SPLIT_SHAPES)
def test_matmul_split_k_slices(qk_lib, cuda, qtype, M, N, K):
    rng = synth.rng_for(M * 13 + N, K + 1)
    W = synth.weights(rng, qtype, N, K)
    x = synth.activations(rng, M, K)
    ref = oracle.matmul(QT[qtype], W, x, N, K)
    check_close(gpu_matmul(qk_lib, qtype, W, x, N, K, cuda), ref, "split %s M%d N%d K%d" % (qtype, M, N, K))


@pytest.mark.parametrize("M,N,K", [(48, 512, 4096), (112, 256, 6144)])
def test_gateup_split_k_slices(qk_lib, cuda, M, N, K):
    import torch
    rng = synth.rng_for(M * 3 + N, K + 2)
    Wg = synth.q4k_weights(rng, N, K)
    Wu = synth.q4k_weights(rng, N, K)
    x = synth.activations(rng, M, K)
    y = torch.empty(M, N, dtype=torch.float16, device=cuda)
    qk_lib.qk_gateup_swiglu_q4k(_dev(Wg, cuda), _dev(Wu, cuda), _x_dev(x, cuda), y, M, N, K)
    qk_lib.qk_get_device_status()
    ref = oracle.gateup_swiglu(Wg, Wu, x, N, K)
    check_close_f16out(y.float().cpu().numpy().astype(np.float64), ref, "split gateup M%d N%d K%d" % (M, N, K))


# ---------------------------------------------------------------------------
# Boundary checks that need a device
# ---------------------------------------------------------------------------
def test_alias_and_host_pointer_rejected(qk_lib, cuda):
    import torch
    L = qk_lib.lib()
    W = torch.zeros(128 * 144, dtype=torch.uint8, device=cuda)
    x = torch.zeros(4 * 256, dtype=torch.float16, device=cuda)
    y = torch.zeros(4 * 128, dtype=torch.float32, device=cuda)
    s = torch.cuda.current_stream().cuda_stream
    assert L.qk_matmul_q4k(W.data_ptr(), x.data_ptr(), W.data_ptr(), 4, 128, 256, s) == -7  # y aliases W
    host = np.zeros(1 << 16, np.uint8)
    hp = (host.ctypes.data + 15) & ~15
    assert L.qk_matmul_q4k(hp, x.data_ptr(), y.data_ptr(), 4, 128, 256, s) == -8  # pageable host memory
    assert L.qk_matmul_q4k(W.data_ptr(), x.data_ptr(), y.data_ptr(), 4, 128, 256, s) == 0
    assert L.qk_get_device_status(s) == 0


# ---------------------------------------------------------------------------
# Grouped calls
# ---------------------------------------------------------------------------
def test_batch_decode_layer_matches_single_calls(qk_lib, cuda):
    """The seven M = 1 linears of a layer in one grouped launch: bit-identical to
    the single-problem calls, and within the bar of the oracle."""
    import torch
    probs, singles, refs = [], [], []
    for tag, lin, M in synth.workloads()["decode_layer_m1"].linears:
        rng = synth.rng_for(11, tag)
        W = synth.weights(rng, lin.qtype, lin.N, lin.K)
        x = synth.activations(rng, M, lin.K)
        Wd, xd = _dev(W, cuda), _x_dev(x, cuda)
        y = torch.full((M, lin.N), float("nan"), device=cuda)
        probs.append(dict(qtype=lin.qtype, blocks=Wd, x_f16=xd, y=y, M=M, N=lin.N, K=lin.K))
        refs.append(oracle.matmul(QT[lin.qtype], W, x, lin.N, lin.K))
        singles.append(gpu_matmul(qk_lib, lin.qtype, W, x, lin.N, lin.K, cuda))
    qk_lib.qk_matmul_batch(probs)
    qk_lib.qk_get_device_status()
    for p, ref, single in zip(probs, refs, singles):
        got = p["y"].cpu().numpy().astype(np.float64)
        assert np.array_equal(got, single)
        check_close(got, ref, "batch N%d K%d" % (p["N"], p["K"]))


def test_batch_mixed_and_gateup(qk_lib, cuda):
    """M = 1 gate/up + SwiGLU, an M > 1 problem, an empty problem and >8 GEMVs in one call."""
    import torch
    rng = synth.rng_for(12, 0)
    K, N = 1024, 256
    Wg, Wu = synth.q4k_weights(rng, N, K), synth.q4k_weights(rng, N, K)
    x1 = synth.activations(rng, 1, K)
    yg = torch.empty(1, N, dtype=torch.float16, device=cuda)
    probs = [dict(qtype="q4k", blocks=_dev(Wg, cuda), up_blocks=_dev(Wu, cuda), x_f16=_x_dev(x1, cuda), y=yg, M=1,
                  N=N, K=K)]
    x40 = synth.activations(rng, 40, K)
    W6 = synth.q6k_weights(rng, 200, K)
    y40 = torch.empty(40, 200, device=cuda)
    probs.append(dict(qtype="q6k", blocks=_dev(W6, cuda), x_f16=_x_dev(x40, cuda), y=y40, M=40, N=200, K=K))
    probs.append(dict(qtype="q4k", blocks=_dev(Wg, cuda), x_f16=_x_dev(x1, cuda), y=torch.empty(1, 0, device=cuda),
                      M=1, N=0, K=K))
    smalls = []
    for i in range(9):
        W = synth.weights(rng, "q4k" if i % 2 else "q6k", 48 + 16 * i, K)
        x = synth.activations(rng, 1, K)
        y = torch.empty(1, W.shape[0], device=cuda)
        smalls.append((W, x, y, "q4k" if i % 2 else "q6k"))
        probs.append(dict(qtype=smalls[-1][3], blocks=_dev(W, cuda), x_f16=_x_dev(x, cuda), y=y, M=1, N=W.shape[0],
                          K=K))
    qk_lib.qk_matmul_batch(probs)
    qk_lib.qk_get_device_status()
    check_close_f16out(yg.float().cpu().numpy().astype(np.float64), oracle.gateup_swiglu(Wg, Wu, x1, N, K), "gu M1")
    check_close(y40.cpu().numpy().astype(np.float64), oracle.matmul(oracle.Q6K, W6, x40, 200, K), "q6k M40")
    for W, x, y, qt in smalls:
        check_close(y.cpu().numpy().astype(np.float64), oracle.matmul(QT[qt], W, x, W.shape[0], K), "small")


def test_batch_alias_between_entries_rejected(qk_lib, cuda):
    import torch
    W = torch.zeros(128 * 144, dtype=torch.uint8, device=cuda)
    x = torch.zeros(256, dtype=torch.float16, device=cuda)
    y = torch.zeros(128, dtype=torch.float32, device=cuda)
    p = dict(qtype="q4k", blocks=W, x_f16=x, y=y, M=1, N=128, K=256)
    with pytest.raises(qk_lib.QKError) as e:
        qk_lib.qk_matmul_batch([p, dict(p)])  # two entries write the same y
    assert e.value.status == -7


def test_gateup_decode_m1(qk_lib, cuda):
    """qk_gateup_swiglu_q4k at M = 1 (the grouped-GEMV gate/up path) at full size."""
    import torch
    rng = synth.rng_for(13, 0)
    N, K = 8192, 3072
    Wg, Wu = synth.q4k_weights(rng, N, K), synth.q4k_weights(rng, N, K)
    x = synth.activations(rng, 1, K)
    y = torch.empty(1, N, dtype=torch.float16, device=cuda)
    qk_lib.qk_gateup_swiglu_q4k(_dev(Wg, cuda), _dev(Wu, cuda), _x_dev(x, cuda), y, 1, N, K)
    qk_lib.qk_get_device_status()
    check_close_f16out(y.float().cpu().numpy().astype(np.float64), oracle.gateup_swiglu(Wg, Wu, x, N, K), "gu M1")


# ---------------------------------------------------------------------------
# Failure path: a bounded wait that runs out (no fault, no unbounded wait)
# ---------------------------------------------------------------------------
def test_wait_timeout_is_reported_and_the_context_stays_usable(qk_lib, cuda):
    """A kernel whose only mbarrier wait can never complete gives up after its
    wall-clock limit; the host reads QK_ERR_TIMEOUT, the status is cleared, and
    the next call runs and checks out."""
    import time
    import torch
    t0 = time.perf_counter()
    qk_lib.qk_debug_wait_timeout(20_000_000)  # 20 ms
    with pytest.raises(qk_lib.QKError) as e:
        qk_lib.qk_get_device_status()
    assert e.value.status == -5
    assert time.perf_counter() - t0 >= 0.02
    qk_lib.qk_get_device_status()  # read once, then cleared
    rng = synth.rng_for(21, 0)
    W = synth.q4k_weights(rng, 128, 512)
    x = synth.activations(rng, 3, 512)
    y = torch.empty(3, 128, dtype=torch.float32, device=cuda)
    qk_lib.qk_matmul_q4k(_dev(W, cuda), _x_dev(x, cuda), y, 3, 128, 512)
    qk_lib.qk_get_device_status()
    check_close(y.cpu().numpy().astype(np.float64), oracle.matmul(QT["q4k"], W, x, 128, 512), "after timeout")


# ---------------------------------------------------------------------------
# M = 1 problems whose K the GEMV cannot stage run on the tensor-core GEMM
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("qtype,N,K", [("q6k", 200, 6912), ("q6k", 70, 26624), ("q4k", 50, 35840), ("q4k", 33, 2304)])
def test_decode_largest_k_on_the_gemv(qk_lib, cuda, qtype, N, K):
    """K at the decode GEMV's limits: whole Q6_K rows of an odd block count
    (rows 2 mod 4 bytes aligned), 8-block Q6_K chunks, 5-block Q4_K chunks,
    and two-tile stages with an odd last tile."""
    assert qk_lib.qk_decode_uses_gemv(qtype, K)
    rng = synth.rng_for(43, K)
    W = synth.weights(rng, qtype, N, K)
    x = synth.activations(rng, 1, K)
    ref = oracle.matmul(QT[qtype], W, x, N, K)
    check_close(gpu_matmul(qk_lib, qtype, W, x, N, K, cuda), ref, "%s M1 N%d K%d on the GEMV" % (qtype, N, K))


@pytest.mark.parametrize("qtype,N,K", [("q6k", 200, 8448), ("q4k", 130, 65536)])
def test_decode_fallback_to_gemm(qk_lib, cuda, qtype, N, K):
    assert not qk_lib.qk_decode_uses_gemv(qtype, K)
    rng = synth.rng_for(41, K)
    W = synth.weights(rng, qtype, N, K)
    x = synth.activations(rng, 1, K)
    ref = oracle.matmul(QT[qtype], W, x, N, K)
    check_close(gpu_matmul(qk_lib, qtype, W, x, N, K, cuda), ref, "%s M1 K%d on the GEMM" % (qtype, K))


def test_decode_gateup_at_the_gemv_limit(qk_lib, cuda):
    """Fused gate/up at M = 1 with the longest rows the decode GEMV stages
    (K = 35072 with 8 compute warps), and one super-block beyond (GEMM)."""
    import torch
    N = 96
    for K, on_gemv in ((35072, True), (35328, False)):
        assert qk_lib.qk_decode_uses_gemv("q4k", K, gateup=True) == on_gemv
        rng = synth.rng_for(43, K)
        Wg, Wu = synth.q4k_weights(rng, N, K), synth.q4k_weights(rng, N, K)
        x = synth.activations(rng, 1, K)
        y = torch.empty(1, N, dtype=torch.float16, device=cuda)
        qk_lib.qk_gateup_swiglu_q4k(_dev(Wg, cuda), _dev(Wu, cuda), _x_dev(x, cuda), y, 1, N, K)
        qk_lib.qk_get_device_status()
        check_close_f16out(y.float().cpu().numpy().astype(np.float64), oracle.gateup_swiglu(Wg, Wu, x, N, K),
                           "gate/up M1 K%d" % K)


def test_decode_gateup_fallback_to_gemm(qk_lib, cuda):
    import torch
    N, K = 192, 65536
    assert not qk_lib.qk_decode_uses_gemv("q4k", K, gateup=True)
    rng = synth.rng_for(42, K)
    Wg, Wu = synth.q4k_weights(rng, N, K), synth.q4k_weights(rng, N, K)
    x = synth.activations(rng, 1, K)
    y = torch.empty(1, N, dtype=torch.float16, device=cuda)
    qk_lib.qk_gateup_swiglu_q4k(_dev(Wg, cuda), _dev(Wu, cuda), _x_dev(x, cuda), y, 1, N, K)
    qk_lib.qk_get_device_status()
    check_close_f16out(y.float().cpu().numpy().astype(np.float64), oracle.gateup_swiglu(Wg, Wu, x, N, K),
                       "gate/up M1 K%d on the GEMM" % K)


def test_batch_mixed_k_group(qk_lib, cuda):
    """M = 1 problems of different K share one launch (each keeps its own plan,
    the launch takes the largest shared-memory size); a Q6_K at K = 16640 and
    a Q4_K at K = 36864 fit no GEMV plan and run on the GEMM.  Every result is
    bit-identical to its single-problem call: the order of every addition
    depends on the problem's shape only."""
    import torch
    assert qk_lib.qk_decode_uses_gemv("q4k", 6144, gateup=True) and qk_lib.qk_decode_uses_gemv("q6k", 16384)
    assert not qk_lib.qk_decode_uses_gemv("q6k", 16640) and not qk_lib.qk_decode_uses_gemv("q4k", 36864)
    rng = synth.rng_for(43, 0)
    probs, checks = [], []
    Wg, Wu = synth.q4k_weights(rng, 128, 6144), synth.q4k_weights(rng, 128, 6144)
    xg = synth.activations(rng, 1, 6144)
    yg = torch.empty(1, 128, dtype=torch.float16, device=cuda)
    Wgd, Wud, xgd = _dev(Wg, cuda), _dev(Wu, cuda), _x_dev(xg, cuda)
    probs.append(dict(qtype="q4k", blocks=Wgd, up_blocks=Wud, x_f16=xgd, y=yg, M=1, N=128, K=6144))
    singles = []
    for qt, N, K in (("q6k", 64, 16384), ("q6k", 64, 16640), ("q4k", 256, 3072), ("q4k", 48, 36864)):
        W = synth.weights(rng, qt, N, K)
        x = synth.activations(rng, 1, K)
        y = torch.empty(1, N, dtype=torch.float32, device=cuda)
        probs.append(dict(qtype=qt, blocks=_dev(W, cuda), x_f16=_x_dev(x, cuda), y=y, M=1, N=N, K=K))
        checks.append((y, oracle.matmul(QT[qt], W, x, N, K), "%s K%d" % (qt, K)))
        singles.append(gpu_matmul(qk_lib, qt, W, x, N, K, cuda))
    ys = torch.empty(1, 128, dtype=torch.float16, device=cuda)
    qk_lib.qk_gateup_swiglu_q4k(Wgd, Wud, xgd, ys, 1, 128, 6144)
    qk_lib.qk_matmul_batch(probs)
    qk_lib.qk_get_device_status()
    assert torch.equal(yg, ys)
    check_close_f16out(yg.float().cpu().numpy().astype(np.float64), oracle.gateup_swiglu(Wg, Wu, xg, 128, 6144),
                       "gate/up K6144")
    for (y, ref, what), single in zip(checks, singles):
        got = y.cpu().numpy().astype(np.float64)
        assert np.array_equal(got, single), what
        check_close(got, ref, what)


# ---------------------------------------------------------------------------
# Stream order around the decode kernel's programmatic dependent launch
# ---------------------------------------------------------------------------
def _long_kernel(cuda):
    """A few hundred microseconds of unrelated work on the current stream."""
    import torch
    buf = torch.empty(256 << 20, dtype=torch.uint8, device=cuda)
    return lambda: buf.fill_(7)


def test_decode_reads_x_written_just_before(qk_lib, cuda):
    """x written by the kernel right before a decode call is the x it reads:
    the decode kernel may be scheduled while that kernel runs (programmatic
    dependent launch) but reads memory only after it has finished.  x starts
    as NaN, so reading it early would show."""
    import torch
    rng = synth.rng_for(51, 0)
    probs, refs, xs_new = [], [], []
    for qt, N, K in (("q4k", 200, 3072), ("q6k", 96, 8192)):
        W = synth.weights(rng, qt, N, K)
        x = synth.activations(rng, 1, K)
        xd = torch.full((1, K), float("nan"), dtype=torch.float16, device=cuda)
        xs_new.append((xd, _x_dev(x, cuda).view(torch.float16)))
        y = torch.full((1, N), float("nan"), device=cuda)
        probs.append(dict(qtype=qt, blocks=_dev(W, cuda), x_f16=xd, y=y, M=1, N=N, K=K))
        refs.append(oracle.matmul(QT[qt], W, x, N, K))
    longk = _long_kernel(cuda)
    torch.cuda.synchronize()
    longk()
    for xd, xn in xs_new:
        xd.copy_(xn)
    qk_lib.qk_matmul_batch(probs)
    qk_lib.qk_get_device_status()
    for p, ref in zip(probs, refs):
        check_close(p["y"].cpu().numpy().astype(np.float64), ref, "x after a kernel, %s" % p["qtype"])


def test_decode_reads_weights_written_just_before(qk_lib, cuda):
    """Weights written by the kernel right before the call are the ones the
    decode kernel reads (they start as zeros, which would give y = 0)."""
    import torch
    rng = synth.rng_for(52, 0)
    N, K = 256, 3072
    W = synth.weights(rng, "q4k", N, K)
    x = synth.activations(rng, 1, K)
    Wn = _dev(W, cuda)
    Wd = torch.zeros_like(Wn)
    y = torch.full((1, N), float("nan"), device=cuda)
    longk = _long_kernel(cuda)
    torch.cuda.synchronize()
    longk()
    Wd.copy_(Wn)
    qk_lib.qk_matmul_batch([dict(qtype="q4k", blocks=Wd, x_f16=_x_dev(x, cuda), y=y, M=1, N=N, K=K)])
    qk_lib.qk_get_device_status()
    check_close(y.cpu().numpy().astype(np.float64), oracle.matmul(QT["q4k"], W, x, N, K), "weights after a kernel")


def test_decode_chain_back_to_back(qk_lib, cuda):
    """The decode layer's linears launched back to back, each reading an x
    written by a copy kernel right before it: every result matches the
    oracle."""
    import torch
    rng = synth.rng_for(53, 0)
    K = synth.HIDDEN
    steps = []
    for lin in synth.layer_linears(0):
        W = synth.weights(rng, lin.qtype, lin.N, lin.K)
        x = synth.activations(rng, 1, lin.K)
        xd = torch.full((1, lin.K), float("nan"), dtype=torch.float16, device=cuda)
        y = torch.full((1, lin.N), float("nan"), device=cuda)
        steps.append((dict(qtype=lin.qtype, blocks=_dev(W, cuda), x_f16=xd, y=y, M=1, N=lin.N, K=lin.K),
                      _x_dev(x, cuda).view(torch.float16), oracle.matmul(QT[lin.qtype], W, x, lin.N, lin.K), lin.name))
    torch.cuda.synchronize()
    for p, xn, _, _ in steps:
        p["x_f16"].copy_(xn)
        qk_lib.qk_matmul_batch([p])
    qk_lib.qk_get_device_status()
    for p, _, ref, name in steps:
        check_close(p["y"].cpu().numpy().astype(np.float64), ref, "back-to-back chain " + name)


# ---------------------------------------------------------------------------
# RMSNorm in front of the linears
# ---------------------------------------------------------------------------
EPS = 1e-5


def gamma_vec(rng, K):
    """Norm weights fp16(1 + 0.1 N(0,1)): the synthetic recipe of this suite."""
    return (1.0 + 0.1 * rng.standard_normal(K)).astype(np.float16)


def scratch_for(qk, problems, cuda):
    import torch
    need = 0
    for qt, M, K, gu in problems:
        need = max(need, qk.qk_rmsnorm_scratch_bytes(qt, M, K, gu))
    return torch.empty(max(need // 2, 1), dtype=torch.float16, device=cuda) if need else None


@pytest.mark.parametrize("qtype", ["q4k", "q6k"])
@pytest.mark.parametrize("M,N,K", [(1, 200, 3072), (1, 64, 8192), (5, 130, 1024), (16, 96, 3072), (40, 160, 1024),
                                   (300, 128, 512), (12, 64, 8192)])
def test_rmsnorm_matmul(qk_lib, cuda, qtype, M, N, K):
    """y = (RMSNorm(x) * gamma) . W^T: fused into the GEMV's x staging for
    M <= 8 where it fits, through the scratch buffer and the GEMM otherwise."""
    import torch
    rng = synth.rng_for(M + 3 * N, K + 7)
    W = synth.weights(rng, qtype, N, K)
    x = synth.activations(rng, M, K)
    g = gamma_vec(rng, K)
    sc = scratch_for(qk_lib, [(qtype, M, K, False)], cuda)
    assert (sc is None) == qk_lib.qk_uses_gemv(qtype, M, K)
    y = torch.empty(M, N, dtype=torch.float32, device=cuda)
    fn = qk_lib.qk_rmsnorm_matmul_q4k if qtype == "q4k" else qk_lib.qk_rmsnorm_matmul_q6k
    fn(_dev(W, cuda), _x_dev(x, cuda), _x_dev(g, cuda), EPS, y, M, N, K, scratch=sc)
    qk_lib.qk_get_device_status()
    ref = oracle.rmsnorm_matmul(QT[qtype], W, x, g, EPS, N, K)
    check_close(y.cpu().numpy().astype(np.float64), ref, "rmsnorm %s M%d N%d K%d" % (qtype, M, N, K))


@pytest.mark.parametrize("M", [1, 8, 16, 100])
def test_rmsnorm_gateup(qk_lib, cuda, M):
    import torch
    N, K = 160, 3072
    rng = synth.rng_for(M, 91)
    Wg, Wu = synth.q4k_weights(rng, N, K), synth.q4k_weights(rng, N, K)
    x = synth.activations(rng, M, K)
    g = gamma_vec(rng, K)
    sc = scratch_for(qk_lib, [("q4k", M, K, True)], cuda)
    y = torch.empty(M, N, dtype=torch.float16, device=cuda)
    qk_lib.qk_rmsnorm_gateup_swiglu_q4k(_dev(Wg, cuda), _dev(Wu, cuda), _x_dev(x, cuda), _x_dev(g, cuda), EPS, y, M,
                                        N, K, scratch=sc)
    qk_lib.qk_get_device_status()
    ref = oracle.rmsnorm_gateup_swiglu(Wg, Wu, x, g, EPS, N, K)
    check_close_f16out(y.float().cpu().numpy().astype(np.float64), ref, "rmsnorm gate/up M%d" % M)


@pytest.mark.parametrize("M", [1, 16, 64])
def test_rmsnorm_batch_qkv(qk_lib, cuda, M):
    """q, k, v share x and one RMSNorm: grouped on the GEMV (M <= 8), or
    normalized once into the scratch for the three GEMMs (M = 16, 64)."""
    import torch
    rng = synth.rng_for(M, 92)
    K = 3072
    x = synth.activations(rng, M, K)
    g = gamma_vec(rng, K)
    xd, gd = _x_dev(x, cuda), _x_dev(g, cuda)
    probs, refs = [], []
    for qt, N in (("q4k", 256), ("q4k", 128), ("q6k", 128)):
        W = synth.weights(rng, qt, N, K)
        y = torch.full((M, N), float("nan"), device=cuda)
        probs.append(dict(qtype=qt, blocks=_dev(W, cuda), x_f16=xd, y=y, M=M, N=N, K=K))
        refs.append(oracle.rmsnorm_matmul(QT[qt], W, x, g, EPS, N, K))
    sc = scratch_for(qk_lib, [(p["qtype"], M, K, False) for p in probs], cuda)
    qk_lib.qk_rmsnorm_matmul_batch(probs, gd, EPS, scratch=sc)
    qk_lib.qk_get_device_status()
    for p, ref in zip(probs, refs):
        check_close(p["y"].cpu().numpy().astype(np.float64), ref, "rmsnorm batch %s M%d" % (p["qtype"], M))


def test_rmsnorm_decode_layer(qk_lib, cuda):
    """The decode layer's linears with their norms (config 1 at M = 1): q, k, v
    behind one RMSNorm, the fused gate/up behind another; checked in full."""
    import torch
    rng = synth.rng_for(93, 0)
    K = synth.HIDDEN
    x1, x2 = synth.activations(rng, 1, K), synth.activations(rng, 1, K)
    g1, g2 = gamma_vec(rng, K), gamma_vec(rng, K)
    lins = synth.layer_linears(0)
    probs, refs = [], []
    for lin in lins[:3]:
        W = synth.weights(rng, lin.qtype, lin.N, lin.K)
        y = torch.empty(1, lin.N, device=cuda)
        probs.append(dict(qtype=lin.qtype, blocks=_dev(W, cuda), x_f16=_x_dev(x1, cuda), y=y, M=1, N=lin.N, K=K))
        refs.append(oracle.rmsnorm_matmul(QT[lin.qtype], W, x1, g1, EPS, lin.N, K))
    qk_lib.qk_rmsnorm_matmul_batch(probs, _x_dev(g1, cuda), EPS)
    Wg, Wu = synth.q4k_weights(rng, synth.FFN, K), synth.q4k_weights(rng, synth.FFN, K)
    yg = torch.empty(1, synth.FFN, dtype=torch.float16, device=cuda)
    qk_lib.qk_rmsnorm_gateup_swiglu_q4k(_dev(Wg, cuda), _dev(Wu, cuda), _x_dev(x2, cuda), _x_dev(g2, cuda), EPS, yg,
                                        1, synth.FFN, K)
    qk_lib.qk_get_device_status()
    for p, ref in zip(probs, refs):
        check_close(p["y"].cpu().numpy().astype(np.float64), ref, "rmsnorm " + p["qtype"])
    check_close_f16out(yg.float().cpu().numpy().astype(np.float64),
                       oracle.rmsnorm_gateup_swiglu(Wg, Wu, x2, g2, EPS, synth.FFN, K), "rmsnorm gate/up M1")


def test_rmsnorm_prefill_gateup_m1024(qk_lib, cuda):
    """Config 2 behind its RMSNorm: M = 1024 through the scratch and the GEMM
    (sampled output features)."""
    import torch
    rng = synth.rng_for(94, 0)
    M, N, K = 1024, synth.FFN, synth.HIDDEN
    Wg, Wu = synth.q4k_weights(rng, N, K), synth.q4k_weights(rng, N, K)
    x = synth.activations(rng, M, K)
    g = gamma_vec(rng, K)
    sc = scratch_for(qk_lib, [("q4k", M, K, True)], cuda)
    assert sc is not None and sc.numel() * 2 == M * K * 2
    y = torch.empty(M, N, dtype=torch.float16, device=cuda)
    qk_lib.qk_rmsnorm_gateup_swiglu_q4k(_dev(Wg, cuda), _dev(Wu, cuda), _x_dev(x, cuda), _x_dev(g, cuda), EPS, y, M,
                                        N, K, scratch=sc)
    qk_lib.qk_get_device_status()
    rows = sample_rows(N, 48, 94)
    ref = oracle.rmsnorm_gateup_swiglu(Wg, Wu, x, g, EPS, N, K, rows=rows)
    check_close_f16out(y.float().cpu().numpy().astype(np.float64)[:, rows], ref, "rmsnorm gate/up M1024")


def test_rmsnorm_rejects_missing_scratch_and_bad_arguments(qk_lib, cuda):
    import torch
    L = qk_lib.lib()
    M, N, K = 64, 128, 512
    W = torch.zeros(N * 2 * 144, dtype=torch.uint8, device=cuda)
    x = torch.zeros(M * K, dtype=torch.float16, device=cuda)
    g = torch.ones(K, dtype=torch.float16, device=cuda)
    y = torch.zeros(M * N, dtype=torch.float32, device=cuda)
    sc = torch.zeros(M * K, dtype=torch.float16, device=cuda)
    s = torch.cuda.current_stream().cuda_stream
    args = lambda gm, eps, scr, yy: (W.data_ptr(), x.data_ptr(), gm, eps, scr, yy, M, N, K, s)
    assert L.qk_rmsnorm_matmul_q4k(*args(g.data_ptr(), 1e-5, None, y.data_ptr())) == -1      # GEMM needs scratch
    assert L.qk_rmsnorm_matmul_q4k(*args(None, 1e-5, sc.data_ptr(), y.data_ptr())) == -1     # no gamma
    assert L.qk_rmsnorm_matmul_q4k(*args(g.data_ptr(), -1.0, sc.data_ptr(), y.data_ptr())) == -3
    assert L.qk_rmsnorm_matmul_q4k(*args(g.data_ptr(), float("nan"), sc.data_ptr(), y.data_ptr())) == -3
    assert L.qk_rmsnorm_matmul_q4k(*args(g.data_ptr(), 1e-5, x.data_ptr(), y.data_ptr())) == -7  # scratch = x
    assert L.qk_rmsnorm_matmul_q4k(*args(g.data_ptr(), 1e-5, sc.data_ptr(), y.data_ptr())) == 0
    assert L.qk_get_device_status(s) == 0


# ---------------------------------------------------------------------------
# Edge cases of the number formats
# ---------------------------------------------------------------------------
def _q4k_const_blocks(N, K, d, sc, q, dmin=0.0, mn=0):
    """Q4_K blocks whose every sub-block has scale sc, min mn and every quant q."""
    nb = N * (K // 256)
    blk = np.zeros((nb, 144), np.uint8)
    blk[:, 0:2] = np.array([d], np.float16).view(np.uint8)
    blk[:, 2:4] = np.array([dmin], np.float16).view(np.uint8)
    s = np.zeros(12, np.uint8)
    for j in range(8):  # pack sc / mn of every sub-block (GGUF 6-bit packing)
        if j < 4:
            s[j] |= sc & 63
            s[j + 4] |= mn & 63
        else:
            s[j + 4] |= (sc & 0xF) | ((mn & 0xF) << 4)
            s[j - 4] |= (sc >> 4) << 6
            s[j] |= (mn >> 4) << 6
    blk[:, 4:16] = s
    blk[:, 16:144] = q | (q << 4)
    return blk.reshape(N, -1)


def test_gemm_fp16_weight_range_boundary(qk_lib, cuda):
    """The tensor-core path (M > 16) builds each weight in fp16: d*sc*q up to
    65504 is representable (d = 69, sc = 63, q = 15: 65205) and matches the
    oracle; past it (d = 70: 66150) the weight is +inf there, while the GEMV
    (fp32 scales) stays finite and exact.  include/qk.h states the limit."""
    N, K, M = 32, 512, 40
    x = np.ones((M, K), np.float16) * np.float16(2.0 ** -12)
    W = _q4k_const_blocks(N, K, 69.0, 63, 15)
    ref = oracle.matmul(oracle.Q4K, W, x, N, K)
    check_close(gpu_matmul(qk_lib, "q4k", W, x, N, K, cuda), ref, "q4k d*sc*q = 65205 on the GEMM")
    W = _q4k_const_blocks(N, K, 70.0, 63, 15)
    ref = oracle.matmul(oracle.Q4K, W, x, N, K)
    assert np.isfinite(ref).all()
    import torch
    y = torch.empty(M, N, dtype=torch.float32, device=cuda)
    qk_lib.qk_matmul_q4k(_dev(W, cuda), _x_dev(x, cuda), y, M, N, K)
    qk_lib.qk_get_device_status()
    assert not np.isfinite(y.cpu().numpy()).any()   # +inf weights: the documented fp16 limit
    check_close(gpu_matmul(qk_lib, "q4k", W, x[:1], N, K, cuda), ref[:1], "q4k d*sc*q = 66150 on the GEMV")


@pytest.mark.parametrize("qtype", ["q4k", "q6k"])
@pytest.mark.parametrize("M", [1, 8, 64])
def test_nonfinite_scale_fields(qk_lib, cuda, qtype, M):
    """A block whose d (or dmin) is inf or NaN makes its row non-finite on every
    path, as in the oracle; the other rows still match the oracle."""
    rng = synth.rng_for(71, M)
    N, K = 48, 512
    W = synth.weights(rng, qtype, N, K).reshape(-1, 144 if qtype == "q4k" else 210).copy()
    bad_rows = [3, 17, 40]
    per_row = K // 256
    for r, v in zip(bad_rows, (np.inf, -np.inf, np.nan)):
        off = 0 if qtype == "q4k" else 208
        W[r * per_row, off:off + 2] = np.array([v], np.float16).view(np.uint8)
    W = W.reshape(N, -1)
    x = synth.activations(rng, M, K)
    ref = oracle.matmul(QT[qtype], W, x, N, K)
    import torch
    y = torch.empty(M, N, dtype=torch.float32, device=cuda)
    (qk_lib.qk_matmul_q4k if qtype == "q4k" else qk_lib.qk_matmul_q6k)(_dev(W, cuda), _x_dev(x, cuda), y, M, N, K)
    qk_lib.qk_get_device_status()
    got = y.cpu().numpy().astype(np.float64)
    assert not np.isfinite(ref[:, bad_rows]).any()
    assert not np.isfinite(got[:, bad_rows]).any()
    good = [n for n in range(N) if n not in bad_rows]
    check_close(got[:, good], ref[:, good], "%s M%d finite rows" % (qtype, M))


def test_random_shapes(qk_lib, cuda):
    """Seeded random shapes (M 1..600, N 1..700, K = 256 * 1..40) for both
    formats and the fused gate/up, every kernel path and tile width."""
    import torch
    rng = np.random.default_rng(2026)
    for case in range(24):
        M = int(rng.choice([1, 2, 5, 9, 16, 17, 31, 64, 100, 257, 600])) if case % 3 else int(rng.integers(1, 601))
        N = int(rng.integers(1, 701))
        K = 256 * int(rng.integers(1, 41))
        kind = ("q4k", "q6k", "gateup")[case % 3]
        r = synth.rng_for(900 + case, 0)
        x = synth.activations(r, M, K)
        # the oracle on every row while it stays cheap, else on 48 sampled rows
        rows = None if M * N * K <= 3e7 else sample_rows(N, 48, 900 + case)
        if kind == "gateup":
            Wg, Wu = synth.q4k_weights(r, N, K), synth.q4k_weights(r, N, K)
            y = torch.empty(M, N, dtype=torch.float16, device=cuda)
            qk_lib.qk_gateup_swiglu_q4k(_dev(Wg, cuda), _dev(Wu, cuda), _x_dev(x, cuda), y, M, N, K)
            qk_lib.qk_get_device_status()
            got = y.float().cpu().numpy().astype(np.float64)
            check_close_f16out(got if rows is None else got[:, rows], oracle.gateup_swiglu(Wg, Wu, x, N, K, rows=rows),
                               "random gate/up M%d N%d K%d" % (M, N, K))
        else:
            W = synth.weights(r, kind, N, K)
            check_close(gpu_matmul(qk_lib, kind, W, x, N, K, cuda, rows=rows),
                        oracle.matmul(QT[kind], W, x, N, K, rows=rows), "random %s M%d N%d K%d" % (kind, M, N, K))
