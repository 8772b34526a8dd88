"""Host-only checks of the tensor-core GEMM's launch plans (no GPU needed:
qk_gemm_plan is a host query), over every linear of the model at the sweep's
token counts and a range of other sizes.

- Tensor memory: tcgen05.alloc waits, without a time limit, until enough
  columns are free, so the CTAs that shared memory lets share an SM must fit
  in its 512 columns together (a CTA stuck in alloc would hold up its whole
  split-K cluster at the cluster barrier).
- Shared memory: the request stays within the 227 KB a CTA may have.
- Rings: a single-tensor x ring deeper than 4 is even (the two issuers take
  alternate K steps and each keeps to its own slots), and a Q6_K plan has 4 A
  stages with an even done ring max(x, A) (its halves wait on the done
  barrier of their own steps; an odd ring can stall, see test_ring_model.py).
"""
import pytest

import quantized_q4_matmul_gb300 as qk
from tests import synth

SWEEP_M = (9, 16, 17, 100, 128, 200, 256, 257, 512, 1000, 1024, 2048, 4096)
SMEM_LIMIT = 227 * 1024


def shapes():
    seen = {(lin.qtype, lin.N, lin.K, False) for _, lin in synth.model_linears()}
    seen.add((synth.Q4K, synth.FFN, synth.HIDDEN, True))  # fused gate/up
    for K in (256, 768, 4096, 12288):
        for N in (128, 1000, 5000):
            seen.add((synth.Q4K, N, K, False))
            seen.add((synth.Q6K, N, K, False))
    return sorted(seen)


def qname(qtype):
    return "q4k" if qtype == synth.Q4K else "q6k"


@pytest.mark.parametrize("qtype,N,K,gateup", shapes())
def test_plans_fit_tensor_and_shared_memory(qtype, N, K, gateup):
    for M in SWEEP_M:
        p = qk.qk_gemm_plan(qname(qtype), M, N, K, gateup)
        assert p["token_tile"] % 16 == 0 and 16 <= p["token_tile"] <= 256
        assert p["tmem_cols"] in (32, 64, 128, 256, 512)
        assert p["max_ctas_per_sm"] >= 1
        assert p["max_ctas_per_sm"] * p["tmem_cols"] <= 512, (M, p)
        assert p["smem_bytes"] <= SMEM_LIMIT, (M, p)
        if not gateup and p["x_stages"] > 4:
            assert p["x_stages"] % 2 == 0, (M, p)
        if qtype == synth.Q6K:
            assert p["a_stages"] == 4, (M, p)
            assert max(p["x_stages"], p["a_stages"]) % 2 == 0, (M, p)
        if gateup:
            assert not p["a_in_tmem"] and p["x_stages"] <= 4
            # a third A stage before a fourth x stage (measured faster wherever both fit)
            if p["token_tile"] <= 240:
                assert p["x_stages"] >= 3 and p["a_stages"] >= 3, (M, p)
