"""Seeded synthetic inputs in the GGUF Q4_K / Q6_K block layout.

This module only draws random numbers and lays bytes out in the block formats;
it holds none of the dequantize / matmul arithmetic.  Both the CUDA path and
the oracle read the bytes it produces, so the two sides always see identical
inputs.

Distributions (DAMASCUS project overview, "[06] the target", fixes the model
shapes; the value distributions are the workload recipe this project uses for
synthetic Llama-3.2-3B-shaped weights, since no model file is available):

* Q4_K block (144 B): fp16 d, fp16 dmin, 12 packed bytes of 6-bit scales and
  mins, 128 bytes of nibbles.  Nibbles are uniform 0..15 (uniform bytes).  The
  12 scale/min bytes are drawn as uniform bytes: every 6-bit field the format
  packs into them (8 scales, 8 mins) then comes out uniform on 0..63 and
  independent of the others, which is the stated distribution without this
  module having to implement the packing.  d and dmin are fp16(|N(0,1)| * 1e-4)
  (round to nearest even, so about half of them are fp16 subnormals).
* Q6_K block (210 B): 128 bytes ql and 64 bytes qh uniform, 16 int8 scales
  uniform on -32..63, fp16 d = fp16(|N(0,1)| * 1e-4).
* Activations: fp16(N(0,1)), or fp16(silu(z1) * z2) for the down-projection
  input of the prefill workload.

Every array is drawn from ``numpy.random.default_rng([seed, *tags])`` so each
tensor of a workload has its own reproducible stream.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

QK = 256
Q4K, Q6K = "q4k", "q6k"
BLOCK_BYTES = {Q4K: 144, Q6K: 210}

# Llama-3.2-3B (DAMASCUS project overview, "[06] the target").
N_LAYERS = 28
HIDDEN = 3072
FFN = 8192
N_HEADS = 24
N_KV_HEADS = 8
HEAD_DIM = 128
VOCAB = 128256
KV_DIM = N_KV_HEADS * HEAD_DIM  # 1024

# Q4_K_M mix: layers whose down projection is stored as Q6_K.
DOWN_Q6K_LAYERS = (0, 1, 2, 5, 8, 11, 14, 17, 20, 23, 24, 25, 26, 27)


def rng_for(seed: int, *tags: int) -> np.random.Generator:
    return np.random.default_rng([int(seed), *[int(t) for t in tags]])


def fp16_scale(rng: np.random.Generator, n: int) -> np.ndarray:
    """fp16(|N(0,1)| * 1e-4), as raw little-endian bytes [n][2]."""
    v = (np.abs(rng.standard_normal(n)) * 1e-4).astype(np.float16)
    return v.view(np.uint8).reshape(n, 2)


def q4k_weights(rng: np.random.Generator, N: int, K: int) -> np.ndarray:
    """N rows of K/256 Q4_K blocks: uint8 [N][K/256*144]."""
    assert K % QK == 0
    nb = N * (K // QK)
    qs = rng.integers(0, 256, size=(nb, 128), dtype=np.uint8)
    sm = rng.integers(0, 256, size=(nb, 12), dtype=np.uint8)
    d = fp16_scale(rng, nb)
    dmin = fp16_scale(rng, nb)
    blk = np.empty((nb, 144), dtype=np.uint8)
    blk[:, 0:2] = d
    blk[:, 2:4] = dmin
    blk[:, 4:16] = sm
    blk[:, 16:144] = qs
    return blk.reshape(N, (K // QK) * 144)


def q6k_weights(rng: np.random.Generator, N: int, K: int) -> np.ndarray:
    """N rows of K/256 Q6_K blocks: uint8 [N][K/256*210]."""
    assert K % QK == 0
    nb = N * (K // QK)
    ql = rng.integers(0, 256, size=(nb, 128), dtype=np.uint8)
    qh = rng.integers(0, 256, size=(nb, 64), dtype=np.uint8)
    sc = rng.integers(-32, 64, size=(nb, 16), dtype=np.int8)
    d = fp16_scale(rng, nb)
    blk = np.empty((nb, 210), dtype=np.uint8)
    blk[:, 0:128] = ql
    blk[:, 128:192] = qh
    blk[:, 192:208] = sc.view(np.uint8)
    blk[:, 208:210] = d
    return blk.reshape(N, (K // QK) * 210)


def weights(rng: np.random.Generator, qtype: str, N: int, K: int) -> np.ndarray:
    return q4k_weights(rng, N, K) if qtype == Q4K else q6k_weights(rng, N, K)


def activations(rng: np.random.Generator, M: int, K: int) -> np.ndarray:
    return rng.standard_normal((M, K)).astype(np.float16)


def swiglu_activations(rng: np.random.Generator, M: int, K: int) -> np.ndarray:
    """fp16(silu(z1) * z2), z1, z2 ~ N(0,1): the input distribution of a down projection."""
    z1 = rng.standard_normal((M, K))
    z2 = rng.standard_normal((M, K))
    return (z1 / (1.0 + np.exp(-z1)) * z2).astype(np.float16)


def weight_bytes(qtype: str, N: int, K: int) -> int:
    return N * (K // QK) * BLOCK_BYTES[qtype]


@dataclass(frozen=True)
class Linear:
    name: str
    qtype: str
    N: int  # output features
    K: int  # input features


def layer_linears(layer: int) -> list:
    """The seven quantized linears of one decoder layer under the Q4_K_M mix."""
    down_t = Q6K if layer in DOWN_Q6K_LAYERS else Q4K
    return [
        Linear("attn_q", Q4K, HIDDEN, HIDDEN),
        Linear("attn_k", Q4K, KV_DIM, HIDDEN),
        Linear("attn_v", Q6K, KV_DIM, HIDDEN),
        Linear("attn_output", Q4K, HIDDEN, HIDDEN),
        Linear("ffn_gate", Q4K, FFN, HIDDEN),
        Linear("ffn_up", Q4K, FFN, HIDDEN),
        Linear("ffn_down", down_t, HIDDEN, FFN),
    ]


LM_HEAD = Linear("output", Q6K, VOCAB, HIDDEN)


def model_linears() -> list:
    """(layer, Linear) for all 28 layers plus the tied LM head (layer -1)."""
    out = []
    for layer in range(N_LAYERS):
        out += [(layer, lin) for lin in layer_linears(layer)]
    out.append((-1, LM_HEAD))
    return out


# ----------------------------------------------------------------------------
# The five workloads.
# ----------------------------------------------------------------------------
@dataclass
class Workload:
    name: str
    description: str
    linears: list = field(default_factory=list)  # [(tag, Linear, M)]


def workloads() -> dict:
    decode_layer = [(i, lin, 1) for i, lin in enumerate(layer_linears(0))]  # layer 0: down is Q6_K
    w = {
        "attn_q_m16": Workload(
            "attn_q_m16", "single Q4_K matmul, M=16, K=3072, N=3072",
            [(0, Linear("attn_q", Q4K, HIDDEN, HIDDEN), 16)]),
        "decode_layer_m1": Workload(
            "decode_layer_m1", "decode GEMV M=1 over one layer's seven linears", decode_layer),
        "prefill_gateup_swiglu_m1024": Workload(
            "prefill_gateup_swiglu_m1024", "fused gate/up + SwiGLU, M=1024, K=3072, N_ff=8192, Q4_K",
            [(0, Linear("ffn_gate", Q4K, FFN, HIDDEN), 1024), (1, Linear("ffn_up", Q4K, FFN, HIDDEN), 1024)]),
        "prefill_down_v_m1024": Workload(
            "prefill_down_v_m1024", "Q6_K down 8192->3072 and attn_v 3072->1024 at M=1024",
            [(0, Linear("ffn_down", Q6K, HIDDEN, FFN), 1024), (1, Linear("attn_v", Q6K, KV_DIM, HIDDEN), 1024)]),
    }
    return w


SWEEP_M = (1, 16, 128, 512, 1024, 2048)
