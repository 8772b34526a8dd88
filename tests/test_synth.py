"""The seeded input recipe: shapes, byte totals and value distributions (no GPU)."""
import numpy as np

import oracle
from tests import synth


def test_model_mix_matches_the_pages_file_size():
    # DAMASCUS project overview, terminal demo: "Q4_K_M · 1.9 GiB".  The Q4_K_M
    # reading (Q6_K for attn_v, 14 of 28 down projections and the tied LM head,
    # Q4_K elsewhere) must reproduce that size from the block byte counts.
    total = sum(synth.weight_bytes(lin.qtype, lin.N, lin.K) for _, lin in synth.model_linears())
    assert total == 2_022_193_152
    assert round(total / 2**30, 1) == 1.9
    assert len(synth.DOWN_Q6K_LAYERS) == synth.N_LAYERS // 2


def test_layer_shapes():
    lins = {l.name: l for l in synth.layer_linears(0)}
    assert (lins["attn_q"].N, lins["attn_q"].K) == (3072, 3072)
    assert (lins["attn_k"].N, lins["attn_v"].N) == (1024, 1024)
    assert (lins["ffn_gate"].N, lins["ffn_up"].N, lins["ffn_down"].K) == (8192, 8192, 8192)
    assert lins["attn_v"].qtype == synth.Q6K and lins["ffn_down"].qtype == synth.Q6K
    assert synth.layer_linears(3)[-1].qtype == synth.Q4K
    assert synth.weight_bytes(synth.Q4K, 3072, 3072) == 3072 * 12 * 144


def test_seeded_reproducible():
    a = synth.q4k_weights(synth.rng_for(0, 1), 8, 512)
    b = synth.q4k_weights(synth.rng_for(0, 1), 8, 512)
    c = synth.q4k_weights(synth.rng_for(1, 1), 8, 512)
    assert np.array_equal(a, b) and not np.array_equal(a, c)


def test_q4k_distributions():
    from tests.oracle_pins import q4k_scale_bit_table
    W = synth.q4k_weights(synth.rng_for(0, 2), 2048, 2048).reshape(-1, 144)
    d = W[:, 0:2].copy().view(np.float16).astype(np.float64).ravel()
    assert (d >= 0).all() and abs(np.median(d) - 0.6745e-4) < 0.05e-4
    nib = np.concatenate([W[:, 16:] & 15, W[:, 16:] >> 4]).ravel()
    assert np.bincount(nib, minlength=16).min() > 0.9 * nib.size / 16
    # every packed 6-bit scale / min field is uniform on 0..63
    sm = W[:, 4:16].astype(np.int64)
    fields = {}
    for (byte, bit), (f, j, fb) in q4k_scale_bit_table().items():
        fields.setdefault((f, j), np.zeros(len(W), np.int64))
        fields[(f, j)] |= ((sm[:, byte] >> bit) & 1) << fb
    for v in fields.values():
        h = np.bincount(v, minlength=64)
        assert h.size == 64 and h.min() > 0.7 * len(W) / 64


def test_q6k_distributions():
    W = synth.q6k_weights(synth.rng_for(0, 3), 256, 2048).reshape(-1, 210)
    sc = W[:, 192:208].view(np.int8)
    assert sc.min() == -32 and sc.max() == 63
    w = oracle.dequant(oracle.Q6K, W[:64])
    assert np.isfinite(w).all()
