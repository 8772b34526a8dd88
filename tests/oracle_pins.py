"""Pins that tie the CPU oracle to facts outside itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError on
a mismatch.  ``test_oracle_pins.py`` runs them on the oracle; the mutant test
runs them on deliberately broken copies of the oracle to show that each
plausible mistake is caught by at least one pin.

What the pins rest on:
* IEEE binary16 widening: numpy's float16 -> float32 conversion (a library
  routine) for all 65536 bit patterns.
* Block layouts: the hand-written tables in ``tests/golden`` (public GGUF Q4_K /
  Q6_K definitions; the DAMASCUS pages name the formats in "Building DAMASCUS",
  "Read the model, then reproduce its operations", but print no layout) drive
  an independent table-lookup decoder and one-hot bit-placement checks.
* Worked blocks with hand-derived scales, closed forms (all-zero / all-max
  quants), one-hot and all-ones activations, a float64 library matmul,
  linearity, row permutation and the SwiGLU closed form via scipy's expit.
* RMSNorm: hand-worked examples (tests/golden/rmsnorm_worked.txt), the closed
  form of a constant vector, unit mean square and exact invariance to scaling
  x by a power of two, a one-hot gamma, and the composition with the matmul
  and the SwiGLU against float64 library routines.
* GQA attention: one visible position returns its value row exactly; equal
  keys (or scale 0) give the mean of the visible value rows; a dominant key
  returns its value row within the softmax's closed-form remainder; shifting
  every key by one vector changes nothing; head h reads key/value head
  h // (H / H_kv); future positions are never read; and a float64 numpy
  restatement (einsum, scipy softmax, explicit causal mask) on random inputs.
"""
from __future__ import annotations

import os
import re

import numpy as np

from tests import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
Q4K, Q6K = 0, 1


def _lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.strip() for ln in f if ln.strip() and not ln.lstrip().startswith("#")]


def _rng(a):
    lo, hi = (int(v) for v in a.split("-")) if "-" in a else (int(a), int(a))
    return list(range(lo, hi + 1))


# ---------------------------------------------------------------------------
# Golden tables
# ---------------------------------------------------------------------------
def q4k_scale_bit_table():
    """{(byte, bit): (field, subblock, field_bit)} from q4k_scale_bits.txt."""
    table = {}
    for ln in _lines("q4k_scale_bits.txt"):
        byte, rest = ln.split(":")
        for bit, dest in enumerate(rest.split()):
            m = re.fullmatch(r"(sc|m)(\d)\.(\d)", dest)
            table[(int(byte), bit)] = (m.group(1), int(m.group(2)), int(m.group(3)))
    assert len(table) == 96
    return table


def q4k_quant_table():
    """[(qs_byte, nibble_shift, weight)] from q4k_quant_map.txt (256 entries)."""
    out = []
    for ln in _lines("q4k_quant_map.txt"):
        b, lo, hi = ln.split()
        for byte, wl, wh in zip(_rng(b), _rng(lo), _rng(hi)):
            out += [(byte, 0, wl), (byte, 4, wh)]
    assert sorted(w for _, _, w in out) == list(range(256))
    return out


def q6k_quant_table():
    """(ql entries [(byte, shift, weight)], qh entries [(byte, shift, weight)])."""
    ql, qh = [], []
    for ln in _lines("q6k_quant_map.txt"):
        parts = ln.split()
        if parts[0] == "ql":
            for byte, wl, wh in zip(_rng(parts[1]), _rng(parts[2]), _rng(parts[3])):
                ql += [(byte, 0, wl), (byte, 4, wh)]
        else:
            cols = [_rng(p) for p in parts[2:6]]
            for idx, byte in enumerate(_rng(parts[1])):
                for pair in range(4):
                    qh.append((byte, 2 * pair, cols[pair][idx]))
    assert sorted(w for _, _, w in ql) == list(range(256))
    assert sorted(w for _, _, w in qh) == list(range(256))
    return ql, qh


# ---------------------------------------------------------------------------
# An independent, table-driven decoder (numpy, fp32 steps one at a time)
# ---------------------------------------------------------------------------
def _f16(b2):
    return np.ascontiguousarray(b2).view(np.float16).astype(np.float32).reshape(-1)


def table_fields_q4k(blocks):
    """(d, dmin, sc[nb, 256], m[nb, 256], q[nb, 256]) per weight, via the tables."""
    blocks = np.asarray(blocks, dtype=np.uint8).reshape(-1, 144)
    nb = blocks.shape[0]
    d = _f16(blocks[:, 0:2])
    dmin = _f16(blocks[:, 2:4])
    sm = blocks[:, 4:16].astype(np.int64)
    sc = np.zeros((nb, 8), np.int64)
    mn = np.zeros((nb, 8), np.int64)
    for (byte, bit), (field, j, fbit) in q4k_scale_bit_table().items():
        v = ((sm[:, byte] >> bit) & 1) << fbit
        if field == "sc":
            sc[:, j] |= v
        else:
            mn[:, j] |= v
    # weight-major work arrays (one contiguous row per byte / weight), transposed at the end
    q = np.zeros((256, nb), np.int16)
    qs = np.ascontiguousarray(blocks[:, 16:144].T).astype(np.int16)
    for byte, shift, w in q4k_quant_table():
        q[w] = (qs[byte] >> shift) & 0xF
    j = np.arange(256) // 32
    return d, dmin, sc[:, j], mn[:, j], np.ascontiguousarray(q.T)


@np.errstate(invalid="ignore", over="ignore")
def table_decode_q4k(blocks):
    d, dmin, sc, mn, q = table_fields_q4k(blocks)
    dsc = (d[:, None] * sc.astype(np.float32)).astype(np.float32)
    dmn = (dmin[:, None] * mn.astype(np.float32)).astype(np.float32)
    t = (dsc * q.astype(np.float32)).astype(np.float32)
    return (t - dmn).astype(np.float32).reshape(-1)


def table_fields_q6k(blocks):
    """(d, sc[nb, 256], q[nb, 256]) per weight, q already minus 32, via the tables."""
    blocks = np.asarray(blocks, dtype=np.uint8).reshape(-1, 210)
    nb = blocks.shape[0]
    ql_b = np.ascontiguousarray(blocks[:, 0:128].T).astype(np.int16)
    qh_b = np.ascontiguousarray(blocks[:, 128:192].T).astype(np.int16)
    sc = blocks[:, 192:208].view(np.int8).astype(np.float32)
    d = _f16(blocks[:, 208:210])
    lo = np.zeros((256, nb), np.int16)
    hi = np.zeros((256, nb), np.int16)
    ql_t, qh_t = q6k_quant_table()
    for byte, shift, w in ql_t:
        lo[w] = (ql_b[byte] >> shift) & 0xF
    for byte, shift, w in qh_t:
        hi[w] = (qh_b[byte] >> shift) & 0x3
    q = np.ascontiguousarray(((lo | (hi << 4)) - 32).T)
    return d, sc[:, np.arange(256) // 16], q


@np.errstate(invalid="ignore", over="ignore")
def table_decode_q6k(blocks):
    d, sc, q = table_fields_q6k(blocks)
    dsc = (d[:, None] * sc).astype(np.float32)
    return (dsc * q.astype(np.float32)).astype(np.float32).reshape(-1)


def same_bits(a, b):
    """fp32 equality bit for bit, NaN == NaN of any payload."""
    a = np.asarray(a, np.float32)
    b = np.asarray(b, np.float32)
    both_nan = np.isnan(a) & np.isnan(b)
    eq = (a.view(np.uint32) == b.view(np.uint32)) | both_nan
    return bool(eq.all())


# ---------------------------------------------------------------------------
# Block builders for hand-made cases
# ---------------------------------------------------------------------------
def _half_bytes(v):
    return np.array([v], dtype=np.float16).view(np.uint8)


def q4k_block(d=1.0, dmin=1.0, scales=None, qs=None):
    blk = np.zeros(144, np.uint8)
    blk[0:2] = _half_bytes(d)
    blk[2:4] = _half_bytes(dmin)
    if scales is not None:
        blk[4:16] = scales
    if qs is not None:
        blk[16:144] = qs
    return blk


def q6k_block(d=1.0, scales=None, ql=None, qh=None):
    blk = np.zeros(210, np.uint8)
    if ql is not None:
        blk[0:128] = ql
    if qh is not None:
        blk[128:192] = qh
    if scales is not None:
        blk[192:208] = np.asarray(scales, np.int8).view(np.uint8)
    blk[208:210] = _half_bytes(d)
    return blk


# ---------------------------------------------------------------------------
# Pins
# ---------------------------------------------------------------------------
def pin_half_to_float(O):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float32)
    got = np.array([O.half_to_float(int(b)) for b in bits], dtype=np.float32)
    assert same_bits(got, ref)
    nan = np.isnan(ref)
    # NaN keeps its sign bit
    assert ((got.view(np.uint32)[nan] >> 31) == (bits[nan] >> 15)).all()


def pin_q4k_scale_bits(O):
    """Each of the 96 scale/min bits lands on the sub-block and field of the table."""
    for (byte, bit), (field, j, fbit) in q4k_scale_bit_table().items():
        s = np.zeros(12, np.uint8)
        s[byte] = 1 << bit
        if field == "sc":
            w = O.dequant(Q4K, q4k_block(d=1.0, dmin=0.0, scales=s, qs=np.full(128, 0x11, np.uint8)))
            expect = np.zeros(256, np.float32)
            expect[32 * j:32 * j + 32] = float(1 << fbit)
        else:
            w = O.dequant(Q4K, q4k_block(d=0.0, dmin=1.0, scales=s, qs=np.zeros(128, np.uint8)))
            expect = np.zeros(256, np.float32)
            expect[32 * j:32 * j + 32] = -float(1 << fbit)
        assert np.array_equal(w + 0.0, expect), (byte, bit)


def pin_q4k_quant_map(O):
    """A single non-zero nibble shows up at exactly the weight the table names."""
    ones = np.array([1, 1, 1, 1, 0, 0, 0, 0, 1, 1, 1, 1], np.uint8)  # all scales 1, all mins 0
    for byte, shift, wi in q4k_quant_table():
        qs = np.zeros(128, np.uint8)
        qs[byte] = 0xF << shift
        w = O.dequant(Q4K, q4k_block(d=1.0, dmin=1.0, scales=ones, qs=qs))
        expect = np.zeros(256, np.float32)
        expect[wi] = 15.0
        assert np.array_equal(w, expect), (byte, shift, wi)


def pin_q4k_worked_block(O):
    lines = _lines("q4k_worked_block.txt")
    scales = np.array([int(h, 16) for h in lines[0].split(":")[1].split()], np.uint8)
    scm = [tuple(int(v) for v in ln.split(":")[1].split()) for ln in lines[1:9]]
    qs = np.array([(b % 16) | ((15 - b % 16) << 4) for b in range(128)], np.uint8)
    w = O.dequant(Q4K, q4k_block(d=1.0, dmin=0.5, scales=scales, qs=qs))
    q = np.zeros(256, np.int64)
    for byte, shift, wi in q4k_quant_table():
        q[wi] = (int(qs[byte]) >> shift) & 0xF
    expect = np.array([scm[i // 32][0] * q[i] - 0.5 * scm[i // 32][1] for i in range(256)], np.float32)
    assert np.array_equal(w, expect)


def pin_q4k_closed_forms(O):
    """All-zero quants give -dmin*m_j; all-15 quants give 15*d*sc_j - dmin*m_j."""
    lines = _lines("q4k_worked_block.txt")
    scales = np.array([int(h, 16) for h in lines[0].split(":")[1].split()], np.uint8)
    scm = [tuple(int(v) for v in ln.split(":")[1].split()) for ln in lines[1:9]]
    for d, dmin in [(0.000123, 0.0000456), (3.5, -1.25), (6.0e-8, 65504.0)]:
        dh = np.float32(np.float16(d))
        mh = np.float32(np.float16(dmin))
        w0 = O.dequant(Q4K, q4k_block(d=d, dmin=dmin, scales=scales, qs=np.zeros(128, np.uint8)))
        w15 = O.dequant(Q4K, q4k_block(d=d, dmin=dmin, scales=scales, qs=np.full(128, 0xFF, np.uint8)))
        for i in range(256):
            sc, m = scm[i // 32]
            dmn = np.float32(mh * np.float32(m))
            assert w0[i] == np.float32(np.float32(dh * np.float32(sc)) * np.float32(0)) - dmn
            assert w15[i] == np.float32(np.float32(dh * np.float32(sc)) * np.float32(15)) - dmn


def pin_q6k_quant_map(O):
    ones = np.ones(16, np.int8)
    ql_t, qh_t = q6k_quant_table()
    for byte, shift, wi in ql_t:
        ql = np.zeros(128, np.uint8)
        ql[byte] = 0xF << shift
        w = O.dequant(Q6K, q6k_block(d=1.0, scales=ones, ql=ql))
        expect = np.full(256, -32.0, np.float32)
        expect[wi] = -17.0
        assert np.array_equal(w, expect), ("ql", byte, shift)
    for byte, shift, wi in qh_t:
        for val in (1, 2, 3):
            qh = np.zeros(64, np.uint8)
            qh[byte] = val << shift
            w = O.dequant(Q6K, q6k_block(d=1.0, scales=ones, qh=qh))
            expect = np.full(256, -32.0, np.float32)
            expect[wi] = -32.0 + 16 * val
            assert np.array_equal(w, expect), ("qh", byte, shift, val)


def pin_q6k_scale_map(O):
    for t in range(16):
        sc = np.zeros(16, np.int8)
        sc[t] = -3
        w = O.dequant(Q6K, q6k_block(d=1.0, scales=sc))
        expect = np.zeros(256, np.float32)
        expect[16 * t:16 * t + 16] = 96.0  # (-3) * (0 - 32)
        assert np.array_equal(w + 0.0, expect), t


def pin_q6k_worked_block(O):
    lines = _lines("q6k_worked_block.txt")
    sc = [int(v) for v in lines[0].split(":")[1].split()]
    qg = [int(v) for v in lines[1].split(":")[1].split()]
    w = O.dequant(Q6K, q6k_block(d=1.0, scales=sc, ql=np.full(128, 0x0F, np.uint8),
                                  qh=np.full(64, 0x1B, np.uint8)))
    expect = np.array([sc[i // 16] * qg[i // 32] for i in range(256)], np.float32)
    assert np.array_equal(w, expect)


def pin_q6k_closed_forms(O):
    sc = np.array([5, -7, 63, -32, 1, 0, 17, -1, 9, 33, -20, 2, 44, -9, 3, 12], np.int8)
    for d in (0.000123, -2.5, 6.0e-8):
        dh = np.float32(np.float16(d))
        lo = O.dequant(Q6K, q6k_block(d=d, scales=sc))
        hi = O.dequant(Q6K, q6k_block(d=d, scales=sc, ql=np.full(128, 0xFF, np.uint8),
                                       qh=np.full(64, 0xFF, np.uint8)))
        for i in range(256):
            dsc = np.float32(dh * np.float32(sc[i // 16]))
            assert lo[i] == np.float32(dsc * np.float32(-32))
            assert hi[i] == np.float32(dsc * np.float32(31))


def random_blocks(qtype, n, seed):
    """Synthetic blocks plus raw random bytes (any fp16 scale, incl. inf / NaN / subnormal)."""
    rng = synth.rng_for(seed, 991)
    bb = 144 if qtype == Q4K else 210
    gen = synth.q4k_weights if qtype == Q4K else synth.q6k_weights
    a = gen(rng, n // 2, 256).reshape(-1, bb)
    b = rng.integers(0, 256, size=(n - n // 2, bb), dtype=np.uint8)
    return np.concatenate([a, b])


def pin_bruteforce_vs_table_decoder(O, n=100_000, seed=7, chunk=4096):
    """The oracle against the table decoder, bit for bit, on n random blocks
    (decoded in chunks: a few small working arrays instead of several
    hundred MB of fresh memory)."""
    for qtype, dec in ((Q4K, table_decode_q4k), (Q6K, table_decode_q6k)):
        blocks = random_blocks(qtype, n, seed + qtype)
        for c in range(0, n, chunk):
            part = blocks[c:c + chunk]
            assert same_bits(O.dequant(qtype, part), dec(part)), (qtype, c)


@np.errstate(invalid="ignore", over="ignore")
def pin_dequant_correctly_rounded(O, n=8192, seed=3):
    """Every weight is the exact real value of its formula, rounded once to fp32.

    The products are exact in fp32: an fp16 scale has 11 significant bits, a
    Q4_K scale or min 6 and a quant 4 (21 bits in all); a Q6_K int8 scale has
    at most 7 significant bits and |q - 32| <= 32 at most 5 (23 bits).  So a
    Q6_K weight is exact, and a Q4_K weight has a single rounding, at the
    subtraction.  The reference value is computed in fp64 (exact for the
    products; fp64 to fp32 double rounding is innocuous for one subtraction of
    fp32 values, 53 >= 2*24 + 2) and compared bit for bit.  The order in which
    the products are formed, or a fused multiply-add at the subtraction,
    therefore cannot change a bit."""
    b4 = random_blocks(Q4K, n, seed)
    d, dmin, sc, mn, q = table_fields_q4k(b4)
    exact = (d[:, None].astype(np.float64) * sc * q - dmin[:, None].astype(np.float64) * mn)
    assert same_bits(O.dequant(Q4K, b4), exact.astype(np.float32).reshape(-1))
    b6 = random_blocks(Q6K, n, seed + 1)
    d, sc, q = table_fields_q6k(b6)
    exact = d[:, None].astype(np.float64) * sc.astype(np.float64) * q
    finite = np.isfinite(exact)
    assert (exact[finite] == exact[finite].astype(np.float32)).all()  # no rounding at all
    assert same_bits(O.dequant(Q6K, b6), exact.astype(np.float32).reshape(-1))


def _mat(qtype, N, K, seed):
    rng = synth.rng_for(seed, 5)
    W = synth.q4k_weights(rng, N, K) if qtype == Q4K else synth.q6k_weights(rng, N, K)
    dec = table_decode_q4k if qtype == Q4K else table_decode_q6k
    return W, dec(W).reshape(N, K)


def pin_matmul_onehot(O):
    """x = e_k picks column k of the dequantized weights, exactly."""
    for qtype in (Q4K, Q6K):
        N, K = 37, 512
        W, Wf = _mat(qtype, N, K, 11)
        ks = np.array([0, 1, 31, 32, 63, 64, 255, 256, 300, 511])
        x = np.zeros((ks.size, K), np.float16)
        x[np.arange(ks.size), ks] = 1.0
        y = O.matmul(qtype, W, x, N, K)
        assert np.array_equal(y, Wf[:, ks].T.astype(np.float64))
        # a scaled one-hot: x = 2^-3 e_k scales exactly
        y2 = O.matmul(qtype, W, (x * np.float16(0.125)).astype(np.float16), N, K)
        assert np.array_equal(y2, Wf[:, ks].T.astype(np.float64) * 0.125)


def pin_matmul_ones_rowsum(O):
    """x = ones gives the exact row sums of the dequantized weights (math.fsum)."""
    import math
    for qtype in (Q4K, Q6K):
        N, K = 19, 768
        W, Wf = _mat(qtype, N, K, 12)
        y = O.matmul(qtype, W, np.ones((1, K), np.float16), N, K)[0]
        exact = np.array([math.fsum(Wf[n].astype(np.float64)) for n in range(N)])
        mag = np.abs(Wf.astype(np.float64)).sum(axis=1)
        assert (np.abs(y - exact) <= 1e-13 * mag).all()


def pin_matmul_vs_numpy_f64(O):
    for qtype in (Q4K, Q6K):
        N, K, M = 64, 1024, 5
        W, Wf = _mat(qtype, N, K, 13)
        x = synth.activations(synth.rng_for(13, 6), M, K)
        y = O.matmul(qtype, W, x, N, K)
        ref = x.astype(np.float64) @ Wf.astype(np.float64).T
        scale = np.abs(x.astype(np.float64)) @ np.abs(Wf.astype(np.float64)).T
        assert (np.abs(y - ref) <= 1e-13 * scale + 1e-300).all()


def pin_matmul_rows_and_permutation(O):
    """Row subsets and row permutations of W permute the outputs exactly."""
    for qtype in (Q4K, Q6K):
        N, K, M = 40, 512, 3
        W, _ = _mat(qtype, N, K, 14)
        x = synth.activations(synth.rng_for(14, 6), M, K)
        y = O.matmul(qtype, W, x, N, K)
        perm = synth.rng_for(14, 7).permutation(N)
        yp = O.matmul(qtype, W.reshape(N, -1)[perm], x, N, K)
        assert np.array_equal(yp, y[:, perm])
        sub = np.array([39, 0, 17, 17, 5])
        assert np.array_equal(O.matmul(qtype, W, x, N, K, rows=sub), y[:, sub])


def pin_matmul_linearity(O):
    """y(x1 + x2) = y(x1) + y(x2) for fp16 inputs whose sum is exact in fp16."""
    for qtype in (Q4K, Q6K):
        N, K = 16, 512
        W, _ = _mat(qtype, N, K, 15)
        rng = synth.rng_for(15, 8)
        x1 = rng.integers(-64, 64, size=(2, K)).astype(np.float16)
        x2 = rng.integers(-64, 64, size=(2, K)).astype(np.float16)
        y1 = O.matmul(qtype, W, x1, N, K)
        y2 = O.matmul(qtype, W, x2, N, K)
        y12 = O.matmul(qtype, W, (x1 + x2).astype(np.float16), N, K)
        assert np.allclose(y12, y1 + y2, rtol=1e-12, atol=1e-12)
        # K-ordering: reversing the K blocks of W and of x together leaves y unchanged
        nb = K // 256
        Wr = W.reshape(N, nb, -1)[:, ::-1].reshape(N, -1)
        xr = x1.reshape(2, nb, 256)[:, ::-1].reshape(2, K)
        assert np.allclose(O.matmul(qtype, Wr, xr, N, K), y1, rtol=1e-12, atol=1e-12)


def pin_gateup_swiglu(O):
    from scipy.special import expit
    N, K, M = 24, 768, 4
    rng = synth.rng_for(16, 9)
    Wg = synth.q4k_weights(rng, N, K)
    Wu = synth.q4k_weights(rng, N, K)
    x = synth.activations(rng, M, K)
    out, g, u = O.gateup_swiglu(Wg, Wu, x, N, K, return_gu=True)
    assert np.array_equal(g, O.matmul(Q4K, Wg, x, N, K))
    assert np.array_equal(u, O.matmul(Q4K, Wu, x, N, K))
    assert np.allclose(out, g * expit(g) * u, rtol=1e-14, atol=1e-300)
    # silu(0) = 0: an all-zero activation row gives exactly zero
    z = O.gateup_swiglu(Wg, Wu, np.zeros((1, K), np.float16), N, K)
    assert np.array_equal(z, np.zeros_like(z))
    # gate and up swapped is not the same function (guards a swapped operand)
    sw = O.gateup_swiglu(Wu, Wg, x, N, K)
    assert not np.allclose(sw, out)


# ---------------------------------------------------------------------------
# RMSNorm in front of a linear
# ---------------------------------------------------------------------------
def pin_rmsnorm_worked(O):
    for ln in _lines("rmsnorm_worked.txt"):
        eps, xs, gs, want = (p.split() for p in ln.split("|"))
        x = np.array([float(v) for v in xs], np.float16)
        g = np.array([float(v) for v in gs], np.float16)
        got = O.rmsnorm(x.reshape(1, -1), g, float(eps[0]))[0]
        exp = np.array([float(v) for v in want])
        assert np.allclose(got, exp, rtol=1e-15, atol=0), (ln, got)


def pin_rmsnorm_constant_vector(O):
    """x = c everywhere, gamma = 1: xhat = sign(c) / sqrt(1 + eps / c^2)."""
    K = 3072
    for c in (0.5, -2.0, 0.0009765625, 100.0):
        for eps in (0.0, 1e-5, 1e-2):
            x = np.full((1, K), c, np.float16)
            got = O.rmsnorm(x, np.ones(K, np.float16), eps)[0]
            want = np.sign(c) / np.sqrt(1.0 + eps / (c * c))
            assert np.allclose(got, want, rtol=1e-14, atol=0), (c, eps, got[0], want)


def pin_rmsnorm_unit_mean_square_and_scale_invariance(O):
    rng = synth.rng_for(61, 0)
    K = 3072
    x = synth.activations(rng, 3, K)
    one = np.ones(K, np.float16)
    a = O.rmsnorm(x, one, 0.0)
    assert np.allclose((a ** 2).mean(axis=1), 1.0, rtol=1e-12)
    # scaling x by 4 scales the sum of squares by 16 and the root by 4, all
    # exactly: the output is bit-identical
    b = O.rmsnorm((x.astype(np.float32) * 4).astype(np.float16), one, 0.0)
    assert np.array_equal(a, b)


def pin_rmsnorm_gamma_onehot(O):
    rng = synth.rng_for(62, 0)
    K = 512
    x = synth.activations(rng, 2, K)
    rms = np.sqrt((x.astype(np.float64) ** 2).mean(axis=1) + 1e-5)
    for k in (0, 7, K - 1):
        g = np.zeros(K, np.float16)
        g[k] = 1
        out = O.rmsnorm(x, g, 1e-5)
        assert np.count_nonzero(out[:, np.arange(K) != k]) == 0
        assert np.allclose(out[:, k], x[:, k].astype(np.float64) / rms, rtol=1e-14)


def pin_rmsnorm_matmul_composition(O):
    """The normalized linear equals a float64 library matmul of the oracle's
    dequantized weights with its normalized activations (and the SwiGLU of two
    such, through scipy's expit), with eps large enough to matter."""
    from scipy.special import expit
    rng = synth.rng_for(63, 0)
    K, N, eps = 512, 40, 1e-2
    x = (synth.activations(rng, 3, K).astype(np.float32) * 0.05).astype(np.float16)
    g = (1.0 + 0.1 * rng.standard_normal(K)).astype(np.float16)
    xn = O.rmsnorm(x, g, eps)
    for qt in (Q4K, Q6K):
        W = synth.weights(rng, "q4k" if qt == Q4K else "q6k", N, K)
        w = O.dequant(qt, W).astype(np.float64).reshape(N, K)
        got = O.rmsnorm_matmul(qt, W, x, g, eps, N, K)
        ref = xn @ w.T
        assert np.all(np.abs(got - ref) <= 1e-13 * (np.abs(xn) @ np.abs(w).T))
    Wg, Wu = synth.q4k_weights(rng, N, K), synth.q4k_weights(rng, N, K)
    G = xn @ O.dequant(Q4K, Wg).astype(np.float64).reshape(N, K).T
    U = xn @ O.dequant(Q4K, Wu).astype(np.float64).reshape(N, K).T
    got = O.rmsnorm_gateup_swiglu(Wg, Wu, x, g, eps, N, K)
    assert np.allclose(got, G * expit(G) * U, rtol=1e-10, atol=1e-12 * np.abs(G * U).max())


# ---------------------------------------------------------------------------
# Q8 activations (int8 per block of 32 with one fp32 scale; the reading this
# project takes, the pages have no such variant)
# ---------------------------------------------------------------------------
def pin_q8_worked_block(O):
    """A hand-worked block: amax 127/128 gives d = 1/128 exactly, so x / d is
    exact and ties round away from zero; an all-zero block has d = 0, q = 0."""
    x = np.zeros((1, 64), np.float16)
    vals = {0: 127 / 128, 1: 5 / 256, 2: -5 / 256, 3: 1 / 256, 4: -1 / 256, 5: 3 / 256, 6: 64 / 128,
            7: -127 / 128, 8: 1 / 1024}
    for i, v in vals.items():
        x[0, i] = v
    q, d = O.quantize_q8(x)
    assert d[0, 0] == np.float32(1 / 128) and d[0, 1] == 0.0
    want = {0: 127, 1: 3, 2: -3, 3: 1, 4: -1, 5: 2, 6: 64, 7: -127, 8: 0}
    for i in range(32):
        assert q[0, i] == want.get(i, 0), (i, q[0, i])
    assert not q[0, 32:].any()


def _grid_x(rng, M, K, e):
    """x = 2^-e * q with q integer in [-127, 127] and |q| = 127 somewhere in
    every block of 32: exactly representable in fp16 and on its own int8 grid."""
    q = rng.integers(-127, 128, size=(M, K))
    for m in range(M):
        for b in range(K // 32):
            q[m, 32 * b + rng.integers(0, 32)] = 127 if rng.integers(0, 2) else -127
    return (q * 2.0 ** -e).astype(np.float16), q


def pin_q8_grid_reproduces_fp16(O):
    """x already on its int8 grid: the Q8 matmul is the fp16 matmul, bit for bit."""
    rng = synth.rng_for(71, 0)
    K, N = 512, 24
    x, qx = _grid_x(rng, 3, K, 9)
    q, d = O.quantize_q8(x)
    assert np.array_equal(q, qx) and np.all(d == np.float32(2.0 ** -9))
    for qt in (Q4K, Q6K):
        W = synth.weights(rng, "q4k" if qt == Q4K else "q6k", N, K)
        assert np.array_equal(O.q8_matmul(qt, W, x, N, K), O.matmul(qt, W, x, N, K))


def pin_q8_error_bound_and_composition(O):
    """Random activations: every element within half a step of its int8 value
    (|x - d q| <= d / 2), the matmul equal to a float64 library product of the
    dequantized weights with d * q, and within sum_b (d_b / 2) sum_k |w_k| of
    the fp16 matmul."""
    rng = synth.rng_for(72, 0)
    K, N = 768, 40
    x = synth.activations(rng, 4, K)
    q, d = O.quantize_q8(x)
    dk = np.repeat(d.astype(np.float64), 32, axis=1)
    xq = dk * q
    xf = x.astype(np.float64)
    assert np.all(np.abs(xf - xq) <= dk / 2 * (1 + 1e-6))
    assert np.all(np.abs(q) <= 127)
    for qt in (Q4K, Q6K):
        W = synth.weights(rng, "q4k" if qt == Q4K else "q6k", N, K)
        w = O.dequant(qt, W).astype(np.float64).reshape(N, K)
        got = O.q8_matmul(qt, W, x, N, K)
        ref = xq @ w.T
        assert np.all(np.abs(got - ref) <= 1e-13 * (np.abs(xq) @ np.abs(w).T))
        bound = (dk / 2) @ np.abs(w).T
        assert np.all(np.abs(got - O.matmul(qt, W, x, N, K)) <= bound * (1 + 1e-9) + 1e-300)


def pin_q8_gateup_composition(O):
    """The int8-activation gate/up + SwiGLU equals silu(G) * U of the two
    int8-activation matmuls (through scipy's expit)."""
    from scipy.special import expit
    rng = synth.rng_for(74, 0)
    K, N = 512, 24
    x = synth.activations(rng, 2, K)
    Wg, Wu = synth.q4k_weights(rng, N, K), synth.q4k_weights(rng, N, K)
    G, U = O.q8_matmul(Q4K, Wg, x, N, K), O.q8_matmul(Q4K, Wu, x, N, K)
    assert np.allclose(O.q8_gateup_swiglu(Wg, Wu, x, N, K), G * expit(G) * U, rtol=1e-12,
                       atol=1e-14 * np.abs(G * U).max())


def pin_q8_power_of_two_scaling(O):
    """Doubling x keeps every q and doubles every d exactly, so y doubles exactly."""
    rng = synth.rng_for(73, 0)
    K, N = 256, 16
    x = (synth.activations(rng, 2, K).astype(np.float32) * 0.25).astype(np.float16)
    x2 = (x.astype(np.float32) * 2).astype(np.float16)
    q1, d1 = O.quantize_q8(x)
    q2, d2 = O.quantize_q8(x2)
    assert np.array_equal(q1, q2) and np.array_equal(d2, d1 * 2)
    W = synth.weights(rng, "q6k", N, K)
    assert np.array_equal(O.q8_matmul(Q6K, W, x2, N, K), 2 * O.q8_matmul(Q6K, W, x, N, K))


# ---------------------------------------------------------------------------
# GQA attention over a KV cache
# ---------------------------------------------------------------------------
def _attn_inputs(rng, M, H, Hkv, D, Lmax, lo=-3, hi=4):
    """Small-integer fp16 inputs (exact in fp16 and in every fp64 dot product)."""
    q = rng.integers(lo, hi, size=(M, H, D)).astype(np.float16)
    k = rng.integers(lo, hi, size=(Hkv, Lmax, D)).astype(np.float16)
    v = rng.integers(-8, 9, size=(Hkv, Lmax, D)).astype(np.float16)
    return q, k, v


def pin_attn_single_position(O):
    """Query at position 0 (one visible key): the output is v_0, exactly."""
    rng = synth.rng_for(71, 0)
    q, k, v = _attn_inputs(rng, 1, 4, 2, 8, 3)
    out = O.gqa_attention(q, k, v, 4, 2, 0, 0.37)
    for h in range(4):
        assert np.array_equal(out[0, h], v[h // 2, 0].astype(np.float64))


def pin_attn_uniform_weights(O):
    """Equal keys, or scale 0: every visible position weighs 1/n, so each row
    is the mean of the value rows 0 .. pos (math.fsum / n)."""
    import math
    rng = synth.rng_for(72, 0)
    H, Hkv, D, M, pos0 = 6, 3, 8, 5, 2
    q, k, v = _attn_inputs(rng, M, H, Hkv, D, pos0 + M)
    keq = np.broadcast_to(k[:, :1, :], k.shape).copy()
    for kk, scale in ((keq, 0.5), (k, 0.0)):
        out = O.gqa_attention(q, kk, v, H, Hkv, pos0, scale)
        for i in range(M):
            n = pos0 + i + 1
            for h in range(H):
                g = h // (H // Hkv)
                want = [math.fsum(float(v[g, j, d]) for j in range(n)) / n for d in range(D)]
                assert np.allclose(out[i, h], want, rtol=0, atol=1e-12), (i, h)


def pin_attn_dominant_key(O):
    """One key aligned with q far above the others: the output is that key's
    value row, up to the softmax remainder (n - 1) * exp(-margin) * max|v|."""
    H, Hkv, D, L = 2, 1, 4, 6
    q = np.zeros((1, H, D), np.float16)
    q[0, :, 0] = 8
    k = np.zeros((Hkv, L, D), np.float16)
    k[0, 3, 0] = 8                      # s_3 = 64 * scale, every other s_j = 0
    v = np.arange(Hkv * L * D, dtype=np.float16).reshape(Hkv, L, D)
    scale = 0.75                        # margin 48
    out = O.gqa_attention(q, k, v, H, Hkv, L - 1, scale)
    bound = (L - 1) * np.exp(-64 * scale) * float(np.abs(v).max()) * 2
    for h in range(H):
        assert np.max(np.abs(out[0, h] - v[0, 3])) <= bound


def pin_attn_key_shift_invariance(O):
    """Adding one vector u to every key adds scale * q.u to every score of a
    query, which the softmax removes: the outputs do not change."""
    rng = synth.rng_for(73, 0)
    H, Hkv, D, M, pos0 = 4, 2, 8, 4, 3
    q, k, v = _attn_inputs(rng, M, H, Hkv, D, pos0 + M)
    u = rng.integers(-2, 3, size=(Hkv, 1, D)).astype(np.float16)
    a = O.gqa_attention(q, k, v, H, Hkv, pos0, 0.3)
    b = O.gqa_attention(q, (k + u).astype(np.float16), v, H, Hkv, pos0, 0.3)
    assert np.max(np.abs(a - b)) <= 1e-12 * float(np.abs(v).max())


def pin_attn_gqa_head_mapping(O):
    """Head h of an (H, H_kv) call equals a one-head call on key/value head
    h // (H / H_kv) alone."""
    rng = synth.rng_for(74, 0)
    H, Hkv, D, M, pos0 = 6, 2, 8, 3, 1
    q, k, v = _attn_inputs(rng, M, H, Hkv, D, pos0 + M)
    out = O.gqa_attention(q, k, v, H, Hkv, pos0, 0.2)
    for h in range(H):
        g = h // (H // Hkv)
        one = O.gqa_attention(np.ascontiguousarray(q[:, h:h + 1]), k[g:g + 1], v[g:g + 1], 1, 1, pos0, 0.2)
        assert np.array_equal(out[:, h], one[:, 0]), h


def pin_attn_causal(O):
    """Query i never reads positions after pos0 + i: changing them (and the
    cache beyond the last query) leaves its row unchanged."""
    rng = synth.rng_for(75, 0)
    H, Hkv, D, M, pos0, Lmax = 4, 2, 8, 4, 2, 9
    q, k, v = _attn_inputs(rng, M, H, Hkv, D, Lmax)
    a = O.gqa_attention(q, k, v, H, Hkv, pos0, 0.4)
    for i in range(M):
        k2, v2 = k.copy(), v.copy()
        k2[:, pos0 + i + 1:] = 3
        v2[:, pos0 + i + 1:] = -7
        b = O.gqa_attention(q, k2, v2, H, Hkv, pos0, 0.4, qrows=[i])
        assert np.array_equal(a[i], b[0]), i


def pin_attn_vs_numpy(O):
    """Random fp16 inputs against a float64 numpy restatement."""
    from scipy.special import softmax
    rng = synth.rng_for(76, 0)
    H, Hkv, D, M, pos0, Lmax = 6, 2, 16, 5, 7, 14
    q = rng.standard_normal((M, H, D)).astype(np.float16)
    k = rng.standard_normal((Hkv, Lmax, D)).astype(np.float16)
    v = rng.standard_normal((Hkv, Lmax, D)).astype(np.float16)
    scale = 1 / np.sqrt(D)
    out = O.gqa_attention(q, k, v, H, Hkv, pos0, scale)
    kk = np.repeat(k.astype(np.float64), H // Hkv, axis=0)  # [H][Lmax][D]
    vv = np.repeat(v.astype(np.float64), H // Hkv, axis=0)
    s = scale * np.einsum("mhd,hjd->mhj", q.astype(np.float64), kk)
    visible = np.arange(Lmax)[None, :] <= (pos0 + np.arange(M))[:, None]
    s = np.where(visible[:, None, :], s, -np.inf)
    want = np.einsum("mhj,hjd->mhd", softmax(s, axis=-1), vv)
    assert np.allclose(out, want, rtol=0, atol=1e-12)


ALL_PINS = [
    pin_attn_single_position, pin_attn_uniform_weights, pin_attn_dominant_key, pin_attn_key_shift_invariance,
    pin_attn_gqa_head_mapping, pin_attn_causal, pin_attn_vs_numpy,
    pin_q8_worked_block, pin_q8_grid_reproduces_fp16, pin_q8_error_bound_and_composition,
    pin_q8_power_of_two_scaling, pin_q8_gateup_composition,
    pin_rmsnorm_worked, pin_rmsnorm_constant_vector, pin_rmsnorm_unit_mean_square_and_scale_invariance,
    pin_rmsnorm_gamma_onehot, pin_rmsnorm_matmul_composition,
    pin_half_to_float,
    pin_q4k_scale_bits,
    pin_q4k_quant_map,
    pin_q4k_worked_block,
    pin_q4k_closed_forms,
    pin_q6k_quant_map,
    pin_q6k_scale_map,
    pin_q6k_worked_block,
    pin_q6k_closed_forms,
    pin_bruteforce_vs_table_decoder,
    pin_dequant_correctly_rounded,
    pin_matmul_onehot,
    pin_matmul_ones_rowsum,
    pin_matmul_vs_numpy_f64,
    pin_matmul_rows_and_permutation,
    pin_matmul_linearity,
    pin_gateup_swiglu,
]
