"""A CPU model of the decode GEMV's arithmetic, checked against the oracle.

The GEMV multiplies raw quants on the warp tensor instruction mma.m16n8k16.
- A quant OR-ed into the mantissa of fp16 1024.0 is the exact value 1024 + F·q,
  with F = 1 or 16 by nibble position.
- x is replicated over the 8 MMA columns.
- So every lane holds D = 1024·Sx + F·Σq·x for its rows g and g+8, per sub-block.
- Lane tig turns the D of one sub-block into Σ w·x with the block's scale and
  min: (d·sc/F)·D − Sx·(1024·d·sc/F + dmin·m). For Q6_K the second term is
  32·d·sc.
- Two lane shuffles sum the four sub-blocks of a half.

This model runs those steps for one 16-row × 256-weight unit:
- the MMA fragment layout of the PTX ISA (A row-major, B column-major, f32
  accumulators);
- the operand bit tricks and the k-permuted x pairs;
- the 16-wide x sums;
- the lane's sub-block choice.

It compares the result with the oracle's dequantized weights times x. The
model restates the method, so it checks the arithmetic the kernel relies on
(exact integer operands, the scale identity, the byte, k and lane mapping),
not the compiled kernel, which the GPU parity tests cover.
"""
import numpy as np
import pytest

import oracle
from tests import synth

MAGIC = 0x64006400


def f16pair(word):
    v = np.array([word & 0xFFFF, (word >> 16) & 0xFFFF], np.uint16).view(np.float16)
    return float(v[0]), float(v[1])


def u32(b, off):
    return int(b[off]) | (int(b[off + 1]) << 8) | (int(b[off + 2]) << 16) | (int(b[off + 3]) << 24)


def f16_at(b, off):
    return float(np.array([int(b[off]) | (int(b[off + 1]) << 8)], np.uint16).view(np.float16)[0])


def mma(afrag, bfrag):
    """m16n8k16 with f16 A (a0: row g, k 2t..2t+1; a1: row g+8; a2/a3: k + 8) and
    f16 B (b0: k 2t..2t+1, column g; b1: k + 8); returns each lane's (c0..c3):
    rows g, g, g+8, g+8 and columns 2t, 2t+1, 2t, 2t+1."""
    A = np.zeros((16, 16))
    B = np.zeros((16, 8))
    for lane in range(32):
        g, t = lane >> 2, lane & 3
        a0, a1, a2, a3 = afrag[lane]
        A[g, 2 * t:2 * t + 2] = f16pair(a0)
        A[g + 8, 2 * t:2 * t + 2] = f16pair(a1)
        A[g, 2 * t + 8:2 * t + 10] = f16pair(a2)
        A[g + 8, 2 * t + 8:2 * t + 10] = f16pair(a3)
        b0, b1 = bfrag[lane]
        B[2 * t:2 * t + 2, g] = f16pair(b0)
        B[2 * t + 8:2 * t + 10, g] = f16pair(b1)
    D = A @ B  # the products are exact in fp64 as in fp32: small integers times fp16
    return [(D[l >> 2, 2 * (l & 3)], D[l >> 2, 2 * (l & 3) + 1], D[(l >> 2) + 8, 2 * (l & 3)],
             D[(l >> 2) + 8, 2 * (l & 3) + 1]) for l in range(32)]


def stage_x(x):
    """k-permuted pairs xp[k/4] = (x[k] | x[k+2] << 16, x[k+1] | x[k+3] << 16) and 16-wide sums."""
    xb = x.view(np.uint16).astype(np.uint32)
    xp = [(int(xb[4 * q]) | (int(xb[4 * q + 2]) << 16), int(xb[4 * q + 1]) | (int(xb[4 * q + 3]) << 16))
          for q in range(x.size // 4)]
    sx16 = [float(np.float32(x[16 * i:16 * i + 16].astype(np.float32).sum())) for i in range(x.size // 16)]
    return xp, sx16


def lane_sum(y):
    """The two xor shuffles over tig: each row's total from its four lanes."""
    out = np.zeros(16)
    for lane in range(32):
        g = lane >> 2
        out[g] += y[lane][0]
        out[g + 8] += y[lane][1]
    return out


def model_q4k(W, x):
    xp, sx16 = stage_x(x)
    y = [[0.0, 0.0] for _ in range(32)]
    lop = lambda v, m: (v & m) | MAGIC
    for U in range(2):
        D = {}
        for i in range(2):
            G = 2 * U + i
            acc_c = [np.zeros(4) for _ in range(32)]
            acc_e = [np.zeros(4) for _ in range(32)]
            for hh in range(2):
                fc, fe, blo, bhi = [], [], [], []
                for lane in range(32):
                    g, tig = lane >> 2, lane & 3
                    v0 = u32(W[g], 16 + 32 * G + 8 * tig + 4 * hh)
                    v1 = u32(W[g + 8], 16 + 32 * G + 8 * tig + 4 * hh)
                    s0, s1 = v0 >> 8, v1 >> 8
                    fc.append((lop(v0, 0x000F000F), lop(v1, 0x000F000F), lop(s0, 0x000F000F), lop(s1, 0x000F000F)))
                    fe.append((lop(v0, 0x00F000F0), lop(v1, 0x00F000F0), lop(s0, 0x00F000F0), lop(s1, 0x00F000F0)))
                    blo.append(xp[16 * G + 2 * tig + hh])        # k = 64G + 8tig + 4hh
                    bhi.append(xp[16 * G + 8 + 2 * tig + hh])    # k + 32: the high nibbles
                for lane, (c, e) in enumerate(zip(mma(fc, blo), mma(fe, bhi))):
                    acc_c[lane] += c
                    acc_e[lane] += e
            for lane in range(32):
                D[(lane, i, 0)], D[(lane, i, 1)] = acc_c[lane], acc_e[lane]
        for lane in range(32):
            g, tig = lane >> 2, lane & 3
            j = 4 * U + tig                    # the lane's sub-block: group 2U + tig/2, nibble tig%2
            Dv = D[(lane, tig >> 1, tig & 1)]
            inv_f = 1 / 16 if tig & 1 else 1.0
            sx = sx16[2 * j] + sx16[2 * j + 1]
            for r, row in enumerate((W[g], W[g + 8])):
                s = row[4:16]
                if j < 4:
                    sc, mn = s[j] & 63, s[j + 4] & 63
                else:
                    sc = (s[j + 4] & 0xF) | ((s[j - 4] >> 6) << 4)
                    mn = (s[j + 4] >> 4) | ((s[j] >> 6) << 4)
                a = f16_at(row, 0) * int(sc) * inv_f
                k = 1024 * a + f16_at(row, 2) * int(mn)
                y[lane][r] += a * Dv[2 * r] - k * sx        # replicated x: c0 == c1, c2 == c3
    return lane_sum(y)


def q6_operands(wl, wh, g6):
    wl8 = wl >> 8
    up = ((wh << 2) if g6 & 1 else (wh << 4)) & 0xFFFFFFFF
    dn = (wh >> 6) if g6 & 1 else (wh >> 4)
    if g6 < 2:
        return (wl & 0x000F000F) | (up & 0x00300030) | MAGIC, (wl8 & 0x000F000F) | (dn & 0x00300030) | MAGIC
    return (wl & 0x00F000F0) | (up & 0x03000300) | MAGIC, (wl8 & 0x00F000F0) | (dn & 0x03000300) | MAGIC


def model_q6k(W, x):
    xp, sx16 = stage_x(x)
    y = [[0.0, 0.0] for _ in range(32)]
    for H in range(2):
        D = {}
        for tt in range(8):
            g6, s = (tt >> 1) & 3, tt & 1
            li = 2 * (g6 & 1) + s
            fr, bx = [], []
            for lane in range(32):
                g, tig = lane >> 2, lane & 3
                ops = []
                for row in (W[g], W[g + 8]):
                    wl = u32(row, 64 * H + 32 * (li >> 1) + 16 * (li & 1) + 4 * tig)
                    wh = u32(row, 128 + 32 * H + 16 * s + 4 * tig)
                    ops.append(q6_operands(wl, wh, g6))
                fr.append((ops[0][0], ops[1][0], ops[0][1], ops[1][1]))
                bx.append(xp[4 * (8 * H + tt) + tig])          # k = 16(8H + tt) + 4tig
            for lane, c in enumerate(mma(fr, bx)):
                D[(lane, tt)] = c
        for lane in range(32):
            g, tig = lane >> 2, lane & 3
            for u in range(2):                  # scale groups 8H + 4u + tig; F = 16 for u = 1
                tt = 4 * u + tig
                Dv = D[(lane, tt)]
                inv_f = 1 / 16 if u else 1.0
                sx = sx16[8 * H + tt]
                for r, row in enumerate((W[g], W[g + 8])):
                    dsc = f16_at(row, 208) * int(np.int8(np.uint8(row[192 + 8 * H + tt])))
                    a = dsc * inv_f
                    y[lane][r] += a * Dv[2 * r] - (1024 * a + 32 * dsc) * sx
    return lane_sum(y)


@pytest.mark.parametrize("qtype", ["q4k", "q6k"])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_gemv_mma_formulation_matches_the_oracle(qtype, seed):
    O = oracle.Oracle(oracle.build())
    rng = synth.rng_for(seed, 55)
    W = synth.weights(rng, qtype, 16, 256)
    x = synth.activations(rng, 1, 256)[0]
    bb = 144 if qtype == "q4k" else 210
    rows = W.reshape(16, bb)
    got = model_q4k(rows, x) if qtype == "q4k" else model_q6k(rows, x)
    ref = O.matmul(oracle.Q4K if qtype == "q4k" else oracle.Q6K, W, x.reshape(1, -1), 16, 256)[0]
    # fp64 model of fp32 hardware sums: the residue is the 1024·Sx cancellation only
    assert np.abs(got - ref).max() <= 1e-4 * np.sqrt(np.mean(ref ** 2))


def test_magic_operands_are_exact():
    """1024 + F·q for every 4-bit q (F = 1, 16) and every 6-bit Q6_K q (F = 1, 16)
    is exact in fp16: the operands carry the quants without rounding."""
    for q in range(16):
        assert f16pair(((q << 16) | q) | MAGIC) == (1024.0 + q, 1024.0 + q)
        assert f16pair((((q << 4) << 16) | (q << 4)) | MAGIC) == (1024.0 + 16 * q, 1024.0 + 16 * q)
    for q6 in range(64):
        lo, hi = q6 & 0xF, q6 >> 4
        assert f16pair(lo | (hi << 4) | MAGIC)[0] == 1024.0 + q6                    # F = 1: bits 0..5
        assert f16pair((lo << 4) | (hi << 8) | MAGIC)[0] == 1024.0 + 16 * q6        # F = 16: bits 4..9
