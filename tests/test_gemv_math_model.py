"""A CPU model of the decode GEMV's arithmetic, checked against the oracle.

The GEMV multiplies raw quants on the warp tensor instruction mma.m16n8k16.
- A quant OR-ed into the mantissa of fp16 1024.0 is the exact value 1024 + F·q,
  with F = 1 or 16 by nibble position (Q6_K: the 6-bit quant, F = 1 or 16).
- Lane (g, t) feeds its 4 k-slots of every MMA from one byte group: B half 0
  (k-slots 2t, 2t+1) from one sub-block, B half 1 (2t+8, 2t+9) from another.
- Column 2t of B holds x only at lane t's half-0 slots, column 2t+1 only at its
  half-1 slots; every other entry is zero.  The B operands come from an x table
  in shared memory: a lane whose column takes x from lane group g >> 1 reads
  its entry, every other lane reads a zero region.
- So lane (g, t) receives in D[g][2t] and D[g][2t+1] the sums over exactly its
  own two sub-blocks, for rows g and g+8, and applies their scales:
    Q4_K: (d·sc/F)·(D − 1024·Sx) − (dmin·m)·Sx
    Q6_K: (d·sc/F)·(D − (1024 + 32F)·Sx)
  with Sx the sum of x over the lane's k-slots of that sub-block.

This model runs those steps for one 16-row × 256-weight block: the x-table
entries and sums as the kernel builds them, each lane's table or zero-region
address, the operand bit operations, the MMA fragment layout of the PTX ISA
(A row-major, B column-major, f32 accumulators) and the per-lane scale decode
(the packed 6-bit fields with lane-dependent shifts, the exact fp32 2^23
conversion).  It compares the row sums with the oracle's dequantized weights
times x.  The model restates the method, so it checks the arithmetic and the
index mapping the kernel relies on, not the compiled kernel, which the GPU
parity tests cover.  Planted mistakes in the model show that each part is
load-bearing.
"""
import numpy as np
import pytest

import oracle
from tests import synth

MAGIC = 0x64006400
FMAGIC = 0x4B000000
M32 = 0xFFFFFFFF


def f16pair(word):
    v = np.array([word & 0xFFFF, (word >> 16) & 0xFFFF], np.uint16).view(np.float16)
    return float(v[0]), float(v[1])


def u32(b, off):
    return int(b[off]) | (int(b[off + 1]) << 8) | (int(b[off + 2]) << 16) | (int(b[off + 3]) << 24)


def f16_at(b, off):
    return float(np.array([int(b[off]) | (int(b[off + 1]) << 8)], np.uint16).view(np.float16)[0])


def f32(bits):
    return float(np.array([bits & M32], np.uint32).view(np.float32)[0])


def prmt(a, b, sel):
    """PTX prmt.b32 (default mode): byte i of the result is byte sel_i of {b, a}."""
    src = [(a >> (8 * i)) & 0xFF for i in range(4)] + [(b >> (8 * i)) & 0xFF for i in range(4)]
    return sum(src[(sel >> (4 * i)) & 7] << (8 * i) for i in range(4))


def lop(v, mask, orv=MAGIC):
    return (v & mask) | orv


def mma(afrag, bfrag, acc):
    """m16n8k16 with f16 A (a0: row g, k 2t..2t+1; a1: row g+8; a2/a3: k + 8) and
    f16 B (b0: k 2t..2t+1, column g; b1: k + 8), accumulating into each lane's
    (c0..c3): rows g, g, g+8, g+8 and columns 2t, 2t+1, 2t, 2t+1."""
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
    for l in range(32):
        g, t = l >> 2, l & 3
        acc[l] += np.array([D[g, 2 * t], D[g, 2 * t + 1], D[g + 8, 2 * t], D[g + 8, 2 * t + 1]])


# ---------------------------------------------------------------------------
# The x table and the sums, as the kernel's table build writes them
# ---------------------------------------------------------------------------
def entry_base(qtype, v, t, e):
    if qtype == "q4k":
        return 64 * t + 32 * e + 4 * v
    h, P, u = v >> 2, (v >> 1) & 1, v & 1
    return 128 * h + 64 * P + 32 * e + 8 * t + 4 * u


def build_tables(qtype, x, mistakes=()):
    """x table entries [v][t][e] -> 4 words, and the sums table."""
    xb = x.view(np.uint16).astype(np.int64)
    xf = x.astype(np.float32)
    xt = {}
    for v in range(8):
        for t in range(4):
            for e in range(2):
                k = entry_base(qtype, v, t, e)
                wa = int(xb[k]) | (int(xb[k + 1]) << 16)
                wb = int(xb[k + 2]) | (int(xb[k + 3]) << 16)
                p0, p1 = prmt(wa, wb, 0x5410), prmt(wa, wb, 0x7632)  # (x0, x2), (x1, x3)
                if "swap_pairs" in mistakes:
                    p0, p1 = p1, p0
                xt[(v, t, e)] = (p0, 0, p1, 0) if e == 0 else (0, p0, 0, p1)
    if qtype == "q4k":
        sx = {}
        for t in range(4):
            for e in range(2):
                s = float(np.float32(xf[64 * t + 32 * e:64 * t + 32 * e + 32].sum(dtype=np.float32)))
                sx[(t, e)] = (s, -1024.0 * s)
        return xt, sx
    ns = {}
    for h in range(2):
        for t in range(4):
            for j in range(4):
                s = float(xf[128 * h + 32 * j + 8 * t:128 * h + 32 * j + 8 * t + 8].sum(dtype=np.float32))
                F = 16 if j >= 2 else 1
                ns[(h, t, j)] = -(1024.0 + 32.0 * F) * s
    return xt, ns


def b_operand(xt, lane, v, mistakes=()):
    """The 4 words lane `lane` loads for word v: its table entry or the zero region."""
    g, t = lane >> 2, lane & 3
    reads_x = (g >> 1) == t
    if "all_lanes_read_x" in mistakes:
        reads_x = True
    return xt[(v, t, g & 1)] if reads_x else (0, 0, 0, 0)


# ---------------------------------------------------------------------------
# Q4_K
# ---------------------------------------------------------------------------
def q4_scales(row, tig, mistakes=()):
    """(a0, a1, m0, m1) of the lane's sub-blocks 2t and 2t+1 as the kernel decodes them."""
    A, B, C = u32(row, 4), u32(row, 8), u32(row, 12)
    hi = tig >= 2
    sh = 16 * (tig & 1)
    shA = sh + (2 if hi else 0)
    shL = sh + (4 if hi else 0)
    if "no_high_bits" in mistakes:
        shA = sh + 6
    L1, L2 = (C if hi else A), (C if hi else B)
    sc2 = ((L1 >> sh) & 0x0F0F) | ((A >> shA) & 0x3030)
    mn2 = ((L2 >> shL) & 0x0F0F) | ((B >> shA) & 0x3030)
    fs0, fs1 = f32(prmt(sc2, FMAGIC, 0x7440)), f32(prmt(sc2, FMAGIC, 0x7441))
    fm0, fm1 = f32(prmt(mn2, FMAGIC, 0x7440)), f32(prmt(mn2, FMAGIC, 0x7441))
    d, dmin = f16_at(row, 0), f16_at(row, 2)
    d16 = d * 0.0625
    # fma(d, 2^23 + v, -d * 2^23) is d * v exactly
    return d * (fs0 - 2 ** 23), d16 * (fs1 - 2 ** 23), dmin * (fm0 - 2 ** 23), dmin * (fm1 - 2 ** 23)


def model_q4k(W, x, mistakes=()):
    xt, sx = build_tables("q4k", x, mistakes)
    acc = [np.zeros(4) for _ in range(32)]
    for v in range(8):
        for p in range(2):
            af, bf = [], []
            for lane in range(32):
                g, tig = lane >> 2, lane & 3
                w0 = u32(W[g], 16 + 32 * tig + 4 * v) >> (8 * p)
                w1 = u32(W[g + 8], 16 + 32 * tig + 4 * v) >> (8 * p)
                lo, hi = 0x000F000F, 0x00F000F0
                if "swap_nibbles" in mistakes:
                    lo, hi = hi, lo
                af.append((lop(w0, lo), lop(w1, lo), lop(w0, hi), lop(w1, hi)))
                xb = b_operand(xt, lane, v, mistakes)
                bf.append((xb[2 * p], xb[2 * p + 1]))
            mma(af, bf, acc)
    y = np.zeros(16)
    for lane in range(32):
        g, tig = lane >> 2, lane & 3
        s0, n0 = sx[(tig, 0)]
        s1, n1 = sx[(tig, 1)]
        for r, row in enumerate((W[g], W[g + 8])):
            a0, a1, m0, m1 = q4_scales(row, tig, mistakes)
            c0, c1 = acc[lane][2 * r], acc[lane][2 * r + 1]
            y[g + 8 * r] += a0 * (c0 + n0) + a1 * (c1 + n1) - m0 * s0 - m1 * s1
    return y


# ---------------------------------------------------------------------------
# Q6_K
# ---------------------------------------------------------------------------
def q6op(X, H, lo, hi):
    return (X & lo) | (H & hi) | MAGIC


def model_q6k(W, x, mistakes=()):
    xt, ns = build_tables("q6k", x, mistakes)
    acc = {(h, P): [np.zeros(4) for _ in range(32)] for h in range(2) for P in range(2)}
    for h in range(2):
        for u in range(2):
            for p in range(2):
                for P in range(2):
                    af, bf = [], []
                    for lane in range(32):
                        g, tig = lane >> 2, lane & 3
                        ops = []
                        for row in (W[g], W[g + 8]):
                            o = 8 * tig + 4 * u
                            X0 = u32(row, 64 * h + o) >> (8 * p)
                            X1 = u32(row, 64 * h + 32 + o) >> (8 * p)
                            H = u32(row, 128 + 32 * h + o) >> (8 * p)
                            H4, H2 = (H << 4) & M32, (H << 2) & M32
                            if P == 0:
                                ops.append((q6op(X0, H4, 0x000F000F, 0x00300030), q6op(X1, H2, 0x000F000F, 0x00300030)))
                            else:
                                ops.append((q6op(X0, H4, 0x00F000F0, 0x03000300), q6op(X1, H2, 0x00F000F0, 0x03000300)))
                        af.append((ops[0][0], ops[1][0], ops[0][1], ops[1][1]))
                        xb = b_operand(xt, lane, 4 * h + 2 * P + u, mistakes)
                        bf.append((xb[2 * p], xb[2 * p + 1]))
                    mma(af, bf, acc[(h, P)])
    y = np.zeros(16)
    for lane in range(32):
        g, tig = lane >> 2, lane & 3
        s = tig >> 1
        sel0, sel1 = 0x7440 | s, 0x7440 | (s + 2)
        for r, row in enumerate((W[g], W[g + 8])):
            d = f16_at(row, 208)
            for h in range(2):
                for P in range(2):
                    dF = d * 0.0625 if P else d
                    if "no_f" in mistakes:
                        dF = d
                    Sw = u32(row, 192 + 4 * (2 * h + P)) ^ 0x80808080
                    for e, sel in ((0, sel0), (1, sel1)):
                        a = dF * (f32(prmt(Sw, FMAGIC, sel)) - 2 ** 23) - 128.0 * dF
                        c = acc[(h, P)][lane][2 * r + e]
                        y[g + 8 * r] += a * (c + ns[(h, tig, 2 * P + e)])
    return y


# ---------------------------------------------------------------------------
# Several tokens: the MMA columns carry tokens (8 per n-tile)
# ---------------------------------------------------------------------------
def xp_pairs(x):
    """k-permuted pairs xp[k/4] = ((x[k], x[k+2]), (x[k+1], x[k+3])) as words."""
    xb = x.view(np.uint16).astype(np.int64)
    return [(prmt(int(xb[4 * q]) | (int(xb[4 * q + 1]) << 16), int(xb[4 * q + 2]) | (int(xb[4 * q + 3]) << 16), 0x5410),
             prmt(int(xb[4 * q]) | (int(xb[4 * q + 1]) << 16), int(xb[4 * q + 2]) | (int(xb[4 * q + 3]) << 16), 0x7632))
            for q in range(x.size // 4)]


def model_q4k_tn(W, X, NT, mistakes=()):
    """Lane (g, t) owns bytes 8t .. 8t+7 of each 32-byte group G; the two
    words feed the k-slots of sub-block 2G (low nibbles) and 2G+1 (high); the
    lane's own sub-blocks 2t, 2t+1 reach the quad through shuffles."""
    M = X.shape[0]
    xps = [xp_pairs(X[m]) for m in range(M)]
    sx = [[float(X[m, 32 * j:32 * j + 32].astype(np.float32).sum(dtype=np.float32)) for j in range(8)]
          for m in range(M)]
    y = np.zeros((16, M))
    dec = {}
    for lane in range(32):
        g, tig = lane >> 2, lane & 3
        for r, row in enumerate((W[g], W[g + 8])):
            a0, a1, m0, m1 = q4_scales(row, tig)
            dec[(lane, r)] = (a0, a1, 1024 * a0 + m0, 1024 * a1 + m1)
    for G in range(4):
        for sb in range(2):
            j = 2 * G + sb
            accs = [[np.zeros(4) for _ in range(32)] for _ in range(NT)]
            for hh in range(2):
                af, bfs = [], [[] for _ in range(NT)]
                for lane in range(32):
                    g, tig = lane >> 2, lane & 3
                    w0 = u32(W[g], 16 + 32 * G + 8 * tig + 4 * hh)
                    w1 = u32(W[g + 8], 16 + 32 * G + 8 * tig + 4 * hh)
                    mask = 0x00F000F0 if sb else 0x000F000F
                    af.append((lop(w0, mask), lop(w1, mask), lop(w0 >> 8, mask), lop(w1 >> 8, mask)))
                    for nt in range(NT):
                        tok = 8 * nt + g
                        q = (64 * G + 32 * sb + 8 * tig + 4 * hh) // 4
                        bfs[nt].append(xps[tok][q] if tok < M else (0, 0))
                for nt in range(NT):
                    mma(af, bfs[nt], accs[nt])
            for lane in range(32):
                g, tig = lane >> 2, lane & 3
                src = (lane & ~3) | (j >> 1)
                if "wrong_owner" in mistakes:
                    src = (lane & ~3) | (j & 3)
                e = j & 1
                for nt in range(NT):
                    for i in range(4):
                        r, tok = i >> 1, 8 * nt + 2 * tig + (i & 1)
                        a, k = dec[(src, r)][e], dec[(src, r)][2 + e]
                        if tok < M:
                            y[g + 8 * r, tok] += a * accs[nt][lane][i] - k * sx[tok][j]
    return y


def model_q6k_tn(W, X, NT, mistakes=()):
    M = X.shape[0]
    xps = [xp_pairs(X[m]) for m in range(M)]
    sx = [[float(X[m, 16 * q:16 * q + 16].astype(np.float32).sum(dtype=np.float32)) for q in range(16)]
          for m in range(M)]
    y = np.zeros((16, M))
    dec = {}
    for lane in range(32):
        g, tig = lane >> 2, lane & 3
        for r, row in enumerate((W[g], W[g + 8])):
            dF = f16_at(row, 208) * (0.0625 if tig & 1 else 1.0)
            dec[(lane, r)] = [dF * int(np.int8(np.uint8(row[192 + 4 * tig + i]))) for i in range(4)]
    for h in range(2):
        for sb in range(2):
            for j in range(4):
                grp = 8 * h + 2 * j + sb
                af, bfs = [], [[] for _ in range(NT)]
                for lane in range(32):
                    g, tig = lane >> 2, lane & 3
                    ops = []
                    for row in (W[g], W[g + 8]):
                        o = 16 * sb + 4 * tig
                        X0 = u32(row, 64 * h + 32 * (j & 1) + o)
                        H = u32(row, 128 + 32 * h + o)
                        lo, hi = (0x000F000F, 0x00300030) if j < 2 else (0x00F000F0, 0x03000300)
                        shl = 4 if j % 2 == 0 else 2
                        ops.append((q6op(X0, (H << shl) & M32, lo, hi), q6op(X0 >> 8, ((H >> 8) << shl) & M32, lo, hi)))
                    af.append((ops[0][0], ops[1][0], ops[0][1], ops[1][1]))
                    for nt in range(NT):
                        tok = 8 * nt + g
                        q = (128 * h + 32 * j + 16 * sb + 4 * tig) // 4
                        bfs[nt].append(xps[tok][q] if tok < M else (0, 0))
                accs = [[np.zeros(4) for _ in range(32)] for _ in range(NT)]
                for nt in range(NT):
                    mma(af, bfs[nt], accs[nt])
                kf = 1024.0 + 32.0 * (16 if j >= 2 else 1)
                for lane in range(32):
                    g, tig = lane >> 2, lane & 3
                    src = (lane & ~3) | (grp >> 2)
                    for nt in range(NT):
                        for i in range(4):
                            r, tok = i >> 1, 8 * nt + 2 * tig + (i & 1)
                            a = dec[(src, r)][grp & 3]
                            if tok < M:
                                y[g + 8 * r, tok] += a * accs[nt][lane][i] - a * kf * sx[tok][grp]
    return y


@pytest.mark.parametrize("qtype", ["q4k", "q6k"])
@pytest.mark.parametrize("M", [2, 8, 11, 16])
def test_gemv_token_columns_match_the_oracle(qtype, M):
    O = oracle.Oracle(oracle.build())
    rng = synth.rng_for(M, 56)
    W = synth.weights(rng, qtype, 16, 256)
    X = synth.activations(rng, M, 256)
    rows = W.reshape(16, 144 if qtype == "q4k" else 210)
    NT = 1 if M <= 8 else 2
    got = (model_q4k_tn if qtype == "q4k" else model_q6k_tn)(rows, X, NT)
    ref = O.matmul(oracle.Q4K if qtype == "q4k" else oracle.Q6K, W, X, 16, 256).T
    assert np.abs(got - ref).max() <= 1e-5 * np.sqrt(np.mean(ref ** 2))


def test_token_columns_planted_mistake_fails():
    O = oracle.Oracle(oracle.build())
    rng = synth.rng_for(3, 56)
    W = synth.weights(rng, "q4k", 16, 256)
    X = synth.activations(rng, 4, 256)
    got = model_q4k_tn(W.reshape(16, 144), X, 1, ("wrong_owner",))
    ref = O.matmul(oracle.Q4K, W, X, 16, 256).T
    assert np.abs(got - ref).max() > 1e-2 * np.sqrt(np.mean(ref ** 2))


def run(qtype, seed, mistakes=()):
    O = oracle.Oracle(oracle.build())
    rng = synth.rng_for(seed, 55)
    W = synth.weights(rng, qtype, 16, 256)
    x = synth.activations(rng, 1, 256)[0]
    bb = 144 if qtype == "q4k" else 210
    rows = W.reshape(16, bb)
    got = model_q4k(rows, x, mistakes) if qtype == "q4k" else model_q6k(rows, x, mistakes)
    ref = O.matmul(oracle.Q4K if qtype == "q4k" else oracle.Q6K, W, x.reshape(1, -1), 16, 256)[0]
    return np.abs(got - ref).max() / np.sqrt(np.mean(ref ** 2))


@pytest.mark.parametrize("qtype", ["q4k", "q6k"])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_gemv_column_layout_matches_the_oracle(qtype, seed):
    # fp64 model of fp32 hardware sums: the residue is the 1024·Sx cancellation only
    assert run(qtype, seed) <= 1e-5


@pytest.mark.parametrize("qtype,mistake", [
    ("q4k", "swap_pairs"), ("q4k", "all_lanes_read_x"), ("q4k", "swap_nibbles"), ("q4k", "no_high_bits"),
    ("q6k", "swap_pairs"), ("q6k", "all_lanes_read_x"), ("q6k", "no_f"),
])
def test_planted_mistakes_fail(qtype, mistake):
    """Each part of the layout is load-bearing: a plausible slip in any of them
    (pair order, the zero region, nibble halves, the high scale bits, the F
    factor) breaks agreement with the oracle."""
    assert run(qtype, 0, (mistake,)) > 1e-2


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


def test_scale_decode_covers_every_sub_block():
    """The lane-dependent shifts decode the packed 6-bit scale and min of every
    sub-block: for each lane group t, sub-blocks 2t and 2t+1 of a block whose
    12 packed bytes are random agree with the format's own unpacking rule."""
    rng = np.random.default_rng(5)
    for _ in range(200):
        row = np.zeros(144, np.uint8)
        row[0:2] = np.array([1.0], np.float16).view(np.uint8)
        row[2:4] = np.array([1.0], np.float16).view(np.uint8)
        row[4:16] = rng.integers(0, 256, 12)
        s = row[4:16].astype(int)
        for t in range(4):
            a0, a1, m0, m1 = q4_scales(row, t)
            for j, a, m in ((2 * t, a0, m0), (2 * t + 1, a1 * 16, m1)):
                if j < 4:
                    sc, mn = s[j] & 63, s[j + 4] & 63
                else:
                    sc = (s[j + 4] & 0xF) | ((s[j - 4] >> 6) << 4)
                    mn = (s[j + 4] >> 4) | ((s[j] >> 6) << 4)
                assert (a, m) == (sc, mn)
