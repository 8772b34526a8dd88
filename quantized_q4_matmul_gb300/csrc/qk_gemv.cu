// qk_gemv.cu -- the GEMV for M <= 8 tokens: y[m][n] = sum_k x[m][k] * w[n][k]
// for Q4_K and Q6_K weights, one or several independent problems per launch.
//
// Source: DAMASCUS project overview, "[01] the thesis" (decode handles one
// token at a time with matrix-vector products whose speed is set by streaming
// the weights from memory) and "[04] one decode step"; "Building DAMASCUS",
// "Prefill and decode need different performance questions".
//
// The kernel is HBM-bound by design: every packed weight byte is read once.
//   * Streaming: the weights of 16 consecutive rows are contiguous, so a
//     producer warp copies whole 16-row tiles (two adjacent tiles, or the
//     gate and the up tile, per stage; for long rows 16-row x cb-block chunks,
//     one copy per row) with bulk asynchronous copies into a ring of
//     shared-memory stages.
//   * Arithmetic: the warp tensor instruction mma.sync m16n8k16 (fp16 x fp16,
//     fp32 accumulate) multiplies raw quants: a 4-bit quant OR-ed into the
//     mantissa of fp16 1024.0 is the exact value 1024 + F*q (F = 1 or 16 by
//     nibble position; Q6_K: the 6-bit quant, F = 1 or 16), and its product
//     with an fp16 activation is exact.
//   * One token, column layout: the MMA's 8 columns do not hold copies of x.
//     Lane (g, t) of the warp feeds the 4 k-slots it owns in every MMA from
//     one byte group of the block: the slots of its B half 0 belong to one
//     sub-block (Q4_K low nibbles; Q6_K one scale group), those of half 1 to
//     another.  Column 2t holds x only at lane t's half-0 slots and column
//     2t+1 only at its half-1 slots (every other B entry is zero), so the
//     accumulator lane (g, t) receives, D[g][2t] and D[g][2t+1], is the sum
//     over exactly its own two sub-blocks, for rows g and g+8.  Each lane then
//     applies the scales of those two sub-blocks.  The zero B entries come
//     from a zero region: a lane whose column takes no x reads zeros.
//   * Several tokens: the MMA columns carry tokens (see q4_block_tn).
//   * Per sub-block, with Sx the sum of x over the lane's k-slots of it:
//       Q4_K: sum(w*x) = (d*sc/F) * (D - 1024*Sx) - (dmin*m) * Sx
//       Q6_K: sum(w*x) = (d*sc/F) * (D - (1024 + 32F)*Sx)
//   * Reduction: compute warp w takes the blocks j = w mod kDW of every tile
//     and leaves its sums of a finished tile in the stage's partials slot;
//     the producer adds the kDW warps' sums in warp order before it refills
//     the stage and writes y.  The order of every addition depends on the
//     problem's shape only (deterministic, and the same alone or grouped).
// Q6_K blocks are 210 bytes, so a block can start 2 mod 4 bytes into shared
// memory; its words then come from aligned loads and funnel shifts.  Problem
// kind 1 is the fused gate/up + SwiGLU: a stage holds the gate tile and the up
// tile of the same rows, and the epilogue writes fp16(silu(g)*u).
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>

#include "qk_device.cuh"
#include "qk_internal.h"

namespace qk {

__device__ uint32_t g_gemv_status = 0;

namespace {

constexpr uint32_t kMagic = 0x64006400u;   // fp16x2 (1024.0, 1024.0)
constexpr uint32_t kFMagic = 0x4B000000u;  // fp32 2^23: 0x4B0000XX is 2^23 + XX

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Shared-memory loads through 32-bit shared-window addresses.
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ float4 ldsf4(uint32_t a) {
  const uint4 v = lds128(a);
  return make_float4(__uint_as_float(v.x), __uint_as_float(v.y), __uint_as_float(v.z), __uint_as_float(v.w));
}

__device__ __forceinline__ float half_lo(uint32_t v) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(v & 0xFFFFu)));
}

// Two consecutive 4-byte words starting at shared address a, which is 4-byte
// aligned (A2 = false) or 2 mod 4 (A2 = true: three aligned loads, two funnel
// shifts).
template <bool A2>
__device__ __forceinline__ void lds_run2(uint32_t a, uint32_t& w0, uint32_t& w1) {
  if constexpr (!A2) {
    w0 = lds32(a);
    w1 = lds32(a + 4);
  } else {
    const uint32_t t0 = lds32(a - 2), t1 = lds32(a + 2), t2 = lds32(a + 6);
    w0 = __funnelshift_r(t0, t1, 16);
    w1 = __funnelshift_r(t1, t2, 16);
  }
}

// Per-lane constants of the decode layout.
struct Lane {
  int g, tig;
  uint32_t xt_off;     // offset of the lane's x-table entry inside a block's table, or its zero-region offset
  uint32_t xt_stride;  // bytes per block for lanes that read x, 0 for lanes that read zeros
  // Q4_K scale decode (sub-blocks 2t, 2t+1): shifts for the packed 6-bit fields
  uint32_t sh, shA, shL;
  bool hi;             // sub-blocks 4..7
  // Q6_K scale group offset s = t >> 1 and the byte selectors of its two scales per word
  uint32_t sel0, sel1;
};

// ---------------------------------------------------------------------------
// Q4_K, one 256-weight block of rows g (row address r0) and g+8 (r1).
// Lane t owns byte group t (quant bytes 32t .. 32t+31: low nibbles are
// sub-block 2t, high nibbles sub-block 2t+1).  Word v (bytes 4v .. 4v+3) feeds
// two MMAs: p = 0 the bytes 0 and 2, p = 1 the bytes 1 and 3 (shifted down by
// 8).  In each, a0/a1 (k-slots 2t, 2t+1) carry the low nibbles (F = 1) and
// a2/a3 (k-slots 2t+8, 2t+9) the high nibbles (F = 16) of the same two bytes.
// The x-table entry of word v holds the B operands of both MMAs.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void q4_row_scales(uint4 h, float c0, float c1, float4 sx, const Lane& L, uint32_t fmagic,
                                              float& y) {
  const uint32_t A = h.y, B = h.z, C = h.w;
  const uint32_t L1 = L.hi ? C : A, L2 = L.hi ? C : B;
  // bytes 0, 1: the 6-bit scale (min) of sub-blocks 2t and 2t+1
  const uint32_t sc2 = ((L1 >> L.sh) & 0x0F0Fu) | ((A >> L.shA) & 0x3030u);
  const uint32_t mn2 = ((L2 >> L.shL) & 0x0F0Fu) | ((B >> L.shA) & 0x3030u);
  // 2^23 + v as fp32 bit patterns; fma(d, 2^23 + v, -d * 2^23) = d * v exactly
  const float fs0 = __uint_as_float(prmt(sc2, fmagic, 0x7440u)), fs1 = __uint_as_float(prmt(sc2, fmagic, 0x7441u));
  const float fm0 = __uint_as_float(prmt(mn2, fmagic, 0x7440u)), fm1 = __uint_as_float(prmt(mn2, fmagic, 0x7441u));
  const float d = half_lo(h.x), dmin = half_lo(h.x >> 16);
  const float d16 = d * 0.0625f;
  const float a0 = fmaf(d, fs0, d * -8388608.0f);          // d*sc0
  const float a1 = fmaf(d16, fs1, d16 * -8388608.0f);      // d*sc1/16
  const float m0 = fmaf(dmin, fm0, dmin * -8388608.0f);    // dmin*m0
  const float m1 = fmaf(dmin, fm1, dmin * -8388608.0f);    // dmin*m1
  y = fmaf(a0, c0 + sx.y, y);
  y = fmaf(a1, c1 + sx.w, y);
  y = fmaf(-m0, sx.x, y);
  y = fmaf(-m1, sx.z, y);
}

__device__ __forceinline__ void q4_block(uint32_t r0, uint32_t r1, uint32_t xa, uint32_t sxa, const Lane& L,
                                         uint32_t magic, uint32_t fmagic, float& y0, float& y1) {
  // Every load of the block first (the loads and MMAs keep their source
  // order), so that their latencies overlap.
  const uint32_t o = 16u + 32u * (uint32_t)L.tig;
  const uint4 qa = lds128(r0 + o), qb = lds128(r0 + o + 16), qc = lds128(r1 + o), qd = lds128(r1 + o + 16);
  uint4 xb[8];
#pragma unroll
  for (int v = 0; v < 8; ++v) xb[v] = lds128(xa + 128u * (uint32_t)v);
  const float4 sx = ldsf4(sxa);  // (Sx, -1024 Sx) of sub-blocks 2t and 2t+1
  const uint4 h0 = lds128(r0), h1 = lds128(r1);
  const uint32_t w0[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
  const uint32_t w1[8] = {qc.x, qc.y, qc.z, qc.w, qd.x, qd.y, qd.z, qd.w};
  // four independent accumulation chains (MMA m = 2v + p goes to chain m % 4)
  float acc[4][4];
#pragma unroll
  for (int c = 0; c < 4; ++c)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[c][i] = 0.f;
#pragma unroll
  for (int v = 0; v < 8; ++v) {
    const uint32_t s0 = w0[v] >> 8, s1 = w1[v] >> 8;
    mma16816(acc[(2 * v) & 3], lop_and_or<0x000F000Fu>(w0[v], magic), lop_and_or<0x000F000Fu>(w1[v], magic),
             lop_and_or<0x00F000F0u>(w0[v], magic), lop_and_or<0x00F000F0u>(w1[v], magic), xb[v].x, xb[v].y);
    mma16816(acc[(2 * v + 1) & 3], lop_and_or<0x000F000Fu>(s0, magic), lop_and_or<0x000F000Fu>(s1, magic),
             lop_and_or<0x00F000F0u>(s0, magic), lop_and_or<0x00F000F0u>(s1, magic), xb[v].z, xb[v].w);
  }
  float c[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) c[i] = (acc[0][i] + acc[1][i]) + (acc[2][i] + acc[3][i]);
  q4_row_scales(h0, c[0], c[1], sx, L, fmagic, y0);
  q4_row_scales(h1, c[2], c[3], sx, L, fmagic, y1);
}

// ---------------------------------------------------------------------------
// Q6_K, one block of rows g (r0) and g+8 (r1).  Weight 128h + 32j + l (half
// h, field j = 0..3, l = 0..31) takes its low 4 bits from byte
// 64h + 32(j & 1) + l (low nibble for j < 2, high for j >= 2) and its high 2
// bits from bits 2j of byte 128 + 32h + l; its scale group is 8h + 2j +
// (l >= 16).  Lane t owns l = 8t .. 8t+7 of every half and field, so all its
// weights of a (half, field) share the scale group 8h + 2j + (t >> 1).  Pass
// P = 0 takes fields j = 0 (B half 0, F = 1) and 1 (B half 1, F = 1), pass
// P = 1 fields 2 and 3 (F = 16).  Word u (l = 8t + 4u .. 8t + 4u + 3) feeds two
// MMAs, p = 0 (bytes 0 and 2) and p = 1 (bytes 1 and 3).
// ---------------------------------------------------------------------------
struct Q6Row {
  uint32_t ql0[2][2], ql1[2][2], qh[2][2];  // [h][u]
  uint32_t S[4];                            // the 16 int8 scales
  uint32_t dw;                              // low half: d
};

template <bool A2>
__device__ __forceinline__ void q6_load_row(uint32_t b, int tig, Q6Row& q) {
  const uint32_t o = 8u * (uint32_t)tig;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    lds_run2<A2>(b + 64u * h + o, q.ql0[h][0], q.ql0[h][1]);
    lds_run2<A2>(b + 64u * h + 32u + o, q.ql1[h][0], q.ql1[h][1]);
    lds_run2<A2>(b + 128u + 32u * h + o, q.qh[h][0], q.qh[h][1]);
  }
  if constexpr (!A2) {
#pragma unroll
    for (int i = 0; i < 4; ++i) q.S[i] = lds32(b + 192u + 4u * i);
    q.dw = lds32(b + 208);
  } else {
    uint32_t t[6];
#pragma unroll
    for (int i = 0; i < 6; ++i) t[i] = lds32(b + 190u + 4u * i);
#pragma unroll
    for (int i = 0; i < 4; ++i) q.S[i] = __funnelshift_r(t[i], t[i + 1], 16);
    q.dw = __funnelshift_r(t[4], t[5], 16);
  }
}

// (X & lo_mask) | (H & hi_mask) | magic in two LOP3s.
template <uint32_t LO, uint32_t HI>
__device__ __forceinline__ uint32_t q6op(uint32_t X, uint32_t H, uint32_t magic) {
  return lop_and_or<LO>(X, lop_and_or<HI>(H, magic));
}

// Scales of one row for pass (h, P): y += (d*sc/F) * (c + nS) for the lane's
// two fields j = 2P (c_a) and 2P + 1 (c_b).
__device__ __forceinline__ void q6_row_scales(uint32_t Sw, float dF, float c_a, float c_b, float ns_a, float ns_b,
                                              const Lane& L, uint32_t fmagic, float& y) {
  const uint32_t u = Sw ^ 0x80808080u;  // int8 + 128 as unsigned bytes
  const float f0 = __uint_as_float(prmt(u, fmagic, L.sel0)), f1 = __uint_as_float(prmt(u, fmagic, L.sel1));
  const float ndF = dF * -8388608.0f;
  const float a0 = fmaf(-128.0f, dF, fmaf(dF, f0, ndF));  // dF * sc exactly
  const float a1 = fmaf(-128.0f, dF, fmaf(dF, f1, ndF));
  y = fmaf(a0, c_a + ns_a, y);
  y = fmaf(a1, c_b + ns_b, y);
}

__device__ __forceinline__ void q6_block(uint32_t r0, uint32_t r1, uint32_t xa, uint32_t sxa, const Lane& L,
                                         uint32_t magic, uint32_t fmagic, float& y0, float& y1) {
  // The loads branch per lane on the block's alignment (rows g and g+8 share
  // it); the warp reconverges before the MMAs, which need every lane.
  Q6Row q, r;
  if ((r0 & 3u) == 0) {
    q6_load_row<false>(r0, L.tig, q);
    q6_load_row<false>(r1, L.tig, r);
  } else {
    q6_load_row<true>(r0, L.tig, q);
    q6_load_row<true>(r1, L.tig, r);
  }
  __syncwarp();
  uint4 xb[8];  // entry v = 4h + 2P + u
#pragma unroll
  for (int v = 0; v < 8; ++v) xb[v] = lds128(xa + 128u * (uint32_t)v);
  const float4 ns0 = ldsf4(sxa), ns1 = ldsf4(sxa + 64u);  // -(1024 + 32F) * Sx of fields 0..3, per half
  float acc[2][2][4];
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int P = 0; P < 2; ++P)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[h][P][i] = 0.f;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const uint4 xb0 = xb[4 * h + u];      // P = 0
      const uint4 xb1 = xb[4 * h + 2 + u];  // P = 1
#pragma unroll
      for (int p = 0; p < 2; ++p) {
        const int sh = 8 * p;
        const uint32_t X0 = q.ql0[h][u] >> sh, X1 = q.ql1[h][u] >> sh, H = q.qh[h][u] >> sh;
        const uint32_t Y0 = r.ql0[h][u] >> sh, Y1 = r.ql1[h][u] >> sh, G = r.qh[h][u] >> sh;
        const uint32_t H4 = H << 4, H2 = H << 2, G4 = G << 4, G2 = G << 2;
        const uint32_t b0a = p ? xb0.z : xb0.x, b1a = p ? xb0.w : xb0.y;
        const uint32_t b0b = p ? xb1.z : xb1.x, b1b = p ? xb1.w : xb1.y;
        // P = 0: fields 0 (low nibble of ql0, qh bits 0-1) and 1 (low nibble of ql1, qh bits 2-3)
        mma16816(acc[h][0], q6op<0x000F000Fu, 0x00300030u>(X0, H4, magic),
                 q6op<0x000F000Fu, 0x00300030u>(Y0, G4, magic), q6op<0x000F000Fu, 0x00300030u>(X1, H2, magic),
                 q6op<0x000F000Fu, 0x00300030u>(Y1, G2, magic), b0a, b1a);
        // P = 1: fields 2 (high nibble of ql0, qh bits 4-5) and 3 (high nibble of ql1, qh bits 6-7)
        mma16816(acc[h][1], q6op<0x00F000F0u, 0x03000300u>(X0, H4, magic),
                 q6op<0x00F000F0u, 0x03000300u>(Y0, G4, magic), q6op<0x00F000F0u, 0x03000300u>(X1, H2, magic),
                 q6op<0x00F000F0u, 0x03000300u>(Y1, G2, magic), b0b, b1b);
      }
    }
  }
  const float dq = half_lo(q.dw), dr = half_lo(r.dw);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const float4 ns = h ? ns1 : ns0;
#pragma unroll
    for (int P = 0; P < 2; ++P) {
      const float fq = P ? dq * 0.0625f : dq, fr = P ? dr * 0.0625f : dr;
      const float na = P ? ns.z : ns.x, nb = P ? ns.w : ns.y;
      q6_row_scales(q.S[2 * h + P], fq, acc[h][P][0], acc[h][P][1], na, nb, L, fmagic, y0);
      q6_row_scales(r.S[2 * h + P], fr, acc[h][P][2], acc[h][P][3], na, nb, L, fmagic, y1);
    }
  }
}

// ---------------------------------------------------------------------------
// Several tokens (2 <= M <= 8): the MMA columns carry tokens.  Lane (g, t)
// supplies B for token 8*nt + g of n-tile nt from that token's k-permuted x
// (or from the zero region for a token beyond M).  Every k-slot of one MMA
// lies in one sub-block (Q4_K) or scale group (Q6_K), so after its MMAs lane
// (g, t) holds that sub-block's sums for rows g, g+8 and tokens 8nt + 2t,
// 8nt + 2t + 1, and adds scale * D - k * Sx for each:
//   Q4_K: scale = d*sc/F, k = 1024*scale + dmin*m
//   Q6_K: scale = d*sc/F, k = (1024 + 32F)*scale
// Each lane decodes the scales of two sub-blocks (Q4_K) or four groups (Q6_K)
// of its two rows, and the others reach it through shuffles within the
// lane's quad.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void q4_row_decode(uint4 h, const Lane& L, uint32_t fmagic, float& a0, float& a1,
                                              float& k0, float& k1) {
  const uint32_t A = h.y, B = h.z, C = h.w;
  const uint32_t L1 = L.hi ? C : A, L2 = L.hi ? C : B;
  const uint32_t sc2 = ((L1 >> L.sh) & 0x0F0Fu) | ((A >> L.shA) & 0x3030u);
  const uint32_t mn2 = ((L2 >> L.shL) & 0x0F0Fu) | ((B >> L.shA) & 0x3030u);
  const float fs0 = __uint_as_float(prmt(sc2, fmagic, 0x7440u)), fs1 = __uint_as_float(prmt(sc2, fmagic, 0x7441u));
  const float fm0 = __uint_as_float(prmt(mn2, fmagic, 0x7440u)), fm1 = __uint_as_float(prmt(mn2, fmagic, 0x7441u));
  const float d = half_lo(h.x), dmin = half_lo(h.x >> 16);
  const float d16 = d * 0.0625f;
  a0 = fmaf(d, fs0, d * -8388608.0f);                                // d*sc0
  a1 = fmaf(d16, fs1, d16 * -8388608.0f);                            // d*sc1/16
  k0 = fmaf(1024.0f, a0, fmaf(dmin, fm0, dmin * -8388608.0f));       // 1024*a0 + dmin*m0
  k1 = fmaf(1024.0f, a1, fmaf(dmin, fm1, dmin * -8388608.0f));       // 1024*a1 + dmin*m1
}

template <int NT>
__device__ __forceinline__ void q4_block_tn(uint32_t r0, uint32_t r1, const uint32_t (&xa)[NT], uint32_t sxa,
                                            const Lane& L, int lane, uint32_t magic, uint32_t fmagic,
                                            float (&y)[NT][4]) {
  constexpr int MT = 8 * NT;
  float a0[2], a1[2], k0[2], k1[2];  // [row g / g+8]: the lane's sub-blocks 2t, 2t+1
  q4_row_decode(lds128(r0), L, fmagic, a0[0], a1[0], k0[0], k1[0]);
  q4_row_decode(lds128(r1), L, fmagic, a0[1], a1[1], k0[1], k1[1]);
  const int quad = lane & ~3;
  const uint32_t o = 16u + 8u * (uint32_t)L.tig;
#pragma unroll
  for (int G = 0; G < 4; ++G) {
    const uint2 wa = lds64(r0 + o + 32u * G), wb = lds64(r1 + o + 32u * G);
#pragma unroll
    for (int sb = 0; sb < 2; ++sb) {
      const int j = 2 * G + sb;
      float acc[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[nt][i] = 0.f;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const uint32_t w0 = hh ? wa.y : wa.x, w1 = hh ? wb.y : wb.x;
        const uint32_t s0 = w0 >> 8, s1 = w1 >> 8;
        uint32_t A0, A1, A2, A3;
        if (sb == 0) {
          A0 = lop_and_or<0x000F000Fu>(w0, magic);
          A1 = lop_and_or<0x000F000Fu>(w1, magic);
          A2 = lop_and_or<0x000F000Fu>(s0, magic);
          A3 = lop_and_or<0x000F000Fu>(s1, magic);
        } else {
          A0 = lop_and_or<0x00F000F0u>(w0, magic);
          A1 = lop_and_or<0x00F000F0u>(w1, magic);
          A2 = lop_and_or<0x00F000F0u>(s0, magic);
          A3 = lop_and_or<0x00F000F0u>(s1, magic);
        }
        const uint32_t koff = 2u * (uint32_t)(64 * G + 32 * sb + 4 * hh) + 16u * (uint32_t)L.tig;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const uint2 b = lds64(xa[nt] + koff);
          mma16816(acc[nt], A0, A1, A2, A3, b.x, b.y);
        }
      }
      // the scale and offset of sub-block j for rows g and g+8, from lane t = j / 2 of the quad
      const int src = quad | (j >> 1);
      const float sa0 = __shfl_sync(0xffffffffu, (j & 1) ? a1[0] : a0[0], src);
      const float sa1 = __shfl_sync(0xffffffffu, (j & 1) ? a1[1] : a0[1], src);
      const float sk0 = __shfl_sync(0xffffffffu, (j & 1) ? k1[0] : k0[0], src);
      const float sk1 = __shfl_sync(0xffffffffu, (j & 1) ? k1[1] : k0[1], src);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const uint2 sxw = lds64(sxa + 4u * (uint32_t)(j * MT + 8 * nt + 2 * L.tig));
        const float sx0 = __uint_as_float(sxw.x), sx1 = __uint_as_float(sxw.y);
        y[nt][0] = fmaf(sa0, acc[nt][0], fmaf(-sk0, sx0, y[nt][0]));
        y[nt][1] = fmaf(sa0, acc[nt][1], fmaf(-sk0, sx1, y[nt][1]));
        y[nt][2] = fmaf(sa1, acc[nt][2], fmaf(-sk1, sx0, y[nt][2]));
        y[nt][3] = fmaf(sa1, acc[nt][3], fmaf(-sk1, sx1, y[nt][3]));
      }
    }
  }
}

// A 4-byte word at shared address a: 4-byte aligned (A2 = false) or 2 mod 4.
template <bool A2>
__device__ __forceinline__ uint32_t lds_word(uint32_t a) {
  if constexpr (!A2) {
    return lds32(a);
  } else {
    return __funnelshift_r(lds32(a - 2), lds32(a + 2), 16);
  }
}

// The lane's words of one Q6_K row for the multi-token layout: for half h and
// 16-weight column s, ql words of fields 0/2 (c = 0) and 1/3 (c = 1) and the qh
// word at l = 16s + 4t; the lane's four scales (groups 4t .. 4t+3) and d.
struct Q6RowTn {
  uint32_t x0[2][2], x1[2][2], qh[2][2];  // [h][s]
  uint32_t sc;                            // int8 scales of groups 4t .. 4t+3
  uint32_t dw;
};

template <bool A2>
__device__ __forceinline__ void q6_load_row_tn(uint32_t b, int tig, Q6RowTn& q) {
  const uint32_t o = 4u * (uint32_t)tig;
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      q.x0[h][s] = lds_word<A2>(b + 64u * h + 16u * s + o);
      q.x1[h][s] = lds_word<A2>(b + 64u * h + 32u + 16u * s + o);
      q.qh[h][s] = lds_word<A2>(b + 128u + 32u * h + 16u * s + o);
    }
  q.sc = lds_word<A2>(b + 192u + o);
  q.dw = lds_word<A2>(b + 208u);
}

// The lane's four scales as fp32 d*sc/F: groups 4t + i, i = 0..3, share the
// field parity (t odd: fields 2, 3, F = 16).
__device__ __forceinline__ void q6_decode_tn(const Q6RowTn& q, int tig, float (&a)[4]) {
  const float dF = (tig & 1) ? half_lo(q.dw) * 0.0625f : half_lo(q.dw);
#pragma unroll
  for (int i = 0; i < 4; ++i) a[i] = dF * (float)(int8_t)((q.sc >> (8 * i)) & 0xFFu);
}

template <int NT>
__device__ __forceinline__ void q6_block_tn(uint32_t r0, uint32_t r1, const uint32_t (&xa)[NT], uint32_t sxa,
                                            const Lane& L, int lane, uint32_t magic, float (&y)[NT][4]) {
  constexpr int MT = 8 * NT;
  Q6RowTn q, r;
  if ((r0 & 3u) == 0) {
    q6_load_row_tn<false>(r0, L.tig, q);
    q6_load_row_tn<false>(r1, L.tig, r);
  } else {
    q6_load_row_tn<true>(r0, L.tig, q);
    q6_load_row_tn<true>(r1, L.tig, r);
  }
  __syncwarp();
  float aq[4], ar[4];
  q6_decode_tn(q, L.tig, aq);
  q6_decode_tn(r, L.tig, ar);
  const int quad = lane & ~3;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
#pragma unroll
    for (int s = 0; s < 2; ++s) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int grp = 8 * h + 2 * j + s;
        const uint32_t X = (j & 1) ? q.x1[h][s] : q.x0[h][s], Y = (j & 1) ? r.x1[h][s] : r.x0[h][s];
        const uint32_t H = q.qh[h][s], G = r.qh[h][s];
        const uint32_t X8 = X >> 8, Y8 = Y >> 8, H8 = H >> 8, G8 = G >> 8;
        uint32_t A0, A1, A2, A3;
        if (j == 0) {
          A0 = q6op<0x000F000Fu, 0x00300030u>(X, H << 4, magic);
          A1 = q6op<0x000F000Fu, 0x00300030u>(Y, G << 4, magic);
          A2 = q6op<0x000F000Fu, 0x00300030u>(X8, H8 << 4, magic);
          A3 = q6op<0x000F000Fu, 0x00300030u>(Y8, G8 << 4, magic);
        } else if (j == 1) {
          A0 = q6op<0x000F000Fu, 0x00300030u>(X, H << 2, magic);
          A1 = q6op<0x000F000Fu, 0x00300030u>(Y, G << 2, magic);
          A2 = q6op<0x000F000Fu, 0x00300030u>(X8, H8 << 2, magic);
          A3 = q6op<0x000F000Fu, 0x00300030u>(Y8, G8 << 2, magic);
        } else if (j == 2) {
          A0 = q6op<0x00F000F0u, 0x03000300u>(X, H << 4, magic);
          A1 = q6op<0x00F000F0u, 0x03000300u>(Y, G << 4, magic);
          A2 = q6op<0x00F000F0u, 0x03000300u>(X8, H8 << 4, magic);
          A3 = q6op<0x00F000F0u, 0x03000300u>(Y8, G8 << 4, magic);
        } else {
          A0 = q6op<0x00F000F0u, 0x03000300u>(X, H << 2, magic);
          A1 = q6op<0x00F000F0u, 0x03000300u>(Y, G << 2, magic);
          A2 = q6op<0x00F000F0u, 0x03000300u>(X8, H8 << 2, magic);
          A3 = q6op<0x00F000F0u, 0x03000300u>(Y8, G8 << 2, magic);
        }
        const uint32_t koff = 2u * (uint32_t)(128 * h + 32 * j + 16 * s) + 8u * (uint32_t)L.tig;
        float acc[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[nt][i] = 0.f;
          const uint2 b = lds64(xa[nt] + koff);
          mma16816(acc[nt], A0, A1, A2, A3, b.x, b.y);
        }
        // the scale of group grp (rows g, g+8) from lane t = grp / 4 of the quad
        const int src = quad | (grp >> 2);
        const float sa0 = __shfl_sync(0xffffffffu, aq[grp & 3], src);
        const float sa1 = __shfl_sync(0xffffffffu, ar[grp & 3], src);
        const float kf = j >= 2 ? 1024.0f + 32.0f * 16.0f : 1024.0f + 32.0f;
        const float sk0 = sa0 * kf, sk1 = sa1 * kf;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const uint2 sxw = lds64(sxa + 4u * (uint32_t)(grp * MT + 8 * nt + 2 * L.tig));
          const float sx0 = __uint_as_float(sxw.x), sx1 = __uint_as_float(sxw.y);
          y[nt][0] = fmaf(sa0, acc[nt][0], fmaf(-sk0, sx0, y[nt][0]));
          y[nt][1] = fmaf(sa0, acc[nt][1], fmaf(-sk0, sx1, y[nt][1]));
          y[nt][2] = fmaf(sa1, acc[nt][2], fmaf(-sk1, sx0, y[nt][2]));
          y[nt][3] = fmaf(sa1, acc[nt][3], fmaf(-sk1, sx1, y[nt][3]));
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------
// Sleep between polls of the producer's waits, in ns (0: poll back to back).
#ifndef QK_GEMV_BACKOFF_NS
#define QK_GEMV_BACKOFF_NS 0
#endif
constexpr uint32_t kBackoffNs = QK_GEMV_BACKOFF_NS;
// Compute warps per CTA; one more warp streams.  8 measured faster than 12
// or 16 in steady state (a layer's grouped launch 20.1 vs 20.6 and 21.5 us,
// a 131072 x 3072 Q4_K GEMV 49.4 vs 51.3 and 54.2 us).
#ifndef QK_DECODE_WARPS
#define QK_DECODE_WARPS 8
#endif
constexpr int kDW = QK_DECODE_WARPS;
constexpr int kDCompute = 32 * kDW;
constexpr int kDThreads = 32 * (kDW + 1);
constexpr uint32_t kXtBlock = 1024;  // x-table bytes per 256-weight block
constexpr uint32_t kZeroBytes = 1024;

constexpr uint32_t round128(size_t v) { return (uint32_t)((v + 127) / 128 * 128); }
// Sums table bytes per block: Q4_K [t][Sx, -1024 Sx, Sx', -1024 Sx'], Q6_K [h][t][4 fields].
constexpr uint32_t sx_block_bytes(int qtype) { return qtype == kQ4K ? 64u : 128u; }

struct GemvProb {
  const uint8_t* w[2];  // weights (gate for kind 1), up weights (kind 1)
  const uint16_t* x;
  void* y;
  int M;                // tokens (1 for the decode layout)
  const uint16_t* gamma;  // RMSNorm prologue: fp16 gamma[K], or null for none
  float eps;
  int N, K, qtype, kind;
  int pair;             // one tensor, whole rows: a stage holds two adjacent 16-row tiles
  int cb;               // K blocks per chunk (a stage holds 16 rows x cb blocks per weight tensor)
  int stages;           // pipeline depth of this problem's CTAs
  uint32_t stage_bytes;
  uint32_t ctl_off, red_off, ring_off;  // shared-memory layout of this problem's CTAs
  uint32_t rawx_off, gamma_off;         // where the bulk copies of x and gamma land
  int tiles, cta_begin, ctas;
};

struct GemvBatch {
  GemvProb p[kMaxGemvProbs];
  int count;
};

// RMSNorm prologue (DAMASCUS project overview, "[04] one decode step": an
// RMSNorm comes before the QKV projections and the SwiGLU FFN), over x staged
// in shared memory at xs: every compute thread sums the squares of its 8-value
// chunks c = tid, tid + 32 NW, ... of each token, the warps reduce them in a
// fixed shuffle tree into rss[m][warp], and after a barrier thread m adds the
// warps in order: rnorm[m] = 1 / sqrt(mean_k x[m][k]^2 + eps), fp32.
template <int NW>
__device__ void rms_partials(uint32_t xs, int M, int K, float* rss, int tid) {
  const int warp = tid >> 5, lane = tid & 31;
  const int nc = K / 8;
  for (int m = 0; m < M; ++m) {
    float ss = 0.f;
    for (int c = tid; c < nc; c += 32 * NW) {
      const uint4 v = lds128(xs + (uint32_t)m * (uint32_t)(2 * K) + 16u * c);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float a = half_lo(w[i]), b = half_lo(w[i] >> 16);
        ss = fmaf(b, b, fmaf(a, a, ss));
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) rss[m * NW + warp] = ss;
  }
}

// Four fp16 values of x (two words) times r * gamma, rounded to fp16.
__device__ __forceinline__ uint2 norm4(uint2 v, uint2 g, float r) {
  uint2 o;
  const __half2 a = __floats2half2_rn(half_lo(v.x) * r * half_lo(g.x), half_lo(v.x >> 16) * r * half_lo(g.x >> 16));
  const __half2 b = __floats2half2_rn(half_lo(v.y) * r * half_lo(g.y), half_lo(v.y >> 16) * r * half_lo(g.y >> 16));
  o.x = *reinterpret_cast<const uint32_t*>(&a);
  o.y = *reinterpret_cast<const uint32_t*>(&b);
  return o;
}

// Build the x table and the sums table of one problem from x staged in shared
// memory at xs (gs: gamma staged there too, or 0 for no RMSNorm prologue; all
// compute threads; the caller synchronises them afterwards).
//   Q4_K entry (block, word v, lane group t, e): base k = 64t + 32e + 4v.
//   Q6_K entry (block, v = 4h + 2P + u, t, e):   base k = 128h + 64P + 32e + 8t + 4u.
// An entry holds x[k], x[k+2] / x[k+1], x[k+3] as fp16 pairs: for e = 0 in
// words 0 and 2 (B half 0 of the MMAs p = 0, 1), for e = 1 in words 1 and 3.
template <int QT>
__device__ void build_x_table(uint32_t xs, uint32_t gs, const float* rnorm, int K, uint32_t xt, uint32_t sx,
                              uint32_t zero, int tid) {
  const int nb = K / kQK;
  const int nent = nb * 64;  // entries, each from 4 consecutive x values
  for (int i = tid; i < nent; i += kDCompute) {
    int blk, t, e, v, k;
    uint32_t dst;
    if constexpr (QT == kQ4K) {
      // i = ((blk * 4 + t) * 2 + e) * 8 + v: the 8 entries of one sub-block are adjacent lanes
      v = i & 7;
      e = (i >> 3) & 1;
      t = (i >> 4) & 3;
      blk = i >> 6;
      k = 64 * t + 32 * e + 4 * v;
      dst = xt + (uint32_t)blk * kXtBlock + 128u * v + 32u * t + 16u * e;
    } else {
      // i = ((((blk * 2 + h) * 2 + P) * 4 + t) * 2 + e) * 2 + u: the two entries of a field sum are adjacent
      const int u = i & 1;
      e = (i >> 1) & 1;
      t = (i >> 2) & 3;
      const int P = (i >> 4) & 1, h = (i >> 5) & 1;
      blk = i >> 6;
      v = 4 * h + 2 * P + u;
      k = 128 * h + 64 * P + 32 * e + 8 * t + 4 * u;
      dst = xt + (uint32_t)blk * kXtBlock + 128u * v + 32u * t + 16u * e;
    }
    const uint32_t off = 2u * (uint32_t)(blk * kQK + k);
    uint2 q = lds64(xs + off);
    if (gs) q = norm4(q, lds64(gs + off), rnorm[0]);
    const uint32_t p0 = prmt(q.x, q.y, 0x5410u), p1 = prmt(q.x, q.y, 0x7632u);  // (x0, x2), (x1, x3)
    if (e == 0)
      sts128_u(dst, p0, 0u, p1, 0u);
    else
      sts128_u(dst, 0u, p0, 0u, p1);
    float s = (half_lo(q.x) + half_lo(q.x >> 16)) + (half_lo(q.y) + half_lo(q.y >> 16));
    if constexpr (QT == kQ4K) {
      s += __shfl_xor_sync(0xffffffffu, s, 1);
      s += __shfl_xor_sync(0xffffffffu, s, 2);
      s += __shfl_xor_sync(0xffffffffu, s, 4);
      if (v == 0) {
        const uint32_t a = sx + (uint32_t)blk * 64u + 16u * t + 8u * e;
        asm volatile("st.shared.v2.f32 [%0], {%1, %2};" ::"r"(a), "f"(s), "f"(-1024.0f * s) : "memory");
      }
    } else {
      s += __shfl_xor_sync(0xffffffffu, s, 1);
      if ((i & 1) == 0) {
        const int P = (i >> 4) & 1, h = (i >> 5) & 1;
        const float c = P ? -(1024.0f + 32.0f * 16.0f) : -(1024.0f + 32.0f);
        const uint32_t a = sx + (uint32_t)blk * 128u + 64u * h + 16u * t + 4u * (2 * P + e);
        asm volatile("st.shared.f32 [%0], %1;" ::"r"(a), "f"(c * s) : "memory");
      }
    }
  }
  for (int i = tid; i < (int)(kZeroBytes / 16); i += kDCompute) sts128_u(zero + 16u * i, 0u, 0u, 0u, 0u);
}

// Several tokens: token m's x (bulk-copied to xt + 2K m) rearranged in place
// into k-permuted fp16 pairs, xp_m[k/4] = { (x[k], x[k+2]), (x[k+1], x[k+3]) },
// and the sums table
// [block][sub-block (Q4_K, 32 weights) or scale group (Q6_K, 16)][MT tokens]
// (zero for tokens beyond M).
template <int QT, int MT>
__device__ void build_x_table_tn(uint32_t gs, const float* rnorm, int M, int K, uint32_t xt, uint32_t sx,
                                 uint32_t zero, int tid) {
  constexpr int kSub = QT == kQ4K ? 8 : 16;      // sums per block
  constexpr int kPer = QT == kQ4K ? 8 : 4;       // 4-value groups per sum
  const int nq = K / 4;
  for (int i = tid; i < M * nq; i += kDCompute) {  // nq is a multiple of 64: a warp never straddles tokens
    const int m = i / nq, q = i - m * nq;
    const uint32_t a = xt + (uint32_t)m * (uint32_t)(2 * K) + 8u * q;  // x copied here; rearranged in place
    uint2 v = lds64(a);
    if (gs) v = norm4(v, lds64(gs + 8u * q), rnorm[m]);
    asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(a), "r"(prmt(v.x, v.y, 0x5410u)),
                 "r"(prmt(v.x, v.y, 0x7632u))
                 : "memory");
    float s = (half_lo(v.x) + half_lo(v.x >> 16)) + (half_lo(v.y) + half_lo(v.y >> 16));
    s += __shfl_xor_sync(0xffffffffu, s, 1);
    s += __shfl_xor_sync(0xffffffffu, s, 2);
    if (kPer == 8) s += __shfl_xor_sync(0xffffffffu, s, 4);
    if ((q & (kPer - 1)) == 0) {
      const int sub = q / kPer;  // global sub-block / group index: block sub / kSub, slot sub % kSub
      asm volatile("st.shared.f32 [%0], %1;" ::"r"(sx + 4u * (uint32_t)(sub * MT + m)), "f"(s) : "memory");
    }
  }
  const int nsums = (K / kQK) * kSub;
  for (int i = tid; i < nsums * (MT - M); i += kDCompute) {
    const int sub = i / (MT - M), m = M + i % (MT - M);
    asm volatile("st.shared.f32 [%0], %1;" ::"r"(sx + 4u * (uint32_t)(sub * MT + m)), "f"(0.0f) : "memory");
  }
  for (int i = tid; i < (int)(kZeroBytes / 16); i += kDCompute) sts128_u(zero + 16u * i, 0u, 0u, 0u, 0u);
}

// ---------------------------------------------------------------------------
// The kernel (MT token slots: 1 or 8)
// ---------------------------------------------------------------------------
// A producer warp streams stages into a ring with bulk copies of whole
// 16-row tiles (two adjacent tiles of one tensor, or the gate and the up tile,
// per stage), or of 16-row x cb-block chunks with one copy per row: a few
// large copies per stage keep the copy engine and DRAM efficient.  A unit is
// 16 rows x one 256-weight block of one tensor; compute warp w takes the
// units of block j = w, w + kDW, ... of every tile, so each warp's share of a
// tile is fixed by j alone.  A warp adds its units in j order, leaves its row
// (x token) sums of a finished tile in the stage's partials slot, and
// releases the stage.  Before refilling a stage the producer adds the kDW warps' sums of
// the tile(s) it held, in warp order, and writes y (fp32, or fp16
// silu(gate) * up).  No atomic and no barrier among compute warps: each only
// waits for its stage to land.  The order of every addition depends on the
// problem's shape only, so a problem launched alone or grouped gives the same
// bits.
constexpr int kDMaxStages = 8;
#ifndef QK_DECODE_PDL
#define QK_DECODE_PDL 1
#endif
#ifndef QK_DECODE_PIECE
#define QK_DECODE_PIECE 8192
#endif
constexpr uint32_t kDPiece = QK_DECODE_PIECE;  // bytes per bulk copy of a whole-row stage

struct DecodeCtl {
  uint64_t full[kDMaxStages];   // stage landed (producer arrival + copy bytes)
  uint64_t empty[kDMaxStages];  // stage released by the kDW compute warps
  uint64_t x_full;              // x (and gamma) copied into shared memory
  uint32_t abort_flag;
  float rnorm[kMaxGemvM];       // RMSNorm prologue: 1 / sqrt(mean(x^2) + eps) per token
  float rss[kMaxGemvM][kDW];    // its per-warp sums of squares
};

// ---------------------------------------------------------------------------
// Q8 activations (one token): x is quantized per block of 32 to int8 with one
// fp32 scale, d = amax / 127 and q = round(x / d) (IEEE fp32 division, ties
// away from zero, clamped to +-127; d = 0 gives q = 0), and the products run
// as integer dot products (dp4a: four int8 x times four quant bytes, int32
// sum).  Per sub-block (Q4_K) or scale group (Q6_K) the integer sum is scaled
// once in fp32.  x table: the int8 x in k order (K bytes), then per 32-block
// {d, sum of q over its first 16 k, over its last 16, 0} (16 bytes).
// ---------------------------------------------------------------------------
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

__device__ void build_x_table_q8(uint32_t xs, int K, uint32_t xq, uint32_t dt, int tid) {
  const int warp = tid >> 5, lane = tid & 31;
  for (int b = warp; b < K / 32; b += kDW) {
    uint32_t h;
    asm volatile("ld.shared.u16 %0, [%1];" : "=r"(h) : "r"(xs + 2u * (uint32_t)(32 * b + lane)));
    const float v = half_lo(h);
    float a = fabsf(v);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    const float d = __fdiv_rn(a, 127.0f);
    int q = 0;
    if (d != 0.0f) q = (int)fminf(fmaxf(roundf(__fdiv_rn(v, d)), -127.0f), 127.0f);
    asm volatile("st.shared.s8 [%0], %1;" ::"r"(xq + (uint32_t)(32 * b + lane)), "r"(q) : "memory");
    int s = q;
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);  // within each half of the warp
    if (lane == 0) {
      asm volatile("st.shared.v2.f32 [%0], {%1, %2};" ::"r"(dt + 16u * (uint32_t)b), "f"(d), "f"((float)s)
                   : "memory");
    } else if (lane == 16) {
      asm volatile("st.shared.v2.f32 [%0], {%1, %2};" ::"r"(dt + 16u * (uint32_t)b + 8u), "f"((float)s), "f"(0.0f)
                   : "memory");
    }
  }
}

// One Q4_K block of row r (address rb), lane half s (sub-blocks 4s .. 4s+3):
// y += sum over those sub-blocks of d_x * (d*sc*IDOT - dmin*m*ISUM).
__device__ __forceinline__ void q4_block_q8(uint32_t rb, uint32_t xa, uint32_t da, int s, float& y) {
  const uint4 h = lds128(rb);
  uint4 w4[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) w4[i] = lds128(rb + 16u + 64u * (uint32_t)s + 16u * (uint32_t)i);
  uint4 x4[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) x4[i] = lds128(xa + 16u * (uint32_t)i);
  float4 D[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) D[i] = ldsf4(da + 16u * (uint32_t)i);
  const uint32_t w[16] = {w4[0].x, w4[0].y, w4[0].z, w4[0].w, w4[1].x, w4[1].y, w4[1].z, w4[1].w,
                          w4[2].x, w4[2].y, w4[2].z, w4[2].w, w4[3].x, w4[3].y, w4[3].z, w4[3].w};
  const uint32_t X[32] = {x4[0].x, x4[0].y, x4[0].z, x4[0].w, x4[1].x, x4[1].y, x4[1].z, x4[1].w,
                          x4[2].x, x4[2].y, x4[2].z, x4[2].w, x4[3].x, x4[3].y, x4[3].z, x4[3].w,
                          x4[4].x, x4[4].y, x4[4].z, x4[4].w, x4[5].x, x4[5].y, x4[5].z, x4[5].w,
                          x4[6].x, x4[6].y, x4[6].z, x4[6].w, x4[7].x, x4[7].y, x4[7].z, x4[7].w};
  int acc[4] = {0, 0, 0, 0};  // sub-blocks 4s + t
#pragma unroll
  for (int v = 0; v < 8; ++v) {
    const uint32_t a = w[v], b = w[8 + v];  // groups 2s and 2s+1, bytes 4v .. 4v+3
    acc[0] = dp4a_us(a & 0x0F0F0F0Fu, X[v], acc[0]);
    acc[1] = dp4a_us((a >> 4) & 0x0F0F0F0Fu, X[8 + v], acc[1]);
    acc[2] = dp4a_us(b & 0x0F0F0F0Fu, X[16 + v], acc[2]);
    acc[3] = dp4a_us((b >> 4) & 0x0F0F0F0Fu, X[24 + v], acc[3]);
  }
  const float d = half_lo(h.x), dmin = half_lo(h.x >> 16);
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    // sub-block j = 4s + t: bytes s[0..3] = h.y, s[4..7] = h.z, s[8..11] = h.w
    uint32_t sc, m;
    if (s == 0) {
      sc = (h.y >> (8 * t)) & 63u;
      m = (h.z >> (8 * t)) & 63u;
    } else {
      sc = ((h.w >> (8 * t)) & 15u) | (((h.y >> (8 * t + 6)) & 3u) << 4);
      m = ((h.w >> (8 * t + 4)) & 15u) | (((h.z >> (8 * t + 6)) & 3u) << 4);
    }
    const float dsc = d * (float)sc, dmn = dmin * (float)m;
    y = fmaf(D[t].x, fmaf(dsc, (float)acc[t], -dmn * (D[t].y + D[t].z)), y);
  }
}

// Two consecutive words at shared address a (4-byte aligned, or 2 mod 4).
__device__ __forceinline__ void lds_pair(uint32_t a, bool a2, uint32_t& w0, uint32_t& w1) {
  if (!a2) {
    w0 = lds32(a);
    w1 = lds32(a + 4);
  } else {
    const uint32_t t0 = lds32(a - 2), t1 = lds32(a + 2), t2 = lds32(a + 6);
    w0 = __funnelshift_r(t0, t1, 16);
    w1 = __funnelshift_r(t1, t2, 16);
  }
}

// One Q6_K block of row r (address rb), lane half h (weights 128h .. 128h+127,
// scale groups 8h .. 8h+7): y += sum over the 8 groups of
// d_x * d * sc * (IDOT(q6 + 32) - 32 * ISUM).
__device__ __forceinline__ void q6_block_q8(uint32_t rb, uint32_t xa, uint32_t da, int h, float& y) {
  const bool a2 = (rb & 3u) != 0;
  uint32_t A[8], B[8], H[8];
#pragma unroll
  for (int v = 0; v < 8; v += 2) {
    lds_pair(rb + 64u * (uint32_t)h + 4u * (uint32_t)v, a2, A[v], A[v + 1]);
    lds_pair(rb + 64u * (uint32_t)h + 32u + 4u * (uint32_t)v, a2, B[v], B[v + 1]);
    lds_pair(rb + 128u + 32u * (uint32_t)h + 4u * (uint32_t)v, a2, H[v], H[v + 1]);
  }
  uint32_t S[2], dw0, dw1;
  lds_pair(rb + 192u + 8u * (uint32_t)h, a2, S[0], S[1]);
  lds_pair(rb + 204u, a2, dw0, dw1);  // bytes 204..211: d is bytes 208..209
  uint4 x4[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) x4[i] = lds128(xa + 16u * (uint32_t)i);
  float4 D[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) D[i] = ldsf4(da + 16u * (uint32_t)i);
  const uint32_t X[32] = {x4[0].x, x4[0].y, x4[0].z, x4[0].w, x4[1].x, x4[1].y, x4[1].z, x4[1].w,
                          x4[2].x, x4[2].y, x4[2].z, x4[2].w, x4[3].x, x4[3].y, x4[3].z, x4[3].w,
                          x4[4].x, x4[4].y, x4[4].z, x4[4].w, x4[5].x, x4[5].y, x4[5].z, x4[5].w,
                          x4[6].x, x4[6].y, x4[6].z, x4[6].w, x4[7].x, x4[7].y, x4[7].z, x4[7].w};
  int acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};  // [field g6][half of l]
#pragma unroll
  for (int v = 0; v < 8; ++v) {
    const int hl = v >> 2;
    const uint32_t a = A[v], b = B[v], q = H[v];
    // 6-bit quants + 32 of fields 0..3 for l = 4v .. 4v+3, as unsigned bytes
    const uint32_t q0 = (a & 0x0F0F0F0Fu) | ((q << 4) & 0x30303030u);
    const uint32_t q1 = (b & 0x0F0F0F0Fu) | ((q << 2) & 0x30303030u);
    const uint32_t q2 = ((a >> 4) & 0x0F0F0F0Fu) | (q & 0x30303030u);
    const uint32_t q3 = ((b >> 4) & 0x0F0F0F0Fu) | ((q >> 2) & 0x30303030u);
    acc[0 + hl] = dp4a_us(q0, X[v], acc[0 + hl]);
    acc[2 + hl] = dp4a_us(q1, X[8 + v], acc[2 + hl]);
    acc[4 + hl] = dp4a_us(q2, X[16 + v], acc[4 + hl]);
    acc[6 + hl] = dp4a_us(q3, X[24 + v], acc[6 + hl]);
  }
  const float d = half_lo(dw1);  // bytes 208..209 are the low half of the second word
#pragma unroll
  for (int g6 = 0; g6 < 4; ++g6) {
#pragma unroll
    for (int hl = 0; hl < 2; ++hl) {
      const int gi = 2 * g6 + hl;  // scale group 8h + gi
      const int sc = (int)(int8_t)((S[gi >> 2] >> (8 * (gi & 3))) & 0xFFu);
      const float isum = hl ? D[g6].z : D[g6].y;
      y = fmaf(D[g6].x * (d * (float)sc), fmaf(-32.0f, isum, (float)acc[2 * g6 + hl]), y);
    }
  }
}

__device__ __forceinline__ float quad_sum(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 1);
  return v + __shfl_xor_sync(0xffffffffu, v, 2);
}

// Stage geometry of a decode problem (P.pair: two tiles of one tensor per
// stage; P.cb: blocks per stage and row, nb for whole rows).
template <int QT, int MT, bool Q8X>
__device__ __forceinline__ void decode_problem(const GemvProb& P, int cta, uint8_t* smem) {
  static_assert(!Q8X || MT == 1, "int8 activations: one token");
  constexpr int kBB = QT == kQ4K ? kQ4KBytes : kQ6KBytes;
  constexpr int NT = MT / 8;  // several tokens: 8-token n-tiles of the MMA
  const int K = P.K, N = P.N, nb = K / kQK, cb = P.cb, S = P.stages;
  const int nten = 1 + P.kind, pair = P.pair;
  const int ncomb = pair ? 2 : nten;  // row sets per stage: two tiles, or gate and up
  const int redw = ncomb * 16 * MT;   // partial floats per warp and stage
  const int64_t RB = (int64_t)nb * kBB;
  const int nchunks = nb / cb;
  const uint32_t SB = P.stage_bytes;
  const uint32_t comb_bytes = (uint32_t)(16 * cb * kBB);  // one row set's share of a stage
  const uint32_t pitch = cb == nb ? (uint32_t)RB : (uint32_t)(cb * kBB);
  const int tps = pair ? 2 : 1;  // tiles per stage
  const int t0 = (int)((int64_t)cta * P.tiles / P.ctas), t1 = (int)((int64_t)(cta + 1) * P.tiles / P.ctas);
  const int groups = (t1 - t0 + tps - 1) / tps;  // stages' worth of tiles
  const int steps = groups * nchunks;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  DecodeCtl* ctl = reinterpret_cast<DecodeCtl*>(smem + P.ctl_off);
  const uint32_t base = smem_u32(smem);
  uint8_t* const ring = smem + P.ring_off;
  // partials: [S][kDW][row set (ncomb)][16 rows][MT tokens], as the plan sizes them
  float* const red = reinterpret_cast<float*>(smem + P.red_off);
  const int M = P.M;
  void* const yout = P.y;

  if (tid < S) {
    mbar_init(&ctl->full[tid], 1);
    mbar_init(&ctl->empty[tid], kDW);
  }
  if (tid == 0) {
    ctl->abort_flag = 0u;
    mbar_init(&ctl->x_full, 1);
  }
  fence_mbar_init();
  __syncthreads();

  if (warp == kDW) {
    // ------------------------------------------------------------ producer
    // Lane 0 copies; all lanes add the partial sums of finished tiles.
    auto finish = [&](int st) {  // the tile(s) of step st, if its chunk was the last
      const int s = st % S, g = st / nchunks;
      if (st % nchunks != nchunks - 1) return;
      const float* q = red + (size_t)s * (kDW * redw);
      // output (row set c, row r, token m) at lane + 32 i
      for (int o = lane; o < ncomb * 16 * MT; o += 32) {
        const int c = o / (16 * MT), r = (o / MT) % 16, m = o % MT;
        const int tile = t0 + g * tps + (pair ? c : 0);
        const int n = tile * 16 + r;
        if (m >= M || n >= N || tile >= t1 || (nten == 2 && c == 1)) continue;
        float v = 0.f;
        for (int w = 0; w < kDW; ++w) v += q[w * redw + o];
        if (nten == 2) {
          float u = 0.f;
          for (int w = 0; w < kDW; ++w) u += q[w * redw + 16 * MT + o];
          static_cast<__half*>(yout)[(size_t)m * N + n] = __float2half_rn(v / (1.0f + __expf(-v)) * u);
        } else {
          static_cast<float*>(yout)[(size_t)m * N + n] = v;
        }
      }
    };
    bool ok = true;
    // Copies of step st into stage st % S, issued from several lanes at once
    // (the copy engine works on several requests in parallel): whole rows as
    // pieces of at most kDPiece bytes of each tensor's span, chunks as one row
    // per lane.  The compute warps read a stage with plain loads; its refill
    // is an async-proxy write, ordered after their reads by the proxy fence.
    auto issue = [&](int st) {
      const int s = st % S;
      const int g = st / nchunks, chunk = st % nchunks;
      const int n0 = (t0 + g * tps) * 16;
      uint8_t* dst = ring + (size_t)s * SB;
      if (cb == nb) {
        // whole rows: a tensor's rows n0 .. n0 + rows - 1 are one span
        const int rows = min(16 * tps, min(t1 * 16, N) - n0);
        const int64_t span = (int64_t)rows * RB;
        const uint32_t bulk = (uint32_t)(span & ~int64_t(15));
        const int np = (int)((bulk + kDPiece - 1) / kDPiece);  // pieces per tensor
        if (lane == 0) {
          for (int t = 0; t < nten; ++t) {
            const uint8_t* src = (t ? P.w[1] : P.w[0]) + (int64_t)n0 * RB;
            uint8_t* d = dst + (size_t)t * comb_bytes;
            for (int64_t b = bulk; b < span; b += 2)  // the tensor's last bytes (span % 16 != 0)
              *reinterpret_cast<uint16_t*>(d + b) = *reinterpret_cast<const uint16_t*>(src + b);
          }
          mbar_arrive_expect_tx(&ctl->full[s], bulk * (uint32_t)nten);
        }
        __syncwarp();
        for (int i = lane; i < np * nten; i += 32) {
          const int t = i / np, pc = i - t * np;
          const uint32_t o = (uint32_t)pc * kDPiece, len = min(kDPiece, bulk - o);
          fence_proxy_async_smem();
          bulk_copy_g2s(dst + (size_t)t * comb_bytes + o, (t ? P.w[1] : P.w[0]) + (int64_t)n0 * RB + o, len,
                        &ctl->full[s]);
        }
      } else {
        // a K chunk: one copy per row of cb blocks (16-byte aligned by construction)
        const int rows = min(16, N - n0);
        const uint32_t row_bytes = (uint32_t)(cb * kBB);
        if (lane == 0) mbar_arrive_expect_tx(&ctl->full[s], row_bytes * (uint32_t)(rows * nten));
        __syncwarp();
        for (int i = lane; i < rows * nten; i += 32) {
          const int t = i / rows, r = i - t * rows;
          fence_proxy_async_smem();
          bulk_copy_g2s(dst + (size_t)t * comb_bytes + (size_t)r * row_bytes,
                        (t ? P.w[1] : P.w[0]) + (int64_t)(n0 + r) * RB + (int64_t)chunk * cb * kBB, row_bytes,
                        &ctl->full[s]);
        }
      }
    };
    int issued = 0;
#if QK_DECODE_PDL
    // Launched as a programmatic dependent: the next kernel may be scheduled
    // now (it waits for this grid before touching memory), and this warp, the
    // only one that touches global memory, reads weights, x and gamma and
    // writes y only after the grids this one depends on have finished.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
#endif
    if (lane == 0) {
      // one token: x lands in its own buffer for the x-table build; several:
      // x lands in the table area and is rearranged in place
      const uint32_t xbytes = (uint32_t)(2 * K) * (uint32_t)M, gbytes = P.gamma ? (uint32_t)(2 * K) : 0u;
      mbar_arrive_expect_tx(&ctl->x_full, xbytes + gbytes);
      bulk_copy_g2s(smem + P.rawx_off, P.x, xbytes, &ctl->x_full);
      if (gbytes) bulk_copy_g2s(smem + P.gamma_off, P.gamma, gbytes, &ctl->x_full);
    }
    for (int st = 0; st < steps; ++st) {
      const int s = st % S;
      if (st >= S) {
        ok = ok && mbar_wait<kBackoffNs>(&ctl->empty[s], (uint32_t)((st / S) - 1) & 1u, &ctl->abort_flag,
                                          &g_gemv_status);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        finish(st - S);
        __syncwarp();
      }
      issue(st);
      ++issued;
      __syncwarp();
    }
    // the last stages: wait for their release, then finish their tiles
    for (int st = max(0, steps - S); ok && st < steps; ++st) {
      ok = ok && mbar_wait<kBackoffNs>(&ctl->empty[st % S], (uint32_t)(st / S) & 1u, &ctl->abort_flag,
                                        &g_gemv_status);
      ok = __all_sync(0xffffffffu, ok);
      if (ok) finish(st);
      __syncwarp();
    }
    if (lane == 0 && !ok) {
      // drain: copies still in flight land before the CTA exits
      for (int i = 1; i <= S && i <= issued; ++i)
        mbar_wait(&ctl->full[(issued - i) % S], (uint32_t)((issued - i) / S) & 1u, &ctl->abort_flag, &g_gemv_status,
                  true);
    }
    return;
  }

  // -------------------------------------------------------------- compute
  const uint32_t xs = base + P.rawx_off, gs = P.gamma ? base + P.gamma_off : 0u;
  const uint32_t zero = base + P.ctl_off - kZeroBytes;
  // the sums table follows the x table: nb KB of B operands (one token), or
  // the k-permuted x of MT tokens
  const uint32_t sxt = base + (MT == 1 ? (uint32_t)nb * kXtBlock : (uint32_t)MT * (uint32_t)(2 * K));
  bool ok = mbar_wait(&ctl->x_full, 0u, &ctl->abort_flag, &g_gemv_status);
  if (P.gamma) {
    rms_partials<kDW>(xs, M, K, &ctl->rss[0][0], tid);
    asm volatile("bar.sync 1, %0;" ::"n"(kDCompute) : "memory");
    if (tid < M) {
      float t = 0.f;
      for (int w = 0; w < kDW; ++w) t += ctl->rss[tid][w];
      ctl->rnorm[tid] = 1.0f / sqrtf(t / (float)K + P.eps);
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kDCompute) : "memory");
  }
  if constexpr (Q8X)
    build_x_table_q8(xs, K, base, base + (uint32_t)K, tid);
  else if constexpr (MT == 1)
    build_x_table<QT>(xs, gs, ctl->rnorm, K, base, sxt, zero, tid);
  else
    build_x_table_tn<QT, MT>(gs, ctl->rnorm, M, K, base, sxt, zero, tid);
  asm volatile("bar.sync 1, %0;" ::"n"(kDCompute) : "memory");

  Lane L;
  L.g = lane >> 2;
  L.tig = lane & 3;
  L.hi = L.tig >= 2;
  L.sh = 16u * (uint32_t)(L.tig & 1);
  L.shA = L.sh + (L.hi ? 2u : 0u);
  L.shL = L.sh + (L.hi ? 4u : 0u);
  uint32_t magic, fmagic;
  asm volatile("mov.b32 %0, %1;" : "=r"(magic) : "n"(kMagic));
  asm volatile("mov.b32 %0, %1;" : "=r"(fmagic) : "n"(kFMagic));
  const uint32_t ring_s = base + P.ring_off + (uint32_t)L.g * pitch;

  if constexpr (Q8X) {
    // lane (r, s): row r of the 16, weights 128s .. 128s+127 of every block
    const int r = lane & 15, hs = lane >> 4;
    const uint32_t ring_r = base + P.ring_off + (uint32_t)r * pitch;
    const uint32_t xq = base + 128u * (uint32_t)hs, dq = base + (uint32_t)K + 64u * (uint32_t)hs;
    float a0 = 0.f, a1 = 0.f;  // row r of row set 0, of row set 1 (this half)
    for (int st = 0; st < steps; ++st) {
      const int s = st % S, chunk = st % nchunks;
      if (ok) ok = mbar_wait(&ctl->full[s], (uint32_t)(st / S) & 1u, &ctl->abort_flag, &g_gemv_status);
      const int j0 = chunk * cb;
      int b = warp - j0 % kDW;
      if (b < 0) b += kDW;
      const uint32_t stg = ring_r + (uint32_t)s * SB;
      for (; ok && b < cb; b += kDW) {
        const int j = j0 + b;
        const uint32_t rb = stg + (uint32_t)(b * kBB);
        const uint32_t xa = xq + 256u * (uint32_t)j, da = dq + 128u * (uint32_t)j;
        if constexpr (QT == kQ4K) {
          q4_block_q8(rb, xa, da, hs, a0);
          if (ncomb == 2) q4_block_q8(rb + comb_bytes, xa, da, hs, a1);
        } else {
          q6_block_q8(rb, xa, da, hs, a0);
          if (ncomb == 2) q6_block_q8(rb + comb_bytes, xa, da, hs, a1);
        }
      }
      if (chunk == nchunks - 1) {
        const float p0 = a0 + __shfl_xor_sync(0xffffffffu, a0, 16), p1 = a1 + __shfl_xor_sync(0xffffffffu, a1, 16);
        if (lane < 16) {
          float* q = red + ((size_t)s * kDW + warp) * redw;
          q[r] = p0;
          if (ncomb == 2) q[16 + r] = p1;
        }
        a0 = a1 = 0.f;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->empty[s]);
    }
  } else if constexpr (MT == 1) {
    {
      const int e = L.g & 1;
      const bool reads_x = (L.g >> 1) == L.tig;
      L.xt_off = reads_x ? 32u * (uint32_t)L.tig + 16u * (uint32_t)e : 32u * (uint32_t)(((L.g >> 1) + 2) & 3);
      L.xt_stride = reads_x ? kXtBlock : 0u;
    }
    {
      const uint32_t sv = (uint32_t)(L.tig >> 1);
      L.sel0 = 0x7440u | sv;
      L.sel1 = 0x7440u | (sv + 2);
    }
    const uint32_t xt_lane = (L.xt_stride ? base : zero) + L.xt_off;
    const uint32_t sx_lane = sxt + 16u * (uint32_t)L.tig;
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;  // rows g, g+8 of row set 0, then of row set 1
    for (int st = 0; st < steps; ++st) {
      const int s = st % S, chunk = st % nchunks;
      if (ok) ok = mbar_wait(&ctl->full[s], (uint32_t)(st / S) & 1u, &ctl->abort_flag, &g_gemv_status);
      // this warp's blocks of the chunk: j = chunk * cb + b with j mod kDW = warp
      const int j0 = chunk * cb;
      int b = warp - j0 % kDW;
      if (b < 0) b += kDW;
      const uint32_t stg = ring_s + (uint32_t)s * SB;
      for (; ok && b < cb; b += kDW) {
        const int j = j0 + b;
        const uint32_t r0 = stg + (uint32_t)(b * kBB);
        const uint32_t xa = xt_lane + (uint32_t)j * L.xt_stride;
        const uint32_t sxa = sx_lane + (uint32_t)j * sx_block_bytes(QT);
        if constexpr (QT == kQ4K) {
          q4_block(r0, r0 + 8u * pitch, xa, sxa, L, magic, fmagic, a0, a1);
          if (ncomb == 2) q4_block(r0 + comb_bytes, r0 + comb_bytes + 8u * pitch, xa, sxa, L, magic, fmagic, a2, a3);
        } else {
          q6_block(r0, r0 + 8u * pitch, xa, sxa, L, magic, fmagic, a0, a1);
          if (ncomb == 2) q6_block(r0 + comb_bytes, r0 + comb_bytes + 8u * pitch, xa, sxa, L, magic, fmagic, a2, a3);
        }
      }
      if (chunk == nchunks - 1) {
        // tile(s) done: this warp's row sums to the stage's partials slot
        const float p0 = quad_sum(a0), p1 = quad_sum(a1), p2 = quad_sum(a2), p3 = quad_sum(a3);
        if (L.tig == 0) {
          float* q = red + ((size_t)s * kDW + warp) * redw;
          q[L.g] = p0;
          q[L.g + 8] = p1;
          if (ncomb == 2) {
            q[16 + L.g] = p2;
            q[16 + L.g + 8] = p3;
          }
        }
        a0 = a1 = a2 = a3 = 0.f;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->empty[s]);
    }
  } else {
    // Several tokens: lane (g, t) supplies B for token 8 nt + g of n-tile nt
    // (the zero region for a token beyond M) and accumulates rows g, g+8 x
    // tokens 8 nt + 2t, 8 nt + 2t + 1 of each row set; every k-slot of an MMA
    // lies in one sub-block, so no lanes are summed afterwards.
    uint32_t xbase[NT], xstride[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int tok = 8 * nt + L.g;
      xbase[nt] = tok < M ? base + (uint32_t)tok * (uint32_t)(2 * K) : zero;
      xstride[nt] = tok < M ? 2u * kQK : 0u;
    }
    constexpr int kSub = QT == kQ4K ? 8 : 16;
    float ya[NT][4], yb[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) ya[nt][i] = yb[nt][i] = 0.f;
    for (int st = 0; st < steps; ++st) {
      const int s = st % S, chunk = st % nchunks;
      if (ok) ok = mbar_wait(&ctl->full[s], (uint32_t)(st / S) & 1u, &ctl->abort_flag, &g_gemv_status);
      const int j0 = chunk * cb;
      int b = warp - j0 % kDW;
      if (b < 0) b += kDW;
      const uint32_t stg = ring_s + (uint32_t)s * SB;
      for (; ok && b < cb; b += kDW) {
        const int j = j0 + b;
        const uint32_t r0 = stg + (uint32_t)(b * kBB);
        uint32_t xa[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) xa[nt] = xbase[nt] + (uint32_t)j * xstride[nt];
        const uint32_t sxa = sxt + (uint32_t)j * (uint32_t)(kSub * MT * 4);
        if constexpr (QT == kQ4K) {
          q4_block_tn<NT>(r0, r0 + 8u * pitch, xa, sxa, L, lane, magic, fmagic, ya);
          if (ncomb == 2)
            q4_block_tn<NT>(r0 + comb_bytes, r0 + comb_bytes + 8u * pitch, xa, sxa, L, lane, magic, fmagic, yb);
        } else {
          q6_block_tn<NT>(r0, r0 + 8u * pitch, xa, sxa, L, lane, magic, ya);
          if (ncomb == 2) q6_block_tn<NT>(r0 + comb_bytes, r0 + comb_bytes + 8u * pitch, xa, sxa, L, lane, magic, yb);
        }
      }
      if (chunk == nchunks - 1) {
        float* q = red + ((size_t)s * kDW + warp) * redw;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int row = L.g + 8 * (i >> 1), tok = 8 * nt + 2 * L.tig + (i & 1);
            q[row * MT + tok] = ya[nt][i];
            if (ncomb == 2) q[16 * MT + row * MT + tok] = yb[nt][i];
            ya[nt][i] = yb[nt][i] = 0.f;
          }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->empty[s]);
    }
  }
}

template <int MT, bool Q8X>
__global__ void __launch_bounds__(kDThreads, 1) gemv_decode_kernel(const __grid_constant__ GemvBatch B) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  int i = 0;
  while (i + 1 < B.count && (int)blockIdx.x >= B.p[i + 1].cta_begin) ++i;
  const GemvProb& P = B.p[i];
  const int cta = (int)blockIdx.x - P.cta_begin;
  if (P.qtype == kQ4K)
    decode_problem<kQ4K, MT, Q8X>(P, cta, smem);
  else
    decode_problem<kQ6K, MT, Q8X>(P, cta, smem);
}

}  // namespace

int gemv_max_m() { return kMaxGemvM; }

uint32_t gemv_take_status() {
  uint32_t v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_gemv_status, sizeof(v)) != cudaSuccess) return 0;
  cudaMemcpyToSymbol(g_gemv_status, &zero, sizeof(zero));
  v |= take_debug_status();
  return v;
}

namespace {

constexpr size_t kGemvSmem = 227 * 1024;
// Relative compute cost per packed byte, for splitting CTAs among the problems
// of a grouped launch: a Q6_K block's 6-bit assembly takes ~1.4x the logic
// instructions per byte of a Q4_K block, and a decode CTA streams Q6_K at
// 0.5-0.75x its Q4_K rate (per-CTA timelines on GB300: 18-26 vs 34 GB/s);
// 1.7 balanced the grouped decode layer best.
#ifndef QK_Q6_COST
#define QK_Q6_COST 1.7
#endif
constexpr double kQ6CostPerByte = QK_Q6_COST;

// The token slots of the kernel that runs M tokens: 1 (decode layout) or 8.
int slots_for(int64_t M) { return M <= 1 ? 1 : 8; }

// The plan of one problem, from its shape only (so grouping problems never
// changes how one of them is computed).  Layout:
//   one token:     [x table | sums | zero region | control | x | gamma | partials[S] | ring[S]]
//   several (MT):  [k-permuted x of MT tokens | sums | zero region | control | gamma | partials[S] | ring[S]]
// (several tokens: x is copied straight into the table area and rearranged
// in place).  Stage geometry, first that fits: two adjacent whole tiles of
// one tensor per stage (one token only) with at least 3 stages; whole tiles
// (gate and up together) with 3; the largest 16-byte-aligned chunk of cb
// blocks with 4, then 3; then the same with 2 stages (several tokens: with 2
// stages from the start).
bool plan_decode_problem(const GemvDesc& d, GemvProb& P, size_t* smem_out) {
  memset(&P, 0, sizeof(P));
  if (d.M < 1 || d.M > kMaxGemvM || d.N <= 0 || d.N >= ((int64_t)1 << 31) || d.K <= 0 || d.K % kQK != 0 ||
      d.K >= ((int64_t)1 << 31))
    return false;
  P.w[0] = static_cast<const uint8_t*>(d.w0);
  P.w[1] = static_cast<const uint8_t*>(d.w1);
  P.x = d.x;
  P.y = d.y;
  P.M = (int)d.M;
  P.gamma = d.gamma;
  P.eps = d.eps;
  P.N = (int)d.N;
  P.K = (int)d.K;
  P.qtype = d.qtype;
  P.kind = d.w1 ? 1 : 0;
  const int mt = slots_for(d.M);
  const int nb = P.K / kQK, nten = 1 + P.kind;
  const int bb = P.qtype == kQ4K ? kQ4KBytes : kQ6KBytes;
  const int64_t RB = (int64_t)nb * bb;
  P.tiles = (P.N + 15) / 16;
  if (d.q8x && (mt != 1 || d.gamma)) return false;  // int8 activations: one token, no RMSNorm prologue
  const size_t xt = d.q8x   ? round128((size_t)P.K + (size_t)(P.K / 32) * 16)
                    : mt == 1 ? round128((size_t)nb * (kXtBlock + sx_block_bytes(P.qtype)))
                              : round128((size_t)mt * 2 * P.K + (size_t)nb * (P.qtype == kQ4K ? 8 : 16) * mt * 4);
  P.ctl_off = (uint32_t)(xt + kZeroBytes);
  const uint32_t after_ctl = P.ctl_off + round128(sizeof(DecodeCtl));
  P.rawx_off = mt == 1 ? after_ctl : 0u;
  P.gamma_off = mt == 1 ? after_ctl + round128((size_t)2 * P.K) : after_ctl;
  P.red_off = P.gamma_off + (P.gamma ? round128((size_t)2 * P.K) : 0);
  const bool can_pair = mt == 1 && !P.kind && P.tiles >= 2;
  auto red_stage = [&](bool two) { return round128((size_t)kDW * (two ? 2 : nten) * 16 * mt * sizeof(float)); };
  const size_t fixed = (size_t)P.red_off + 128;  // + base alignment
  if (fixed >= kGemvSmem) return false;
  const size_t avail = kGemvSmem - fixed;
  auto stages_for = [&](size_t stage_bytes, bool two) {
    return (int)std::min<size_t>(kDMaxStages, avail / (round128(stage_bytes) + red_stage(two)));
  };
  int cb = 0, S = 0, pair = 0;
  // Several tokens keep large partials per stage and a large x table: there
  // two big stages beat more small ones (copies below ~1 KB stream slowly).
  for (int want : {mt == 1 ? 3 : 2, 2}) {
    if (can_pair && stages_for((size_t)32 * RB, true) >= want) {
      cb = nb, pair = 1, S = stages_for((size_t)32 * RB, true);
      break;
    }
    if (stages_for((size_t)16 * RB * nten, false) >= want) {
      cb = nb, S = stages_for((size_t)16 * RB * nten, false);
      break;
    }
    for (int w2 : {want + (mt == 1 ? 1 : 0), want}) {
      for (int c = nb - 1; c >= 1 && !cb; --c) {
        if (nb % c != 0 || (c * bb) % 16 != 0 || RB % 16 != 0) continue;
        if (stages_for((size_t)16 * c * bb * nten, false) >= w2)
          cb = c, S = stages_for((size_t)16 * c * bb * nten, false);
      }
      if (cb) break;
    }
    if (cb) break;
  }
  if (!cb) return false;
  P.cb = cb;
  P.pair = pair;
  P.stages = S;
  P.stage_bytes = round128((size_t)16 * cb * bb * (pair ? 2 : nten));
  P.ring_off = (uint32_t)(P.red_off + (size_t)S * red_stage(pair != 0));
  *smem_out = (size_t)P.ring_off + (size_t)S * P.stage_bytes + 128;
  return *smem_out <= kGemvSmem;
}

// One grouped GEMV launch (problems of the same token-slot count): every
// problem keeps its own plan and the launch takes the largest shared-memory
// size.  The CTAs (one per SM, `sms` of them) go one at a time to the
// problem whose busiest CTA has the most work (tiles times tile bytes times
// the format's compute cost per byte).
bool plan_gemv(const GemvDesc* d, int count, int sms, GemvBatch* out, size_t* smem_out) {
  if (count <= 0 || count > kMaxGemvProbs) return false;
  GemvBatch& B = *out;
  memset(&B, 0, sizeof(B));
  B.count = count;
  double tile_cost[kMaxGemvProbs];
  size_t smem = 0;
  for (int i = 0; i < count; ++i) {
    size_t s = 0;
    if (slots_for(d[i].M) != slots_for(d[0].M) || d[i].q8x != d[0].q8x) return false;
    if (!plan_decode_problem(d[i], B.p[i], &s)) return false;
    smem = std::max(smem, s);
    const int bb = B.p[i].qtype == kQ4K ? kQ4KBytes : kQ6KBytes;
    const double cost = B.p[i].qtype == kQ4K ? 1.0 : kQ6CostPerByte;
    tile_cost[i] = 16.0 * (B.p[i].K / kQK) * bb * (1 + B.p[i].kind) * cost;
    B.p[i].ctas = 1;
  }
  *smem_out = smem;
  const int budget = std::max(count, sms);
  for (int used = count; used < budget; ++used) {
    int best = -1;
    double best_load = 0.0;
    for (int i = 0; i < count; ++i) {
      if (B.p[i].ctas >= B.p[i].tiles) continue;
      const double load = (double)((B.p[i].tiles + B.p[i].ctas - 1) / B.p[i].ctas) * tile_cost[i];
      if (load > best_load) {
        best_load = load;
        best = i;
      }
    }
    if (best < 0) break;
    ++B.p[best].ctas;
  }
  int begin = 0;
  for (int i = 0; i < count; ++i) {
    B.p[i].cta_begin = begin;
    begin += B.p[i].ctas;
  }
  return true;
}

template <int MT, bool Q8X>
cudaError_t launch_decode(const GemvBatch& B, size_t smem, cudaStream_t s) {
  static PerDeviceFlag attr;  // the shared-memory limit is a per-device function attribute
  const int dev = current_device();
  if (!attr.done(dev)) {
    cudaError_t e =
        cudaFuncSetAttribute(gemv_decode_kernel<MT, Q8X>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGemvSmem);
    if (e != cudaSuccess) return e;
    attr.mark(dev);
  }
  int ctas = 0;
  for (int i = 0; i < B.count; ++i) ctas += B.p[i].ctas;
#if QK_DECODE_PDL
  // Programmatic dependent launch: the CTAs of this grid may be scheduled
  // while the previous kernel on the stream finishes (they wait for it in
  // griddepcontrol.wait before reading anything), which hides the launch
  // and the set-up of consecutive calls.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)ctas);
  cfg.blockDim = dim3(kDThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, gemv_decode_kernel<MT, Q8X>, B);
  return e != cudaSuccess ? e : cudaGetLastError();
#else
  gemv_decode_kernel<MT, Q8X><<<ctas, kDThreads, smem, s>>>(B);
  return cudaGetLastError();
#endif
}

}  // namespace

bool gemv_plan_fits(const GemvDesc* d, int count) {
  GemvBatch B;
  size_t smem = 0;
  return plan_gemv(d, count, 152, &B, &smem);  // the SM count splits CTAs; it does not decide the fit
}

int gemv_slots(int64_t M) { return slots_for(M); }

// Launch one grouped GEMV (see plan_gemv).
cudaError_t launch_gemv_batch(const GemvDesc* d, int count, cudaStream_t s) {
  GemvBatch B;
  size_t smem = 0;
  if (!plan_gemv(d, count, device_sms(), &B, &smem)) return cudaErrorInvalidConfiguration;
  switch (slots_for(d[0].M)) {
    case 1: return d[0].q8x ? launch_decode<1, true>(B, smem, s) : launch_decode<1, false>(B, smem, s);
    default: return launch_decode<8, false>(B, smem, s);
  }
}

cudaError_t launch_gemv(QType t, const void* W, const uint16_t* x, float* y, int64_t N, int64_t K,
                        cudaStream_t s) {
  GemvDesc d{t, W, nullptr, x, y, 1, N, K, nullptr, 0.f};
  return launch_gemv_batch(&d, 1, s);
}

}  // namespace qk
