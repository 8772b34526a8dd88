// qk_gemv.cu -- decode GEMV (M = 1): y[n] = sum_k x[k] * w[n][k] for Q4_K and
// Q6_K weights.
//
// Source: DAMASCUS project overview, "[01] the thesis" (decode is one token at
// a time, GEMV-heavy and limited by streaming the weights from memory) and
// "[04] one decode step"; "Building DAMASCUS", "Prefill and decode need
// different performance questions".
//
// The kernel is HBM-bound: every packed weight byte is read once, by TMA, into
// shared memory, and the arithmetic stays well under the bandwidth budget:
//
//   * a warp owns whole 16-row tiles and streams their K slices through a
//     private two-stage shared-memory pipeline filled by tensor-map TMA loads
//     (Q4_K: one box of 16 rows x 2 blocks; Q6_K: one box per residue of a
//     group of g rows whose byte stride is 16-aligned, like the prefill GEMM),
//     so each weight byte crosses the memory system once, in full sectors;
//   * the inner products use the warp tensor instruction mma.sync m16n8k16
//     (fp16 x fp16, fp32 accumulate) as a dot-product engine: a 4-bit quant
//     OR-ed into the mantissa of fp16 1024.0 is the exact value 1024 + F*q (F =
//     1 or 16 by nibble position, no shifts), its product with an fp16
//     activation is exact and the sum fp32;
//   * x is replicated across the 8 MMA columns, so every lane holds the sum
//     D = 1024*Sx + F*sum(q*x) of its two rows for the current sub-block, and
//     sum(w*x) = (d*sc/F)*D - Sx*(1024*d*sc/F + dmin*m) (Q4_K) or
//     (d*sc/F)*D - Sx*(1024*d*sc/F + 32*d*sc) (Q6_K), Sx being the sum of the
//     sub-block's activations, staged once per CTA with a k-permuted fp16 x;
//   * lane tig applies the scales of a quarter of the sub-blocks; the two
//     partial sums of a row meet in two shuffles (deterministic).
// Q6_K blocks are 210 bytes, so every other block is 2 mod 4 bytes into its
// window: its words come from two aligned shared-memory loads and a funnel
// shift.  Shared-memory row pitches (288 B, 432 B) and the Q6_K row order
// (MMA row r <-> weight row 2r or 2r+1 for g = 2) make the fragment reads of
// a warp bank-conflict free.
//
// One launch runs up to kMaxGemvProbs independent problems (qk_matmul_batch):
// each owns a contiguous range of CTAs sized by its share of the weight
// bytes.  Problem kind 1 is the fused gate/up + SwiGLU: a warp streams the gate
// rows then the up rows of its tile and writes fp16(silu(g) * u).
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

constexpr uint32_t kMagic = 0x64006400u;  // fp16x2 (1024.0, 1024.0)

struct GemvProb {
  CUtensorMap tm[2];  // weights (gate for kind 1), up weights (kind 1)
  const uint8_t* w[2];
  const uint16_t* x;
  void* y;
  int N, K, qtype, kind;
  int g;          // Q6_K: weight rows per tensor-map row (1 for Q4_K)
  int rows_tma;   // rows covered by the tensor map; rows past it are copied by hand
  int pitch;      // shared-memory bytes per row slot (the box width)
  int region;     // shared-memory bytes per residue region (128-byte aligned)
  int stage;      // shared-memory bytes per pipeline stage
  int tiles, cta_begin, ctas;
};

struct GemvBatch {
  GemvProb p[kMaxGemvProbs];
  int count;
};

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float half_lo(uint32_t v) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(v & 0xFFFFu)));
}

__device__ __forceinline__ float pick4(const float (&v)[4], int i) {
  float r = v[0];
  r = i == 1 ? v[1] : r;
  r = i == 2 ? v[2] : r;
  r = i == 3 ? v[3] : r;
  return r;
}

// ---------------------------------------------------------------------------
// x staging: xp[k/4] = { fp16x2(x[k], x[k+2]), fp16x2(x[k+1], x[k+3]) } (the
// MMA k-slot order used below) and sx16[i] = sum of x[16i .. 16i+15] in fp32.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void stage_x(const uint16_t* __restrict__ x, int K, uint2* xp, float* sx16) {
  const int nq = K / 4;  // a multiple of 64
  for (int i = threadIdx.x; i < nq; i += blockDim.x) {
    const uint2 v = *reinterpret_cast<const uint2*>(x + 4 * i);
    uint2 o;
    o.x = prmt(v.x, v.y, 0x5410u);  // x0 | x2 << 16
    o.y = prmt(v.x, v.y, 0x7632u);  // x1 | x3 << 16
    xp[i] = o;
    float s = (half_lo(v.x) + half_lo(v.x >> 16)) + (half_lo(v.y) + half_lo(v.y >> 16));
    s += __shfl_xor_sync(0xffffffffu, s, 1);
    s += __shfl_xor_sync(0xffffffffu, s, 2);
    if ((i & 3) == 0) sx16[i >> 2] = s;
  }
}

// ---------------------------------------------------------------------------
// Q4_K: lane (g, tig) handles rows g, g+8.  In 64-weight group G (sub-blocks
// 2G, 2G+1, quant bytes 32G..32G+31) the lane owns bytes 8*tig .. 8*tig+7,
// i.e. words hh = 0, 1 at 8*tig + 4*hh.  Word hh feeds one MMA per sub-block:
//   k-slots 2tig, 2tig+1  <- bytes 0, 2 of the word  (k = 8tig+4hh + 0, 2)
//   k-slots 2tig+8, +9    <- bytes 1, 3              (k = 8tig+4hh + 1, 3)
// Low nibbles (mask 0x000F000F, F = 1) give sub-block 2G, high nibbles (mask
// 0x00F000F0, F = 16) sub-block 2G+1.
// ---------------------------------------------------------------------------
struct Q4Scales {
  float a_lo, c_lo, a_hi, c_hi;
};

// Scale/min of sub-blocks 2*tig and 2*tig+1 from a block header.
__device__ __forceinline__ Q4Scales q4k_lane_scales(uint4 hdr, int tig) {
  const float d = half_lo(hdr.x);
  const float dmin = half_lo(hdr.x >> 16);
  Q4Scales r;
#pragma unroll
  for (int side = 0; side < 2; ++side) {
    const int j = 2 * tig + side;
    const int jj = j & 3;
    uint32_t sc, mn;
    if (j < 4) {
      sc = (hdr.y >> (8 * jj)) & 63u;
      mn = (hdr.z >> (8 * jj)) & 63u;
    } else {
      const uint32_t lo = (hdr.w >> (8 * jj)) & 0xFFu;
      sc = (lo & 0xFu) | (((hdr.y >> (8 * jj + 6)) & 3u) << 4);
      mn = (lo >> 4) | (((hdr.z >> (8 * jj + 6)) & 3u) << 4);
    }
    const float dsc = d * (float)sc;
    const float dmn = dmin * (float)mn;
    if (side == 0) {
      r.a_lo = dsc;
      r.c_lo = fmaf(1024.0f, dsc, dmn);
    } else {
      r.a_hi = dsc * 0.0625f;
      r.c_hi = fmaf(64.0f, dsc, dmn);
    }
  }
  return r;
}

// Registers holding one block of each of the lane's two rows.
template <int QT>
struct BlockRegs;

template <>
struct BlockRegs<kQ4K> {
  uint4 h0, h1;      // d, dmin, packed scales of rows g, g+8
  uint2 q0[4], q1[4];  // quant bytes 32G + 8tig .. +7, G = 0..3
};

// Block registers from shared memory: blk0 / blk1 = the block of the lane's
// two rows inside their stage slots (16-byte aligned for Q4_K).
__device__ __forceinline__ void load_block(BlockRegs<kQ4K>& r, const uint8_t* blk0, const uint8_t* blk1, int tig) {
  r.h0 = *reinterpret_cast<const uint4*>(blk0);
  r.h1 = *reinterpret_cast<const uint4*>(blk1);
#pragma unroll
  for (int G = 0; G < 4; ++G) {
    r.q0[G] = *reinterpret_cast<const uint2*>(blk0 + 16 + 32 * G + 8 * tig);
    r.q1[G] = *reinterpret_cast<const uint2*>(blk1 + 16 + 32 * G + 8 * tig);
  }
}

__device__ __forceinline__ void compute_block(const BlockRegs<kQ4K>& r, const uint2* xpb, const float* sxb, int tig,
                                              float& y0, float& y1) {
  float dlo0[4], dlo1[4], dhi0[4], dhi1[4];
#pragma unroll
  for (int G = 0; G < 4; ++G) {
    float c[4] = {0.f, 0.f, 0.f, 0.f}, e[4] = {0.f, 0.f, 0.f, 0.f};
    const uint4 xlo = *reinterpret_cast<const uint4*>(xpb + 16 * G + 2 * tig);      // k = 64G + 8tig + {0..7}
    const uint4 xhi = *reinterpret_cast<const uint4*>(xpb + 16 * G + 8 + 2 * tig);  // k + 32
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const uint32_t w0 = hh ? r.q0[G].y : r.q0[G].x;
      const uint32_t w1 = hh ? r.q1[G].y : r.q1[G].x;
      const uint32_t s0 = w0 >> 8, s1 = w1 >> 8;
      const uint32_t bl0 = hh ? xlo.z : xlo.x, bl1 = hh ? xlo.w : xlo.y;
      const uint32_t bh0 = hh ? xhi.z : xhi.x, bh1 = hh ? xhi.w : xhi.y;
      mma16816(c, (w0 & 0x000F000Fu) | kMagic, (w1 & 0x000F000Fu) | kMagic, (s0 & 0x000F000Fu) | kMagic,
               (s1 & 0x000F000Fu) | kMagic, bl0, bl1);
      mma16816(e, (w0 & 0x00F000F0u) | kMagic, (w1 & 0x00F000F0u) | kMagic, (s0 & 0x00F000F0u) | kMagic,
               (s1 & 0x00F000F0u) | kMagic, bh0, bh1);
    }
    dlo0[G] = c[0];
    dlo1[G] = c[2];
    dhi0[G] = e[0];
    dhi1[G] = e[2];
  }
  // This lane applies the scales of group G = tig (sub-blocks 2tig, 2tig+1).
  const Q4Scales r0 = q4k_lane_scales(r.h0, tig);
  const Q4Scales r1 = q4k_lane_scales(r.h1, tig);
  const float2 sx = make_float2(sxb[4 * tig] + sxb[4 * tig + 1], sxb[4 * tig + 2] + sxb[4 * tig + 3]);
  y0 = fmaf(r0.a_lo, pick4(dlo0, tig), y0);
  y0 = fmaf(-r0.c_lo, sx.x, y0);
  y0 = fmaf(r0.a_hi, pick4(dhi0, tig), y0);
  y0 = fmaf(-r0.c_hi, sx.y, y0);
  y1 = fmaf(r1.a_lo, pick4(dlo1, tig), y1);
  y1 = fmaf(-r1.c_lo, sx.x, y1);
  y1 = fmaf(r1.a_hi, pick4(dhi1, tig), y1);
  y1 = fmaf(-r1.c_hi, sx.y, y1);
}

// ---------------------------------------------------------------------------
// Q6_K: scale group t (16 weights, t = 8h + 2*g6 + s) takes its low 4 bits
// from quant bytes 64h + 32(g6&1) + 16s + l (low nibble if g6 < 2) and its
// high 2 bits from bits 2*g6 of byte 128 + 32h + 16s + l, l = 0..15.  Lane tig
// owns l = 4tig .. 4tig+3 (one word of each).  The fp16 operand is 1024 + F*q6
// with F = 1 (g6 < 2: nibble in bits 0-3, high bits moved to 4-5) or F = 16
// (g6 >= 2: nibble in bits 4-7, high bits moved to 8-9).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void q6k_operands(uint32_t wl, uint32_t wh, int g6, uint32_t& r0, uint32_t& r2) {
  const uint32_t wl8 = wl >> 8;
  const uint32_t up = (g6 & 1) ? (wh << 2) : (wh << 4);
  const uint32_t dn = (g6 & 1) ? (wh >> 6) : (wh >> 4);
  if (g6 < 2) {
    r0 = (wl & 0x000F000Fu) | (up & 0x00300030u) | kMagic;
    r2 = (wl8 & 0x000F000Fu) | (dn & 0x00300030u) | kMagic;
  } else {
    r0 = (wl & 0x00F000F0u) | (up & 0x03000300u) | kMagic;
    r2 = (wl8 & 0x00F000F0u) | (dn & 0x03000300u) | kMagic;
  }
}

template <>
struct BlockRegs<kQ6K> {
  uint32_t ql0[8], ql1[8], qh0[4], qh1[4];  // the lane's quant words of rows g, g+8
  uint32_t sc0, sc1;                        // int8 scales t = 4u + tig, u = 0..3 (byte u)
  uint32_t d;                               // fp16 d of row g (low half) and row g+8 (high half)
};

// 4-byte word at a 2-byte-aligned shared-memory address.
__device__ __forceinline__ uint32_t lds_u32_a2(const uint8_t* p) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  const uint32_t* w = reinterpret_cast<const uint32_t*>(a & ~uintptr_t(3));
  const uint32_t odd = (uint32_t)(a >> 1) & 1u;
  return __funnelshift_r(w[0], w[odd], 16u * odd);
}

__device__ __forceinline__ void load_block(BlockRegs<kQ6K>& r, const uint8_t* blk0, const uint8_t* blk1, int tig) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {  // i = 4h + 2p + s: byte 64h + 32p + 16s + 4tig
    const int off = 64 * (i >> 2) + 32 * ((i >> 1) & 1) + 16 * (i & 1) + 4 * tig;
    r.ql0[i] = lds_u32_a2(blk0 + off);
    r.ql1[i] = lds_u32_a2(blk1 + off);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {  // i = 2h + s: byte 128 + 32h + 16s + 4tig
    const int off = 128 + 32 * (i >> 1) + 16 * (i & 1) + 4 * tig;
    r.qh0[i] = lds_u32_a2(blk0 + off);
    r.qh1[i] = lds_u32_a2(blk1 + off);
  }
  uint32_t s0 = 0, s1 = 0;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    s0 |= (uint32_t)blk0[192 + 4 * u + tig] << (8 * u);
    s1 |= (uint32_t)blk1[192 + 4 * u + tig] << (8 * u);
  }
  r.sc0 = s0;
  r.sc1 = s1;
  r.d = (uint32_t)*reinterpret_cast<const uint16_t*>(blk0 + 208) |
        ((uint32_t)*reinterpret_cast<const uint16_t*>(blk1 + 208) << 16);
}

__device__ __forceinline__ void compute_block(const BlockRegs<kQ6K>& r, const uint2* xpb, const float* sxb, int tig,
                                              float& y0, float& y1) {
  float d0[16], d1[16];
#pragma unroll
  for (int t = 0; t < 16; ++t) {
    const int h = t >> 3, g6 = (t >> 1) & 3, s = t & 1;
    const int li = 4 * h + 2 * (g6 & 1) + s, hi = 2 * h + s;
    uint32_t a0, a2, a1, a3;
    q6k_operands(r.ql0[li], r.qh0[hi], g6, a0, a2);
    q6k_operands(r.ql1[li], r.qh1[hi], g6, a1, a3);
    const uint2 b = xpb[4 * t + tig];
    float c[4] = {0.f, 0.f, 0.f, 0.f};
    mma16816(c, a0, a1, a2, a3, b.x, b.y);
    d0[t] = c[0];
    d1[t] = c[2];
  }
  // Scales: lane tig applies scale groups t = 4u + tig.
  const float dA = half_lo(r.d), dB = half_lo(r.d >> 16);
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int t = 4 * u + tig;
    // 1/F: scale group t = 4u + tig has g6 = (2u + tig/2) & 3, which is >= 2 exactly for odd u.
    const float inv_f = (u & 1) ? 0.0625f : 1.0f;
    const float dsc0 = dA * (float)(int8_t)((r.sc0 >> (8 * u)) & 0xFFu);
    const float dsc1 = dB * (float)(int8_t)((r.sc1 >> (8 * u)) & 0xFFu);
    float v0[4] = {d0[4 * u], d0[4 * u + 1], d0[4 * u + 2], d0[4 * u + 3]};
    float v1[4] = {d1[4 * u], d1[4 * u + 1], d1[4 * u + 2], d1[4 * u + 3]};
    const float sxt = sxb[t];
    const float a0 = dsc0 * inv_f, a1 = dsc1 * inv_f;
    y0 = fmaf(a0, pick4(v0, tig), y0);
    y0 = fmaf(-fmaf(1024.0f, a0, 32.0f * dsc0), sxt, y0);
    y1 = fmaf(a1, pick4(v1, tig), y1);
    y1 = fmaf(-fmaf(1024.0f, a1, 32.0f * dsc1), sxt, y1);
  }
}

// ---------------------------------------------------------------------------
// The kernel.
// ---------------------------------------------------------------------------
constexpr int kGemvWarps = 8;
constexpr int kSliceBlocks = 2;  // K blocks per pipeline stage

struct GemvShared {
  uint64_t full[kGemvWarps][2];
  uint32_t abort_flag;
};

// Weight row held by MMA row r (0..15) of a tile: identity, except for Q6_K
// with g = 2, where MMA rows 0..7 take the even rows and 8..15 the odd rows so
// the eight rows read by one instruction sit in one residue region.
__device__ __forceinline__ int tile_row(int r, int g) { return g == 2 ? 2 * (r & 7) + (r >> 3) : r; }

// Shared-memory slot of tile row rho (0..15) inside a stage.
__device__ __forceinline__ uint32_t row_slot(const GemvProb& P, int rho) {
  return (uint32_t)(rho % P.g) * (uint32_t)P.region + (uint32_t)(rho / P.g) * (uint32_t)P.pitch;
}

// Byte offset of block b0 of tile row rho inside its slot (the misalignment of
// the box start: 0 for Q4_K, (n * row_bytes + 210 * b0) mod 16 for Q6_K).
template <int QT>
__device__ __forceinline__ int slot_mis(int64_t RB, int n, int b0) {
  if constexpr (QT == kQ4K) return 0;
  return (int)(((int64_t)n * RB + (int64_t)b0 * kQ6KBytes) & 15);
}

template <int QT>
__device__ __forceinline__ void run_gemv_problem(const GemvProb& P, int cta, uint8_t* smem, uint8_t* stages,
                                                 GemvShared* sh) {
  const int K = P.K, N = P.N, nb = K / kQK;
  const uint2* xp = reinterpret_cast<const uint2*>(smem);
  const float* sx16 = reinterpret_cast<const float*>(smem + 2 * K);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, tig = lane & 3;
  constexpr int kBB = QT == kQ4K ? kQ4KBytes : kQ6KBytes;
  const int64_t RB = (int64_t)nb * kBB;
  const int nten = P.kind == 1 ? 2 : 1;
  const int nslices = (nb + kSliceBlocks - 1) / kSliceBlocks;
  // Tiles of this CTA, then of this warp.
  const int c0 = (int)((int64_t)cta * P.tiles / P.ctas), c1 = (int)((int64_t)(cta + 1) * P.tiles / P.ctas);
  const int t0 = c0 + (int)((int64_t)warp * (c1 - c0) / kGemvWarps);
  const int t1 = c0 + (int)((int64_t)(warp + 1) * (c1 - c0) / kGemvWarps);
  const int steps = (t1 - t0) * nten * nslices;
  uint8_t* const my_stages = stages + (size_t)(2 * warp) * P.stage;  // this warp's two stages
  uint64_t* full = sh->full[warp];
  volatile uint32_t* abort_flag = &sh->abort_flag;

  // Issue the TMA boxes of step `st` into stage `b` (lane 0 only).
  auto issue = [&](int st, int b) {
    const int slice = st % nslices;
    const int ten = (st / nslices) % nten;
    const int tile = t0 + st / (nslices * nten);
    const int n0 = tile * 16;
    const int b0 = slice * kSliceBlocks;
    const bool tma = n0 < P.rows_tma;
    mbar_arrive_expect_tx(&full[b], tma ? (uint32_t)(16 * P.pitch) : 0u);
    if (tma) {
      for (int j = 0; j < P.g; ++j) {
        const int64_t off = (int64_t)j * RB + (int64_t)b0 * kBB;  // byte offset inside a map row
        tma_load_2d(my_stages + (size_t)b * P.stage + (uint32_t)j * P.region, &P.tm[ten],
                    (int32_t)((off & ~int64_t(15)) >> 3),
                    n0 / P.g, &full[b]);
      }
    }
  };

  if (lane == 0 && steps > 0) issue(0, 0);
  float y0 = 0.f, y1 = 0.f, z0 = 0.f, z1 = 0.f;
  bool ok = true;
  for (int st = 0; st < steps && ok; ++st) {
    const int b = st & 1;
    const int slice = st % nslices;
    const int ten = (st / nslices) % nten;
    const int tile = t0 + st / (nslices * nten);
    const int n0 = tile * 16;
    const int b0 = slice * kSliceBlocks;
    if (lane == 0 && st + 1 < steps) issue(st + 1, b ^ 1);
    ok = mbar_wait(&full[b], (uint32_t)(st >> 1) & 1u, abort_flag, &g_gemv_status);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) break;
    uint8_t* stg = my_stages + (size_t)b * P.stage;
    // Rows past the tensor map (only the last rows of a Q6_K tensor whose row
    // count is not a multiple of g): copy their slice bytes by hand.
    if (QT == kQ6K && n0 + 16 > P.rows_tma) {
      const uint8_t* W = P.w[ten];
      for (int rho = 0; rho < 16; ++rho) {
        const int n = n0 + rho;
        if (n < P.rows_tma || n >= N) continue;
        const int64_t src0 = (int64_t)n * RB + (int64_t)b0 * kBB;
        const int64_t rem = RB - (int64_t)b0 * kBB;
        const int64_t len = rem < (int64_t)kSliceBlocks * kBB ? rem : (int64_t)kSliceBlocks * kBB;
        uint8_t* dst = stg + row_slot(P, rho) + slot_mis<QT>(RB, n, b0);
        for (int64_t i = 2 * lane; i < len; i += 64)
          *reinterpret_cast<uint16_t*>(dst + i) = *reinterpret_cast<const uint16_t*>(W + src0 + i);
      }
      __syncwarp();
    }
    const int r0 = tile_row(g, P.g), r1 = tile_row(g + 8, P.g);
    const uint8_t* s0 = stg + row_slot(P, r0) + slot_mis<QT>(RB, min(n0 + r0, N - 1), b0);
    const uint8_t* s1 = stg + row_slot(P, r1) + slot_mis<QT>(RB, min(n0 + r1, N - 1), b0);
    float& a0 = ten ? z0 : y0;
    float& a1 = ten ? z1 : y1;
#pragma unroll
    for (int bb = 0; bb < kSliceBlocks; ++bb) {
      const int blk = b0 + bb;
      if (blk < nb) {
        BlockRegs<QT> r;
        load_block(r, s0 + bb * kBB, s1 + bb * kBB, tig);
        compute_block(r, xp + 64 * blk, sx16 + 16 * blk, tig, a0, a1);
      }
    }
    fence_proxy_async_smem();  // our reads of this stage precede the TMA that refills it
    __syncwarp();
    if (slice == nslices - 1 && ten == nten - 1) {  // tile done
      y0 += __shfl_xor_sync(0xffffffffu, y0, 1);
      y0 += __shfl_xor_sync(0xffffffffu, y0, 2);
      y1 += __shfl_xor_sync(0xffffffffu, y1, 1);
      y1 += __shfl_xor_sync(0xffffffffu, y1, 2);
      if (P.kind == 1) {
        z0 += __shfl_xor_sync(0xffffffffu, z0, 1);
        z0 += __shfl_xor_sync(0xffffffffu, z0, 2);
        z1 += __shfl_xor_sync(0xffffffffu, z1, 1);
        z1 += __shfl_xor_sync(0xffffffffu, z1, 2);
      }
      if (tig == 0) {
        const int n_a = n0 + r0, n_b = n0 + r1;
        if (P.kind == 1) {
          __half* y = static_cast<__half*>(P.y);
          if (n_a < N) y[n_a] = __float2half_rn(y0 / (1.0f + __expf(-y0)) * z0);
          if (n_b < N) y[n_b] = __float2half_rn(y1 / (1.0f + __expf(-y1)) * z1);
        } else {
          float* y = static_cast<float*>(P.y);
          if (n_a < N) y[n_a] = y0;
          if (n_b < N) y[n_b] = y1;
        }
      }
      y0 = y1 = z0 = z1 = 0.f;
    }
  }
  // Drain: the copy issued for the step after an early exit must land first.
  if (!ok && lane == 0) {
    for (int b = 0; b < 2; ++b) mbar_wait(&full[b], 0u, abort_flag, &g_gemv_status, true);
  }
}

__global__ void __launch_bounds__(32 * kGemvWarps) gemv_tma_kernel(const __grid_constant__ GemvBatch B) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  int i = 0;
  while (i + 1 < B.count && (int)blockIdx.x >= B.p[i + 1].cta_begin) ++i;
  const GemvProb& P = B.p[i];
  const int cta = (int)blockIdx.x - P.cta_begin;
  const uint32_t x_bytes = ((uint32_t)(2 * P.K + P.K / 4) + 127u) & ~127u;
  uint8_t* stages = smem + x_bytes;
  GemvShared* sh = reinterpret_cast<GemvShared*>(stages + (size_t)(2 * kGemvWarps) * P.stage);
  if (threadIdx.x < 2 * kGemvWarps) mbar_init(&sh->full[threadIdx.x >> 1][threadIdx.x & 1], 1);
  if (threadIdx.x == 0) {
    sh->abort_flag = 0;
    prefetch_tmap(&P.tm[0]);
    if (P.kind == 1) prefetch_tmap(&P.tm[1]);
  }
  fence_mbar_init();
  __syncthreads();
  // The first TMA of each warp could go out before x is staged; staging is
  // short next to a weight fetch, so it simply comes first.
  stage_x(P.x, P.K, reinterpret_cast<uint2*>(smem), reinterpret_cast<float*>(smem + 2 * P.K));
  __syncthreads();
  if (P.qtype == kQ4K)
    run_gemv_problem<kQ4K>(P, cta, smem, stages, sh);
  else
    run_gemv_problem<kQ6K>(P, cta, smem, stages, sh);
}

int g_sms = 0;

int sm_count() {
  if (!g_sms) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&g_sms, cudaDevAttrMultiProcessorCount, dev);
    if (g_sms <= 0) g_sms = 148;
  }
  return g_sms;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// Weight tensor map: rows of g weight rows (g * row_bytes is 16-aligned) of
// 8-byte elements; one box = `pitch` bytes of 16/g such rows.
bool make_weight_map(CUtensorMap* tm, const void* w, int64_t N, int64_t RB, int g, int pitch) {
  EncodeTiledFn enc = encode_fn();
  if (!enc || N / g <= 0) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)(g * RB / 8), (cuuint64_t)(N / g)};
  const cuuint64_t strides[1] = {(cuuint64_t)(g * RB)};
  const cuuint32_t box[2] = {(cuuint32_t)(pitch / 8), (cuuint32_t)(16 / g)};
  const cuuint32_t estr[2] = {1, 1};
  return enc(tm, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<void*>(w), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int gemv_max_m() { return 1; }

uint32_t gemv_take_status() {
  uint32_t v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_gemv_status, sizeof(v)) != cudaSuccess) return 0;
  cudaMemcpyToSymbol(g_gemv_status, &zero, sizeof(zero));
  return v;
}

// Launch one grouped GEMV: per problem the tensor map(s) and stage geometry;
// CTAs (one or two per SM, by shared memory) split across problems in
// proportion to their weight bytes.
cudaError_t launch_gemv_batch(const GemvDesc* d, int count, cudaStream_t s) {
  if (count <= 0 || count > kMaxGemvProbs) return cudaErrorInvalidValue;
  GemvBatch B;
  memset(&B, 0, sizeof(B));
  B.count = count;
  double total = 0;
  int64_t bytes[kMaxGemvProbs];
  size_t smem = 0;
  for (int i = 0; i < count; ++i) {
    GemvProb& P = B.p[i];
    P.w[0] = static_cast<const uint8_t*>(d[i].w0);
    P.w[1] = static_cast<const uint8_t*>(d[i].w1);
    P.x = d[i].x;
    P.y = d[i].y;
    P.N = (int)d[i].N;
    P.K = (int)d[i].K;
    P.qtype = d[i].qtype;
    P.kind = d[i].w1 ? 1 : 0;
    const int nb = P.K / kQK;
    const int64_t RB = (int64_t)nb * (P.qtype == kQ4K ? kQ4KBytes : kQ6KBytes);
    if (P.qtype == kQ4K) {
      P.g = 1;
      P.pitch = kSliceBlocks * kQ4KBytes;  // 288 B: 72 words = 8 mod 32, conflict-free 8-byte reads
      P.region = 16 * P.pitch;
    } else {
      int g = 1;
      while (g < 8 && (g * RB) % 16) g *= 2;
      P.g = g;
      // 2 blocks (420 B) plus the window's misalignment (<= 12 when row_bytes is
      // a multiple of 4, else <= 14), rounded up to 16 bytes.
      P.pitch = (RB % 4 == 0) ? 432 : 448;
      P.region = ((16 / g) * P.pitch + 127) / 128 * 128;
    }
    P.stage = P.g * P.region;
    P.rows_tma = (P.N / P.g) * P.g;
    for (int t = 0; t < 1 + P.kind; ++t)
      if (P.rows_tma > 0 && !make_weight_map(&P.tm[t], P.w[t], P.N, RB, P.g, P.pitch))
        return cudaErrorInvalidValue;
    P.tiles = (P.N + 15) / 16;
    bytes[i] = (int64_t)P.N * RB * (1 + P.kind);
    total += (double)bytes[i];
    const size_t x_bytes = ((size_t)(2 * P.K + P.K / 4) + 127) / 128 * 128;
    smem = std::max(smem, x_bytes + (size_t)(2 * kGemvWarps) * P.stage + sizeof(GemvShared) + 128);
  }
  const int per_sm = std::max<int>(1, (int)((227 * 1024) / smem));
  const int budget = std::max(count, sm_count() * std::min(per_sm, 2));
  int used = 0;
  for (int i = 0; i < count; ++i) {
    const int max_ctas = std::max(1, (B.p[i].tiles + kGemvWarps - 1) / kGemvWarps);
    int c = (int)((double)budget * (double)bytes[i] / total);
    c = std::max(1, std::min(c, max_ctas));
    B.p[i].ctas = c;
    used += c;
  }
  for (bool again = true; again && used < budget;) {  // leftover CTAs to the busiest problems
    again = false;
    int best = -1;
    double best_load = 0.0;
    for (int i = 0; i < count; ++i) {
      const int max_ctas = std::max(1, (B.p[i].tiles + kGemvWarps - 1) / kGemvWarps);
      const double load = (double)bytes[i] / B.p[i].ctas;
      if (B.p[i].ctas < max_ctas && load > best_load) {
        best_load = load;
        best = i;
      }
    }
    if (best >= 0) {
      ++B.p[best].ctas;
      ++used;
      again = true;
    }
  }
  int begin = 0;
  for (int i = 0; i < count; ++i) {
    B.p[i].cta_begin = begin;
    begin += B.p[i].ctas;
  }
  static size_t smem_set = 0;
  if (smem > 48 * 1024 && smem > smem_set) {
    cudaError_t e = cudaFuncSetAttribute(gemv_tma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         227 * 1024);
    if (e != cudaSuccess) return e;
    smem_set = 227 * 1024;
  }
  gemv_tma_kernel<<<begin, 32 * kGemvWarps, smem, s>>>(B);
  return cudaGetLastError();
}

cudaError_t launch_gemv(QType t, const void* W, const uint16_t* x, float* y, int64_t N, int64_t K,
                        cudaStream_t s) {
  GemvDesc d{t, W, nullptr, x, y, N, K};
  return launch_gemv_batch(&d, 1, s);
}

}  // namespace qk
