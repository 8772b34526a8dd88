// qk_gemv.cu -- decode GEMV (M = 1): y[n] = sum_k x[k] * w[n][k] for Q4_K and
// Q6_K weights.
//
// Source: DAMASCUS project overview, "[01] the thesis" (decode is one token at
// a time, GEMV-heavy and limited by streaming the weights from memory) and
// "[04] one decode step"; "Building DAMASCUS", "Prefill and decode need
// different performance questions".
//
// The kernel is HBM-bound: every packed weight byte is read once.  To keep
// the arithmetic well under the bandwidth budget the inner products run on
// the warp-level tensor instruction mma.sync m16n8k16 (fp16 x fp16, fp32
// accumulate) used as a dot-product engine, with the block scales applied
// after each sub-block instead of per weight:
//
//   * a warp owns 16 weight rows (lane g = lane/4 holds rows g and g+8);
//   * each 4-bit quant q becomes the fp16 value 1024 + F*q by OR-ing the
//     nibble into the mantissa of 1024.0 (F = 1 or 16 depending on where the
//     nibble sits, no shifts needed); the product with an fp16 activation is
//     exact and the sum is fp32;
//   * x is replicated across the 8 MMA columns, so every lane holds the sum
//     D = 1024*Sx + F*sum(q*x) of its two rows for the current sub-block, and
//     the block math gives  sum(w*x) = (d*sc/F)*D - Sx*(1024*d*sc/F + dmin*m)
//     (Q4_K) or (d*sc/F)*D - Sx*(1024*d*sc/F + 32*d*sc) (Q6_K), Sx being the
//     sum of the sub-block's activations (computed once per CTA);
//   * lane tig applies the scales of a quarter of the sub-blocks, so no scale
//     is decoded twice; partial sums meet in two shuffles and one fixed-order
//     pass over the warps that split K.  The result is deterministic.
//
// Packed rows are read with 8-byte (Q4_K) or 4-byte (Q6_K) loads that each
// cover whole 32-byte sectors across the warp.  Q6_K blocks are 210 bytes and
// therefore only 2-byte aligned; their words are assembled from two aligned
// loads and a funnel shift.
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
  const uint8_t* w0;  // weights (gate for kind 1)
  const uint8_t* w1;  // up weights (kind 1), else null
  const uint16_t* x;
  void* y;
  int N, K, qtype, kind;
  int ks, units, cta_begin, ctas;
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

// 4-byte little-endian load from a 2-byte-aligned address inside the buffer.
__device__ __forceinline__ uint32_t ld_u32_a2(const uint8_t* p) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  const uint32_t* w = reinterpret_cast<const uint32_t*>(a & ~uintptr_t(3));
  const uint32_t odd = (uint32_t)(a >> 1) & 1u;
  const uint32_t lo = __ldg(w);
  const uint32_t hi = __ldg(w + odd);  // same word when aligned: never reads past the block
  return __funnelshift_r(lo, hi, 16u * odd);
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

__device__ __forceinline__ void load_block(BlockRegs<kQ4K>& r, const uint8_t* blk0, const uint8_t* blk1, int tig) {
  r.h0 = __ldg(reinterpret_cast<const uint4*>(blk0));
  r.h1 = __ldg(reinterpret_cast<const uint4*>(blk1));
#pragma unroll
  for (int G = 0; G < 4; ++G) {
    r.q0[G] = ldg_stream8(blk0 + 16 + 32 * G + 8 * tig);
    r.q1[G] = ldg_stream8(blk1 + 16 + 32 * G + 8 * tig);
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

__device__ __forceinline__ void load_block(BlockRegs<kQ6K>& r, const uint8_t* blk0, const uint8_t* blk1, int tig) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {  // i = 4h + 2p + s: byte 64h + 32p + 16s + 4tig
    const int off = 64 * (i >> 2) + 32 * ((i >> 1) & 1) + 16 * (i & 1) + 4 * tig;
    r.ql0[i] = ld_u32_a2(blk0 + off);
    r.ql1[i] = ld_u32_a2(blk1 + off);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {  // i = 2h + s: byte 128 + 32h + 16s + 4tig
    const int off = 128 + 32 * (i >> 1) + 16 * (i & 1) + 4 * tig;
    r.qh0[i] = ld_u32_a2(blk0 + off);
    r.qh1[i] = ld_u32_a2(blk1 + off);
  }
  uint32_t s0 = 0, s1 = 0;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    s0 |= (uint32_t)__ldg(blk0 + 192 + 4 * u + tig) << (8 * u);
    s1 |= (uint32_t)__ldg(blk1 + 192 + 4 * u + tig) << (8 * u);
  }
  r.sc0 = s0;
  r.sc1 = s1;
  r.d = (uint32_t)__ldg(reinterpret_cast<const uint16_t*>(blk0 + 208)) |
        ((uint32_t)__ldg(reinterpret_cast<const uint16_t*>(blk1 + 208)) << 16);
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
// The grouped kernel.  One launch runs up to kMaxGemvProbs independent M = 1
// problems (e.g. the seven linears of a decoder layer).  Each problem owns a
// contiguous range of CTAs, sized by its share of the total weight bytes, so
// every CTA stages one x and the whole launch finishes together.  A CTA has 8
// warps: `ks` warps split the K blocks of a 16-row tile and `tpc` = 8 / ks
// tiles are processed side by side; the CTA walks its contiguous range of
// such units, every warp loading the next block (or the next unit's first
// block) while it computes the current one.  Partial sums of the ks warps of
// a tile meet in shared memory in a fixed order (deterministic).
//
// Problem kind 1 is the fused gate/up + SwiGLU: sub-tile 0 holds rows of the
// gate weights, sub-tile 1 the same rows of the up weights, and the epilogue
// writes fp16(silu(g) * u).
// ---------------------------------------------------------------------------
constexpr int kGemvWarps = 8;

template <int QT>
__device__ __forceinline__ void run_gemv_problem(const GemvProb& P, int cta, uint8_t* smem) {
  const int K = P.K, N = P.N, ks = P.ks, tpc = kGemvWarps / P.ks;
  uint2* xp = reinterpret_cast<uint2*>(smem);
  float* sx16 = reinterpret_cast<float*>(smem + 2 * K);
  float* red = sx16 + K / 16;

  const int nb = K / kQK;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, tig = lane & 3;
  const int sub = warp / ks, kslice = warp % ks;
  const int bpw = nb / ks;
  const int b_begin = kslice * bpw;
  constexpr int kBB = QT == kQ4K ? kQ4KBytes : kQ6KBytes;
  const int64_t RB = (int64_t)nb * kBB;
  const int ntiles = (N + 15) / 16;
  // Units of this CTA: [u_begin, u_end).  A unit is tpc tiles (or, for gate/up,
  // one tile of each weight tensor).
  const int u_begin = (int)((int64_t)cta * P.units / P.ctas);
  const int u_end = (int)((int64_t)(cta + 1) * P.units / P.ctas);
  const bool gu = P.kind == 1;
  const uint8_t* Wsub = (gu && sub == 1) ? P.w1 : P.w0;

  auto tile_of = [&](int u) { return gu ? u : u * tpc + sub; };
  auto row_ptr = [&](int tile, int which) {
    const int r = min(tile * 16 + g + 8 * which, N - 1);
    return Wsub + r * RB;
  };

  BlockRegs<QT> cur;
  if (u_begin < u_end && tile_of(u_begin) < ntiles)
    load_block(cur, row_ptr(tile_of(u_begin), 0) + b_begin * kBB, row_ptr(tile_of(u_begin), 1) + b_begin * kBB,
               tig);
  stage_x(P.x, K, xp, sx16);
  __syncthreads();

  for (int u = u_begin; u < u_end; ++u) {
    const int tile = tile_of(u);
    float y0 = 0.f, y1 = 0.f;
    if (tile < ntiles) {
      const uint8_t* row0 = row_ptr(tile, 0);
      const uint8_t* row1 = row_ptr(tile, 1);
      const int tile_next = tile_of(u + 1);
      for (int b = b_begin; b < b_begin + bpw; ++b) {
        BlockRegs<QT> nxt;
        if (b + 1 < b_begin + bpw) {
          load_block(nxt, row0 + (b + 1) * kBB, row1 + (b + 1) * kBB, tig);
        } else if (u + 1 < u_end && tile_next < ntiles) {
          load_block(nxt, row_ptr(tile_next, 0) + b_begin * kBB, row_ptr(tile_next, 1) + b_begin * kBB, tig);
        }
        compute_block(cur, xp + 64 * b, sx16 + 16 * b, tig, y0, y1);
        cur = nxt;
      }
    }
    y0 += __shfl_xor_sync(0xffffffffu, y0, 1);
    y0 += __shfl_xor_sync(0xffffffffu, y0, 2);
    y1 += __shfl_xor_sync(0xffffffffu, y1, 1);
    y1 += __shfl_xor_sync(0xffffffffu, y1, 2);
    if (tig == 0) {
      red[warp * 16 + g] = y0;
      red[warp * 16 + g + 8] = y1;
    }
    __syncthreads();
    if (!gu) {
      if (threadIdx.x < 16 * tpc) {
        const int t = threadIdx.x >> 4, r = threadIdx.x & 15;
        float acc = 0.f;
        for (int w = 0; w < ks; ++w) acc += red[(t * ks + w) * 16 + r];
        const int row = (u * tpc + t) * 16 + r;
        if (row < N) static_cast<float*>(P.y)[row] = acc;
      }
    } else if (threadIdx.x < 16) {
      const int r = threadIdx.x;
      float gs = 0.f, us = 0.f;
      for (int w = 0; w < ks; ++w) {
        gs += red[w * 16 + r];
        us += red[(ks + w) * 16 + r];
      }
      const int row = u * 16 + r;
      if (row < N) static_cast<__half*>(P.y)[row] = __float2half_rn(gs / (1.0f + __expf(-gs)) * us);
    }
    __syncthreads();
  }
}

__global__ void __maxnreg__(128) gemv_batch_kernel(const __grid_constant__ GemvBatch B) {
  extern __shared__ __align__(16) uint8_t smem[];
  int i = 0;
  while (i + 1 < B.count && (int)blockIdx.x >= B.p[i + 1].cta_begin) ++i;
  const GemvProb& P = B.p[i];
  const int cta = (int)blockIdx.x - P.cta_begin;
  if (P.qtype == kQ4K)
    run_gemv_problem<kQ4K>(P, cta, smem);
  else
    run_gemv_problem<kQ6K>(P, cta, smem);
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

}  // namespace

int gemv_max_m() { return 1; }

uint32_t gemv_take_status() {
  uint32_t v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_gemv_status, sizeof(v)) != cudaSuccess) return 0;
  cudaMemcpyToSymbol(g_gemv_status, &zero, sizeof(zero));
  return v;
}

// Launch one grouped GEMV.  ks = the largest of 8, 4, 2, 1 dividing the block
// count (gate/up: at most 4, so a CTA holds one gate and one up tile).  CTAs:
// two per SM (256 threads x 128 registers), split across problems in
// proportion to their weight bytes.
cudaError_t launch_gemv_batch(const GemvDesc* d, int count, cudaStream_t s) {
  GemvBatch B;
  memset(&B, 0, sizeof(B));
  B.count = count;
  double total = 0;
  int64_t bytes[kMaxGemvProbs];
  size_t smem = 0;
  for (int i = 0; i < count; ++i) {
    GemvProb& P = B.p[i];
    P.w0 = static_cast<const uint8_t*>(d[i].w0);
    P.w1 = static_cast<const uint8_t*>(d[i].w1);
    P.x = d[i].x;
    P.y = d[i].y;
    P.N = (int)d[i].N;
    P.K = (int)d[i].K;
    P.qtype = d[i].qtype;
    P.kind = d[i].w1 ? 1 : 0;
    const int nb = P.K / kQK;
    int ks = 1;
    for (int c = (P.kind ? 4 : 8); c >= 1; c /= 2)
      if (nb % c == 0) {
        ks = c;
        break;
      }
    if (P.kind) {
      if (nb % 4) return cudaErrorInvalidValue;  // gate/up needs one gate + one up tile per CTA
      ks = 4;
    }
    P.ks = ks;
    const int tpc = kGemvWarps / ks;
    const int ntiles = (P.N + 15) / 16;
    P.units = P.kind ? ntiles : (ntiles + tpc - 1) / tpc;
    bytes[i] = (int64_t)P.N * nb * (P.qtype == kQ4K ? kQ4KBytes : kQ6KBytes) * (P.kind ? 2 : 1);
    total += (double)bytes[i];
    smem = std::max(smem, (size_t)2 * P.K + (size_t)P.K / 4 + (size_t)kGemvWarps * 16 * sizeof(float));
  }
  const int budget = std::max(count, sm_count() * 2);
  int used = 0;
  for (int i = 0; i < count; ++i) {
    int c = (int)((double)budget * (double)bytes[i] / total);
    c = std::max(1, std::min(c, B.p[i].units));
    B.p[i].ctas = c;
    used += c;
  }
  // Hand leftover CTAs to the problems with the most units per CTA.
  for (bool again = true; again && used < budget;) {
    again = false;
    int best = -1;
    double best_load = 1.0;
    for (int i = 0; i < count; ++i) {
      const double load = (double)B.p[i].units / B.p[i].ctas;
      if (B.p[i].ctas < B.p[i].units && load > best_load) {
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
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(gemv_batch_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  gemv_batch_kernel<<<begin, 32 * kGemvWarps, smem, s>>>(B);
  return cudaGetLastError();
}

cudaError_t launch_gemv(QType t, const void* W, const uint16_t* x, float* y, int64_t N, int64_t K,
                        cudaStream_t s) {
  GemvDesc d{t, W, nullptr, x, y, N, K};
  return launch_gemv_batch(&d, 1, s);
}

}  // namespace qk
