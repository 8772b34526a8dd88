// qk_gemv.cu -- decode GEMV (M = 1): y[n] = sum_k x[k] * w[n][k] for Q4_K and
// Q6_K weights, one or several independent problems per launch.
//
// Source: DAMASCUS project overview, "[01] the thesis" (decode is one token at
// a time, GEMV-heavy and limited by streaming the weights from memory) and
// "[04] one decode step"; "Building DAMASCUS", "Prefill and decode need
// different performance questions".
//
// The kernel is HBM-bound: every packed weight byte is read once.
//   * Streaming: the weights of 16 consecutive rows are contiguous, so one
//     producer warp fetches a whole 16-row tile (or, for long rows, a 16-row x
//     cb-block chunk, one copy per row) with bulk asynchronous copies into a
//     ring of 2..8 shared-memory stages; with 100+ KB in flight per SM the HBM
//     latency is hidden without holding data in registers.
//   * Arithmetic: 12 compute warps split a stage into blocks (16 rows x 256
//     weights; the two 128-weight halves are independent straight-line code).  The inner products use the warp tensor instruction
//     mma.sync m16n8k16 (fp16 x fp16, fp32 accumulate) as a dot-product
//     engine: a 4-bit quant OR-ed into the mantissa of fp16 1024.0 is the exact
//     value 1024 + F*q (F = 1 or 16 by nibble position, no shifts), its product
//     with an fp16 activation is exact and the sum fp32.  x is replicated over
//     the 8 MMA columns, so every lane holds D = 1024*Sx + F*sum(q*x) of its
//     rows g and g+8 for each sub-block, and
//       sum(w*x) = (d*sc/F)*D - Sx*(1024*d*sc/F + dmin*m)        (Q4_K)
//       sum(w*x) = (d*sc/F)*D - Sx*(1024*d*sc/F + 32*d*sc)       (Q6_K)
//     with Sx the sub-block's sum of x.  Lane tig (0..3) applies the scales
//     of one quarter of each half's sub-blocks, so no scale is decoded twice.  A k-permuted fp16 copy of x and the sums Sx are staged once per
//     CTA in shared memory.
//   * Reduction: partial sums meet in two shuffles and one fixed-order pass
//     over the compute warps per tile (deterministic).
// Q6_K blocks are 210 bytes, so a block can start 2 mod 4 bytes into shared
// memory; its words then come from two aligned loads and a funnel shift.
// Problem kind 1 is the fused gate/up + SwiGLU: a stage holds the gate tile
// and the up tile of the same rows, and the epilogue writes fp16(silu(g)*u).
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
__device__ __forceinline__ float ldsf(uint32_t a) { return __uint_as_float(lds32(a)); }
__device__ __forceinline__ float2 ldsf2(uint32_t a) {
  const uint2 v = lds64(a);
  return make_float2(__uint_as_float(v.x), __uint_as_float(v.y));
}

// 4-byte word at shared address a: 4-byte aligned (A2 = false) or 2 mod 4
// (A2 = true: two aligned loads and a funnel shift).
template <bool A2>
__device__ __forceinline__ uint32_t lds_word(uint32_t a) {
  if constexpr (!A2) {
    return lds32(a);
  } else {
    return __funnelshift_r(lds32(a - 2), lds32(a + 2), 16);
  }
}

__device__ __forceinline__ float half_lo(uint32_t v) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(v & 0xFFFFu)));
}

// v[i] for a lane-dependent i in 0..3.
__device__ __forceinline__ float pick4(float v0, float v1, float v2, float v3, int i) {
  const float a = (i & 1) ? v1 : v0;
  const float b = (i & 1) ? v3 : v2;
  return (i & 2) ? b : a;
}

// ---------------------------------------------------------------------------
// Q4_K half-block U (sub-blocks 4U .. 4U+3, quant bytes 64U .. 64U+63) of the
// lane's rows g (block at shared address b0) and g+8 (b1).  In 64-weight group
// G (sub-blocks 2G, 2G+1, quant bytes 32G .. 32G+31) the lane owns bytes
// 8*tig .. 8*tig+7, i.e. words hh = 0, 1 at 8*tig + 4*hh.  Word hh feeds one
// MMA per sub-block:
//   k-slots 2tig, 2tig+1  <- bytes 0, 2 of the word  (k = 8tig+4hh + 0, 2)
//   k-slots 2tig+8, +9    <- bytes 1, 3              (k = 8tig+4hh + 1, 3)
// which is the order of the permuted x pairs xp[k/4] = {(x0,x2), (x1,x3)}.
// Low nibbles (mask 0x000F000F, F = 1) give sub-block 2G, high nibbles (mask
// 0x00F000F0, F = 16) sub-block 2G+1.  Lane tig then scales sub-block
// j = 4U + tig of both rows.
// ---------------------------------------------------------------------------
template <int U>
__device__ __forceinline__ void q4_half(uint32_t b0, uint32_t b1, uint32_t xa, uint32_t sxa, int tig, uint32_t magic,
                                        float& y0, float& y1) {
  float D[2][2][4];  // [G - 2U][lo, hi][mma regs]
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int G = 2 * U + i;
    const uint2 w0 = lds64(b0 + 16 + 32 * G + 8 * tig);
    const uint2 w1 = lds64(b1 + 16 + 32 * G + 8 * tig);
    const uint4 xlo = lds128(xa + 8 * (16 * G + 2 * tig));      // k = 64G + 8tig + 0..7
    const uint4 xhi = lds128(xa + 8 * (16 * G + 8 + 2 * tig));  // k + 32
    float c[4] = {0.f, 0.f, 0.f, 0.f}, e[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const uint32_t v0 = hh ? w0.y : w0.x, v1 = hh ? w1.y : w1.x;
      const uint32_t s0 = v0 >> 8, s1 = v1 >> 8;
      mma16816(c, lop_and_or<0x000F000Fu>(v0, magic), lop_and_or<0x000F000Fu>(v1, magic),
               lop_and_or<0x000F000Fu>(s0, magic), lop_and_or<0x000F000Fu>(s1, magic), hh ? xlo.z : xlo.x,
               hh ? xlo.w : xlo.y);
      mma16816(e, lop_and_or<0x00F000F0u>(v0, magic), lop_and_or<0x00F000F0u>(v1, magic),
               lop_and_or<0x00F000F0u>(s0, magic), lop_and_or<0x00F000F0u>(s1, magic), hh ? xhi.z : xhi.x,
               hh ? xhi.w : xhi.y);
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      D[i][0][r] = c[r];
      D[i][1][r] = e[r];
    }
  }
  // Sub-block j = 4U + tig: group G = 2U + (tig >> 1), nibble tig & 1.
  const float d0 = pick4(D[0][0][0], D[0][1][0], D[1][0][0], D[1][1][0], tig);
  const float d1 = pick4(D[0][0][2], D[0][1][2], D[1][0][2], D[1][1][2], tig);
  const uint4 h0 = lds128(b0), h1 = lds128(b1);
  const int sh = 8 * tig;
  uint32_t sc0, mn0, sc1, mn1;
  if constexpr (U == 0) {
    sc0 = (h0.y >> sh) & 63u;
    mn0 = (h0.z >> sh) & 63u;
    sc1 = (h1.y >> sh) & 63u;
    mn1 = (h1.z >> sh) & 63u;
  } else {
    const uint32_t l0 = h0.w >> sh, l1 = h1.w >> sh;
    sc0 = (l0 & 0xFu) | ((h0.y >> (sh + 2)) & 0x30u);
    mn0 = ((l0 >> 4) & 0xFu) | ((h0.z >> (sh + 2)) & 0x30u);
    sc1 = (l1 & 0xFu) | ((h1.y >> (sh + 2)) & 0x30u);
    mn1 = ((l1 >> 4) & 0xFu) | ((h1.z >> (sh + 2)) & 0x30u);
  }
  const float inv_f = (tig & 1) ? 0.0625f : 1.0f;
  const float2 sxp = ldsf2(sxa + 8 * (4 * U + tig));  // 16-wide x sums of sub-block j
  const float sx = sxp.x + sxp.y;
  const float dsc0 = half_lo(h0.x) * (float)sc0, dmn0 = half_lo(h0.x >> 16) * (float)mn0;
  const float dsc1 = half_lo(h1.x) * (float)sc1, dmn1 = half_lo(h1.x >> 16) * (float)mn1;
  const float a0 = dsc0 * inv_f, a1 = dsc1 * inv_f;
  y0 = fmaf(a0, d0, fmaf(-fmaf(1024.0f, a0, dmn0), sx, y0));
  y1 = fmaf(a1, d1, fmaf(-fmaf(1024.0f, a1, dmn1), sx, y1));
}

// ---------------------------------------------------------------------------
// Q6_K half H (scale groups 8H .. 8H+7, 128 weights).  Scale group t = 8H + tt
// (tt = 2*g6 + s, g6 = 0..3) takes its low 4 bits from quant bytes
// 64H + 32(g6&1) + 16s + l (low nibble if g6 < 2) and its high 2 bits from
// bits 2*g6 of byte 128 + 32H + 16s + l, l = 0..15.  Lane tig owns
// l = 4tig .. 4tig+3 (one word of each).  The fp16 operand is 1024 + F*q6
// with F = 1 (g6 < 2: nibble in bits 0-3, high bits moved to 4-5) or F = 16
// (g6 >= 2: nibble in bits 4-7, high bits moved to 8-9).  Lane tig scales
// groups 8H + tig and 8H + 4 + tig of both rows.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void q6k_operands(uint32_t wl, uint32_t wh, int g6, uint32_t magic, uint32_t& r0,
                                             uint32_t& r2) {
  const uint32_t wl8 = wl >> 8;
  const uint32_t up = (g6 & 1) ? (wh << 2) : (wh << 4);
  const uint32_t dn = (g6 & 1) ? (wh >> 6) : (wh >> 4);
  if (g6 < 2) {
    r0 = lop_and_or<0x000F000Fu>(wl, lop_and_or<0x00300030u>(up, magic));
    r2 = lop_and_or<0x000F000Fu>(wl8, lop_and_or<0x00300030u>(dn, magic));
  } else {
    r0 = lop_and_or<0x00F000F0u>(wl, lop_and_or<0x03000300u>(up, magic));
    r2 = lop_and_or<0x00F000F0u>(wl8, lop_and_or<0x03000300u>(dn, magic));
  }
}

// The lane's words of one Q6_K half for rows g (block at b0) and g+8 (b1):
// loads only, so a caller may pick A2 per lane.
struct Q6Half {
  uint32_t ql0[4], ql1[4], qh0[2], qh1[2];
  uint32_t sc0[2], sc1[2];  // int8 scale words 192 + 8H + 4u (u = 0, 1)
  uint32_t dw0, dw1;        // the words holding d (low half)
};

template <int H, bool A2>
__device__ __forceinline__ void q6_load_half(uint32_t b0, uint32_t b1, int tig, Q6Half& q) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {  // i = 2p + s: byte 64H + 32p + 16s + 4tig
    const uint32_t off = 64 * H + 32 * (i >> 1) + 16 * (i & 1) + 4 * tig;
    q.ql0[i] = lds_word<A2>(b0 + off);
    q.ql1[i] = lds_word<A2>(b1 + off);
  }
#pragma unroll
  for (int s = 0; s < 2; ++s) {  // byte 128 + 32H + 16s + 4tig
    const uint32_t off = 128 + 32 * H + 16 * s + 4 * tig;
    q.qh0[s] = lds_word<A2>(b0 + off);
    q.qh1[s] = lds_word<A2>(b1 + off);
  }
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    q.sc0[u] = lds_word<A2>(b0 + 192 + 8 * H + 4 * u);
    q.sc1[u] = lds_word<A2>(b1 + 192 + 8 * H + 4 * u);
  }
  q.dw0 = lds_word<A2>(b0 + 208);
  q.dw1 = lds_word<A2>(b1 + 208);
}

template <int H>
__device__ __forceinline__ void q6_half(const Q6Half& q, uint32_t xa, uint32_t sxa, int tig, uint32_t magic, float& y0,
                                        float& y1) {
  float d0[8], d1[8];
#pragma unroll
  for (int tt = 0; tt < 8; ++tt) {
    const int g6 = (tt >> 1) & 3, s = tt & 1;
    const int li = 2 * (g6 & 1) + s;
    uint32_t a0, a2, a1, a3;
    q6k_operands(q.ql0[li], q.qh0[s], g6, magic, a0, a2);
    q6k_operands(q.ql1[li], q.qh1[s], g6, magic, a1, a3);
    const uint2 bx = lds64(xa + 8 * (4 * (8 * H + tt) + tig));
    float c[4] = {0.f, 0.f, 0.f, 0.f};
    mma16816(c, a0, a1, a2, a3, bx.x, bx.y);
    d0[tt] = c[0];
    d1[tt] = c[2];
  }
  // Scale groups 8H + tig (u = 0, F = 1) and 8H + 4 + tig (u = 1, F = 16).
  const float dA = half_lo(q.dw0), dB = half_lo(q.dw1);
  const int sh = 8 * tig;
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const float inv_f = u ? 0.0625f : 1.0f;
    const float dsc0 = dA * (float)(int8_t)((q.sc0[u] >> sh) & 0xFFu);
    const float dsc1 = dB * (float)(int8_t)((q.sc1[u] >> sh) & 0xFFu);
    const float v0 = pick4(d0[4 * u], d0[4 * u + 1], d0[4 * u + 2], d0[4 * u + 3], tig);
    const float v1 = pick4(d1[4 * u], d1[4 * u + 1], d1[4 * u + 2], d1[4 * u + 3], tig);
    const float sx = ldsf(sxa + 4 * (8 * H + 4 * u + tig));
    const float a0 = dsc0 * inv_f, a1 = dsc1 * inv_f;
    y0 = fmaf(a0, v0, fmaf(-fmaf(1024.0f, a0, 32.0f * dsc0), sx, y0));
    y1 = fmaf(a1, v1, fmaf(-fmaf(1024.0f, a1, 32.0f * dsc1), sx, y1));
  }
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------
// Compute warps per CTA (measured on GB300: 12 beat 8 and 16 on the decode
// layer; a K = 3072 tile is 12 blocks, one per warp).
#ifndef QK_GEMV_WARPS
#define QK_GEMV_WARPS 12
#endif
constexpr int kComputeWarps = QK_GEMV_WARPS;
// Sleep between polls of the producer's and the reducer's waits, in ns (0:
// poll back to back).  Those two warps share schedulers with compute warps;
// their waits are hidden by the ring and by the double-buffered partials.
#ifndef QK_GEMV_BACKOFF_NS
#define QK_GEMV_BACKOFF_NS 0
#endif
constexpr uint32_t kBackoffNs = QK_GEMV_BACKOFF_NS;
constexpr int kProducerWarp = kComputeWarps;      // streams the weights (and x)
constexpr int kReducerWarp = kComputeWarps + 1;       // sums the compute warps' partials per tile
constexpr int kThreads = 32 * (kComputeWarps + 2);
constexpr int kMaxStages = 8;

struct GemvProb {
  const uint8_t* w[2];  // weights (gate for kind 1), up weights (kind 1)
  const uint16_t* x;
  void* y;
  int N, K, qtype, kind;
  int pair;         // one tensor, whole rows: a stage holds two adjacent 16-row tiles (as two "tensors")
  int cb;           // K blocks per chunk (a stage holds 16 rows x cb blocks per weight tensor)
  int stages;       // pipeline depth of this problem's CTAs
  uint32_t stage_bytes;
  int tiles, cta_begin, ctas;
};

struct GemvBatch {
  GemvProb p[kMaxGemvProbs];
  int count;
};

struct GemvShared;
constexpr uint32_t round128(size_t v) { return (uint32_t)((v + 127) / 128 * 128); }

struct GemvShared {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t x_full;                     // x copied into shared memory
  uint64_t red_full[2];                // every compute warp wrote its partials of a tile (by parity)
  uint64_t red_free[2];                // the reducer has consumed them
  float red[2][kComputeWarps][2][16];  // [tile parity][warp][tensor][row]
  uint32_t abort_flag;
};
constexpr uint32_t kSharedBytes = round128(sizeof(GemvShared));


template <int QT>
__device__ __forceinline__ void run_gemv_problem(const GemvProb& P, int cta, const GemvBatch& B, uint8_t* smem,
                                                 uint8_t* stages, GemvShared* sh) {
  const int K = P.K, N = P.N, nb = K / kQK, cb = P.cb;
  constexpr int kBB = QT == kQ4K ? kQ4KBytes : kQ6KBytes;
  const int64_t RB = (int64_t)nb * kBB;
  // Tiles of a stage: gate and up (kind 1), two adjacent 16-row tiles of one
  // tensor (pair), or one tile.  "tile" below is a stage's worth of rows.
  const int nten = (P.kind == 1 || P.pair) ? 2 : 1;
  const int tile_rows = P.pair ? 32 : 16;
  const int nchunks = nb / cb;  // the host makes cb divide nb
  const int t0 = (int)((int64_t)cta * P.tiles / P.ctas), t1 = (int)((int64_t)(cta + 1) * P.tiles / P.ctas);
  const int steps = (t1 - t0) * nchunks;
  const int S = P.stages;
  const uint32_t SB = P.stage_bytes;
  const uint32_t ten_bytes = (uint32_t)(16 * cb * kBB);  // one tensor's share of a stage
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile uint32_t* abort_flag = &sh->abort_flag;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int st = 0;
      for (; st < steps; ++st) {
        const int s = st % S;
        if (!mbar_wait<kBackoffNs>(&sh->empty[s], ((uint32_t)(st / S) & 1u) ^ 1u, abort_flag, &g_gemv_status))
          break;
        // The compute warps read the stage with plain loads; the refill is an
        // async-proxy write.  The proxy fence after the barrier their releases
        // completed orders those reads before the copy.
        fence_proxy_async_smem();
        const int tile = t0 + st / nchunks, chunk = st % nchunks;
        const int n0 = tile * tile_rows, rows = min(16, N - n0);
        uint8_t* dst = stages + (size_t)s * SB;
        if (cb == nb) {
          // Whole 16-row tiles: rows nt .. nt+rows_t-1 of a tensor are one
          // contiguous span (pair: tile t starts 16 rows further).
          uint32_t total = 0;
          for (int t = 0; t < nten; ++t) {
            const int rows_t = min(16, N - (n0 + (P.pair ? 16 * t : 0)));
            if (rows_t > 0) total += (uint32_t)(((int64_t)rows_t * RB) & ~int64_t(15));
          }
          mbar_expect_tx(&sh->full[s], total);
          for (int t = 0; t < nten; ++t) {
            const int nt = n0 + (P.pair ? 16 * t : 0), rows_t = min(16, N - nt);
            if (rows_t <= 0) continue;
            const int64_t span = (int64_t)rows_t * RB;
            const uint32_t bulk = (uint32_t)(span & ~int64_t(15));
            const uint8_t* src = P.w[P.pair ? 0 : t] + (int64_t)nt * RB;
            uint8_t* d = dst + t * ten_bytes;
            if (bulk) bulk_copy_g2s(d, src, bulk, &sh->full[s]);
            for (int64_t b = bulk; b < span; b += 2)  // last bytes of the tensor (span % 16 != 0)
              *reinterpret_cast<uint16_t*>(d + b) = *reinterpret_cast<const uint16_t*>(src + b);
          }
        } else {
          // A K chunk: one copy per row of cb blocks (16-byte aligned by construction).
          const uint32_t row_bytes = (uint32_t)(cb * kBB);
          mbar_expect_tx(&sh->full[s], row_bytes * (uint32_t)(rows * nten));
          for (int t = 0; t < nten; ++t)
            for (int r = 0; r < rows; ++r)
              bulk_copy_g2s(dst + t * ten_bytes + r * row_bytes,
                            P.w[t] + (int64_t)(n0 + r) * RB + (int64_t)chunk * cb * kBB, row_bytes, &sh->full[s]);
        }
        mbar_arrive(&sh->full[s]);
        // Let the first stage of every CTA land before queueing the rest, so
        // the compute warps start while the other stages stream in.
        if (st == 0 && steps > 1 && !mbar_wait(&sh->full[0], 0u, abort_flag, &g_gemv_status)) {
          ++st;
          break;
        }
      }
      // Drain: the copies issued last have landed before the CTA can exit.
      for (int i = 1; i <= S && i <= st; ++i)
        mbar_wait(&sh->full[(st - i) % S], (uint32_t)((st - i) / S) & 1u, abort_flag, &g_gemv_status, true);
    }
    return;
  }

  if (warp == kReducerWarp) {
    // ------------------------------------------------------------ reducer
    // Tile i's partials sit in red[i & 1]; sum them over the compute warps in
    // a fixed order (deterministic) and write y.
    const int ntiles = t1 - t0;
    for (int i = 0; i < ntiles; ++i) {
      const int par = i & 1;
      if (!mbar_wait<kBackoffNs>(&sh->red_full[par], (uint32_t)(i >> 1) & 1u, abort_flag, &g_gemv_status)) break;
      if (P.kind == 1) {
        if (lane < 16) {
          const int n = (t0 + i) * 16 + lane;
          float gs = 0.f, us = 0.f;
          for (int w = 0; w < kComputeWarps; ++w) gs += sh->red[par][w][0][lane];
          for (int w = 0; w < kComputeWarps; ++w) us += sh->red[par][w][1][lane];
          if (n < N) static_cast<__half*>(P.y)[n] = __float2half_rn(gs / (1.0f + __expf(-gs)) * us);
        }
      } else if (lane < 16 * nten) {  // lane 16t + r: row r of tile t of the stage
        const int t = lane >> 4, r = lane & 15;
        const int n = (t0 + i) * tile_rows + 16 * t + r;
        float gs = 0.f;
        for (int w = 0; w < kComputeWarps; ++w) gs += sh->red[par][w][t][r];
        if (n < N) static_cast<float*>(P.y)[n] = gs;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh->red_free[par]);
    }
    return;
  }

  // -------------------------------------------------------------- compute
  const uint32_t xs = smem_u32(smem);             // permuted x pairs, 8 bytes per 4 k
  const uint32_t sxs = smem_u32(smem + 2 * K);    // 16-wide sums of x
  const uint32_t ring = smem_u32(stages);
  const int g = lane >> 2, tig = lane & 3;
  // fp16x2 (1024, 1024), kept in a register for the LOP3s that build the MMA operands
  uint32_t magic;
  asm volatile("mov.b32 %0, %1;" : "=r"(magic) : "n"(kMagic));
  const uint32_t pitch = (cb == nb) ? (uint32_t)RB : (uint32_t)(cb * kBB);  // bytes per row inside a stage
  float ya0 = 0.f, ya1 = 0.f, yb0 = 0.f, yb1 = 0.f;  // rows g, g+8 of tensor 0 (a) and 1 (b)
  bool ok = true;
  for (int st = 0; st < steps; ++st) {
    const int s = st % S;
    const int chunk = st % nchunks;
    // After a timed-out wait the warp skips the arithmetic but still hands its
    // partials of every tile to the reducer, so the reducer is not left waiting.
    if (ok)
      ok = __all_sync(0xffffffffu, mbar_wait(&sh->full[s], (uint32_t)(st / S) & 1u, abort_flag, &g_gemv_status));
    const uint32_t stg = ring + (uint32_t)s * SB + (uint32_t)g * pitch;
    // Warp w takes whole blocks v = w, w + kComputeWarps, ...: v = t*cb + b; both
    // halves of a block are independent straight-line work (more ILP per warp).
    int t = 0, b = warp;
    while (b >= cb) {
      b -= cb;
      ++t;
    }
    for (int v = warp; ok && v < nten * cb; v += kComputeWarps) {
      const uint32_t b0 = stg + (uint32_t)t * ten_bytes + (uint32_t)(b * kBB);
      const uint32_t b1 = b0 + 8 * pitch;
      const int blk = chunk * cb + b;
      const uint32_t xa = xs + (uint32_t)blk * 512u, sxa = sxs + (uint32_t)blk * 64u;
      float y0 = 0.f, y1 = 0.f, z0 = 0.f, z1 = 0.f;
      if constexpr (QT == kQ4K) {
        q4_half<0>(b0, b1, xa, sxa, tig, magic, y0, y1);
        q4_half<1>(b0, b1, xa, sxa, tig, magic, z0, z1);
      } else {
        const bool a2 = (b0 & 3u) != 0;
        Q6Half q, r;
        if (a2) {
          q6_load_half<0, true>(b0, b1, tig, q);
          q6_load_half<1, true>(b0, b1, tig, r);
        } else {
          q6_load_half<0, false>(b0, b1, tig, q);
          q6_load_half<1, false>(b0, b1, tig, r);
        }
        __syncwarp();
        q6_half<0>(q, xa, sxa, tig, magic, y0, y1);
        q6_half<1>(r, xa, sxa, tig, magic, z0, z1);
      }
      if (t == 0) {
        ya0 += y0 + z0;
        ya1 += y1 + z1;
      } else {
        yb0 += y0 + z0;
        yb1 += y1 + z1;
      }
      b += kComputeWarps;
      while (b >= cb) {
        b -= cb;
        ++t;
      }
    }
    __syncwarp();
    if (ok && lane == 0) mbar_arrive(&sh->empty[s]);
    if (chunk == nchunks - 1) {  // tile done: reduce over lanes, hand the warp's partials to the reducer
      const int ti = st / nchunks, par = ti & 1;
      // red[par] was last used by tile ti - 2: wait until the reducer is done with it.
      if (ti >= 2)
        ok = __all_sync(0xffffffffu, mbar_wait(&sh->red_free[par], (uint32_t)((ti >> 1) - 1) & 1u, abort_flag,
                                               &g_gemv_status)) && ok;
      for (int t = 0; t < nten; ++t) {
        float a = t ? yb0 : ya0, c = t ? yb1 : ya1;
        a += __shfl_xor_sync(0xffffffffu, a, 1);
        a += __shfl_xor_sync(0xffffffffu, a, 2);
        c += __shfl_xor_sync(0xffffffffu, c, 1);
        c += __shfl_xor_sync(0xffffffffu, c, 2);
        if (tig == 0) {
          sh->red[par][warp][t][g] = a;
          sh->red[par][warp][t][g + 8] = c;
        }
      }
      ya0 = ya1 = yb0 = yb1 = 0.f;
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh->red_full[par]);
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1) gemv_stream_kernel(const __grid_constant__ GemvBatch B) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  int i = 0;
  while (i + 1 < B.count && (int)blockIdx.x >= B.p[i + 1].cta_begin) ++i;
  const GemvProb& P = B.p[i];
  const int cta = (int)blockIdx.x - P.cta_begin;
  int kmax = 0;
  for (int j = 0; j < B.count; ++j) kmax = max(kmax, B.p[j].K);
  const uint32_t x_bytes = ((uint32_t)(2 * kmax + kmax / 4) + 127u) & ~127u;
  // [x | barriers and partial sums | ring of this problem's stages]
  GemvShared* sh = reinterpret_cast<GemvShared*>(smem + x_bytes);
  uint8_t* stages = smem + x_bytes + kSharedBytes;
  if (threadIdx.x < (unsigned)P.stages) {
    mbar_init(&sh->full[threadIdx.x], 1);
    mbar_init(&sh->empty[threadIdx.x], kComputeWarps);
  }
  if (threadIdx.x == 0) {
    mbar_init(&sh->x_full, 1);
    for (int p = 0; p < 2; ++p) {
      mbar_init(&sh->red_full[p], kComputeWarps);
      mbar_init(&sh->red_free[p], 1);
    }
    sh->abort_flag = 0;
  }
  fence_mbar_init();
  __syncthreads();
  // x arrives with one bulk copy (the producer then streams the weights) and
  // the compute warps rearrange it in place: xp[k/4] = { fp16x2(x[k], x[k+2]),
  // fp16x2(x[k+1], x[k+3]) }, the MMA k-slot order of the quant words, and
  // sx16[i] = sum of x[16i .. 16i+15] in fp32.
  if (threadIdx.x == 32 * kProducerWarp) {
    mbar_arrive_expect_tx(&sh->x_full, (uint32_t)(2 * P.K));
    bulk_copy_g2s(smem, P.x, (uint32_t)(2 * P.K), &sh->x_full);
  }
  if (threadIdx.x < 32 * kComputeWarps) {
    mbar_wait(&sh->x_full, 0u, &sh->abort_flag, &g_gemv_status);
    const int nq = P.K / 4;
    uint2* xp = reinterpret_cast<uint2*>(smem);
    float* sx16 = reinterpret_cast<float*>(smem + 2 * P.K);
    for (int q = threadIdx.x; q < nq; q += 32 * kComputeWarps) {
      const uint2 v = xp[q];
      uint2 o;
      o.x = prmt(v.x, v.y, 0x5410u);
      o.y = prmt(v.x, v.y, 0x7632u);
      xp[q] = o;
      float s = (half_lo(v.x) + half_lo(v.x >> 16)) + (half_lo(v.y) + half_lo(v.y >> 16));
      s += __shfl_xor_sync(0xffffffffu, s, 1);
      s += __shfl_xor_sync(0xffffffffu, s, 2);
      if ((q & 3) == 0) sx16[q >> 2] = s;
    }
    asm volatile("bar.sync 1, %0;" ::"n"(32 * kComputeWarps) : "memory");
  }
  if (P.qtype == kQ4K)
    run_gemv_problem<kQ4K>(P, cta, B, smem, stages, sh);
  else
    run_gemv_problem<kQ6K>(P, cta, B, smem, stages, sh);
}

}  // namespace

int gemv_max_m() { return 1; }

uint32_t gemv_take_status() {
  uint32_t v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_gemv_status, sizeof(v)) != cudaSuccess) return 0;
  cudaMemcpyToSymbol(g_gemv_status, &zero, sizeof(zero));
  return v;
}

namespace {

constexpr size_t kGemvSmem = 227 * 1024;

// The stage geometry of one grouped GEMV launch (host only, no CUDA call):
// each problem gets its own stages (its CTAs carve their own ring), and the
// CTAs (one per SM, `sms` of them) split across problems in proportion to
// their weight bytes.  False if some problem has no plan that fits shared
// memory (x of the largest K plus at least two stages).
bool plan_gemv(const GemvDesc* d, int count, int sms, GemvBatch* out, size_t* smem_out) {
  if (count <= 0 || count > kMaxGemvProbs) return false;
  GemvBatch& B = *out;
  memset(&B, 0, sizeof(B));
  B.count = count;
  int64_t kmax = 0;
  for (int i = 0; i < count; ++i) kmax = std::max<int64_t>(kmax, d[i].K);
  const size_t x_bytes = ((size_t)(2 * kmax + kmax / 4) + 127) / 128 * 128;
  if (x_bytes + kSharedBytes + 128 >= kGemvSmem) return false;
  const size_t avail = kGemvSmem - x_bytes - kSharedBytes - 128;  // for one CTA's ring
  double total = 0;
  int64_t bytes[kMaxGemvProbs];
  size_t ring = 0;
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
    const int bb = P.qtype == kQ4K ? kQ4KBytes : kQ6KBytes;
    const int nten = 1 + P.kind;
    const int64_t RB = (int64_t)nb * bb;
    // Stage: whole rows (cb = K/256) when three stages fit, else the largest
    // multiple of 8 blocks (8 x 210 B is 16-byte aligned) dividing K/256 that
    // gives three stages.
    int cb = nb;
    if ((size_t)3 * 16 * nten * nb * bb > avail) {
      cb = 0;
      for (int c = 8; c <= nb; c += 8)
        if (nb % c == 0 && (size_t)3 * 16 * nten * c * bb <= avail && (RB % 16) == 0) cb = c;
      if (cb == 0) cb = nb;  // fall back to whole rows with fewer stages
    }
    P.cb = cb;
    // One tensor with whole rows: two adjacent tiles per stage (halves the
    // per-block share of the per-tile reduction) when two such stages fit
    // (measured on GB300: the Q6_K LM head streams ~15 % faster with two
    // paired stages than with five single ones).
    P.pair = (P.kind == 0 && cb == nb && P.N > 16 && 2 * (size_t)round128((size_t)32 * nb * bb) <= avail) ? 1 : 0;
    P.stage_bytes = round128((size_t)16 * (nten + P.pair) * cb * bb);
    P.stages = (int)std::min<size_t>(kMaxStages, avail / P.stage_bytes);
    if (P.stages < 2) return false;
    ring = std::max(ring, (size_t)P.stages * P.stage_bytes);
    P.tiles = (P.N + 16 * (1 + P.pair) - 1) / (16 * (1 + P.pair));
    bytes[i] = (int64_t)P.N * RB * nten;
    total += (double)bytes[i];
  }
  *smem_out = x_bytes + kSharedBytes + ring + 128;
  const int budget = std::max(count, sms);
  int used = 0;
  for (int i = 0; i < count; ++i) {
    int c = (int)((double)budget * (double)bytes[i] / total);
    c = std::max(1, std::min(c, B.p[i].tiles));
    B.p[i].ctas = c;
    used += c;
  }
  for (bool again = true; again && used < budget;) {  // leftover CTAs to the busiest problems
    again = false;
    int best = -1;
    double best_load = 0.0;
    for (int i = 0; i < count; ++i) {
      const double load = (double)bytes[i] / B.p[i].ctas;
      if (B.p[i].ctas < B.p[i].tiles && load > best_load) {
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
  return *smem_out <= kGemvSmem;
}

}  // namespace

bool gemv_plan_fits(const GemvDesc* d, int count) {
  GemvBatch B;
  size_t smem = 0;
  return plan_gemv(d, count, 152, &B, &smem);  // the SM count splits CTAs; it does not decide the fit
}

// Launch one grouped GEMV (see plan_gemv).
cudaError_t launch_gemv_batch(const GemvDesc* d, int count, cudaStream_t s) {
  GemvBatch B;
  size_t smem = 0;
  if (!plan_gemv(d, count, device_sms(), &B, &smem)) return cudaErrorInvalidConfiguration;
  static PerDeviceFlag attr;  // the shared-memory limit is a per-device function attribute
  const int dev = current_device();
  if (!attr.done(dev)) {
    cudaError_t e =
        cudaFuncSetAttribute(gemv_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGemvSmem);
    if (e != cudaSuccess) return e;
    attr.mark(dev);
  }
  int ctas = 0;
  for (int i = 0; i < B.count; ++i) ctas += B.p[i].ctas;
  gemv_stream_kernel<<<ctas, kThreads, smem, s>>>(B);
  return cudaGetLastError();
}

cudaError_t launch_gemv(QType t, const void* W, const uint16_t* x, float* y, int64_t N, int64_t K,
                        cudaStream_t s) {
  GemvDesc d{t, W, nullptr, x, y, N, K};
  return launch_gemv_batch(&d, 1, s);
}

}  // namespace qk
