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
// The kernel: one 16-row tile per CTA iteration, `ks` warps split the K blocks.
// Shared memory: xp (2K bytes), sx16 (K/4 bytes), partial sums (ks*16 floats).
// ---------------------------------------------------------------------------
// The kernel: each CTA iteration covers `tpc` 16-row tiles; the `ks` warps of
// a tile split its K/256 blocks.  Each warp issues the loads of its first
// block before the CTA stages x, and loads the next block (or the next tile's
// first block) while it computes the current one.  Shared memory: xp (2K
// bytes), sx16 (K/4 bytes), partial sums (tpc*ks*16 floats).
template <int QT>
__global__ void __maxnreg__(128) gemv_m1_kernel(const uint8_t* __restrict__ W,
                                                      const uint16_t* __restrict__ x, float* __restrict__ y, int N,
                                                      int K, int ks, int tpc) {
  extern __shared__ __align__(16) uint8_t smem[];
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
  const int stride = gridDim.x * tpc;

  auto row_ptr = [&](int tile, int which) {
    const int r = min(tile * 16 + g + 8 * which, N - 1);
    return W + r * RB;
  };

  BlockRegs<QT> cur;
  int tile = blockIdx.x * tpc + sub;
  if (tile < ntiles) load_block(cur, row_ptr(tile, 0) + b_begin * kBB, row_ptr(tile, 1) + b_begin * kBB, tig);
  stage_x(x, K, xp, sx16);
  __syncthreads();

  for (int tile0 = blockIdx.x * tpc; tile0 < ntiles; tile0 += stride) {
    tile = tile0 + sub;
    float y0 = 0.f, y1 = 0.f;
    if (tile < ntiles) {
      const uint8_t* row0 = row_ptr(tile, 0);
      const uint8_t* row1 = row_ptr(tile, 1);
      for (int b = b_begin; b < b_begin + bpw; ++b) {
        BlockRegs<QT> nxt;
        if (b + 1 < b_begin + bpw) {
          load_block(nxt, row0 + (b + 1) * kBB, row1 + (b + 1) * kBB, tig);
        } else if (tile + stride < ntiles) {
          load_block(nxt, row_ptr(tile + stride, 0) + b_begin * kBB, row_ptr(tile + stride, 1) + b_begin * kBB,
                     tig);
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
    if (threadIdx.x < 16 * tpc) {
      const int t = threadIdx.x >> 4, r = threadIdx.x & 15;
      float acc = 0.f;
      for (int w = 0; w < ks; ++w) acc += red[(t * ks + w) * 16 + r];
      const int row = (tile0 + t) * 16 + r;
      if (row < N) y[row] = acc;
    }
    __syncthreads();
  }
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

// Launch shape.  ks warps split the K/256 blocks of a 16-row tile (ks divides
// the block count, ks <= 12); tpc tiles share a CTA when ks is small.  With up
// to 128 registers a thread, an SM holds 512 threads, so a CTA of T threads
// gets floor(512 / T) slots per SM.  Prefer the largest ks (shortest per-warp
// chains, most loads in flight) whose CTAs all fit in one wave.
struct GemvShape {
  int ks, tpc, threads;
  int64_t grid;
};

static GemvShape choose_shape(int64_t N, int nb) {
  const int64_t tiles = (N + 15) / 16;
  const int64_t sms = sm_count();
  GemvShape best{1, 8, 256, 0};
  for (int d = std::min(nb, 12); d >= 1; --d) {
    if (nb % d) continue;
    const int tpc = std::max(1, 4 / d);
    const int threads = 32 * d * tpc;
    const int64_t slots = sms * std::max(1, 512 / threads);
    const int64_t ctas = (tiles + tpc - 1) / tpc;
    if (ctas <= slots) return GemvShape{d, tpc, threads, ctas};
  }
  best.grid = std::min<int64_t>((tiles + best.tpc - 1) / best.tpc, sms * 2);
  return best;
}

cudaError_t launch_gemv(QType t, const void* W, const uint16_t* x, float* y, int64_t N, int64_t K,
                        cudaStream_t s) {
  const int nb = (int)(K / kQK);
  const GemvShape sh = choose_shape(N, nb);
  const size_t smem = (size_t)2 * K + (size_t)K / 4 + (size_t)sh.tpc * sh.ks * 16 * sizeof(float);
  if (t == kQ4K) {
    if (smem > 48 * 1024)
      cudaFuncSetAttribute(gemv_m1_kernel<kQ4K>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    gemv_m1_kernel<kQ4K><<<(int)sh.grid, sh.threads, smem, s>>>(static_cast<const uint8_t*>(W), x, y, (int)N, (int)K,
                                                                sh.ks, sh.tpc);
  } else {
    if (smem > 48 * 1024)
      cudaFuncSetAttribute(gemv_m1_kernel<kQ6K>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    gemv_m1_kernel<kQ6K><<<(int)sh.grid, sh.threads, smem, s>>>(static_cast<const uint8_t*>(W), x, y, (int)N, (int)K,
                                                                sh.ks, sh.tpc);
  }
  return cudaGetLastError();
}

}  // namespace qk
