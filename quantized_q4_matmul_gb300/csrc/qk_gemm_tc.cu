// qk_gemm_tc.cu -- prefill GEMM on the 5th-generation tensor cores (tcgen05):
// y[m][n] = sum_k x[m][k] * w[n][k] with Q4_K / Q6_K weights dequantized on
// the fly, plus the fused gate/up + SwiGLU variant.
//
// Source: DAMASCUS project overview, "[01] the thesis" (prefill takes every
// prompt token in one pass as matrix-matrix products bound by arithmetic, and
// the dequantized weights go straight to the matrix unit, so no fp16 copy of
// them is ever stored) and "[04] one decode step"
// (QKV, SwiGLU FFN, LM head over every prompt position); "Building DAMASCUS",
// "Prefill and decode need different performance questions".
//
// Design (one CTA per 128-weight-row x BN-token output tile, swap-AB so the
// weights are the UMMA A operand with M = 128 and the tokens are N = BN):
//   warp 0      producer: TMA loads of the x tile (BN x 64 fp16, 128-byte
//               swizzle) per 64-wide K step, and (one Q4_K tensor) of the
//               packed blocks of the 128 weight rows per 256-wide super-block.
//   warps 1, 2  UMMA issuers (warp 1 also allocates tensor memory): one thread
//               of each issues tcgen05.mma (kind::f16, fp32 accumulate in
//               TMEM) and tcgen05.commit for its own accumulator: the gate
//               and up tensors, or the even and odd K steps of one tensor.
//   warps 3..   dequantize the packed blocks into fp16 A tiles, written
//               straight into shared memory in the UMMA 128-byte-swizzle
//               K-major layout or into tensor memory (the fp16 weights never
//               touch device memory), then run the epilogue: tcgen05.ld of
//               the accumulator, fp32 y stores or silu(g) * u -> fp16.
//   last warp   (gate/up and Q6_K) copies of the packed blocks, at their own
//               pace.
// Pipelines: packed blocks (P stages, one super-block each), x tiles (SX
// stages) and A tiles (SA stages), the last two released per K step by the
// step's UMMA commit (done barriers, a ring of max(SX, SA)).  Grids that
// would leave half of the SMs idle split K across a thread-block cluster of
// 2..8 CTAs per tile: each CTA owns a slice of the tile's token columns,
// receives the peers' fp32 partials of that slice by bulk shared::cluster
// copies and adds them in rank order (no global scratch, deterministic).
// All waits are bounded mbarrier waits; a timeout raises a device status flag
// and the CTA drains and exits.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>
#include <utility>

#include "qk_device.cuh"
#include "qk_internal.h"

namespace qk {

__device__ uint32_t g_gemm_status = 0;

namespace {

constexpr int kBM = 128;               // weight rows per tile (UMMA M)
constexpr int kBK = 64;                // K per step: one 128-byte swizzle row of fp16
constexpr int kMaxBN = 256;            // tokens per tile (UMMA N), multiple of 16
constexpr int kAStageBytes = kBM * kBK * 2;     // 16 KB
constexpr uint32_t kH2Magic = 0x64646464u;
// UMMA issuer warps.  tcgen05.commit holds its issuing thread until that
// thread's earlier UMMAs have completed, so a single issuer that commits after
// every K step leaves the tensor pipe idle for the commit's latency; two
// issuers, each committing its own steps, keep it fed.  Each issuer owns one
// accumulator (the gate / up tensor, or the even / odd K steps of a single
// tensor, summed in a fixed order in the epilogue), so results stay
// deterministic.
constexpr int kIssuers = 2;

// Q6_K: bytes of the 16-byte-aligned window staged for each 210-byte block
// (the block plus its misalignment, up to 14 bytes, fits in 224).  240 rather
// than 224: at a 60-word pitch the 16-byte loads of 8 consecutive rows cover
// all 32 shared-memory banks (at 56 words every fourth row collided; ncu
// counted 74 % of the Q6_K kernel's shared wavefronts as bank conflicts).
constexpr int kQ6Win = 240;

// Sleep between polls of the copy warps' waits (x tiles and packed blocks),
// in ns; 0 polls back to back.  Those warps share schedulers with dequant
// warps, and their waits are hidden by the rings.
#ifndef QK_GEMM_BACKOFF_NS
#define QK_GEMM_BACKOFF_NS 0
#endif
constexpr uint32_t kCopyBackoffNs = QK_GEMM_BACKOFF_NS;

// Deepest x-tile ring of single-tensor problems (even, <= 8) and deepest
// packed-block ring (<= 4).
#ifndef QK_GEMM_MAX_X
#define QK_GEMM_MAX_X 8
#endif
#ifndef QK_GEMM_MAX_P
#define QK_GEMM_MAX_P 2
#endif

template <int QT, bool GATEUP>
struct Cfg {
  // Dequant warps: two threads per weight row and tensor (each dequantizes
  // half of every K step), i.e. two warps per SM sub-partition per tensor.
  static constexpr int kDqWarps = GATEUP ? 16 : 8;
  // Gate/up and Q6_K: the packed blocks come from a warp of their own, after
  // the dequant warps (measured faster on GB300: the packed copies no longer
  // wait behind the x ring, nor the x copies behind lanes polling for free
  // packed slots); one Q4_K tensor: warp 0 issues both, packed block first.
  static constexpr bool kSplit = GATEUP || QT == kQ6K;
  static constexpr int kThreads = 32 * (1 + kIssuers + kDqWarps + (kSplit ? 1 : 0));
  static constexpr int kDqWarp0 = 1 + kIssuers;  // first dequant warp
  static constexpr int kPackedWarp = kDqWarp0 + kDqWarps;  // with kSplit
  static constexpr int kNumB = GATEUP ? 2 : 1;  // weight tensors per tile
  // Arrivals that complete an A stage: Q4_K threads each write half of every
  // step; Q6_K threads write two of every four steps in full.
  static constexpr int kAArrivals = QT == kQ4K ? 32 * kDqWarps : 32 * kDqWarps / 2;
  // One packed-block stage holds a super-block of the tile's rows per tensor.
  static constexpr int kPSlotBytes = QT == kQ4K ? kBM * kQ4KBytes : kBM * kQ6Win;
};

struct Bars {  // capacity: 8 x / A stages, 4 packed stages
  uint64_t x_full[8];
  uint64_t a_full[8];
  uint64_t done[8];  // done[t % D]: the UMMAs of K step t completed (frees its A and x slots)
  uint64_t p_full[4];
  uint64_t p_empty[4];
  uint64_t acc_full;
  uint64_t peer_full;  // split K: the peers' partial slices of this CTA's token chunks have landed
  uint32_t tmem_base;
  uint32_t abort_flag;
};
constexpr uint32_t kBarsBytes = (sizeof(Bars) + 127) / 128 * 128;

// Shared-memory carve-up for a token tile BN, SX x-tile stages, SA A-tile
// stages and P packed stages (x and A offsets 1024-byte aligned for the
// 128-byte swizzle atoms).
struct Layout {
  uint32_t x_off, x_stage, a_off, p_off, bar_off, total;
};

template <int QT, bool GATEUP, bool AT>
__host__ __device__ inline Layout make_layout(int BN, int SX, int SA, int P) {
  using C = Cfg<QT, GATEUP>;
  Layout L;
  L.x_stage = (uint32_t)BN * kBK * 2;
  L.x_off = 0;
  L.a_off = L.x_off + (uint32_t)SX * L.x_stage;
  L.p_off = L.a_off + (AT ? 0u : (uint32_t)(SA * C::kNumB) * kAStageBytes);
  L.bar_off = L.p_off + (uint32_t)(P * C::kNumB * C::kPSlotBytes);
  L.total = L.bar_off + kBarsBytes + 1024;  // barriers + base alignment slack
  return L;
}



// Split-K exchange geometry.  The tile's BN / 16 token chunks are dealt to the
// ks CTAs of a cluster in contiguous slices; a slot holds one slice's partial
// sums for kNumB tensors: [tensor][128 rows][slice chunks x 16 fp32], rows
// padded by 16 bytes so a warp's 16-byte accesses to 32 consecutive rows
// spread over all banks.
__host__ __device__ inline uint32_t split_slot_pitch(int BN, int ks) {
  return (uint32_t)((BN / 16 + ks - 1) / ks) * 64u + 16u;
}
template <int kNumB>
__host__ __device__ inline uint32_t split_slot_bytes(int BN, int ks) {
  return (uint32_t)kNumB * 128u * split_slot_pitch(BN, ks);
}
// Rank zz's slice is chunks [c(zz), c(zz + 1)) of n = BN / 16, with
// c(zz) = ceil(zz * n / ks) (rank 0 always owns a chunk); with fewer chunks
// than ranks some slices are empty, and those ranks receive nothing.
// min(ks, n) ranks own a slice; below rank zz there are min(zz, c(zz)) owners.
__host__ __device__ inline int split_chunk(int zz, int BN, int ks) { return (zz * (BN / 16) + ks - 1) / ks; }
__host__ __device__ inline bool split_owns(int zz, int BN, int ks) {
  return split_chunk(zz + 1, BN, ks) > split_chunk(zz, BN, ks);
}
// Shared memory of the exchange: an owner keeps ks - 1 receive slots, then
// one send slot per other owner; a rank without a slice only sends, one slot
// per owner from the start of the region.
template <int kNumB>
__host__ __device__ inline uint32_t split_exchange_bytes(int BN, int ks) {
  const int owners = ks < BN / 16 ? ks : BN / 16;
  const int slots = ks - 2 + owners > owners ? ks - 2 + owners : owners;
  return (uint32_t)slots * split_slot_bytes<kNumB>(BN, ks);
}

struct Params {
  const uint8_t* w[2];  // packed weights (gate, up)
  int64_t w_bytes;      // bytes of each weight tensor
  void* y;
  int M, N, K, BN;
  int stages;           // x-tile stages SX
  int astages;          // A-tile stages SA (the dequant may run SA steps ahead of the UMMAs; Q6_K: 4)
  int pstages;          // packed-block pipeline depth P
  int ksplit;           // CTAs of a cluster that split the K range of one tile (1 = no split)
  int q6_group;         // Q6_K: rows per tensor-map row (g: g * row_bytes % 16 == 0)
  int q6_rows_tma;      // Q6_K: rows covered by the tensor map, (N / g) * g
};

__device__ __forceinline__ float h2f(uint32_t bits) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(bits & 0xFFFFu)));
}

__device__ __forceinline__ uint32_t h2_bits(__half2 v) { return *reinterpret_cast<uint32_t*>(&v); }

__device__ __forceinline__ __half2 bits_h2(uint32_t v) { return *reinterpret_cast<__half2*>(&v); }

// Offset of 16-byte chunk j (k = 8j .. 8j+7) of row r in a 128 x 64 fp16 tile
// stored in the UMMA 128-byte-swizzle K-major layout.
__device__ __forceinline__ uint32_t sw128_off(int r, int j) { return (uint32_t)(r * 128 + ((j ^ (r & 7)) << 4)); }

// Four weights from four quant bytes (each < 16) of `b4`: the byte goes into
// the mantissa of 1024.0 (exact fp16 1024 + q), 1024 is subtracted exactly,
// then w = fp16(q * dsc - dmn); the two results hold k, k+1 and k+2, k+3.
__device__ __forceinline__ void q4_emit4(uint32_t b4, __half2 dsc2, __half2 ndmn2, uint4& out0) {
  // b4 holds four quant values (one per byte) for k, k+1, k+2, k+3.
  const __half2 k1024 = __float2half2_rn(1024.0f);
  const __half2 p0 = __hsub2(bits_h2(prmt(b4, kH2Magic, 0x4140u)), k1024);
  const __half2 p1 = __hsub2(bits_h2(prmt(b4, kH2Magic, 0x4342u)), k1024);
  out0.x = h2_bits(__hfma2(p0, dsc2, ndmn2));
  out0.y = h2_bits(__hfma2(p1, dsc2, ndmn2));
}

// Scale and min of sub-block j (0..7) from the 12 packed bytes held in three
// little-endian words s03, s47, s811.
__device__ __forceinline__ void q4_scale_min(uint32_t s03, uint32_t s47, uint32_t s811, int j, float& sc,
                                             float& mn) {
  uint32_t a, b;
  if (j < 4) {
    a = (s03 >> (8 * j)) & 63u;
    b = (s47 >> (8 * j)) & 63u;
  } else {
    const int jj = j - 4;
    const uint32_t lo = (s811 >> (8 * jj)) & 0xFFu;
    a = (lo & 0xFu) | (((s03 >> (8 * jj + 6)) & 3u) << 4);
    b = (lo >> 4) | (((s47 >> (8 * jj + 6)) & 3u) << 4);
  }
  sc = (float)a;
  mn = (float)b;
}

// One thread's share of a Q4_K super-block row, held in registers: the 128
// quant bytes and, for the sub-blocks 2c + PART (c = 0..3) this thread
// dequantizes, fp16x2 (d*sc) and -(dmin*m) (products rounded in fp32 first).
struct Q4Regs {
  uint4 qv[8];
  __half2 dsc[4], ndmn[4];
};

template <int PART>
__device__ __forceinline__ void q4_load(const uint8_t* rowp, Q4Regs& q) {
  const uint4 hdr = *reinterpret_cast<const uint4*>(rowp);
#pragma unroll
  for (int i = 0; i < 8; ++i) q.qv[i] = *reinterpret_cast<const uint4*>(rowp + 16 + 16 * i);
  const float d = h2f(hdr.x), dmin = h2f(hdr.x >> 16);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    float sc, mn;
    q4_scale_min(hdr.y, hdr.z, hdr.w, 2 * c + PART, sc, mn);
    q.dsc[c] = __float2half2_rn(d * sc);
    q.ndmn[c] = __float2half2_rn(-(dmin * mn));
  }
}

// K step c of the row: PART 0 = the low nibbles of quant bytes 32c .. 32c+31
// (sub-block 2c, step-local k 0..31), PART 1 = the high nibbles (sub-block
// 2c+1, k 32..63).  r[4j .. 4j+3] = the 8 fp16 weights of k = 32*PART + 8j ..
// +7 as four k-ordered pairs.
template <int PART>
__device__ __forceinline__ void q4_step(const Q4Regs& q, int c, uint32_t (&r)[16]) {
  const uint4 qa = q.qv[2 * c], qb = q.qv[2 * c + 1];
  const uint32_t wv[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    uint4 t;
    q4_emit4((wv[i] >> (4 * PART)) & 0x0F0F0F0Fu, q.dsc[c], q.ndmn[c], t);
    r[2 * i] = t.x;
    r[2 * i + 1] = t.y;
  }
}

// Q6_K.  The block of a row sits in its smem slot at byte offset MIS (even,
// 0..14: the misalignment of its global address).  The thread reads aligned
// 16-byte vectors and extracts block word j (bytes MIS+4j .. MIS+4j+3 of the
// slot) with compile-time indices and, for MIS % 4 == 2, a funnel shift.
template <int MIS, int N>
__device__ __forceinline__ uint32_t q6_pick(const uint32_t (&v)[N], int byte_in_v) {
  // byte_in_v = MIS + offset relative to the first loaded vector (compile-time)
  const int w = byte_in_v >> 2;
  if ((byte_in_v & 3) == 0) return v[w];
  return __funnelshift_r(v[w], v[w + 1], 16);
}

template <int NV>
__device__ __forceinline__ void lds_vecs(const uint8_t* p, uint32_t (&v)[4 * NV]) {
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const uint4 t = reinterpret_cast<const uint4*>(p)[i];
    v[4 * i] = t.x;
    v[4 * i + 1] = t.y;
    v[4 * i + 2] = t.z;
    v[4 * i + 3] = t.w;
  }
}

// One thread's share of a Q6_K super-block row, K steps 2h and 2h+1 (both read
// ql bytes 64h .. 64h+63 and qh bytes 128+32h .. +31), held in registers.
struct Q6Regs {
  uint32_t ql[16], qh[8];
  uint32_t scw0, scw1;  // int8 scales 8h .. 8h+3 and 8h+4 .. 8h+7
  float d;
};

template <int MIS>
__device__ __forceinline__ void q6_load(const uint8_t* slot, int h, Q6Regs& q) {
  uint32_t vl[20], vh[12], vs[8];
  lds_vecs<5>(slot + 64 * h, vl);         // bytes 64h .. 64h+79
  lds_vecs<3>(slot + 128 + 32 * h, vh);   // bytes 128+32h .. +47
  lds_vecs<2>(slot + 192, vs);            // bytes 192 .. 223
#pragma unroll
  for (int i = 0; i < 16; ++i) q.ql[i] = q6_pick<MIS>(vl, MIS + 4 * i);
#pragma unroll
  for (int i = 0; i < 8; ++i) q.qh[i] = q6_pick<MIS>(vh, MIS + 4 * i);
  q.scw0 = h ? q6_pick<MIS>(vs, MIS + 8) : q6_pick<MIS>(vs, MIS);
  q.scw1 = h ? q6_pick<MIS>(vs, MIS + 12) : q6_pick<MIS>(vs, MIS + 4);
  const uint32_t dw = vs[(16 + MIS) >> 2];
  q.d = h2f(((16 + MIS) & 3) ? (dw >> 16) : dw);
}

__device__ __forceinline__ void q6_load_dispatch(int mis, const uint8_t* slot, int h, Q6Regs& q) {
  switch (mis) {
    case 0: q6_load<0>(slot, h, q); break;
    case 2: q6_load<2>(slot, h, q); break;
    case 4: q6_load<4>(slot, h, q); break;
    case 6: q6_load<6>(slot, h, q); break;
    case 8: q6_load<8>(slot, h, q); break;
    case 10: q6_load<10>(slot, h, q); break;
    case 12: q6_load<12>(slot, h, q); break;
    default: q6_load<14>(slot, h, q); break;
  }
}

// The 64 fp16 weights of K step 2h + SIDE (SIDE 0: low nibbles of ql, SIDE 1:
// high nibbles) as 32 k-ordered pairs r[4j .. 4j+3] = chunk j (k = 8j .. 8j+7).
template <int SIDE>
__device__ __forceinline__ void q6_side(const Q6Regs& q, uint32_t (&r)[32]) {
  const __half2 k1056 = __float2half2_rn(1056.0f);  // 1024 + 32
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int g = 2 * SIDE + (j >> 2);     // 32-weight group within the half
    const int sidx = 4 * SIDE + (j >> 1);  // 16-weight scale group within the half
    const uint32_t scw = sidx < 4 ? q.scw0 : q.scw1;
    const float sc = (float)(int8_t)((scw >> (8 * (sidx & 3))) & 0xFFu);
    const __half2 dsc2 = __float2half2_rn(q.d * sc);
#pragma unroll
    for (int ww = 0; ww < 2; ++ww) {
      const int i = 2 * j + ww;  // ql word: bytes 64h + 4i, step-local k = 4i .. 4i+3
      const uint32_t lo4 = (SIDE ? (q.ql[i] >> 4) : q.ql[i]) & 0x0F0F0F0Fu;
      const uint32_t qhw = q.qh[i & 7];
      const int sh = 4 - 2 * g;  // bits 2g..2g+1 of every byte -> bits 4..5
      const uint32_t hs = sh >= 0 ? (qhw << sh) : (qhw >> (-sh));
      const uint32_t q6 = lo4 | (hs & 0x30303030u);
      const __half2 p0 = __hsub2(bits_h2(prmt(q6, kH2Magic, 0x4140u)), k1056);
      const __half2 p1 = __hsub2(bits_h2(prmt(q6, kH2Magic, 0x4342u)), k1056);
      r[4 * j + 2 * ww] = h2_bits(__hmul2(p0, dsc2));
      r[4 * j + 2 * ww + 1] = h2_bits(__hmul2(p1, dsc2));
    }
  }
}

// Q6_K packed stage layout.  The tensor map views the weights as rows of g
// consecutive weight rows (g * row_bytes is a multiple of 16); box j of a
// stage holds weight rows n0 + g*i + j (i = 0 .. 128/g - 1) at a kQ6Win-byte pitch
// in region j, so every row of region j has the same misalignment
// (j * row_bytes + 210 * kb) mod 16 of its block inside its window.
__device__ __forceinline__ uint32_t q6_region_stride(int g) {
  return (uint32_t)(((128 / g) * kQ6Win + 127) / 128 * 128);
}
__device__ __forceinline__ uint32_t q6_slot(int rho, int g) {
  return (uint32_t)(rho % g) * q6_region_stride(g) + (uint32_t)(rho / g) * kQ6Win;
}

// Row handled by dequant thread t (0..127) of one weight tensor.  Q6_K puts
// rows of the same residue mod g (same misalignment) in a warp, so the
// realignment code path is warp-uniform (for g = 8 a warp holds two residues).
template <int QT>
__device__ __forceinline__ int dq_row(int t, int g) {
  if constexpr (QT == kQ4K) {
    return t;
  } else {
    const int w = t >> 5, i = t & 31;
    if (g <= 4) return g * ((w / g) * 32 + i) + (w % g);
    return 8 * (i & 15) + 2 * w + (i >> 4);
  }
}

// acc[i] += the 16 fp32 values at shared address src (fp32 bits in acc).
__device__ __forceinline__ void add_partial16(uint32_t (&acc)[16], uint32_t src) {
#pragma unroll
  for (int i = 0; i < 16; i += 4) {
    const uint4 v = lds128_u(src + 4 * i);
    acc[i] = __float_as_uint(__uint_as_float(acc[i]) + __uint_as_float(v.x));
    acc[i + 1] = __float_as_uint(__uint_as_float(acc[i + 1]) + __uint_as_float(v.y));
    acc[i + 2] = __float_as_uint(__uint_as_float(acc[i + 2]) + __uint_as_float(v.z));
    acc[i + 3] = __float_as_uint(__uint_as_float(acc[i + 3]) + __uint_as_float(v.w));
  }
}

// Slot and phase parity of a position in a ring of n stages, advanced
// incrementally (the ring depth is a launch parameter: no division per step).
struct RingPos {
  int slot;
  uint32_t phase;
};
__device__ __forceinline__ void ring_advance(RingPos& r, int k, int n) {
  r.slot += k;
  while (r.slot >= n) {
    r.slot -= n;
    r.phase ^= 1u;
  }
}

// The dequant threads' main loop.  Thread (row rho, half PART) dequantizes,
// per K step, half of the step's 64 weights of its row (Q4_K: the nibbles PART
// of sub-block 2c + PART), or for Q6_K the two whole K steps 2*part and
// 2*part + 1 of every super-block (Q6_K uses the runtime `part`; PART is 0).
// A super-block's packed bytes are loaded into registers at once and the
// packed slot released before any conversion, so the producer can refill it
// while the A tiles are written.
template <int QT, bool GATEUP, bool AT, int PART>
__device__ __forceinline__ bool dequant_loop(uint8_t* smem, const Layout& L, Bars* bars, int SA, int D, int P, int nb,
                                             int kb_begin, int nkb, int which, int rho, uint32_t a_lane,
                                             uint32_t a_col0, int n0, int N, int q6g, int part,
                                             volatile uint32_t* abort_flag) {
  using C = Cfg<QT, GATEUP>;
  constexpr int kChunks = QT == kQ4K ? 4 : 8;  // 16-byte chunks of an A-tile row written per K step
  uint32_t off[kChunks];
#pragma unroll
  for (int j = 0; j < kChunks; ++j) off[j] = sw128_off(rho, QT == kQ4K ? 4 * PART + j : j);
  const int64_t RB = (int64_t)nb * (QT == kQ4K ? kQ4KBytes : kQ6KBytes);
  RingPos pos = {0, 0u};   // A slot of K step 4i of this CTA (Q4_K: the current step)
  RingPos ppos = {0, 0u};  // packed stage of super-block i
  // Done barrier of step - SA (ring D >= SA, one lap back at the start, so
  // the first SA waits return at once); Q6_K: of step 4i - SA.
  RingPos dd = {D - SA, 1u};
  bool ok = true;
  for (int i = 0; i < nkb && ok; ++i, ring_advance(ppos, 1, P)) {
    const int kb = kb_begin + i;  // super-block of the row; i counts this CTA's pipeline slots
    const int ps = ppos.slot;
    ok = mbar_wait(&bars->p_full[ps], ppos.phase, abort_flag, &g_gemm_status);
    if (!ok) break;
    const uint8_t* pst = smem + L.p_off + (ps * C::kNumB + which) * C::kPSlotBytes;
    if constexpr (QT == kQ4K) {
      Q4Regs q;
      q4_load<PART>(pst + rho * kQ4KBytes, q);
      mbar_arrive(&bars->p_empty[ps]);  // the producer fences before it refills the slot
#pragma unroll
      for (int c = 0; c < 4; ++c, ring_advance(pos, 1, SA), ring_advance(dd, 1, D)) {
        const int s = pos.slot;
        uint32_t r[16];
        q4_step<PART>(q, c, r);
        // A slot s last held step - SA: wait until its UMMAs completed.
        ok = mbar_wait(&bars->done[dd.slot], dd.phase, abort_flag, &g_gemm_status);
        if constexpr (AT) {
          ok = __all_sync(0xffffffffu, ok);  // tcgen05.st is warp-collective
          if (!ok) break;
          tc_fence_after();
          tmem_st16(a_lane + a_col0 + (uint32_t)((s * C::kNumB + which) * 32 + 16 * PART), r);
          tmem_wait_st();
          tc_fence_before();
        } else {
          if (!ok) break;
          uint8_t* a_tile = smem + L.a_off + (s * C::kNumB + which) * kAStageBytes;
#pragma unroll
          for (int j = 0; j < 4; ++j)
            *reinterpret_cast<uint4*>(a_tile + off[j]) = make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
          fence_proxy_async_smem();
        }
        mbar_arrive(&bars->a_full[s]);
      }
    } else {
      const int n = min(n0 + rho, N - 1);
      const int mis = (int)(((int64_t)n * RB + (int64_t)kb * kQ6KBytes) & 15);
      Q6Regs q;
      q6_load_dispatch(mis, pst + q6_slot(rho, q6g), part, q);
      if constexpr (AT) __syncwarp();  // rows of one warp may differ in alignment (tcgen05.st below is collective)
      mbar_arrive(&bars->p_empty[ps]);
      RingPos sp = pos, sd = dd;  // A slot of K step 4i + 2*part, done barrier of that step - SA
      ring_advance(sp, 2 * part, SA);
      ring_advance(sd, 2 * part, D);
#pragma unroll
      for (int side = 0; side < 2; ++side) {
        if (side == 1) {
          ring_advance(sp, 1, SA);
          ring_advance(sd, 1, D);
        }
        const int s = sp.slot;
        uint32_t r[32];
        if (side == 0)
          q6_side<0>(q, r);
        else
          q6_side<1>(q, r);
        ok = mbar_wait(&bars->done[sd.slot], sd.phase, abort_flag, &g_gemm_status);
        if constexpr (AT) {
          ok = __all_sync(0xffffffffu, ok);  // tcgen05.st is warp-collective
          if (!ok) break;
          tc_fence_after();
          const uint32_t ta = a_lane + a_col0 + (uint32_t)((s * C::kNumB + which) * 32);
          tmem_st16(ta, *reinterpret_cast<const uint32_t(*)[16]>(r));
          tmem_st16(ta + 16, *reinterpret_cast<const uint32_t(*)[16]>(r + 16));
          tmem_wait_st();
          tc_fence_before();
        } else {
          if (!ok) break;
          uint8_t* a_tile = smem + L.a_off + (s * C::kNumB + which) * kAStageBytes;
#pragma unroll
          for (int j = 0; j < 8; ++j)
            *reinterpret_cast<uint4*>(a_tile + off[j]) = make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
          fence_proxy_async_smem();
        }
        mbar_arrive(&bars->a_full[s]);
      }
      ring_advance(pos, 4, SA);
      ring_advance(dd, 4, D);
    }
  }
  return ok;
}

// Copies of super-block kb's packed blocks (the CTA's 128 rows) into the
// packed stage pst, completing on `full`.  Lanes pl = 0 .. np-1 of the calling
// warp share the work: Q4_K, lane 0 alone (one tensor-map box per tensor);
// Q6_K, every lane arrives on `full` (np arrivals).  Q6_K tiles inside the
// tensor map take g boxes (one per residue j); the last tile, if it holds rows
// past (N / g) * g, takes one bulk copy per row of the 16-byte-aligned
// window around its block instead (a window that would run past the
// end of the tensor is shortened and its last bytes copied by plain loads).
template <int QT, bool GATEUP>
__device__ __forceinline__ void issue_packed(uint8_t* pst, uint64_t* full, const CUtensorMap* tm_w0,
                                             const CUtensorMap* tm_w1, const Params& p, int kb, int n0, int nb,
                                             int pl, int np) {
  using C = Cfg<QT, GATEUP>;
  if constexpr (QT == kQ4K) {
    if (pl == 0) {
      mbar_arrive_expect_tx(full, (uint32_t)(C::kNumB * kBM * kQ4KBytes));
      tma_load_2d(pst, tm_w0, kb * kQ4KBytes, n0, full);
      if (GATEUP) tma_load_2d(pst + C::kPSlotBytes, tm_w1, kb * kQ4KBytes, n0, full);
    }
  } else {
    const int g = p.q6_group;
    const int64_t RB = (int64_t)nb * kQ6KBytes;
    if (n0 + kBM <= p.q6_rows_tma) {
      if (pl == 0) {
        mbar_arrive_expect_tx(full, (uint32_t)(kBM * kQ6Win));
        for (int j = 0; j < g; ++j) {
          const int64_t off = (int64_t)j * RB + (int64_t)kb * kQ6KBytes;
          tma_load_2d(pst + (uint32_t)j * q6_region_stride(g), tm_w0, (int32_t)((off & ~int64_t(15)) >> 1), n0 / g,
                      full);
        }
      } else {
        mbar_arrive(full);
      }
    } else {
      uint32_t bytes = 0;
      for (int i = pl; i < kBM; i += np) {
        const int n = n0 + i;
        if (n >= p.N) continue;
        const int64_t gg = (int64_t)n * RB + (int64_t)kb * kQ6KBytes;
        const int64_t lo = gg & ~int64_t(15);
        bytes += (uint32_t)(lo + kQ6Win <= p.w_bytes ? kQ6Win : ((p.w_bytes - lo) & ~int64_t(15)));
      }
      mbar_expect_tx(full, bytes);
      for (int i = pl; i < kBM; i += np) {
        const int n = n0 + i;
        if (n >= p.N) continue;
        const int64_t gg = (int64_t)n * RB + (int64_t)kb * kQ6KBytes;
        const int64_t lo = gg & ~int64_t(15);
        const int64_t len = lo + kQ6Win <= p.w_bytes ? kQ6Win : ((p.w_bytes - lo) & ~int64_t(15));
        uint8_t* dst = pst + q6_slot(i, g);
        bulk_copy_g2s(dst, p.w[0] + lo, (uint32_t)len, full);
        for (int64_t b = lo + len; b < gg + kQ6KBytes; b += 2)  // tail bytes (only at the tensor's end)
          *reinterpret_cast<uint16_t*>(dst + (b - lo)) = *reinterpret_cast<const uint16_t*>(p.w[0] + b);
      }
      fence_proxy_async_smem();  // plain writes into a slot that later refills write through TMA
      mbar_arrive(full);
    }
  }
}

// AT: the dequantized A tiles live in tensor memory (tcgen05.st from the
// dequant threads, UMMA reads A from TMEM) instead of shared memory.  KS: the
// kernel holds the split-K exchange (gate/up launches without split K use a
// KS = false instantiation, which would otherwise spill; single-tensor
// problems always use KS = true, measured faster on GB300 even unsplit).
template <int QT, bool GATEUP, bool AT, bool KS>
__global__ void __launch_bounds__(Cfg<QT, GATEUP>::kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w0,
                   const __grid_constant__ CUtensorMap tm_w1, const Params p) {
  using C = Cfg<QT, GATEUP>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int SX = p.stages, SA = p.astages, P = p.pstages;
  const int D = SX > SA ? SX : SA;  // done-barrier ring
  const Layout L = make_layout<QT, GATEUP, AT>(p.BN, SX, SA, P);
  Bars* bars = reinterpret_cast<Bars*>(smem + L.bar_off);
  volatile uint32_t* abort_flag = &bars->abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * kBM;
  const int m0 = blockIdx.y * p.BN;
  const int nb = p.K / kQK;
  // Split K: CTA z of a cluster of p.ksplit takes super-blocks [kb_begin, kb_begin + nkb).
  const int z = (int)blockIdx.z;
  const int kb_begin = (int)((int64_t)z * nb / p.ksplit);
  const int nkb = (int)((int64_t)(z + 1) * nb / p.ksplit) - kb_begin;
  const int nsteps = nkb * 4;
  const int BN = p.BN;
  const uint32_t x_bytes = (uint32_t)BN * kBK * 2;
  constexpr int kPSlotBytes = C::kPSlotBytes;
  constexpr bool kSplitProducer = C::kSplit;
  constexpr int kPackedLanes = QT == kQ4K ? 1 : 32;  // lanes of the packed warp that issue copies

  if (threadIdx.x == 0) {
    for (int s = 0; s < SX; ++s) mbar_init(&bars->x_full[s], 1);
    for (int s = 0; s < SA; ++s) mbar_init(&bars->a_full[s], C::kAArrivals);
    for (int s = 0; s < D; ++s) mbar_init(&bars->done[s], GATEUP ? kIssuers : 1);  // one commit per issuer of the step
    for (int s = 0; s < P; ++s) {
      mbar_init(&bars->p_full[s], QT == kQ4K ? 1 : 32);
      mbar_init(&bars->p_empty[s], 32 * C::kDqWarps);
    }
    mbar_init(&bars->acc_full, kIssuers);
    mbar_init(&bars->peer_full, 1);
    bars->abort_flag = 0;
    fence_mbar_init();
    if (p.ksplit > 1 && split_owns(z, BN, p.ksplit))  // split K: the ks - 1 partial slices this CTA receives
      mbar_arrive_expect_tx(&bars->peer_full, (uint32_t)(p.ksplit - 1) * split_slot_bytes<C::kNumB>(BN, p.ksplit));
  }
  // Accumulators: one per issuer, BN columns each (gate / up, or even / odd K
  // steps); with AT also SA x kNumB A tiles of 32 columns (128 rows x 64 fp16)
  // after them.
  const uint32_t a_col0 = (uint32_t)(kIssuers * BN);
  const uint32_t need_cols = a_col0 + (AT ? (uint32_t)(SA * C::kNumB * 32) : 0u);
  const uint32_t tmem_cols = need_cols <= 32 ? 32 : need_cols <= 64 ? 64 : need_cols <= 128 ? 128
                             : need_cols <= 256 ? 256 : 512;
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  bool dq_ok = false;  // dequant warps: the accumulators are complete and readable
  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tm_x);
      if (QT == kQ4K || p.q6_rows_tma > 0) prefetch_tmap(&tm_w0);
      if (GATEUP) prefetch_tmap(&tm_w1);
    }
    // x slot of `step` (ring SX) and the done barrier of step - SX (ring D,
    // starting one lap back: the first SX waits return at once).
    int step = 0;
    RingPos xpos = {0, 0u}, dpos = {D - SX, 1u};
    if constexpr (kSplitProducer) {
      // Lane 0 streams the x tiles; the packed warp streams the packed blocks,
      // each at its own pace.
      if (lane == 0) {
        bool ok = true;
        for (; step < nsteps && ok; ++step, ring_advance(xpos, 1, SX), ring_advance(dpos, 1, D)) {
          ok = mbar_wait<kCopyBackoffNs>(&bars->done[dpos.slot], dpos.phase, abort_flag, &g_gemm_status);
          if (!ok) break;
          const int kb = kb_begin + (step >> 2), c = step & 3;
          mbar_arrive_expect_tx(&bars->x_full[xpos.slot], x_bytes);
          tma_load_2d(smem + L.x_off + xpos.slot * L.x_stage, &tm_x, kb * kQK + c * kBK, m0, &bars->x_full[xpos.slot]);
        }
      }
    } else {
      // One loop for both: the packed block of super-block i, then its four x tiles.
      RingPos ppos = {0, 0u};
      bool ok = true;
      for (int i = 0; i < nkb && ok; ++i, ring_advance(ppos, 1, P)) {
        const int kb = kb_begin + i;
        const int ps = ppos.slot;
        ok = mbar_wait<kCopyBackoffNs>(&bars->p_empty[ps], ppos.phase ^ 1u, abort_flag, &g_gemm_status);
        if (!ok) break;
        fence_proxy_async_smem();  // as in the split producer: plain reads before the refill
        issue_packed<QT, GATEUP>(smem + L.p_off + ps * C::kNumB * kPSlotBytes, &bars->p_full[ps], &tm_w0, &tm_w1, p, kb,
                                 n0, nb, lane, 32);
        for (int c = 0; c < 4 && ok; ++c, ++step, ring_advance(xpos, 1, SX), ring_advance(dpos, 1, D)) {
          const int s = xpos.slot;
          ok = mbar_wait<kCopyBackoffNs>(&bars->done[dpos.slot], dpos.phase, abort_flag, &g_gemm_status);
          if (!ok) break;
          if (lane == 0) {
            mbar_arrive_expect_tx(&bars->x_full[s], x_bytes);
            tma_load_2d(smem + L.x_off + s * L.x_stage, &tm_x, kb * kQK + c * kBK, m0, &bars->x_full[s]);
          }
          __syncwarp();
        }
      }
    }
    // Drain: every x copy issued has completed before the CTA exits (the
    // packed-block copies are drained by the dequant warps' waits).
    if (!kSplitProducer || lane == 0) {
      for (int i = 0; i < SX && i < step; ++i) {
        const int st = step - 1 - i;
        mbar_wait(&bars->x_full[st % SX], (uint32_t)(st / SX) & 1u, abort_flag, &g_gemm_status, true);
      }
    }
  } else if (warp <= kIssuers) {
    // ------------------------------------------------------------------ UMMA issuers
    // Issuer i accumulates into columns [i*BN, (i+1)*BN): gate/up -> tensor i
    // in every K step; one tensor -> K steps i, i + kIssuers, ...
    const int iss = warp - 1;
    const uint32_t idesc = umma_idesc_f16(kBM, (uint32_t)BN);
    const uint32_t d_tm = tmem + (uint32_t)(iss * BN);
    const int t_first = GATEUP ? 0 : iss, t_stride = GATEUP ? 1 : kIssuers;
    const int ten = GATEUP ? iss : 0;
    bool ok = true;
    RingPos xs = {0, 0u}, as = {0, 0u}, ds = {0, 0u};  // x slot, A slot and done barrier of `step`
    ring_advance(xs, t_first, SX);
    ring_advance(as, t_first, SA);
    ring_advance(ds, t_first, D);
    for (int step = t_first; step < nsteps && ok;
         step += t_stride, ring_advance(xs, t_stride, SX), ring_advance(as, t_stride, SA), ring_advance(ds, t_stride, D)) {
      const int s = as.slot;
      ok = mbar_wait(&bars->x_full[xs.slot], xs.phase, abort_flag, &g_gemm_status) &&
           mbar_wait(&bars->a_full[s], as.phase, abort_flag, &g_gemm_status);
      if (!ok) break;
      tc_fence_after();
      if (lane == 0) {
        const uint64_t bdesc = umma_desc_sw128(smem_u32(smem + L.x_off + xs.slot * L.x_stage));
        if constexpr (AT) {
          const uint32_t a_tm = tmem + a_col0 + (uint32_t)((s * C::kNumB + ten) * 32);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)  // 16-wide K slice = 8 TMEM columns of A
            umma_f16_ts(d_tm, a_tm + (uint32_t)(8 * kk), bdesc + (uint64_t)(2 * kk), idesc,
                        (step > t_first || kk > 0) ? 1u : 0u);
        } else {
          const uint64_t adesc = umma_desc_sw128(smem_u32(smem + L.a_off + (s * C::kNumB + ten) * kAStageBytes));
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)  // +32 bytes per 16-wide K slice inside the swizzle atom
            umma_f16_ss(d_tm, adesc + (uint64_t)(2 * kk), bdesc + (uint64_t)(2 * kk), idesc,
                        (step > t_first || kk > 0) ? 1u : 0u);
        }
        umma_commit(&bars->done[ds.slot]);
      }
      __syncwarp();
    }
    // acc_full completes once both issuers' UMMAs have completed (it is also
    // committed after an abort, so the wait below always ends); waiting for it
    // here keeps tensor memory allocated until the last UMMA is done.
    if (lane == 0) umma_commit(&bars->acc_full);
    __syncwarp();
    mbar_wait(&bars->acc_full, 0u, abort_flag, &g_gemm_status, true);
  } else if (warp == C::kPackedWarp) {
    // ------------------------------------------------------------------ packed blocks (kSplit)
    // A packed stage is refilled as soon as the dequant threads have released
    // it, whatever the state of the x ring.
    if (lane < kPackedLanes) {
      RingPos ppos = {0, 0u};
      for (int i = 0; i < nkb; ++i, ring_advance(ppos, 1, P)) {
        const int ps = ppos.slot;
        if (!mbar_wait<kCopyBackoffNs>(&bars->p_empty[ps], ppos.phase ^ 1u, abort_flag, &g_gemm_status)) break;
        // The dequant threads read the slot with plain loads; the refill is
        // an async-proxy write.  This proxy fence, after the barrier that
        // their releases completed, orders those reads before the copy
        // (without any fence the copy was seen to overwrite unread bytes).
        fence_proxy_async_smem();
        issue_packed<QT, GATEUP>(smem + L.p_off + ps * C::kNumB * kPSlotBytes, &bars->p_full[ps], &tm_w0, &tm_w1, p,
                                 kb_begin + i, n0, nb, lane, kPackedLanes);
      }
    }
  } else {
    // ------------------------------------------------------------------ dequant + epilogue
    const int t = threadIdx.x - 32 * C::kDqWarp0;  // 0 .. 32*kDqWarps-1
    const int tpt = 32 * C::kDqWarps / C::kNumB;  // threads per weight tensor (256)
    const int which = t / tpt;                    // weight tensor (0 = gate/only, 1 = up)
    const int part = (t % tpt) >> 7;              // which half of the work on this row
    // With A in TMEM a warp may only write its own lane quarter (warp % 4).
    const int rho = AT ? 32 * (warp & 3) + lane : dq_row<QT>(t & 127, p.q6_group);
    const uint32_t a_lane = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    // Q4_K specialises on the nibble half (compile-time shifts); Q6_K takes the
    // half as a runtime value (one copy of its larger code).
    bool ok;
    if (QT == kQ6K || part == 0)
      ok = dequant_loop<QT, GATEUP, AT, 0>(smem, L, bars, SA, D, P, nb, kb_begin, nkb, which, rho, a_lane, a_col0, n0,
                                           p.N, p.q6_group, part, abort_flag);
    else
      ok = dequant_loop<QT, GATEUP, AT, 1>(smem, L, bars, SA, D, P, nb, kb_begin, nkb, which, rho, a_lane, a_col0, n0,
                                           p.N, p.q6_group, part, abort_flag);

    if (ok) ok = mbar_wait(&bars->acc_full, 0u, abort_flag, &g_gemm_status);
    dq_ok = __all_sync(0xffffffffu, ok);  // tcgen05.ld is warp-collective
  }

  // ---------------------------------------------------------------- epilogue
  // Dequant warp w reads TMEM lane quarter w % 4 (rows 32q .. 32q+31); the
  // warps sharing a quarter take alternate 16-column chunks.
  const bool dq_warp = warp >= C::kDqWarp0 && warp < C::kDqWarp0 + C::kDqWarps;
  const int q = warp & 3;
  const int row = q * 32 + lane;
  const int n = n0 + row;
  const uint32_t lane_addr = tmem + ((uint32_t)(q * 32) << 16);
  const int nchunks = BN / 16;
  const int ngroups = C::kDqWarps / 4, grp = (warp - C::kDqWarp0) >> 2;
  // The result of chunk cc: one tensor's value (va), or gate (va) and up (vb).
  auto store_chunk = [&](int cc, const uint32_t (&va)[16], const uint32_t (&vb)[16]) {
    if (n >= p.N) return;
    if constexpr (!GATEUP) {
      float* y = static_cast<float*>(p.y);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int m = m0 + 16 * cc + i;
        if (m < p.M) y[(int64_t)m * p.N + n] = __uint_as_float(va[i]);
      }
    } else {
      __half* y = static_cast<__half*>(p.y);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int m = m0 + 16 * cc + i;
        const float g = __uint_as_float(va[i]), u = __uint_as_float(vb[i]);
        // silu(g) * u with sigmoid(g) = 0.5 + 0.5 tanh(g / 2): one
        // special-function op per element instead of two (exp and a
        // reciprocal); the epilogue was bound by that unit.
        const float hg = 0.5f * g;
        const float o = fmaf(hg, tanh_approx(hg), hg) * u;
        if (m < p.M) y[(int64_t)m * p.N + n] = __float2half_rn(o);
      }
    }
  };
  // This CTA's partial of chunk cc from tensor memory: one tensor, D0 + D1
  // (its even and odd K steps) in va; gate/up, G in va and U in vb.
  auto own_chunk = [&](int cc, uint32_t (&va)[16], uint32_t (&vb)[16]) {
    tmem_ld16(lane_addr + (uint32_t)(16 * cc), va);
    tmem_ld16(lane_addr + (uint32_t)(BN + 16 * cc), vb);
    tmem_wait_ld();
    if constexpr (!GATEUP) {
#pragma unroll
      for (int i = 0; i < 16; ++i) va[i] = __float_as_uint(__uint_as_float(va[i]) + __uint_as_float(vb[i]));
    }
  };
  const int ksplit = KS ? p.ksplit : 1;
  if (KS && ksplit > 1) {
    // Split K, reduce-scatter: CTA zz of the cluster owns the chunks
    // [cz(zz), cz(zz + 1)).  Each CTA writes its partial of every peer's
    // chunks into a send slot of its own stage region (free once its main loop
    // is done); after the first cluster barrier (every CTA past its main loop)
    // one bulk copy per peer moves the slot into that peer's receive slot for
    // this sender, completing on the peer's peer_full (armed at start with the
    // bytes of its ks - 1 incoming slots).  The second cluster barrier, once
    // every owner has seen its slots land, lets the CTAs (the copies' sources)
    // exit; each owner then adds the ks partials of its chunks in rank order
    // (deterministic) from its own tensor and shared memory and writes them.
    // split_chunk without a division per call: num / ks == (num * kinv) >> 16
    // for ks <= 8 and num <= 8 * 16 + 7 (checked for every case on the host)
    const uint32_t kinv = (65536u + (uint32_t)ksplit - 1u) / (uint32_t)ksplit;
    auto cz = [&](int zz) { return (int)(((uint32_t)(zz * nchunks + ksplit - 1) * kinv) >> 16); };
    auto owns = [&](int zz) { return cz(zz + 1) > cz(zz); };
    const uint32_t xbuf = smem_u32(smem);
    const uint32_t pitch = split_slot_pitch(BN, ksplit);
    const uint32_t slot = split_slot_bytes<C::kNumB>(BN, ksplit);
    const bool owner = owns(z);
    auto recv_slot = [&](int dst, int src) { return xbuf + (uint32_t)(src < dst ? src : src - 1) * slot; };
    auto send_slot = [&](int d) {  // d: an owning peer; owners below d: min(d, cz(d))
      const int below = d < cz(d) ? d : cz(d);
      const int j = below - (owner && z < d ? 1 : 0);
      return xbuf + (uint32_t)((owner ? ksplit - 1 : 0) + j) * slot;
    };
    __syncwarp();        // each warp arrives converged (the cluster barrier is .aligned)
    cluster_sync_all();  // every CTA of the cluster is past its main loop
    // an owner whose peers own nothing (fewer chunks than ranks) sends nothing
    const bool sends = (ksplit < nchunks ? ksplit : nchunks) > (owner ? 1 : 0);
    if (dq_warp && sends) {
      if (dq_ok) {
        tc_fence_after();
        for (int d = 0; d < ksplit; ++d) {
          if (d == z || !owns(d)) continue;
          for (int cc = cz(d) + grp; cc < cz(d + 1); cc += ngroups) {
            uint32_t va[16], vb[16];
            own_chunk(cc, va, vb);
            const uint32_t a = send_slot(d) + (uint32_t)row * pitch + (uint32_t)(64 * (cc - cz(d)));
#pragma unroll
            for (int i = 0; i < 4; ++i) sts128_u(a + 16 * i, va[4 * i], va[4 * i + 1], va[4 * i + 2], va[4 * i + 3]);
            if constexpr (GATEUP) {
#pragma unroll
              for (int i = 0; i < 4; ++i)
                sts128_u(a + 128 * pitch + 16 * i, vb[4 * i], vb[4 * i + 1], vb[4 * i + 2], vb[4 * i + 3]);
            }
          }
        }
      }
      fence_proxy_async_smem();  // plain writes, read by the bulk copies (async proxy)
    }
    if (dq_warp) named_bar_sync(1, 32 * C::kDqWarps);  // every send slot of this CTA is written
    if (threadIdx.x == 32 * C::kDqWarp0) {
      // every owning peer always receives from every other rank, so its wait
      // ends (bounded in any case)
      for (int d = 0; d < ksplit; ++d)
        if (d != z && owns(d))
          bulk_copy_s2cluster(mapa_shared(recv_slot(d, z), (uint32_t)d), send_slot(d), slot,
                              mapa_shared(smem_u32(&bars->peer_full), (uint32_t)d));
    }
    if (dq_warp && owner) {
      const bool landed = mbar_wait(&bars->peer_full, 0u, abort_flag, &g_gemm_status, true);
      dq_ok = __all_sync(0xffffffffu, dq_ok && landed);
    }
    __syncwarp();
    cluster_sync_all();  // every copy has landed: the peers may exit
    if (dq_warp && owner && dq_ok) {
      tc_fence_after();
      for (int cc = cz(z) + grp; cc < cz(z + 1); cc += ngroups) {
        uint32_t oa[16], ob[16];
        own_chunk(cc, oa, ob);
        uint32_t va[16], vb[16];
        // rank 0's partial, then ranks 1 .. ks - 1 added in order
#pragma unroll 1
        for (int zz = 0; zz < ksplit; ++zz) {
          if (zz == z) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              va[i] = zz == 0 ? oa[i] : __float_as_uint(__uint_as_float(va[i]) + __uint_as_float(oa[i]));
              if constexpr (GATEUP)
                vb[i] = zz == 0 ? ob[i] : __float_as_uint(__uint_as_float(vb[i]) + __uint_as_float(ob[i]));
            }
          } else {
            const uint32_t src = recv_slot(z, zz) + (uint32_t)row * pitch + (uint32_t)(64 * (cc - cz(z)));
            if (zz == 0) {
#pragma unroll
              for (int i = 0; i < 16; i += 4) {
                const uint4 v = lds128_u(src + 4 * i);
                va[i] = v.x, va[i + 1] = v.y, va[i + 2] = v.z, va[i + 3] = v.w;
              }
              if constexpr (GATEUP) {
#pragma unroll
                for (int i = 0; i < 16; i += 4) {
                  const uint4 v = lds128_u(src + 128 * pitch + 4 * i);
                  vb[i] = v.x, vb[i + 1] = v.y, vb[i + 2] = v.z, vb[i + 3] = v.w;
                }
              }
            } else {
              add_partial16(va, src);
              if constexpr (GATEUP) add_partial16(vb, src + 128 * pitch);
            }
          }
        }
        store_chunk(cc, va, vb);
      }
    }
  } else if (dq_warp && dq_ok) {
    tc_fence_after();
    for (int cc = grp; cc < nchunks; cc += ngroups) {
      uint32_t va[16], vb[16];
      own_chunk(cc, va, vb);
      store_chunk(cc, va, vb);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, tmem_cols);
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up once per process (a function-local
// static: initialised once even when several host threads call at once).
EncodeTiledFn encode_fn() {
  static const EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<EncodeTiledFn>(p);
    cudaGetLastError();
    return nullptr;
  }();
  return fn;
}

bool make_tmap_x(CUtensorMap* tm, const void* x, int64_t M, int64_t K, int BN) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
  const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)BN};
  const cuuint32_t estr[2] = {1, 1};
  return enc(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(x), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Q4_K weights as a byte matrix [N][row_bytes]; one box = one super-block
// (144 bytes) of 128 rows.
bool make_tmap_q4k(CUtensorMap* tm, const void* w, int64_t N, int64_t K) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const int64_t rb = (K / kQK) * kQ4KBytes;
  const cuuint64_t dims[2] = {(cuuint64_t)rb, (cuuint64_t)N};
  const cuuint64_t strides[1] = {(cuuint64_t)rb};
  const cuuint32_t box[2] = {(cuuint32_t)kQ4KBytes, (cuuint32_t)kBM};
  const cuuint32_t estr[2] = {1, 1};
  return enc(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(w), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Q6_K weights as uint16 rows of g consecutive weight rows (g * row_bytes is a
// multiple of 16, as tensor maps require); one box = the kQ6Win-byte window of one
// residue j's blocks for 128/g such rows.
int q6_group(int64_t K) {
  const int64_t rb = (K / kQK) * kQ6KBytes;
  for (int g = 1; g < 8; g *= 2)
    if ((g * rb) % 16 == 0) return g;
  return 8;
}

bool make_tmap_q6k(CUtensorMap* tm, const void* w, int64_t N, int64_t K, int g) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const int64_t rb = (K / kQK) * kQ6KBytes;
  const cuuint64_t dims[2] = {(cuuint64_t)(g * rb / 2), (cuuint64_t)(N / g)};
  const cuuint64_t strides[1] = {(cuuint64_t)(g * rb)};
  const cuuint32_t box[2] = {(cuuint32_t)(kQ6Win / 2), (cuuint32_t)(kBM / g)};
  const cuuint32_t estr[2] = {1, 1};
  return enc(tm, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(w), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Token tile: the multiple of 16 (<= 256) that minimises waves x tile cost,
// where a tile costs its MMA time (~BN) plus a per-tile share (dequantizing
// the 128 x K weight tile and the epilogue) worth about 64 tokens; ties go to
// the larger tile.
int choose_bn(int64_t M, int64_t N) {
  const int64_t ntn = (N + kBM - 1) / kBM;
  if (M <= kMaxBN) return (int)((M + 15) / 16 * 16);
  const int64_t sms = device_sms();
  int best = kMaxBN;
  double best_cost = 1e30;
  for (int bn = kMaxBN; bn >= 128; bn -= 16) {
    const int64_t tiles = ntn * ((M + bn - 1) / bn);
    const int64_t waves = (tiles + sms - 1) / sms;
    const double cost = (double)waves * (bn + 64);
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = bn;
    }
  }
  return best;
}

constexpr int kSmemLimit = 227 * 1024;

template <int QT, bool GATEUP, bool AT, bool KS>
__global__ void gemm_tc_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w0,
                               const __grid_constant__ CUtensorMap tm_w1, const Params p);

// Clusters of c CTAs of the split-K kernel that can be resident at once with
// `smem` bytes of dynamic shared memory each (cached per device and size; 0 if
// the query fails, which disables that split).
template <int QT, bool GATEUP, bool AT>
int max_active_clusters(int c, uint32_t smem) {
  static std::mutex mu;
  static std::map<std::tuple<int, int, uint32_t>, int> cache;
  std::lock_guard<std::mutex> lock(mu);
  const auto key = std::make_tuple(current_device(), c, smem);
  const auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(1, 1, (unsigned)c);
  cfg.blockDim = dim3(Cfg<QT, GATEUP>::kThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = (unsigned)c;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, gemm_tc_kernel<QT, GATEUP, AT, true>, &cfg) != cudaSuccess) {
    cudaGetLastError();  // clear the error; this split size is then not used
    n = 0;
  }
  cache[key] = n;
  return n;
}

// Tensor-memory columns one CTA allocates: one BN-column accumulator per
// issuer and, with A tiles in tensor memory, SA x kNumB tiles of 32 columns,
// rounded up to the power of two tcgen05.alloc takes (the kernel computes the
// same value).
inline uint32_t tmem_cols_for(int BN, int SA, int num_b, bool at) {
  const uint32_t need = (uint32_t)(kIssuers * BN) + (at ? (uint32_t)(SA * num_b * 32) : 0u);
  return need <= 32 ? 32 : need <= 64 ? 64 : need <= 128 ? 128 : need <= 256 ? 256 : 512;
}

// tcgen05.alloc waits until enough tensor-memory columns are free, with no
// time limit, so the CTAs that share an SM must fit in its 512 columns
// together; otherwise one of them can wait forever (in a split-K cluster,
// while its peers hold theirs at the cluster barrier).  Shared memory bounds
// how many CTAs share an SM: `sm_smem` per SM, `reserved` per CTA.  This
// returns the dynamic shared-memory request, at least `smem`, for which at
// most 512 / cols CTAs fit (host only; registers can only lower the count).
uint32_t smem_for_tmem(uint32_t smem, uint32_t cols, uint32_t sm_smem, uint32_t reserved) {
  const uint32_t max_ctas = 512u / cols;
  if (sm_smem / (smem + reserved) <= max_ctas) return smem;
  uint32_t need = sm_smem / (max_ctas + 1) - reserved + 1;
  need = (need + 127u) & ~127u;
  return need > smem ? need : smem;
}

// Shared memory per SM and the per-CTA reservation (the GB300 values when no
// device can be queried).
void sm_smem_limits(uint32_t* sm_smem, uint32_t* reserved) {
  static std::atomic<int64_t> cache[kMaxDevices];
  *sm_smem = 233472;
  *reserved = 1024;
  const int dev = current_device();
  if (dev < 0) return;
  int64_t v = cache[dev].load(std::memory_order_relaxed);
  if (v == 0) {
    int a = 0, b = 0;
    if (cudaDeviceGetAttribute(&a, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&b, cudaDevAttrReservedSharedMemoryPerBlock, dev) == cudaSuccess && a > 0) {
      v = ((int64_t)a << 20) | (int64_t)b;
    } else {
      cudaGetLastError();
      v = ((int64_t)233472 << 20) | 1024;
    }
    cache[dev].store(v, std::memory_order_relaxed);
  }
  *sm_smem = (uint32_t)(v >> 20);
  *reserved = (uint32_t)(v & 0xFFFFF);
}

// The launch plan of one GEMM problem (host only, no kernel launch).
struct TcPlan {
  int BN, SX, SA, P;
  uint32_t smem;       // dynamic shared memory requested per CTA
  uint32_t tmem_cols;  // tensor-memory columns per CTA
  uint32_t bar_off;    // offset of the barrier block (bounds the split-K exchange slots)
};

// Pipeline depths (all measured on GB300).  The K-step rings come first: a
// single-tensor kernel with fewer than 4 x-tile stages ran ~35 % slower.
// Single-tensor problems grow A-tile and x-tile stages alternately, A first,
// up to 4 x stages (x stages alone once a TMEM-capped A ring stops growing),
// then x stages two at a time up to kMaxXDeep.  A per-CTA trace of Q6_K down
// showed the issuers waiting on x tiles (0.4-0.75 us from a tile's load to
// its barrier, and a slot is refilled only once the UMMAs of its previous
// step have completed); 6-8 stages took Q4_K o-proj M = 1024 from 21.0 to
// 19.4 us and Q6_K attn_v M = 128 from 17.4 to 15.2 us, other shapes within
// 2 %.  The ring stays even: the two issuers take alternate K steps, so each
// keeps to its own slots and waits on every phase of them (with an odd ring
// an issuer would skip the phases of the other's steps, and x tiles can land
// out of order, so a parity wait could pass on a slot's previous tile).
// Gate/up grows x stages to 3, then A stages to 3, then x to 4 and A on:
// at 256-token tiles 3 x + 2 A stages ran 12 % faster than 2 + 3, and where
// 3 + 3 fits it ran 2-6 % faster than 4 + 2 from M = 384 to 2048 (20 % at
// M = 192), so among packed-stage counts gate/up ranks min(x, 3), then
// min(A, 3), then the packed stages.  Up to 5 A stages, while shared memory
// (and, with A in tensor memory, TMEM) allows.  Packed-block stages: two where they fit next to 4 x
// stages (cold-cache Q6_K ran faster with two; three or four gained nothing
// in steady state), else one (the dequant threads copy a super-block to
// registers and release its slot at once, so the refill overlaps the
// block's four K steps).
// Q6_K takes 4 A stages.  Its threads write two consecutive K steps of a
// super-block and the two halves of a row alternate.  With SA = 2 a half
// waits on a slot whose previous phase (the other half's step) it never
// saw, so the parity test can pass a phase early (seen on GB300 as wrong
// output once the packed copies ran ahead).  From SA = 3 on, the phase a
// half skips belongs to an earlier step of the same issuer, whose UMMAs
// complete in order, so it has always completed.  Its done-barrier ring
// D = max(SX, SA) is even (4, 6 or 8): the next completion of the slot a half
// waits on is then a later step of the same issuer, which cannot run before
// the half has written its own step (with D = 5 it would be the other half's
// next step, which can complete first, and the wait would never pass).
// Returns false when the A tiles do not fit in tensor memory next to the
// accumulators (the caller then keeps them in shared memory).
template <int QT, bool GATEUP, bool AT>
bool plan_tc(int64_t M, int64_t N, TcPlan* out) {
  using C = Cfg<QT, GATEUP>;
  const int BN = choose_bn(M, N);
  constexpr int kMaxXStages = 4, kMaxAStages = QT == kQ6K ? 4 : 5;
  constexpr int kMaxXDeep = GATEUP ? kMaxXStages : QK_GEMM_MAX_X;
  static_assert(kMaxXDeep <= 8 && kMaxXDeep % 2 == 0, "x ring capacity");
  constexpr int kMaxP = QK_GEMM_MAX_P;
  static_assert(kMaxP >= 1 && kMaxP <= 4, "packed ring capacity");
  auto depths = [&](int P_, int& SX_, int& SA_) {
    auto fits = [&](int sx, int sa) {
      return make_layout<QT, GATEUP, AT>(BN, sx, sa, P_).total <= (uint32_t)kSmemLimit &&
             !(AT && kIssuers * BN + sa * C::kNumB * 32 > 512);
    };
    SX_ = 2;
    SA_ = 2;
    for (bool grew = true; grew;) {
      grew = false;
      if (GATEUP) {  // x to 3, A to 3, then x to 4 and A on
        if (SX_ < 3 && fits(SX_ + 1, SA_)) {
          ++SX_;
          grew = true;
        } else if (SA_ < 3 && fits(SX_, SA_ + 1)) {
          ++SA_;
          grew = true;
        } else if (SX_ < kMaxXStages && fits(SX_ + 1, SA_)) {
          ++SX_;
          grew = true;
        } else if (SA_ < kMaxAStages && fits(SX_, SA_ + 1)) {
          ++SA_;
          grew = true;
        }
      } else if (SA_ == SX_ && SA_ < kMaxAStages && fits(SX_, SA_ + 1)) {
        ++SA_;
        grew = true;
      } else if (SX_ < SA_ && SX_ < kMaxXStages && fits(SX_ + 1, SA_)) {
        ++SX_;
        grew = true;
      }
    }
    if (!GATEUP) {
      while (SX_ < kMaxXStages && fits(SX_ + 1, SA_)) ++SX_;  // x stages past a TMEM-capped A ring
      if (SX_ == kMaxXStages)
        while (SX_ + 2 <= kMaxXDeep && fits(SX_ + 2, SA_)) SX_ += 2;
      if (SX_ & 1) --SX_;  // the issuers alternate: each keeps to its own x slots
    }
  };
  // Packed stages: the most x stages up to 4 first, then the most packed
  // stages up to kMaxP, then the deepest x ring, then the deepest A ring
  // (gate/up: x up to 3, then A up to 3, then packed stages, then x).
  int P = 1, SX = 0, SA = 0;
  auto score = [&](int p_, int sx, int sa) {
    if (GATEUP) return ((std::min(sx, 3) * 8 + std::min(sa, 3)) * 8 + p_) * 16 + sx;
    return ((std::min(sx, kMaxXStages) * 8 + p_) * 16 + sx) * 16 + sa;
  };
  for (int p_ = 1; p_ <= kMaxP; ++p_) {
    int sx, sa;
    depths(p_, sx, sa);
    if (make_layout<QT, GATEUP, AT>(BN, sx, sa, p_).total > (uint32_t)kSmemLimit) continue;
    if (SX == 0 || score(p_, sx, sa) > score(P, SX, SA)) {
      P = p_;
      SX = sx;
      SA = sa;
    }
  }
  if (SX == 0) return false;
  if (AT && (kIssuers * BN + SA * C::kNumB * 32 > 512 || (QT == kQ6K && SA != 4))) return false;
  const Layout L = make_layout<QT, GATEUP, AT>(BN, SX, SA, P);
  uint32_t sm_smem, reserved;
  sm_smem_limits(&sm_smem, &reserved);
  out->BN = BN;
  out->SX = SX;
  out->SA = SA;
  out->P = P;
  out->tmem_cols = tmem_cols_for(BN, SA, C::kNumB, AT);
  out->smem = smem_for_tmem(L.total, out->tmem_cols, sm_smem, reserved);
  out->bar_off = L.bar_off;
  return true;
}

template <int QT, bool GATEUP, bool AT>
cudaError_t launch_tc(const void* W0, const void* W1, const uint16_t* x, void* y, int64_t M, int64_t N, int64_t K,
                      cudaStream_t stream) {
  using C = Cfg<QT, GATEUP>;
  TcPlan pl;
  if (!plan_tc<QT, GATEUP, AT>(M, N, &pl)) {
    if constexpr (AT) return launch_tc<QT, GATEUP, false>(W0, W1, x, y, M, N, K, stream);
    return cudaErrorInvalidConfiguration;
  }
  const int BN = pl.BN, SX = pl.SX, SA = pl.SA, P = pl.P;
  if (QT == kQ6K && SA != 4) return cudaErrorInvalidConfiguration;  // not reached for BN <= 256
  CUtensorMap tx, tw0, tw1;
  memset(&tw0, 0, sizeof(tw0));
  memset(&tw1, 0, sizeof(tw1));
  if (!make_tmap_x(&tx, x, M, K, BN)) return cudaErrorInvalidValue;
  Params p;
  p.q6_group = 1;
  p.q6_rows_tma = 0;
  if (QT == kQ4K) {
    if (!make_tmap_q4k(&tw0, W0, N, K)) return cudaErrorInvalidValue;
    if (GATEUP && !make_tmap_q4k(&tw1, W1, N, K)) return cudaErrorInvalidValue;
  } else {
    p.q6_group = q6_group(K);
    if (N / p.q6_group > 0) {
      if (!make_tmap_q6k(&tw0, W0, N, K, p.q6_group)) return cudaErrorInvalidValue;
      p.q6_rows_tma = (int)((N / p.q6_group) * p.q6_group);
    }
  }
  p.w[0] = static_cast<const uint8_t*>(W0);
  p.w[1] = static_cast<const uint8_t*>(W1);
  p.w_bytes = N * (K / kQK) * (QT == kQ4K ? kQ4KBytes : kQ6KBytes);
  p.y = y;
  p.M = (int)M;
  p.N = (int)N;
  p.K = (int)K;
  p.BN = BN;
  p.stages = SX;
  p.astages = SA;
  p.pstages = P;
  p.ksplit = 1;
  const uint32_t smem = pl.smem;
  if (smem > (uint32_t)kSmemLimit) return cudaErrorInvalidConfiguration;
  static PerDeviceFlag attr_set;  // the shared-memory limit is a per-device function attribute
  const int dev = current_device();
  if (!attr_set.done(dev)) {
    cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<QT, GATEUP, AT, !GATEUP>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(gemm_tc_kernel<QT, GATEUP, AT, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kSmemLimit);
    if (e != cudaSuccess) return e;
    attr_set.mark(dev);
  }
  dim3 grid((unsigned)((N + kBM - 1) / kBM), (unsigned)((M + BN - 1) / BN));
  if (grid.y > 65535u) return cudaErrorInvalidConfiguration;
  // Split K across a cluster when the tiles would leave at least half of the
  // SMs idle (small N or small M): ks CTAs per tile, each with >= 1 super-block,
  // the send and receive slots of the exchange fitting in the stage region, and every
  // tile's cluster resident at once.  The last condition is the device's
  // answer for this kernel and cluster size: clusters must fit inside one GPC,
  // and on GB300 24 clusters of 6 one-CTA-per-SM CTAs did not (a second wave
  // doubled the time of a 24-tile problem).
  // Among the feasible sizes, the one with the fewest super-blocks per CTA
  // (ceil(K/256 / ks): the cluster waits for its slowest CTA), then the
  // smallest (less exchange).
  // A split launch runs one CTA per SM: its shared-memory request is raised so
  // that no two of its CTAs share an SM (small tiles otherwise fit twice, and
  // two CTAs of a cluster on one SM share its tensor pipe: M = 16 splits ran
  // ~1 us slower when the registers allowed it).
  int ks = 1;
  uint32_t split_smem = smem;
  {
    const int64_t tiles = (int64_t)grid.x * grid.y;
    const int64_t nb = K / kQK;
    int64_t best = nb;
    const int64_t sms = device_sms();
    uint32_t sm_smem, reserved;
    sm_smem_limits(&sm_smem, &reserved);
    split_smem = smem_for_tmem(smem, 512u, sm_smem, reserved);
    if (tiles * 2 <= sms && split_smem <= (uint32_t)kSmemLimit)
      for (int c = 2; c <= 8; ++c) {
        const int64_t per = (nb + c - 1) / c;
        if (per < best && tiles * c <= sms && c <= nb &&
            split_exchange_bytes<C::kNumB>(BN, c) <= pl.bar_off &&
            tiles <= max_active_clusters<QT, GATEUP, AT>(c, split_smem)) {
          ks = c;
          best = per;
        }
      }
  }
  p.ksplit = ks;
  if (ks == 1) {
    gemm_tc_kernel<QT, GATEUP, AT, !GATEUP><<<grid, C::kThreads, smem, stream>>>(tx, tw0, tw1, p);
    return cudaGetLastError();
  }
  grid.z = (unsigned)ks;
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = grid;
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = split_smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = (unsigned)ks;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<QT, GATEUP, AT, true>, tx, tw0, tw1, p);
}

// The plan of the instantiation launch_gemm picks (host only).
template <int QT, bool GATEUP, bool AT>
bool plan_for(int64_t M, int64_t N, TcPlan* pl, int* a_in_tmem) {
  if (plan_tc<QT, GATEUP, AT>(M, N, pl)) {
    *a_in_tmem = AT ? 1 : 0;
    return true;
  }
  if constexpr (AT) return plan_for<QT, GATEUP, false>(M, N, pl, a_in_tmem);
  return false;
}

int a_tmem_default() {
  static const int a_tmem = [] {
    const char* e = getenv("QK_A_TMEM");
    return e ? atoi(e) : 1;
  }();
  return a_tmem;
}

}  // namespace

bool encode_tensor_map_f16(void* out, const void* base, int rank, const uint64_t* dims, const uint64_t* strides,
                           const uint32_t* box, bool swizzle128) {
  EncodeTiledFn enc = encode_fn();
  if (!enc || rank < 1 || rank > 5) return false;
  cuuint64_t d[5], st[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
    if (i + 1 < rank) st[i] = strides[i];
  }
  return enc(static_cast<CUtensorMap*>(out), CU_TENSOR_MAP_DATA_TYPE_FLOAT16, (cuuint32_t)rank, const_cast<void*>(base),
             d, st, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

uint32_t gemm_take_status() {
  uint32_t v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_gemm_status, sizeof(v)) != cudaSuccess) return 0;
  cudaMemcpyToSymbol(g_gemm_status, &zero, sizeof(zero));
  v |= take_debug_status();
  return v;
}

cudaError_t launch_gemm(QType t, const void* W, const void* W_up, const uint16_t* x, void* y, int64_t M, int64_t N,
                        int64_t K, bool gateup, cudaStream_t s) {
  // Single-tensor problems keep the dequantized A tiles in tensor memory when
  // they fit next to the accumulators (measured faster on GB300: no A-tile
  // shared-memory writes and UMMA reads); QK_A_TMEM=0 selects shared memory.
  const int a_tmem = a_tmem_default();
  if (gateup) return launch_tc<kQ4K, true, false>(W, W_up, x, y, M, N, K, s);
  if (t == kQ4K) {
    if (a_tmem) return launch_tc<kQ4K, false, true>(W, nullptr, x, y, M, N, K, s);
    return launch_tc<kQ4K, false, false>(W, nullptr, x, y, M, N, K, s);
  }
  if (a_tmem) return launch_tc<kQ6K, false, true>(W, nullptr, x, y, M, N, K, s);
  return launch_tc<kQ6K, false, false>(W, nullptr, x, y, M, N, K, s);
}

bool gemm_plan(QType t, bool gateup, int64_t M, int64_t N, GemmPlanInfo* info) {
  TcPlan pl;
  int at = 0;
  bool ok;
  const int a_tmem = a_tmem_default();
  if (gateup)
    ok = plan_for<kQ4K, true, false>(M, N, &pl, &at);
  else if (t == kQ4K)
    ok = a_tmem ? plan_for<kQ4K, false, true>(M, N, &pl, &at) : plan_for<kQ4K, false, false>(M, N, &pl, &at);
  else
    ok = a_tmem ? plan_for<kQ6K, false, true>(M, N, &pl, &at) : plan_for<kQ6K, false, false>(M, N, &pl, &at);
  if (!ok) return false;
  uint32_t sm_smem, reserved;
  sm_smem_limits(&sm_smem, &reserved);
  info->token_tile = pl.BN;
  info->x_stages = pl.SX;
  info->a_stages = pl.SA;
  info->packed_stages = pl.P;
  info->a_in_tmem = at;
  info->tmem_cols = (int)pl.tmem_cols;
  info->smem_bytes = (int)pl.smem;
  info->max_ctas_per_sm = (int)(sm_smem / (pl.smem + reserved));
  return true;
}

}  // namespace qk
