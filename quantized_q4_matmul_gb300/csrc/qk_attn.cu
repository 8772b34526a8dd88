// qk_attn.cu -- grouped-query attention over a KV cache: the decode step (one
// query token, the cache split over a thread-block cluster) and prefill
// (causal query blocks against streamed key / value tiles on the tensor cores).
//
// Source: DAMASCUS project overview, "[02] the pipeline" (compartment 06: a
// decoder layer is GQA with a KV cache plus the SwiGLU FFN) and "[04] one
// decode step" (after the QKV projections and RoPE, each query head attends
// over the cached keys and values).  The pages print no formula; this
// computes scaled dot-product attention with a softmax over the causally
// visible positions, query head h reading key/value head h / (H / H_kv).
//
// Layouts: q [M][H][128] fp16 (query i at position pos0 + i sees positions
// 0 .. pos0 + i); caches [H_kv][L_max][128] fp16, head-major, so one head's
// positions are contiguous rows of 256 bytes; out [M][H][128] fp32.
//
// Decode (M = 1): a cluster of C CTAs per key/value head splits the visible
// positions into C ranges.  The G query heads of the group are the rows of
// one 16-row MMA tile (mma.sync: the dot products are tiny next to the cache
// bytes).  A copy warp streams 64-position key / value tiles (TMA, 128-byte
// swizzle, six stages deep); warps 0-3 take the even tiles and 4-7 the odd
// ones, each warp 16 positions of a tile, with a running max and sum per head.  The warps' (max, sum, output) partials are combined
// in the CTA and sent to rank 0 over DSMEM, which combines them in rank order.
//
// Prefill (M >= 2) on the 5th-generation tensor cores: one CTA per 128
// queries of one head.  Key and value tiles of 128 positions arrive by TMA
// (two stages each, keys a tile ahead); one thread issues S = Q K^T (UMMA,
// 128 x 128, fp32 in tensor memory, two buffers) and O += P V (P from tensor
// memory, V as an MN-major operand, O in tensor memory); eight softmax warps
// (two per row, half the positions each) turn S into fp16 P with a running
// max that moves only when the row max grows by more than 2^8, so O is rarely
// rescaled.
//
// All waits are bounded; a timeout raises the device status word.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstring>

#include "qk_device.cuh"
#include "qk_internal.h"

namespace qk {

__device__ uint32_t g_attn_status = 0;

namespace {

constexpr int kD = 128;               // head dimension
constexpr int kRowBytes = kD * 2;     // one position of one head, fp16
constexpr int kMaxGroup = 8;          // query heads per key/value head



__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// ---------------------------------------------------------------------------
// Tiles and warp-level MMA helpers (decode)
// ---------------------------------------------------------------------------
constexpr int kPK = 64;                                // positions per key / value tile
constexpr int kPBox = kPK * 128;                       // one 64-dim box: 64 rows x 128 bytes
constexpr int kPTile = 2 * kPBox;                      // 16 KB: a key or value tile

__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// Shared address of 16-byte chunk c (dims 8c .. 8c+7) of row r of a tile
// stored as two 128-byte-swizzled 64-dim boxes.
__device__ __forceinline__ uint32_t tile_addr(uint32_t base, int r, int c) {
  return base + (uint32_t)((c >> 3) * kPBox + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// 2^x with the hardware approximation (relative error about 2^-22, far below
// the fp16 rounding the weights get next; subnormal results flush to zero).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
  const __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// ---------------------------------------------------------------------------
// Decode
// ---------------------------------------------------------------------------
constexpr int kDecWarps = 8;        // two streams of 4 warps (even / odd tiles); a warp takes 16 positions
constexpr int kDecThreads = 32 * (kDecWarps + 1);  // + one copy warp
constexpr int kDecStages = 6;       // key + value tiles in flight (32 KB each)
constexpr int kDecMaxCluster = 8;

struct DecShared {
  uint8_t k[kDecStages][kPTile];     // after the last tile, also the warps' partials
  uint8_t v[kDecStages][kPTile];
  float red[kDecMaxCluster][kMaxGroup][kD + 2];  // rank 0: every CTA's (max, sum, output)
  uint64_t full[kDecStages];
  uint64_t empty[kDecStages];
  uint32_t abort_flag;
};

__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// One query token.  CTA rank r of the cluster for key/value head g takes
// positions [r n / C, (r + 1) n / C) in 64-position tiles; its G query heads
// are the rows of one 16-row MMA tile (rows past G are zero).  Warps 0-3 take
// the even tiles and warps 4-7 the odd ones, warp w positions 16 (w % 4) ..
// +15 of each; every warp keeps its own running max, sum and output.
__global__ void __launch_bounds__(kDecThreads, 1)
    attn_decode_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                       const __half* __restrict__ q, float* __restrict__ out, int G, int64_t n, float scale_log2e,
                       int C) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  DecShared& S = *reinterpret_cast<DecShared*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = lane >> 2, tq = lane & 3;
  const int g = blockIdx.y;
  const uint32_t rank = cluster_rank();
  const int64_t j0 = (int64_t)rank * n / C, j1 = (int64_t)(rank + 1) * n / C;
  const int nt = (int)((j1 - j0 + kPK - 1) / kPK);

  auto issue = [&](int t) {
    const int s = t % kDecStages;
    const int y = (int)(j0 + (int64_t)t * kPK);
    mbar_arrive_expect_tx(&S.full[s], 2u * kPTile);
    tma_load_3d(S.k[s], &tm_k, 0, y, g, &S.full[s]);
    tma_load_3d(S.k[s] + kPBox, &tm_k, 64, y, g, &S.full[s]);
    tma_load_3d(S.v[s], &tm_v, 0, y, g, &S.full[s]);
    tma_load_3d(S.v[s] + kPBox, &tm_v, 64, y, g, &S.full[s]);
  };
  if (threadIdx.x == 0) {
    for (int s = 0; s < kDecStages; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], 4);  // the four warps of the tile's stream
    }
    S.abort_flag = 0;
    fence_mbar_init();
  }
  cluster_sync_all();  // barriers initialised; every CTA of the cluster is running (DSMEM below)

  float (*part)[kMaxGroup][kD + 2] = reinterpret_cast<float (*)[kMaxGroup][kD + 2]>(S.k[0]);
  bool ok = true;
  if (warp == kDecWarps) {
    // ---------------------------------------------------------------- copy warp
    if (lane == 0) {
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      int t = 0;
      for (; t < nt && ok; ++t) {
        if (t >= kDecStages)
          ok = mbar_wait(&S.empty[t % kDecStages], (uint32_t)(t / kDecStages - 1) & 1u, &S.abort_flag,
                         &g_attn_status);
        if (ok) issue(t);
      }
      const int issued = ok ? t : t - 1;
      // Drain: every tile issued has landed before its space is reused or the CTA exits.
      for (int u = (issued > kDecStages ? issued - kDecStages : 0); u < issued; ++u)
        mbar_wait(&S.full[u % kDecStages], (uint32_t)(u / kDecStages) & 1u, &S.abort_flag, &g_attn_status, true);
    }
    __syncwarp();
    __syncthreads();  // (1) the ring is free for the partials
    __syncthreads();  // (2) the partials are written
  } else {
    // ------------------------------------------------------------- compute warps
    const int stream = warp >> 2, slice = warp & 3;
    uint32_t qa[8][4];
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int row = grp + 8 * (i & 1);
        const int col = 16 * kk + 2 * tq + 8 * (i >> 1);
        qa[kk][i] = row < G ? *reinterpret_cast<const uint32_t*>(q + (int64_t)(g * G + row) * kD + col) : 0u;
      }
    float o[16][4];
#pragma unroll
    for (int dn = 0; dn < 16; ++dn)
#pragma unroll
      for (int c = 0; c < 4; ++c) o[dn][c] = 0.f;
    float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};
    const int mat = lane >> 3, mr = lane & 7;
    for (int t = stream; t < nt && ok; t += 2) {
      const int s = t % kDecStages;
      ok = mbar_wait(&S.full[s], (uint32_t)(t / kDecStages) & 1u, &S.abort_flag, &g_attn_status);
      if (!ok) break;
      const uint32_t kb = smem_u32(S.k[s]), vb = smem_u32(S.v[s]);
      float sc[2][4];
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int c = 0; c < 4; ++c) sc[j][c] = 0.f;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        uint32_t b[4];
        ldsm_x4(tile_addr(kb, 16 * slice + 8 * (mat >> 1) + mr, 2 * kk + (mat & 1)), b);
        mma16816(sc[0], qa[kk], b[0], b[1]);
        mma16816(sc[1], qa[kk], b[2], b[3]);
      }
      // scale; positions past this rank's range are the next rank's (or past n)
      const int64_t key0 = j0 + (int64_t)t * kPK + 16 * slice;
      float tmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float v = sc[j][c] * scale_log2e;
          if (key0 + 8 * j + 2 * tq + (c & 1) >= j1) v = -INFINITY;
          sc[j][c] = v;
          tmax[c >> 1] = fmaxf(tmax[c >> 1], v);
        }
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        tmax[r] = fmaxf(tmax[r], __shfl_xor_sync(0xffffffffu, tmax[r], 1));
        tmax[r] = fmaxf(tmax[r], __shfl_xor_sync(0xffffffffu, tmax[r], 2));
        const float mn = fmaxf(mrow[r], tmax[r]);
        // a warp may not have seen a position yet (all of its slice past j1)
        const float corr = mn == -INFINITY ? 1.f : exp2f(mrow[r] - mn);
        mrow[r] = mn;
        lrow[r] *= corr;
#pragma unroll
        for (int dn = 0; dn < 16; ++dn) {
          o[dn][2 * r] *= corr;
          o[dn][2 * r + 1] *= corr;
        }
      }
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const float m = mrow[c >> 1];
          const float p = m == -INFINITY ? 0.f : exp2f(sc[j][c] - m);
          sc[j][c] = p;
          lrow[c >> 1] += p;
        }
      const uint32_t pa[4] = {pack_h2(sc[0][0], sc[0][1]), pack_h2(sc[0][2], sc[0][3]), pack_h2(sc[1][0], sc[1][1]),
                              pack_h2(sc[1][2], sc[1][3])};
#pragma unroll
      for (int dp = 0; dp < 8; ++dp) {
        uint32_t b[4];
        ldsm_x4_t(tile_addr(vb, 16 * slice + 8 * (mat & 1) + mr, 2 * dp + (mat >> 1)), b);
        mma16816(o[2 * dp], pa, b[0], b[1]);
        mma16816(o[2 * dp + 1], pa, b[2], b[3]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.empty[s]);
    }
    __syncthreads();  // (1) every tile is consumed and, after the copy warp's drain, landed
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      lrow[r] += __shfl_xor_sync(0xffffffffu, lrow[r], 1);
      lrow[r] += __shfl_xor_sync(0xffffffffu, lrow[r], 2);
      const int row = grp + 8 * r;
      if (row < G) {
        float* pr = part[warp][row];
        if (tq == 0) {
          pr[0] = mrow[r];
          pr[1] = lrow[r];
        }
#pragma unroll
        for (int dn = 0; dn < 16; ++dn) {
          pr[2 + 8 * dn + 2 * tq] = o[dn][2 * r];
          pr[2 + 8 * dn + 2 * tq + 1] = o[dn][2 * r + 1];
        }
      }
    }
    __syncthreads();  // (2)
    // The CTA's partial (the warps combined in order) into rank 0's slot `rank`.
    const uint32_t red0 = mapa_shared(smem_u32(&S.red[rank][0][0]), 0);
    for (int i = threadIdx.x; i < G * (kD + 2); i += 32 * kDecWarps) {
      const int row = i / (kD + 2), e = i % (kD + 2);
      float M = -INFINITY;
      for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, part[w][row][0]);
      float acc = M;
      if (e > 0) {
        acc = 0.f;
        for (int w = 0; w < kDecWarps; ++w) {
          const float mw = part[w][row][0];
          if (mw != -INFINITY) acc = fmaf(exp2f(mw - M), part[w][row][e], acc);
        }
      }
      st_cluster_f32(red0 + 4u * (uint32_t)i, acc);
    }
  }
  __syncwarp();
  cluster_sync_all();  // every CTA's partial is in rank 0
  if (rank == 0 && warp < kDecWarps) {
    for (int i = threadIdx.x; i < G * kD; i += 32 * kDecWarps) {
      const int row = i / kD, d = i % kD;
      float M = -INFINITY;
      for (int r = 0; r < C; ++r) M = fmaxf(M, S.red[r][row][0]);
      float lsum = 0.f, acc = 0.f;
      for (int r = 0; r < C; ++r) {
        const float c = exp2f(S.red[r][row][0] - M);
        lsum = fmaf(c, S.red[r][row][1], lsum);
        acc = fmaf(c, S.red[r][row][2 + d], acc);
      }
      out[(int64_t)(g * G + row) * kD + d] = acc / lsum;
    }
  }
}

// ---------------------------------------------------------------------------
// Prefill on the 5th-generation tensor cores
// ---------------------------------------------------------------------------
constexpr int kTQ = 128;                   // queries per CTA (UMMA M)
constexpr int kTK = 128;                   // positions per key / value tile
constexpr int kTBox = 128 * 128;           // one 64-wide box of 128 rows of 128 bytes: 16 KB
constexpr int kTTile = 2 * kTBox;          // 32 KB: Q, one key or value tile, or P
constexpr int kTStages = 2;
constexpr int kTParts = 2;                 // softmax warps per TMEM lane quarter (each takes kTCols positions)
constexpr int kTCols = kTK / kTParts;      // 32 positions of S (and columns of O) per softmax thread
constexpr int kTSoftmax = 4 * kTParts;     // softmax warps
constexpr int kTThreads = 32 * (2 + kTSoftmax);  // copy warp, MMA warp, softmax warps

struct TcShared {
  uint8_t q[kTTile];
  uint8_t k[kTStages][kTTile];
  uint8_t v[kTStages][kTTile];
  uint64_t q_full;
  uint64_t k_full[kTStages];
  uint64_t k_empty[kTStages];  // S of the stage's tile is done
  uint64_t v_full[kTStages];
  uint64_t v_empty[kTStages];  // P.V of the stage's tile is done
  uint64_t s_full[2];
  uint64_t s_free[2];
  uint64_t p_full;
  uint64_t pv_done[2];  // P_i.V_i done (P buffer i % 2 free, O holds tiles 0 .. i)
  uint64_t mma_done;
  float rmax[2][kTParts][kTQ];  // [tile parity][part]: each part's row maxima
  float rsum[kTParts][kTQ];     // [part]: row sums at the end
  uint32_t tmem_base;
  uint32_t abort_flag;
};

// UMMA shared-memory descriptor of 16-wide K slice kk (0..7) of a K-major tile
// stored as two 64-wide boxes of 128 rows with the 128-byte swizzle.
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t tile, int kk) {
  return umma_desc_sw128(tile + (uint32_t)((kk >> 2) * kTBox)) + (uint64_t)(2 * (kk & 3));
}

// The same for an MN-major operand (N contiguous): rows are K (positions) of
// 128 bytes = 64 N; the two 64-wide N atoms are kTBox apart (leading byte
// offset) and groups of 8 rows 1024 bytes apart (stride byte offset); slice kk
// starts 16 rows further on.
__device__ __forceinline__ uint64_t mnmajor_desc(uint32_t tile, int kk) {
  const uint32_t a = tile + (uint32_t)(kk * 16 * 128);
  uint64_t d = 0;
  d |= (uint64_t)((a & 0x3FFFFu) >> 4);
  d |= (uint64_t)(kTBox >> 4) << 16;
  d |= (uint64_t)(1024u >> 4) << 32;
  d |= (uint64_t)1u << 46;
  d |= (uint64_t)2u << 61;
  return d;
}

// One CTA: 128 queries of one head.  Warp 0 copies Q once and the key and
// value tiles (two stages each, keys one tile ahead); warp 1 allocates tensor memory and issues the UMMAs:
// S_j = Q K_j^T (128 x 128, fp32 in tensor memory, two buffers) and
// O += P_{j-1} V_{j-1}; warps 2-9 take each S_j, a thread per query row (TMEM
// lane) and half of the 128 positions: row max (the parts of a row meet in
// shared memory), rescale of its part of O in tensor memory when the
// max grew by more than 2^8, P = 2^(s - m) rounded to fp16 into tensor memory
// (the A operand of P.V, two buffers), row sums.
__global__ void __launch_bounds__(kTThreads, 1)
    attn_prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_v, float* __restrict__ out, int H, int G, int64_t M,
                           int64_t pos0, float scale_log2e) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  TcShared& S = *reinterpret_cast<TcShared*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nqb = (int)((M + kTQ - 1) / kTQ);
  // Launch order is x fastest: every head's longest query block first, then
  // the next longest of every head, so the short blocks fill the last wave.
  const int qb = nqb - 1 - (int)blockIdx.y;
  const int h = (int)blockIdx.x, g = h / G;
  const int64_t q0 = (int64_t)qb * kTQ;
  const int64_t last_q = q0 + kTQ - 1 < M - 1 ? q0 + kTQ - 1 : M - 1;
  const int nt = (int)((pos0 + last_q) / kTK) + 1;

  if (threadIdx.x == 0) {
    mbar_init(&S.q_full, 1);
    for (int s = 0; s < kTStages; ++s) {
      mbar_init(&S.k_full[s], 1);
      mbar_init(&S.k_empty[s], 1);
      mbar_init(&S.v_full[s], 1);
      mbar_init(&S.v_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&S.s_full[b], 1);
      mbar_init(&S.s_free[b], kTSoftmax);
    }
    mbar_init(&S.p_full, kTSoftmax);
    mbar_init(&S.pv_done[0], 1);
    mbar_init(&S.pv_done[1], 1);
    mbar_init(&S.mma_done, 1);
    S.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&S.tmem_base, 512);  // S buffers at columns 0 and 128, O at 256, P buffers at 384 and 448
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;
  volatile uint32_t* abort_flag = &S.abort_flag;

  if (warp == 0) {
    // ---------------------------------------------------------------- copy warp
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      mbar_arrive_expect_tx(&S.q_full, (uint32_t)kTTile);
      tma_load_3d(S.q, &tm_q, 0, h, (int)q0, &S.q_full);
      tma_load_3d(S.q + kTBox, &tm_q, 64, h, (int)q0, &S.q_full);
      // Keys run one tile ahead of values: K_j needs S_{j-2} done, V_j needs
      // P_{j-2}.V_{j-2} done.
      bool ok = true;
      int nk = 0, nv = 0;  // tiles issued
      auto issue_k = [&]() {
        const int st = nk & 1;
        if (nk >= kTStages) ok = mbar_wait(&S.k_empty[st], (uint32_t)((nk >> 1) - 1) & 1u, abort_flag, &g_attn_status);
        if (!ok) return;
        mbar_arrive_expect_tx(&S.k_full[st], (uint32_t)kTTile);
        tma_load_3d(S.k[st], &tm_k, 0, nk * kTK, g, &S.k_full[st]);
        tma_load_3d(S.k[st] + kTBox, &tm_k, 64, nk * kTK, g, &S.k_full[st]);
        ++nk;
      };
      auto issue_v = [&]() {
        const int st = nv & 1;
        if (nv >= kTStages) ok = mbar_wait(&S.v_empty[st], (uint32_t)((nv >> 1) - 1) & 1u, abort_flag, &g_attn_status);
        if (!ok) return;
        mbar_arrive_expect_tx(&S.v_full[st], (uint32_t)kTTile);
        tma_load_3d(S.v[st], &tm_v, 0, nv * kTK, g, &S.v_full[st]);
        tma_load_3d(S.v[st] + kTBox, &tm_v, 64, nv * kTK, g, &S.v_full[st]);
        ++nv;
      };
      issue_k();
      for (int j = 0; j < nt && ok; ++j) {
        if (j + 1 < nt) issue_k();
        if (ok) issue_v();
      }
      // Drain: every copy issued has landed before the CTA exits.
      mbar_wait(&S.q_full, 0u, abort_flag, &g_attn_status, true);
      for (int u = (nk > kTStages ? nk - kTStages : 0); u < nk; ++u)
        mbar_wait(&S.k_full[u & 1], (uint32_t)(u >> 1) & 1u, abort_flag, &g_attn_status, true);
      for (int u = (nv > kTStages ? nv - kTStages : 0); u < nv; ++u)
        mbar_wait(&S.v_full[u & 1], (uint32_t)(u >> 1) & 1u, abort_flag, &g_attn_status, true);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------------- UMMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = umma_idesc_f16(kTQ, kTK);
      constexpr uint32_t idesc_pv = umma_idesc_f16(kTQ, 128) | (1u << 16);  // B (V) MN-major
      const uint32_t qa = smem_u32(S.q);
      const uint32_t t_o = tmem + 256u;
      bool ok = mbar_wait(&S.q_full, 0u, abort_flag, &g_attn_status);
      auto pv = [&](int i) {
        ok = ok && mbar_wait(&S.p_full, (uint32_t)i & 1u, abort_flag, &g_attn_status) &&
             mbar_wait(&S.v_full[i & 1], (uint32_t)(i >> 1) & 1u, abort_flag, &g_attn_status);
        if (!ok) return;
        tc_fence_after();
        const uint32_t va = smem_u32(S.v[i & 1]);
        const uint32_t t_p = tmem + 384u + (uint32_t)(64 * (i & 1));  // P: 128 positions as fp16 pairs
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_f16_ts(t_o, t_p + (uint32_t)(8 * kk), mnmajor_desc(va, kk), idesc_pv, (i > 0 || kk > 0) ? 1u : 0u);
        umma_commit(&S.pv_done[i & 1]);
        umma_commit(&S.v_empty[i & 1]);
      };
      int j = 0;
      for (; j < nt && ok; ++j) {
        const int st = j & 1, sb = j & 1;
        ok = mbar_wait(&S.k_full[st], (uint32_t)(j >> 1) & 1u, abort_flag, &g_attn_status);
        if (ok && j >= 2) ok = mbar_wait(&S.s_free[sb], (uint32_t)((j >> 1) - 1) & 1u, abort_flag, &g_attn_status);
        if (!ok) break;
        tc_fence_after();
        const uint32_t ka = smem_u32(S.k[st]);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_f16_ss(tmem + (uint32_t)(sb * kTK), kmajor_desc(qa, kk), kmajor_desc(ka, kk), idesc_s, kk > 0 ? 1u : 0u);
        umma_commit(&S.s_full[sb]);
        umma_commit(&S.k_empty[st]);
        if (j >= 1) pv(j - 1);
      }
      if (ok) pv(nt - 1);
      // every UMMA issued has completed before tensor memory is freed
      umma_commit(&S.mma_done);
      mbar_wait(&S.mma_done, 0u, abort_flag, &g_attn_status, true);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------- softmax warps
    // Every softmax warp runs every iteration and meets the others at the
    // named barriers; after an abort (a wait that timed out) it only skips work.
    const int quarter = warp & 3, part = (warp - 2) >> 2;
    const int r = 32 * quarter + lane;  // query row of the tile = TMEM lane
    const uint32_t lane_off = (uint32_t)(32 * quarter) << 16;
    const uint32_t col0 = (uint32_t)(kTCols * part);  // this part's positions of S and columns of O
    const int64_t qpos = pos0 + q0 + r;
    constexpr int kBarThreads = 32 * kTSoftmax;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nt; ++j) {
      const int sb = j & 1;
      const uint32_t t_s = tmem + lane_off + (uint32_t)(sb * kTK) + col0;
      if (ok) ok = mbar_wait(&S.s_full[sb], (uint32_t)(j >> 1) & 1u, abort_flag, &g_attn_status);
      ok = __all_sync(0xffffffffu, ok);
      const int64_t key0 = (int64_t)j * kTK + col0;
      // positions of this part the row sees: key0 .. key0 + lim - 1
      const int64_t vis = qpos - key0 + 1;
      const int lim = vis >= kTCols ? kTCols : (vis <= 0 ? 0 : (int)vis);
      uint32_t v[kTCols];
      float pmax = -INFINITY;
      // Every position of this part is visible to every row of the warp (a
      // tile below the diagonal): the loops below skip the per-position mask.
      const bool full = __all_sync(0xffffffffu, lim == kTCols);
      if (ok) {
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < kTCols / 16; ++c)
          tmem_ld16(t_s + (uint32_t)(16 * c), *reinterpret_cast<uint32_t(*)[16]>(v + 16 * c));
        tmem_wait_ld();
        // max_e(s_e * c) is c * max_e(s_e) for c >= 0 (rounding is monotonic)
        // and c * min_e(s_e) for c < 0: one multiply per row instead of one
        // per position.  Independent partial extrema keep the chains short.
        float pm[kTCols / 16];
        const bool neg = scale_log2e < 0.0f;
        const float empty = neg ? INFINITY : -INFINITY;
#pragma unroll
        for (int c = 0; c < kTCols / 16; ++c) {
          pm[c] = empty;
          if (full) {
            if (!neg) {
#pragma unroll
              for (int e = 16 * c; e < 16 * c + 16; ++e) pm[c] = fmaxf(pm[c], __uint_as_float(v[e]));
            } else {
#pragma unroll
              for (int e = 16 * c; e < 16 * c + 16; ++e) pm[c] = fminf(pm[c], __uint_as_float(v[e]));
            }
          } else {
#pragma unroll
            for (int e = 16 * c; e < 16 * c + 16; ++e)
              if (e < lim) pm[c] = neg ? fminf(pm[c], __uint_as_float(v[e])) : fmaxf(pm[c], __uint_as_float(v[e]));
          }
        }
        float ext = pm[0];
#pragma unroll
        for (int c = 1; c < kTCols / 16; ++c) ext = neg ? fminf(ext, pm[c]) : fmaxf(ext, pm[c]);
        pmax = lim > 0 ? ext * scale_log2e : -INFINITY;
      }
      // S_j is in registers: its buffer may take S_{j+2}
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.s_free[sb]);
      S.rmax[j & 1][part][r] = pmax;
      named_bar_sync(1, kBarThreads);  // every part's maxima of tile j are written
      float tmax = pmax;
#pragma unroll
      for (int o = 1; o < kTParts; ++o) tmax = fmaxf(tmax, S.rmax[j & 1][(part + o) % kTParts][r]);
      // The reference max moves only when the row max grows by more than 2^8:
      // the weights 2^(s - m) then stay below 256 (fp16 holds them) and O is
      // rescaled rarely; O and l use the same reference, so the result is the
      // same softmax.  All parts of a row take the same decision.
      const bool upd = m == -INFINITY || tmax > m + 8.0f;
      const float mn = upd ? tmax : m;
      const float corr = upd ? exp2f(m - mn) : 1.0f;
      m = mn;
      // P buffer j % 2 is free once P_{j-2}.V_{j-2} is done.
      if (ok && j >= 2) ok = mbar_wait(&S.pv_done[j & 1], (uint32_t)((j >> 1) - 1) & 1u, abort_flag, &g_attn_status);
      ok = __all_sync(0xffffffffu, ok);
      if (ok && j >= 1 && __any_sync(0xffffffffu, corr != 1.0f)) {
        // rescale this part of O once P_{j-1}.V_{j-1} is done
        ok = mbar_wait(&S.pv_done[(j - 1) & 1], (uint32_t)((j - 1) >> 1) & 1u, abort_flag, &g_attn_status);
        ok = __all_sync(0xffffffffu, ok);
        if (ok) {
          tc_fence_after();
          uint32_t w[kTCols];
          const uint32_t t_o = tmem + lane_off + 256u + col0;
#pragma unroll
          for (int c = 0; c < kTCols / 16; ++c)
            tmem_ld16(t_o + (uint32_t)(16 * c), *reinterpret_cast<uint32_t(*)[16]>(w + 16 * c));
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < kTCols; ++e) w[e] = __float_as_uint(__uint_as_float(w[e]) * corr);
#pragma unroll
          for (int c = 0; c < kTCols / 16; ++c)
            tmem_st16(t_o + (uint32_t)(16 * c), *reinterpret_cast<uint32_t(*)[16]>(w + 16 * c));
        }
      }
      if (ok) {
        tc_fence_after();
        // this part's positions as fp16 pairs: P columns (kTCols / 2) * part .. of buffer j % 2
        const uint32_t t_p = tmem + lane_off + 384u + (uint32_t)(64 * (j & 1) + (kTCols / 2) * part);
        float ls = 0.f;
#pragma unroll
        for (int c = 0; c < kTCols / 32; ++c) {
          uint32_t hp[16];
          float lp[2] = {0.f, 0.f};  // two partial sums per 32 positions
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const int e0 = 32 * c + e;
            float p0 = ex2_approx(fmaf(__uint_as_float(v[e0]), scale_log2e, -m));
            float p1 = ex2_approx(fmaf(__uint_as_float(v[e0 + 1]), scale_log2e, -m));
            if (!full) {
              p0 = e0 < lim ? p0 : 0.f;
              p1 = e0 + 1 < lim ? p1 : 0.f;
            }
            lp[(e >> 4) & 1] += p0 + p1;
            hp[e >> 1] = pack_h2(p0, p1);
          }
          tmem_st16(t_p + (uint32_t)(16 * c), hp);
          ls += lp[0] + lp[1];
        }
        tmem_wait_st();
        l = l * corr + ls;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.p_full);
    }
    if (ok) ok = mbar_wait(&S.pv_done[(nt - 1) & 1], (uint32_t)((nt - 1) >> 1) & 1u, abort_flag, &g_attn_status);
    ok = __all_sync(0xffffffffu, ok);
    S.rsum[part][r] = l;
    named_bar_sync(1, kBarThreads);
    if (ok) {
      tc_fence_after();
      const int64_t row = q0 + r;
      float lt = 0.f;
#pragma unroll
      for (int o = 0; o < kTParts; ++o) lt += S.rsum[o][r];
      const float inv = 1.0f / lt;
#pragma unroll 1
      for (int c = 0; c < kTCols / 16; ++c) {
        uint32_t v[16];
        tmem_ld16(tmem + lane_off + 256u + col0 + (uint32_t)(16 * c), v);
        tmem_wait_ld();
        if (row < M) {
          float4* dst = reinterpret_cast<float4*>(out + (row * H + h) * kD + col0 + 16 * c);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            dst[e] = make_float4(__uint_as_float(v[4 * e]) * inv, __uint_as_float(v[4 * e + 1]) * inv,
                                 __uint_as_float(v[4 * e + 2]) * inv, __uint_as_float(v[4 * e + 3]) * inv);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

size_t dec_smem() { return sizeof(DecShared) + 1024; }  // + alignment slack
size_t tc_smem() { return sizeof(TcShared) + 1024; }

}  // namespace

uint32_t attn_take_status() {
  uint32_t v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_attn_status, sizeof(v)) != cudaSuccess) return 0;
  cudaMemcpyToSymbol(g_attn_status, &zero, sizeof(zero));
  v |= take_debug_status();
  return v;
}

cudaError_t launch_gqa_attention(const uint16_t* q, const uint16_t* kc, const uint16_t* vc, float* out, int64_t M,
                                 int H, int Hkv, int64_t pos0, int64_t Lmax, float scale, cudaStream_t s) {
  const int G = H / Hkv;
  const float sl2e = scale * 1.4426950408889634f;
  const __half* qh = reinterpret_cast<const __half*>(q);
  // Tensor maps over [H_kv][visible positions][128] of each cache: positions
  // past the last query read as zero.
  const uint64_t dims[3] = {(uint64_t)kD, (uint64_t)(pos0 + M), (uint64_t)Hkv};
  const uint64_t strides[2] = {(uint64_t)kRowBytes, (uint64_t)Lmax * kRowBytes};
  if (M == 1) {
    const uint32_t box[3] = {64u, (uint32_t)kPK, 1u};
    alignas(64) CUtensorMap tk, tv;
    if (!encode_tensor_map_f16(&tk, kc, 3, dims, strides, box, true) ||
        !encode_tensor_map_f16(&tv, vc, 3, dims, strides, box, true))
      return cudaErrorInvalidValue;
    // Decode: a cluster of C CTAs per key/value head, at least 256 positions each.
    const int64_t n = pos0 + 1;
    int C = (int)((n + 255) / 256);
    C = C < 1 ? 1 : (C > kDecMaxCluster ? kDecMaxCluster : C);
    static PerDeviceFlag attr_set;
    const int dev = current_device();
    if (!attr_set.done(dev)) {
      const cudaError_t e = cudaFuncSetAttribute(attn_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)dec_smem());
      if (e != cudaSuccess) return e;
      attr_set.mark(dev);
    }
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3((unsigned)C, (unsigned)Hkv, 1);
    cfg.blockDim = dim3(kDecThreads);
    cfg.dynamicSmemBytes = dec_smem();
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, attn_decode_kernel, tk, tv, qh, out, G, n, sl2e, C);
  }
  {
    // Q: [M][H][128] as a 3-D map {128, H, M}; a box is 64 dims of one head for 128 queries.
    const uint64_t qd[3] = {(uint64_t)kD, (uint64_t)H, (uint64_t)M};
    const uint64_t qs[2] = {(uint64_t)kRowBytes, (uint64_t)H * kRowBytes};
    const uint32_t qbox[3] = {64u, 1u, (uint32_t)kTQ};
    const uint32_t kvbox[3] = {64u, (uint32_t)kTK, 1u};
    alignas(64) CUtensorMap tq, tk, tv;
    if (!encode_tensor_map_f16(&tq, q, 3, qd, qs, qbox, true) ||
        !encode_tensor_map_f16(&tk, kc, 3, dims, strides, kvbox, true) ||
        !encode_tensor_map_f16(&tv, vc, 3, dims, strides, kvbox, true))
      return cudaErrorInvalidValue;
    static PerDeviceFlag attr_set;
    const int dev = current_device();
    if (!attr_set.done(dev)) {
      const cudaError_t e = cudaFuncSetAttribute(attn_prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)tc_smem());
      if (e != cudaSuccess) return e;
      attr_set.mark(dev);
    }
    const int64_t nqb = (M + kTQ - 1) / kTQ;
    if (nqb > 65535) return cudaErrorInvalidConfiguration;
    const dim3 grid((unsigned)H, (unsigned)nqb);
    attn_prefill_tc_kernel<<<grid, kTThreads, tc_smem(), s>>>(tq, tk, tv, out, H, G, M, pos0, sl2e);
    return cudaGetLastError();
  }
}

}  // namespace qk
