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
// one 16-row MMA tile.  A copy warp streams 64-position key / value tiles
// (the same TMA tiles as prefill, six stages deep); warps 0-3 take the even
// tiles and 4-7 the odd ones, each warp 16 positions of a tile, with a running
// max and sum per head.  The warps' (max, sum, output) partials are combined
// in the CTA and sent to rank 0 over DSMEM, which combines them in rank order.
//
// Prefill (M >= 2): one CTA per 64-query block and group of HPC query heads
// that share a key/value head; 4 warps per head, 16 query rows each.  Key and
// value tiles (64 positions x 128 dims) arrive by TMA with a 128-byte swizzle
// (two 64-dim boxes each), three stages deep; the tensor map's position
// extent is the visible length, so rows past it read as zero.  S = Q K^T and
// O += P V run as mma.sync m16n8k16 (fp16 operands, fp32 accumulation) with
// the online softmax in registers and P re-used from the score fragments.
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
// Prefill
// ---------------------------------------------------------------------------
constexpr int kPQ = 64;                                // queries per CTA and head
constexpr int kPK = 64;                                // positions per key / value tile
constexpr int kPStages = 3;
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

struct PreShared {
  uint8_t k[kPStages][kPTile];
  uint8_t v[kPStages][kPTile];
  uint64_t full[kPStages];
  uint64_t empty[kPStages];
  uint32_t abort_flag;
};

template <int HPC>
__global__ void __launch_bounds__(128 * HPC, 1)
    attn_prefill_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                        const __half* __restrict__ q, float* __restrict__ out, int H, int G, int64_t M, int64_t pos0,
                        float scale_log2e) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte aligned: the 128-byte swizzle pattern repeats every 1024 bytes
  PreShared& S = *reinterpret_cast<PreShared*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr int kWarps = 4 * HPC;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = lane >> 2, tq = lane & 3;
  const int nqb = (int)((M + kPQ - 1) / kPQ);
  const int qb = nqb - 1 - (int)blockIdx.x;  // the longest (latest) query blocks first
  const int h = (int)blockIdx.y * HPC + warp / 4;
  const int g = ((int)blockIdx.y * HPC) / G;
  const int64_t r0 = (int64_t)qb * kPQ + 16 * (warp % 4);  // this warp's first query row
  const int64_t last_q = (int64_t)qb * kPQ + kPQ - 1 < M - 1 ? (int64_t)qb * kPQ + kPQ - 1 : M - 1;
  const int nkt = (int)((pos0 + last_q) / kPK) + 1;  // key tiles the block's last query sees

  auto issue = [&](int kt) {
    const int s = kt % kPStages;
    mbar_arrive_expect_tx(&S.full[s], 2u * kPTile);
    tma_load_3d(S.k[s], &tm_k, 0, kt * kPK, g, &S.full[s]);
    tma_load_3d(S.k[s] + kPBox, &tm_k, 64, kt * kPK, g, &S.full[s]);
    tma_load_3d(S.v[s], &tm_v, 0, kt * kPK, g, &S.full[s]);
    tma_load_3d(S.v[s] + kPBox, &tm_v, 64, kt * kPK, g, &S.full[s]);
  };
  if (threadIdx.x == 0) {
    for (int s = 0; s < kPStages; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], kWarps);
    }
    S.abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    for (int kt = 0; kt < kPStages && kt < nkt; ++kt) issue(kt);
  }
  int issued = kPStages < nkt ? kPStages : nkt;  // thread 0's count of tiles issued
  __syncthreads();

  // Q fragments of rows r0 + grp and r0 + grp + 8 (zero past M).
  uint32_t qa[8][4];
#pragma unroll
  for (int kk = 0; kk < 8; ++kk)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t row = r0 + grp + 8 * (i & 1);
      const int col = 16 * kk + 2 * tq + 8 * (i >> 1);
      qa[kk][i] = row < M ? *reinterpret_cast<const uint32_t*>(q + (row * H + h) * kD + col) : 0u;
    }
  float o[16][4];
#pragma unroll
  for (int dn = 0; dn < 16; ++dn)
#pragma unroll
    for (int c = 0; c < 4; ++c) o[dn][c] = 0.f;
  float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};
  const int64_t qpos[2] = {pos0 + r0 + grp, pos0 + r0 + grp + 8};
  bool ok = true;
  int kt = 0;
  for (; kt < nkt && ok; ++kt) {
    const int s = kt % kPStages;
    ok = mbar_wait(&S.full[s], (uint32_t)(kt / kPStages) & 1u, &S.abort_flag, &g_attn_status);
    if (!ok) break;
    const uint32_t kb = smem_u32(S.k[s]), vb = smem_u32(S.v[s]);
    float sc[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int c = 0; c < 4; ++c) sc[nt][c] = 0.f;
    const int mat = lane >> 3, mr = lane & 7;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        uint32_t b[4];
        ldsm_x4(tile_addr(kb, 16 * np + 8 * (mat >> 1) + mr, 2 * kk + (mat & 1)), b);
        mma16816(sc[2 * np], qa[kk], b[0], b[1]);
        mma16816(sc[2 * np + 1], qa[kk], b[2], b[3]);
      }
    // scale, causal mask, running max
    const int64_t key0 = (int64_t)kt * kPK;
    const bool masked = key0 + kPK - 1 > pos0 + r0;
    float tmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float v = sc[nt][c] * scale_log2e;
        if (masked && key0 + 8 * nt + 2 * tq + (c & 1) > qpos[c >> 1]) v = -INFINITY;
        sc[nt][c] = v;
        tmax[c >> 1] = fmaxf(tmax[c >> 1], v);
      }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      tmax[r] = fmaxf(tmax[r], __shfl_xor_sync(0xffffffffu, tmax[r], 1));
      tmax[r] = fmaxf(tmax[r], __shfl_xor_sync(0xffffffffu, tmax[r], 2));
      const float mn = fmaxf(mrow[r], tmax[r]);
      const float corr = exp2f(mrow[r] - mn);
      mrow[r] = mn;
      lrow[r] *= corr;
#pragma unroll
      for (int dn = 0; dn < 16; ++dn) {
        o[dn][2 * r] *= corr;
        o[dn][2 * r + 1] *= corr;
      }
    }
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float p = exp2f(sc[nt][c] - mrow[c >> 1]);
        sc[nt][c] = p;
        lrow[c >> 1] += p;
      }
    // O += P V
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t pa[4] = {pack_h2(sc[2 * j][0], sc[2 * j][1]), pack_h2(sc[2 * j][2], sc[2 * j][3]),
                              pack_h2(sc[2 * j + 1][0], sc[2 * j + 1][1]), pack_h2(sc[2 * j + 1][2], sc[2 * j + 1][3])};
#pragma unroll
      for (int dp = 0; dp < 8; ++dp) {
        uint32_t b[4];
        ldsm_x4_t(tile_addr(vb, 16 * j + 8 * (mat & 1) + mr, 2 * dp + (mat >> 1)), b);
        mma16816(o[2 * dp], pa, b[0], b[1]);
        mma16816(o[2 * dp + 1], pa, b[2], b[3]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.empty[s]);
    if (threadIdx.x == 0 && kt + kPStages < nkt) {
      ok = mbar_wait(&S.empty[s], (uint32_t)(kt / kPStages) & 1u, &S.abort_flag, &g_attn_status);
      if (ok) {
        issue(kt + kPStages);
        ++issued;
      }
    }
  }
  if (threadIdx.x == 0) {
    // Drain: every tile issued has landed before the CTA exits.
    for (int t = (issued > kPStages ? issued - kPStages : 0); t < issued; ++t)
      mbar_wait(&S.full[t % kPStages], (uint32_t)(t / kPStages) & 1u, &S.abort_flag, &g_attn_status, true);
  }
  if (!ok) return;
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    lrow[r] += __shfl_xor_sync(0xffffffffu, lrow[r], 1);
    lrow[r] += __shfl_xor_sync(0xffffffffu, lrow[r], 2);
  }
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int64_t row = r0 + grp + 8 * r;
    if (row >= M) continue;
    const float inv = 1.0f / lrow[r];
    float* dst = out + (row * H + h) * kD + 2 * tq;
#pragma unroll
    for (int dn = 0; dn < 16; ++dn)
      *reinterpret_cast<float2*>(dst + 8 * dn) = make_float2(o[dn][2 * r] * inv, o[dn][2 * r + 1] * inv);
  }
}

size_t dec_smem() { return sizeof(DecShared) + 1024; }  // + alignment slack
size_t pre_smem() { return sizeof(PreShared) + 1024; }

// Query heads per prefill CTA: the largest divisor of the group size that is
// at most 3 (one tile load serves all of them; 128 threads each).
int heads_per_cta(int G) { return G % 3 == 0 ? 3 : (G % 2 == 0 ? 2 : 1); }

template <int HPC>
cudaError_t launch_prefill(const CUtensorMap& tk, const CUtensorMap& tv, const __half* q, float* out, int H, int G,
                           int64_t M, int64_t pos0, float sl2e, cudaStream_t s) {
  static PerDeviceFlag attr_set;
  const int dev = current_device();
  if (!attr_set.done(dev)) {
    const cudaError_t e = cudaFuncSetAttribute(attn_prefill_kernel<HPC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)pre_smem());
    if (e != cudaSuccess) return e;
    attr_set.mark(dev);
  }
  const dim3 grid((unsigned)((M + kPQ - 1) / kPQ), (unsigned)(H / HPC));
  attn_prefill_kernel<HPC><<<grid, 128 * HPC, pre_smem(), s>>>(tk, tv, q, out, H, G, M, pos0, sl2e);
  return cudaGetLastError();
}

}  // namespace

uint32_t attn_take_status() {
  uint32_t v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_attn_status, sizeof(v)) != cudaSuccess) return 0;
  cudaMemcpyToSymbol(g_attn_status, &zero, sizeof(zero));
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
  const uint32_t box[3] = {64u, (uint32_t)kPK, 1u};
  alignas(64) CUtensorMap tk, tv;
  if (!encode_tensor_map_f16(&tk, kc, 3, dims, strides, box, true) ||
      !encode_tensor_map_f16(&tv, vc, 3, dims, strides, box, true))
    return cudaErrorInvalidValue;
  if (M == 1) {
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
  switch (heads_per_cta(G)) {
    case 3: return launch_prefill<3>(tk, tv, qh, out, H, G, M, pos0, sl2e, s);
    case 2: return launch_prefill<2>(tk, tv, qh, out, H, G, M, pos0, sl2e, s);
    default: return launch_prefill<1>(tk, tv, qh, out, H, G, M, pos0, sl2e, s);
  }
}

}  // namespace qk
