// qk_dequant.cu -- bit-exact fp32 dequantization of Q4_K and Q6_K blocks.
//
// Source: "Building DAMASCUS", "Read the model, then reproduce its
// operations" (the Q4_K / Q6_K dequantizers are checked before anything else
// uses them).  Block layouts are the public GGUF definitions.
//
// Each warp decodes groups of 4 consecutive 256-weight blocks (their loads
// issued together); lane t produces weights 4t..4t+3 and 128+4t..128+4t+3 of
// each block, so each of the warp's two 16-byte streaming stores covers 512
// contiguous bytes: whole 32-byte sectors.  (With lane t writing weights
// 8t..8t+7 as two vectors, each store instruction half-filled every sector it
// touched, and the export ran at 4.2 instead of 5.9 TB/s on GB300.)
// Arithmetic uses __fmul_rn / __fsub_rn, which the compiler never fuses, in
// the order (d*sc)*q - (dmin*m), matching the fp32 expression exactly.  The kernels are HBM-bound: 144 (210) bytes in, 1024 bytes out per
// block.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "qk_device.cuh"
#include "qk_internal.h"

namespace qk {

__device__ uint32_t g_dequant_status = 0;

namespace {

constexpr int kWarpsPerCta = 8;
constexpr int kGroup = 4;  // consecutive blocks per warp and iteration: their loads go out together

__device__ __forceinline__ float half_bits_to_float(uint32_t bits16) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(bits16 & 0xFFFFu)));
}

// Streaming 16-byte store: the output is written once and not read back here.
__device__ __forceinline__ void st_stream16(float* p, float a, float b, float c, float d) {
  asm volatile("st.global.cs.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}

// Sub-block j's 6-bit scale and min of a Q4_K header (scales in hdr.y..w).
__device__ __forceinline__ void q4k_scale_min(uint4 hdr, int j, uint32_t& sc, uint32_t& mn) {
  const uint32_t s03 = hdr.y, s47 = hdr.z, s811 = hdr.w;
  if (j < 4) {
    sc = (s03 >> (8 * j)) & 63u;
    mn = (s47 >> (8 * j)) & 63u;
  } else {
    const int jj = j - 4;
    const uint32_t lo = (s811 >> (8 * jj)) & 0xFFu;
    sc = (lo & 0x0Fu) | (((s03 >> (8 * jj + 6)) & 3u) << 4);
    mn = (lo >> 4) | (((s47 >> (8 * jj + 6)) & 3u) << 4);
  }
}

// One Q4_K block: lane t writes weights 4t .. 4t+3 and 128+4t .. 128+4t+3.
// qa / qb: quant bytes 32(t/16) + 4(t%8) .. +3 and the 4 bytes 64 further on
// (the low nibbles for t % 16 < 8, else the high nibbles).
__device__ __forceinline__ void q4k_lane(uint4 hdr, uint32_t qa, uint32_t qb, int lane, float* out) {
  const float d = half_bits_to_float(hdr.x);
  const float dmin = half_bits_to_float(hdr.x >> 16);
  const int shift = (lane & 8) ? 4 : 0;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    uint32_t sc, mn;
    q4k_scale_min(hdr, 4 * half + (lane >> 3), sc, mn);
    const float dsc = __fmul_rn(d, (float)sc);
    const float dmn = __fmul_rn(dmin, (float)mn);
    const uint32_t word = half ? qb : qa;
    float w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) w[e] = __fsub_rn(__fmul_rn(dsc, (float)((word >> (8 * e + shift)) & 0xFu)), dmn);
    st_stream16(out + 128 * half + 4 * lane, w[0], w[1], w[2], w[3]);
  }
}

// One Q6_K block (staged in shared memory at sb): lane t writes weights
// 4t .. 4t+3 and 128+4t .. 128+4t+3.
__device__ __forceinline__ void q6k_lane(const uint8_t* sb, int lane, float* out) {
  const float d = half_bits_to_float((uint32_t)sb[208] | ((uint32_t)sb[209] << 8));
  const int g = lane >> 3, l0 = 4 * (lane & 7);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const float dsc = __fmul_rn(d, (float)(int8_t)sb[192 + 8 * h + 2 * g + (l0 >> 4)]);
    float w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int l = l0 + e;
      const uint32_t lb = sb[64 * h + 32 * (g & 1) + l];
      const uint32_t lo = g < 2 ? (lb & 0xFu) : (lb >> 4);
      const uint32_t hi = (sb[128 + 32 * h + l] >> (2 * g)) & 3u;
      w[e] = __fmul_rn(dsc, (float)((int)(lo | (hi << 4)) - 32));
    }
    st_stream16(out + 128 * h + 4 * lane, w[0], w[1], w[2], w[3]);
  }
}

// Warp w takes the groups of kGroup consecutive blocks g = w, w + warps, ...
// and issues every load of a group before it converts and stores.
__global__ void __launch_bounds__(kWarpsPerCta * 32) dequant_q4k_kernel(const uint8_t* __restrict__ blocks,
                                                                        int64_t n_blocks, float* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = (int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  const int64_t nwarps = (int64_t)gridDim.x * kWarpsPerCta;
  const int64_t groups = (n_blocks + kGroup - 1) / kGroup;
  for (int64_t gi = warp0; gi < groups; gi += nwarps) {
    const int64_t b0 = gi * kGroup;
    const int nbk = (int)(n_blocks - b0 < kGroup ? n_blocks - b0 : kGroup);
    uint4 hdr[kGroup];
    uint32_t qa[kGroup], qb[kGroup];
#pragma unroll
    for (int i = 0; i < kGroup; ++i) {
      if (i < nbk) {
        const uint8_t* blk = blocks + (b0 + i) * kQ4KBytes;
        hdr[i] = ldg_stream16(blk);  // d, dmin, scales[0..11]
        const uint8_t* q = blk + 16 + 32 * (lane >> 4) + 4 * (lane & 7);
        qa[i] = ldg_stream4(q);
        qb[i] = ldg_stream4(q + 64);
      }
    }
#pragma unroll
    for (int i = 0; i < kGroup; ++i)
      if (i < nbk) q4k_lane(hdr[i], qa[i], qb[i], lane, out + (b0 + i) * kQK);
  }
}

__global__ void __launch_bounds__(kWarpsPerCta * 32) dequant_q6k_kernel(const uint8_t* __restrict__ blocks,
                                                                        int64_t n_blocks, float* __restrict__ out) {
  // kGroup consecutive blocks (840 bytes, 8-byte aligned: 4 * 210 = 8 * 105)
  __shared__ __align__(16) uint2 stage[kWarpsPerCta][kGroup * kQ6KBytes / 8];
  const int lane = threadIdx.x & 31;
  const int wid = threadIdx.x >> 5;
  const int64_t warp0 = (int64_t)blockIdx.x * kWarpsPerCta + wid;
  const int64_t nwarps = (int64_t)gridDim.x * kWarpsPerCta;
  const int64_t groups = (n_blocks + kGroup - 1) / kGroup;
  const uint8_t* sb = reinterpret_cast<const uint8_t*>(stage[wid]);
  for (int64_t gi = warp0; gi < groups; gi += nwarps) {
    const int64_t b0 = gi * kGroup;
    const int nbk = (int)(n_blocks - b0 < kGroup ? n_blocks - b0 : kGroup);
    const uint8_t* src = blocks + b0 * kQ6KBytes;
    if (nbk == kGroup) {
      const uint2* s8 = reinterpret_cast<const uint2*>(src);
      uint2 v[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int i = lane + 32 * k;
        if (i < kGroup * kQ6KBytes / 8) v[k] = ldg_stream8(s8 + i);
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int i = lane + 32 * k;
        if (i < kGroup * kQ6KBytes / 8) stage[wid][i] = v[k];
      }
    } else {
      // the tensor's last, partial group: 2-byte copies of the blocks that exist
      const uint16_t* s2 = reinterpret_cast<const uint16_t*>(src);
      uint16_t* d2 = reinterpret_cast<uint16_t*>(stage[wid]);
      for (int i = lane; i < nbk * kQ6KBytes / 2; i += 32) d2[i] = s2[i];
    }
    __syncwarp();
    for (int i = 0; i < nbk; ++i) q6k_lane(sb + i * kQ6KBytes, lane, out + (b0 + i) * kQK);
    __syncwarp();
  }
}

__global__ void wait_probe_kernel(uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ uint32_t abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&bar, 0u, &abort_flag, &g_dequant_status, false, limit_ns);
}

}  // namespace

cudaError_t launch_wait_probe(uint64_t limit_ns, cudaStream_t s) {
  wait_probe_kernel<<<1, 32, 0, s>>>(limit_ns);
  return cudaGetLastError();
}

uint32_t dequant_take_status() {
  uint32_t v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_dequant_status, sizeof(v)) != cudaSuccess) return 0;
  cudaMemcpyToSymbol(g_dequant_status, &zero, sizeof(zero));
  v |= take_debug_status();
  return v;
}

cudaError_t launch_dequant(QType t, const void* blocks, int64_t n_blocks, float* out, cudaStream_t s) {
  const int sms = device_sms();
  const int64_t groups = (n_blocks + kGroup - 1) / kGroup;
  const int64_t ctas_needed = (groups + kWarpsPerCta - 1) / kWarpsPerCta;
  const int64_t cap = (int64_t)sms * 8;  // the CTAs that fit at once (256 threads each)
  const int grid = (int)(ctas_needed < cap ? ctas_needed : cap);
  if (t == kQ4K)
    dequant_q4k_kernel<<<grid, kWarpsPerCta * 32, 0, s>>>(static_cast<const uint8_t*>(blocks), n_blocks, out);
  else
    dequant_q6k_kernel<<<grid, kWarpsPerCta * 32, 0, s>>>(static_cast<const uint8_t*>(blocks), n_blocks, out);
  return cudaGetLastError();
}

}  // namespace qk
