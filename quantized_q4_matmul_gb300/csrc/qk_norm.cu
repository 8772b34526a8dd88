// qk_norm.cu -- RMSNorm in front of a linear, for the problems the GEMV does
// not take (M > 16, or a K it cannot stage): the normalized activations
//   xhat[m][k] = fp16( x[m][k] * r_m * gamma[k] ),  r_m = 1 / sqrt(mean_k x[m][k]^2 + eps)
// go to a caller-provided fp16 buffer that the tensor-core GEMM then reads.
// (The GEMV computes the same expression inside its x-table build.)
//
// Source: DAMASCUS project overview, "[04] one decode step" (an RMSNorm comes
// before the QKV projections and before the SwiGLU FFN); "Building DAMASCUS",
// "Read the model, then reproduce its operations".
//
// HBM-bound: one CTA per token row reads the row once (16-byte loads kept in
// registers), reduces the sum of squares in a fixed order (fp32, lane partials
// in k order, a shuffle tree, then the warps in order) and writes the row once.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <atomic>

#include "qk_device.cuh"
#include "qk_internal.h"

namespace qk {

namespace {

constexpr int kNormThreads = 256;
constexpr int kNormChunks = 4;  // 8-value chunks per thread kept in registers: K <= 8192 in one pass

__device__ __forceinline__ float hlo(uint32_t v) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(v & 0xFFFFu)));
}

__device__ __forceinline__ uint32_t h2pack(float a, float b) {
  const __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__global__ void __launch_bounds__(kNormThreads) rmsnorm_rows_kernel(const uint16_t* __restrict__ x,
                                                                     const uint16_t* __restrict__ gamma, float eps,
                                                                     uint16_t* __restrict__ out, int K) {
  __shared__ float wsum[kNormThreads / 32];
  __shared__ float r_sh;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const size_t row = (size_t)blockIdx.x * (size_t)K;
  const int nc = K / 8;
  float ss = 0.f;
  uint4 v[kNormChunks];
  // first pass over the chunks this thread keeps (K <= 8 * 256 * kNormChunks)
#pragma unroll
  for (int i = 0; i < kNormChunks; ++i) {
    const int c = tid + i * kNormThreads;
    if (c < nc) {
      v[i] = ldg_stream16(x + row + 8 * c);
      const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float a = hlo(w[j]), b = hlo(w[j] >> 16);
        ss = fmaf(b, b, fmaf(a, a, ss));
      }
    }
  }
  // longer rows: the remaining chunks, read again in the second pass
  for (int c = tid + kNormChunks * kNormThreads; c < nc; c += kNormThreads) {
    const uint4 u = ldg_stream16(x + row + 8 * c);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float a = hlo(w[j]), b = hlo(w[j] >> 16);
      ss = fmaf(b, b, fmaf(a, a, ss));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if (lane == 0) wsum[warp] = ss;
  __syncthreads();
  if (tid == 0) {
    float t = 0.f;
    for (int w = 0; w < kNormThreads / 32; ++w) t += wsum[w];
    r_sh = 1.0f / sqrtf(t / (float)K + eps);
  }
  __syncthreads();
  const float r = r_sh;
  auto emit = [&](int c, uint4 u) {
    const uint4 g = ldg_stream16(gamma + 8 * c);
    uint4 o;
    o.x = h2pack(hlo(u.x) * r * hlo(g.x), hlo(u.x >> 16) * r * hlo(g.x >> 16));
    o.y = h2pack(hlo(u.y) * r * hlo(g.y), hlo(u.y >> 16) * r * hlo(g.y >> 16));
    o.z = h2pack(hlo(u.z) * r * hlo(g.z), hlo(u.z >> 16) * r * hlo(g.z >> 16));
    o.w = h2pack(hlo(u.w) * r * hlo(g.w), hlo(u.w >> 16) * r * hlo(g.w >> 16));
    *reinterpret_cast<uint4*>(out + row + 8 * c) = o;
  };
#pragma unroll
  for (int i = 0; i < kNormChunks; ++i) {
    const int c = tid + i * kNormThreads;
    if (c < nc) emit(c, v[i]);
  }
  for (int c = tid + kNormChunks * kNormThreads; c < nc; c += kNormThreads) emit(c, ldg_stream16(x + row + 8 * c));
}

}  // namespace

// Scratch of qk_rmsnorm_matmul_batch_static, the entry point that allocates
// nothing: the normalized activations of the problems the tensor-core GEMM
// runs.  A file-scope array of fixed size that every GPU loading the library
// holds until the process exits; every call shares it.
static __device__ __align__(256) uint16_t g_static_scratch[kStaticScratchBytes / 2];

// The device address of g_static_scratch on the current device.  In host code
// the array's name is only a host-side stand-in, so its address comes from
// cudaGetSymbolAddress, once per device with that device current, and is kept.
cudaError_t static_scratch_address(void** out) {
  static std::atomic<void*> cache[kMaxDevices];
  const int dev = current_device();
  if (dev < 0) return cudaErrorInvalidDevice;
  void* p = cache[dev].load(std::memory_order_acquire);
  if (!p) {
    const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) return e;
    cache[dev].store(p, std::memory_order_release);
  }
  *out = p;
  return cudaSuccess;
}

cudaError_t launch_rmsnorm_rows(const uint16_t* x, const uint16_t* gamma, float eps, uint16_t* out, int64_t M,
                                int64_t K, cudaStream_t s) {
  if (M <= 0) return cudaSuccess;
  if (M > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  rmsnorm_rows_kernel<<<(unsigned)M, kNormThreads, 0, s>>>(x, gamma, eps, out, (int)K);
  return cudaGetLastError();
}

}  // namespace qk
