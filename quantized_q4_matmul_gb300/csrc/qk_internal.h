// qk_internal.h -- host-side declarations shared by the library's translation
// units (launchers, status words).  Not part of the public C ABI.
#pragma once

#include <atomic>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/qk.h"

namespace qk {

enum QType : int { kQ4K = 0, kQ6K = 1 };

constexpr int kQK = 256;
constexpr int kQ4KBytes = 144;
constexpr int kQ6KBytes = 210;

inline int64_t block_bytes(QType t) { return t == kQ4K ? kQ4KBytes : kQ6KBytes; }

// Host state that CUDA keeps per device (function attributes, SM counts,
// occupancy answers) is cached per device index, for processes that drive
// several GPUs.
constexpr int kMaxDevices = 64;

// The calling thread's current device, or -1 if it cannot be read or is out
// of range.
int current_device();

// The current device's SM count (queried once per device).
int device_sms();

// One bit per device: set once that device's one-time setup has succeeded.
class PerDeviceFlag {
 public:
  bool done(int dev) const { return dev >= 0 && ((bits_.load(std::memory_order_acquire) >> dev) & 1u); }
  void mark(int dev) {
    if (dev >= 0) bits_.fetch_or(uint64_t(1) << dev, std::memory_order_release);
  }

 private:
  std::atomic<uint64_t> bits_{0};
};

// Each translation unit with kernels that can time out owns one device status
// word; these read it (after the stream has been synchronised) and clear it.
// Status bit of a copy that a debug build (QK_DEBUG) skipped (qk_device.cuh).
#ifndef QK_DEV_BAD_COPY
#define QK_DEV_BAD_COPY 4u
#endif
uint32_t dequant_take_status();
uint32_t gemv_take_status();
uint32_t gemm_take_status();

// Launchers.  Arguments are already validated; they return cudaGetLastError().
cudaError_t launch_dequant(QType t, const void* blocks, int64_t n_blocks, float* out, cudaStream_t s);
cudaError_t launch_gemv(QType t, const void* W, const uint16_t* x, float* y, int64_t N, int64_t K,
                        cudaStream_t s);
cudaError_t launch_gemm(QType t, const void* W, const void* W_up, const uint16_t* x, void* y, int64_t M,
                        int64_t N, int64_t K, bool gateup, cudaStream_t s);

// The tensor-core GEMM's launch plan for an M x N problem (host only; the
// fields mirror qk_gemm_plan_info).  False if no plan exists.
struct GemmPlanInfo {
  int token_tile, x_stages, a_stages, packed_stages, a_in_tmem, tmem_cols, smem_bytes, max_ctas_per_sm;
};
bool gemm_plan(QType t, bool gateup, int64_t M, int64_t N, GemmPlanInfo* info);

// RMSNorm rows into an fp16 buffer (problems the GEMV does not take):
// out[m][k] = fp16(x[m][k] / sqrt(mean_k x[m][k]^2 + eps) * gamma[k]).
cudaError_t launch_rmsnorm_rows(const uint16_t* x, const uint16_t* gamma, float eps, uint16_t* out, int64_t M,
                                int64_t K, cudaStream_t s);

// The built-in scratch of qk_rmsnorm_matmul_batch_static (bytes) and its
// device address on the current device (looked up once per device).
constexpr size_t kStaticScratchBytes = size_t(8) << 20;
cudaError_t static_scratch_address(void** out);

// Encode a tiled TMA tensor map of fp16 elements into `out` (a CUtensorMap,
// 64 bytes): `rank` dimensions innermost first, the byte strides of
// dimensions 1.. (rank - 1 of them), the box, and a 128-byte swizzle or none.
// Elements outside the dimensions read as zero.  False if the driver refuses.
bool encode_tensor_map_f16(void* out, const void* base, int rank, const uint64_t* dims, const uint64_t* strides,
                           const uint32_t* box, bool swizzle128);

// GQA attention (qk_gqa_attention); arguments validated.  Device status word.
cudaError_t launch_gqa_attention(const uint16_t* q, const uint16_t* kc, const uint16_t* vc, float* out, int64_t M,
                                 int H, int Hkv, int64_t pos0, int64_t Lmax, float scale, cudaStream_t s);
uint32_t attn_take_status();

// A kernel whose single bounded wait can never complete (see qk_debug_wait_timeout).
cudaError_t launch_wait_probe(uint64_t limit_ns, cudaStream_t s);

// Largest M the GEMV handles (M = 1 in the decode layout, 2..8 with the
// tokens in the MMA columns); larger M goes to the tensor-core GEMM, which
// measured faster there on GB300 (Q4_K 3072 x 3072 at M = 16: 15 vs 24 us).
constexpr int kMaxGemvM = 8;
int gemv_max_m();
// The kernel's token-slot count for M tokens (1 or 8): problems share a
// launch only with problems of the same count.
int gemv_slots(int64_t M);

// One problem of a grouped GEMV launch.  w1 != null makes it the fused
// gate/up + SwiGLU problem (w0 = gate, w1 = up, y fp16), else y is fp32.
constexpr int kMaxGemvProbs = 8;
struct GemvDesc {
  QType qtype;
  const void* w0;
  const void* w1;
  const uint16_t* x;
  void* y;
  int64_t M, N, K;
  const uint16_t* gamma;  // RMSNorm prologue over x (fp16 gamma[K]), or null
  float eps;
  bool q8x = false;       // x quantized to int8 per block of 32 (one token, no gamma)
};
cudaError_t launch_gemv_batch(const GemvDesc* d, int count, cudaStream_t s);

// Whether one grouped GEMV launch can run these problems: each problem's own
// plan (its x table and at least two weight stages) must fit in shared memory
// and all must have the same token-slot count.  Host only (no CUDA call).
// Problems that do not fit run on the GEMM.
bool gemv_plan_fits(const GemvDesc* d, int count);

}  // namespace qk
