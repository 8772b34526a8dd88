// qk_api.cu -- the C ABI of libqk: argument validation and kernel selection.
//
// Every entry point checks its arguments on the host before anything is
// enqueued, so a bad call returns an error code instead of faulting the GPU:
// NULL / misaligned / non-device pointers, shapes (K % 256, negative sizes,
// overflow), output aliasing an input, and the device architecture.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <algorithm>
#include <vector>

#include "../../include/qk.h"
#include "qk_internal.h"

namespace {

using qk::QType;

constexpr int64_t kMaxDim = (int64_t)1 << 31;  // M, N, K each below 2^31
// The GEMM puts token tiles (at least 128 tokens each for M > 256) on the
// grid's y dimension, which holds at most 65535 blocks.
constexpr int64_t kMaxM = (int64_t)65535 * 128;

// sm_103 check, cached per device.
qk_status check_device() {
  static std::atomic<int> checked[qk::kMaxDevices];  // 0 unknown, 1 ok, 2 unsupported
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return QK_ERR_CUDA;
  if (dev < 0 || dev >= qk::kMaxDevices) return QK_ERR_UNSUPPORTED_DEVICE;
  int v = checked[dev].load(std::memory_order_relaxed);
  if (!v) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return QK_ERR_CUDA;
    v = (major == 10 && minor == 3) ? 1 : 2;
    checked[dev].store(v, std::memory_order_relaxed);
  }
  return v == 1 ? QK_OK : QK_ERR_UNSUPPORTED_DEVICE;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The pointer must be readable by the current device: device or managed
// memory of this device, or host memory registered with / allocated by CUDA.
qk_status check_pointer(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return QK_ERR_POINTER;
  }
  if (a.type == cudaMemoryTypeUnregistered) return QK_ERR_POINTER;
  if (a.type == cudaMemoryTypeDevice) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (a.device != dev) return QK_ERR_POINTER;
  }
  if (a.type == cudaMemoryTypeHost && a.devicePointer == nullptr) return QK_ERR_POINTER;
  return QK_OK;
}

bool overlaps(const void* a, int64_t an, const void* b, int64_t bn) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + (uintptr_t)bn && b0 < a0 + (uintptr_t)an;
}

// a * b without overflow, both non-negative; false on overflow past 2^62.
bool mul_ok(int64_t a, int64_t b, int64_t* out) {
  if (a != 0 && b > ((int64_t)1 << 62) / a) return false;
  *out = a * b;
  return true;
}

qk_status map_cuda(cudaError_t e) { return e == cudaSuccess ? QK_OK : QK_ERR_CUDA; }

qk_status dequant(QType t, const void* blocks, int64_t n_blocks, float* out, cudaStream_t s) {
  if (n_blocks < 0) return QK_ERR_SHAPE;
  if (n_blocks == 0) return QK_OK;
  if (!blocks || !out) return QK_ERR_NULL;
  if (!aligned16(blocks) || !aligned16(out)) return QK_ERR_ALIGN;
  int64_t in_bytes, out_elems, out_bytes;
  if (!mul_ok(n_blocks, qk::block_bytes(t), &in_bytes) || !mul_ok(n_blocks, qk::kQK, &out_elems) ||
      !mul_ok(out_elems, 4, &out_bytes))
    return QK_ERR_SHAPE;
  qk_status st = check_device();
  if (st != QK_OK) return st;
  if ((st = check_pointer(blocks)) != QK_OK || (st = check_pointer(out)) != QK_OK) return st;
  if (overlaps(blocks, in_bytes, out, out_bytes)) return QK_ERR_ALIAS;
  return map_cuda(qk::launch_dequant(t, blocks, n_blocks, out, s));
}

struct Checked {
  int64_t w_bytes, x_bytes, y_bytes;
};

// Host-only checks of one problem (no CUDA call); fills the byte extents.
qk_status validate_host(QType t, const void* W, const void* W_up, const uint16_t* x, const void* y, int64_t M,
                        int64_t N, int64_t K, bool gateup, Checked* c) {
  if (M < 0 || N < 0 || K < 0) return QK_ERR_SHAPE;
  if (K == 0 || K % qk::kQK != 0) return QK_ERR_SHAPE;
  if (M > kMaxM || N >= kMaxDim || K >= kMaxDim) return QK_ERR_SHAPE;
  if (gateup && t != qk::kQ4K) return QK_ERR_SHAPE;
  if (M == 0 || N == 0) {
    c->w_bytes = c->x_bytes = c->y_bytes = 0;
    return QK_OK;
  }
  if (!W || !x || !y || (gateup && !W_up)) return QK_ERR_NULL;
  if (!aligned16(W) || !aligned16(x) || !aligned16(y) || (gateup && !aligned16(W_up))) return QK_ERR_ALIGN;
  int64_t x_elems, y_elems;
  if (!mul_ok(N, (K / qk::kQK) * qk::block_bytes(t), &c->w_bytes) || !mul_ok(M, K, &x_elems) ||
      !mul_ok(x_elems, 2, &c->x_bytes) || !mul_ok(M, N, &y_elems) || !mul_ok(y_elems, gateup ? 2 : 4, &c->y_bytes))
    return QK_ERR_SHAPE;
  return QK_OK;
}

// Device-side checks (architecture, pointer kinds, aliasing) after validate_host.
qk_status validate_device(const void* W, const void* W_up, const uint16_t* x, const void* y, int64_t M, int64_t N,
                          bool gateup, const Checked& ck) {
  if (M == 0 || N == 0) return QK_OK;
  const Checked* c = &ck;
  qk_status st = check_device();
  if (st != QK_OK) return st;
  if ((st = check_pointer(W)) != QK_OK || (st = check_pointer(x)) != QK_OK || (st = check_pointer(y)) != QK_OK)
    return st;
  if (gateup && (st = check_pointer(W_up)) != QK_OK) return st;
  if (overlaps(y, c->y_bytes, x, c->x_bytes) || overlaps(y, c->y_bytes, W, c->w_bytes) ||
      (gateup && overlaps(y, c->y_bytes, W_up, c->w_bytes)))
    return QK_ERR_ALIAS;
  return QK_OK;
}

// The GEMV handles M <= 8 when its shared-memory plan fits (the x table of
// M tokens and K plus two weight stages); the tensor-core GEMM takes
// everything else.
bool use_gemv(const qk::GemvDesc& d) { return d.M <= qk::gemv_max_m() && qk::gemv_plan_fits(&d, 1); }

qk_status run(QType t, const void* W, const void* W_up, const uint16_t* x, void* y, int64_t M, int64_t N, int64_t K,
              bool gateup, cudaStream_t s) {
  const qk::GemvDesc d{t, W, gateup ? W_up : nullptr, x, y, M, N, K, nullptr, 0.f};
  if (use_gemv(d)) return map_cuda(qk::launch_gemv_batch(&d, 1, s));
  return map_cuda(qk::launch_gemm(t, W, W_up, x, y, M, N, K, gateup, s));
}

qk_status matmul(QType t, const void* W, const void* W_up, const uint16_t* x, void* y, int64_t M, int64_t N,
                 int64_t K, bool gateup, cudaStream_t s) {
  Checked c;
  qk_status st = validate_host(t, W, W_up, x, y, M, N, K, gateup, &c);
  if (st == QK_OK) st = validate_device(W, W_up, x, y, M, N, gateup, c);
  if (st != QK_OK || M == 0 || N == 0) return st;
  return run(t, W, W_up, x, y, M, N, K, gateup, s);
}

// Host and device checks of a grouped call, including that no y overlaps
// another entry's input or output.
qk_status validate_batch(const qk_matmul_desc* d, int count, std::vector<Checked>& ck) {
  ck.assign((size_t)count, Checked{});
  for (int i = 0; i < count; ++i) {
    if (d[i].qtype != QK_Q4_K && d[i].qtype != QK_Q6_K) return QK_ERR_SHAPE;
    const QType t = d[i].qtype == QK_Q4_K ? qk::kQ4K : qk::kQ6K;
    const qk_status st = validate_host(t, d[i].blocks, d[i].up_blocks, d[i].x_f16, d[i].y, d[i].M, d[i].N, d[i].K,
                                       d[i].up_blocks != nullptr, &ck[(size_t)i]);
    if (st != QK_OK) return st;
  }
  for (int i = 0; i < count; ++i) {
    const qk_status st = validate_device(d[i].blocks, d[i].up_blocks, d[i].x_f16, d[i].y, d[i].M, d[i].N,
                                         d[i].up_blocks != nullptr, ck[(size_t)i]);
    if (st != QK_OK) return st;
  }
  for (int i = 0; i < count; ++i)
    for (int j = 0; j < count; ++j) {
      if (i == j || ck[(size_t)i].y_bytes == 0 || ck[(size_t)j].y_bytes == 0) continue;
      const int64_t wb = ck[(size_t)j].w_bytes;
      if (overlaps(d[i].y, ck[(size_t)i].y_bytes, d[j].y, ck[(size_t)j].y_bytes) ||
          overlaps(d[i].y, ck[(size_t)i].y_bytes, d[j].x_f16, ck[(size_t)j].x_bytes) ||
          overlaps(d[i].y, ck[(size_t)i].y_bytes, d[j].blocks, wb) ||
          (d[j].up_blocks && overlaps(d[i].y, ck[(size_t)i].y_bytes, d[j].up_blocks, wb)))
        return QK_ERR_ALIAS;
    }
  return QK_OK;
}

// Run validated problems.  GEMV problems share launches, up to 8 per launch,
// with the problems of the same token-slot count (M = 1; 2..8); each
// keeps its own plan, so a problem's result does not depend on its group.
// With gamma, every problem's x passes through RMSNorm * gamma first: inside
// the GEMV's x staging, or for GEMM problems into `scratch` (M * K fp16),
// which the GEMM then reads (problems run in order on one stream, so they can
// share the scratch; one x is normalized once for consecutive problems).
qk_status run_batch(const qk_matmul_desc* d, int count, const uint16_t* gamma, float eps, uint16_t* scratch,
                    cudaStream_t s) {
  std::vector<qk::GemvDesc> groups[3];
  auto slot_index = [](int64_t M) { const int k = qk::gemv_slots(M); return k == 1 ? 0 : k == 8 ? 1 : 2; };
  auto flush = [&](int gi) -> qk_status {
    if (groups[gi].empty()) return QK_OK;
    const qk_status st = map_cuda(qk::launch_gemv_batch(groups[gi].data(), (int)groups[gi].size(), s));
    groups[gi].clear();
    return st;
  };
  const uint16_t* normalized = nullptr;  // the x whose rows the scratch holds
  int64_t normalized_m = 0;
  for (int i = 0; i < count; ++i) {
    if (d[i].M == 0 || d[i].N == 0) continue;
    const QType t = d[i].qtype == QK_Q4_K ? qk::kQ4K : qk::kQ6K;
    const bool gu = d[i].up_blocks != nullptr;
    const qk::GemvDesc g{t, d[i].blocks, d[i].up_blocks, d[i].x_f16, d[i].y, d[i].M, d[i].N, d[i].K, gamma, eps};
    if (use_gemv(g)) {
      const int gi = slot_index(d[i].M);
      groups[gi].push_back(g);
      if ((int)groups[gi].size() == qk::kMaxGemvProbs) {
        const qk_status st = flush(gi);
        if (st != QK_OK) return st;
      }
      continue;
    }
    const uint16_t* x = d[i].x_f16;
    if (gamma) {
      if (normalized != d[i].x_f16 || normalized_m != d[i].M) {
        const qk_status st = map_cuda(qk::launch_rmsnorm_rows(d[i].x_f16, gamma, eps, scratch, d[i].M, d[i].K, s));
        if (st != QK_OK) return st;
        normalized = d[i].x_f16;
        normalized_m = d[i].M;
      }
      x = scratch;
    }
    const qk_status st = map_cuda(qk::launch_gemm(t, d[i].blocks, d[i].up_blocks, x, d[i].y, d[i].M, d[i].N, d[i].K,
                                                  gu, s));
    if (st != QK_OK) return st;
  }
  for (int gi = 0; gi < 3; ++gi) {
    const qk_status st = flush(gi);
    if (st != QK_OK) return st;
  }
  return QK_OK;
}

qk_status matmul_batch(const qk_matmul_desc* d, int count, cudaStream_t s) {
  if (count < 0) return QK_ERR_SHAPE;
  if (count == 0) return QK_OK;
  if (!d) return QK_ERR_NULL;
  std::vector<Checked> ck;
  const qk_status st = validate_batch(d, count, ck);
  if (st != QK_OK) return st;
  return run_batch(d, count, nullptr, 0.f, nullptr, s);
}

// Bytes of RMSNorm scratch one problem needs: 0 when the GEMV runs it (the
// norm is fused into its x staging), else M * K fp16.
int64_t norm_scratch_bytes(const qk_matmul_desc& d) {
  if (d.M == 0 || d.N == 0) return 0;
  const QType t = d.qtype == QK_Q4_K ? qk::kQ4K : qk::kQ6K;
  const qk::GemvDesc g{t, d.blocks, d.up_blocks, d.x_f16, d.y, d.M, d.N, d.K, nullptr, 0.f};
  return use_gemv(g) ? 0 : d.M * d.K * 2;
}

qk_status rmsnorm_matmul_batch(const qk_matmul_desc* d, int count, const uint16_t* gamma, float eps, void* scratch,
                               cudaStream_t s) {
  if (count < 0) return QK_ERR_SHAPE;
  if (count == 0) return QK_OK;
  if (!d || !gamma) return QK_ERR_NULL;
  if (!(eps >= 0.0f) || !(eps <= 3.0e38f)) return QK_ERR_SHAPE;  // finite, non-negative
  if (!aligned16(gamma)) return QK_ERR_ALIGN;
  std::vector<Checked> ck;
  qk_status st = validate_batch(d, count, ck);
  if (st != QK_OK) return st;
  int64_t K0 = -1, need = 0;
  for (int i = 0; i < count; ++i) {
    if (d[i].M == 0 || d[i].N == 0) continue;
    if (K0 >= 0 && d[i].K != K0) return QK_ERR_SHAPE;  // one gamma of K values for every problem
    K0 = d[i].K;
    need = std::max(need, norm_scratch_bytes(d[i]));
  }
  if (K0 < 0) return QK_OK;
  if ((st = check_pointer(gamma)) != QK_OK) return st;
  for (int i = 0; i < count; ++i)
    if (ck[(size_t)i].y_bytes && overlaps(d[i].y, ck[(size_t)i].y_bytes, gamma, K0 * 2)) return QK_ERR_ALIAS;
  if (need > 0) {
    if (!scratch) return QK_ERR_NULL;
    if (!aligned16(scratch)) return QK_ERR_ALIGN;
    if ((st = check_pointer(scratch)) != QK_OK) return st;
    if (overlaps(scratch, need, gamma, K0 * 2)) return QK_ERR_ALIAS;
    for (int i = 0; i < count; ++i) {
      const Checked& c = ck[(size_t)i];
      if (c.y_bytes == 0) continue;
      if (overlaps(scratch, need, d[i].x_f16, c.x_bytes) || overlaps(scratch, need, d[i].y, c.y_bytes) ||
          overlaps(scratch, need, d[i].blocks, c.w_bytes) ||
          (d[i].up_blocks && overlaps(scratch, need, d[i].up_blocks, c.w_bytes)))
        return QK_ERR_ALIAS;
    }
  }
  return run_batch(d, count, gamma, eps, static_cast<uint16_t*>(scratch), s);
}

}  // namespace

namespace qk {

int current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
  return dev;
}

int device_sms() {
  static std::atomic<int> sms[kMaxDevices];
  const int dev = current_device();
  if (dev < 0) return 152;
  int v = sms[dev].load(std::memory_order_relaxed);
  if (v <= 0) {
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 152;
    sms[dev].store(v, std::memory_order_relaxed);
  }
  return v;
}

}  // namespace qk

extern "C" {

qk_status qk_dequant_q4k(const void* blocks, int64_t n_blocks, float* out, qk_stream_t stream) {
  return dequant(qk::kQ4K, blocks, n_blocks, out, reinterpret_cast<cudaStream_t>(stream));
}

qk_status qk_dequant_q6k(const void* blocks, int64_t n_blocks, float* out, qk_stream_t stream) {
  return dequant(qk::kQ6K, blocks, n_blocks, out, reinterpret_cast<cudaStream_t>(stream));
}

// int8 activations: validated problems with M <= 1, all on the decode GEMV
// (a problem it cannot stage is refused: there is no other int8 path).
qk_status matmul_batch_q8x(const qk_matmul_desc* d, int count, cudaStream_t s) {
  if (count < 0) return QK_ERR_SHAPE;
  if (count == 0) return QK_OK;
  if (!d) return QK_ERR_NULL;
  for (int i = 0; i < count; ++i)
    if (d[i].M > 1) return QK_ERR_SHAPE;
  std::vector<Checked> ck;
  qk_status st = validate_batch(d, count, ck);
  if (st != QK_OK) return st;
  std::vector<qk::GemvDesc> group;
  for (int i = 0; i < count; ++i) {
    if (d[i].M == 0 || d[i].N == 0) continue;
    qk::GemvDesc g{d[i].qtype == QK_Q4_K ? qk::kQ4K : qk::kQ6K, d[i].blocks, d[i].up_blocks, d[i].x_f16, d[i].y,
                   1, d[i].N, d[i].K, nullptr, 0.f};
    g.q8x = true;
    if (!qk::gemv_plan_fits(&g, 1)) return QK_ERR_SHAPE;
    group.push_back(g);
    if ((int)group.size() == qk::kMaxGemvProbs) {
      if ((st = map_cuda(qk::launch_gemv_batch(group.data(), (int)group.size(), s))) != QK_OK) return st;
      group.clear();
    }
  }
  if (!group.empty()) st = map_cuda(qk::launch_gemv_batch(group.data(), (int)group.size(), s));
  return st;
}

qk_status qk_matmul_batch_q8x(const qk_matmul_desc* descs, int count, qk_stream_t stream) {
  return matmul_batch_q8x(descs, count, reinterpret_cast<cudaStream_t>(stream));
}

qk_status qk_matmul_q8x_q4k(const void* blocks, const uint16_t* x_f16, float* y, int64_t M, int64_t N, int64_t K,
                            qk_stream_t stream) {
  const qk_matmul_desc d{QK_Q4_K, blocks, nullptr, x_f16, y, M, N, K};
  return qk_matmul_batch_q8x(&d, 1, stream);
}

qk_status qk_matmul_q8x_q6k(const void* blocks, const uint16_t* x_f16, float* y, int64_t M, int64_t N, int64_t K,
                            qk_stream_t stream) {
  const qk_matmul_desc d{QK_Q6_K, blocks, nullptr, x_f16, y, M, N, K};
  return qk_matmul_batch_q8x(&d, 1, stream);
}

qk_status qk_matmul_q4k(const void* blocks, const uint16_t* x_f16, float* y, int64_t M, int64_t N, int64_t K,
                        qk_stream_t stream) {
  return matmul(qk::kQ4K, blocks, nullptr, x_f16, y, M, N, K, false, reinterpret_cast<cudaStream_t>(stream));
}

qk_status qk_matmul_q6k(const void* blocks, const uint16_t* x_f16, float* y, int64_t M, int64_t N, int64_t K,
                        qk_stream_t stream) {
  return matmul(qk::kQ6K, blocks, nullptr, x_f16, y, M, N, K, false, reinterpret_cast<cudaStream_t>(stream));
}

qk_status qk_gateup_swiglu_q4k(const void* gate_blocks, const void* up_blocks, const uint16_t* x_f16,
                               uint16_t* y_f16, int64_t M, int64_t N_ff, int64_t K, qk_stream_t stream) {
  return matmul(qk::kQ4K, gate_blocks, up_blocks, x_f16, y_f16, M, N_ff, K, true,
                reinterpret_cast<cudaStream_t>(stream));
}

qk_status qk_matmul_batch(const qk_matmul_desc* descs, int count, qk_stream_t stream) {
  return matmul_batch(descs, count, reinterpret_cast<cudaStream_t>(stream));
}

qk_status qk_rmsnorm_matmul_batch(const qk_matmul_desc* descs, int count, const uint16_t* gamma_f16, float eps,
                                  void* scratch, qk_stream_t stream) {
  return rmsnorm_matmul_batch(descs, count, gamma_f16, eps, scratch, reinterpret_cast<cudaStream_t>(stream));
}

qk_status qk_rmsnorm_matmul_q4k(const void* blocks, const uint16_t* x_f16, const uint16_t* gamma_f16, float eps,
                                void* scratch, float* y, int64_t M, int64_t N, int64_t K, qk_stream_t stream) {
  const qk_matmul_desc d{QK_Q4_K, blocks, nullptr, x_f16, y, M, N, K};
  return qk_rmsnorm_matmul_batch(&d, 1, gamma_f16, eps, scratch, stream);
}

qk_status qk_rmsnorm_matmul_q6k(const void* blocks, const uint16_t* x_f16, const uint16_t* gamma_f16, float eps,
                                void* scratch, float* y, int64_t M, int64_t N, int64_t K, qk_stream_t stream) {
  const qk_matmul_desc d{QK_Q6_K, blocks, nullptr, x_f16, y, M, N, K};
  return qk_rmsnorm_matmul_batch(&d, 1, gamma_f16, eps, scratch, stream);
}

qk_status qk_rmsnorm_gateup_swiglu_q4k(const void* gate_blocks, const void* up_blocks, const uint16_t* x_f16,
                                       const uint16_t* gamma_f16, float eps, void* scratch, uint16_t* y_f16,
                                       int64_t M, int64_t N_ff, int64_t K, qk_stream_t stream) {
  if (!up_blocks && M > 0 && N_ff > 0) return QK_ERR_NULL;
  const qk_matmul_desc d{QK_Q4_K, gate_blocks, up_blocks, x_f16, y_f16, M, N_ff, K};
  return qk_rmsnorm_matmul_batch(&d, 1, gamma_f16, eps, scratch, stream);
}

qk_status qk_rmsnorm_matmul_batch_static(const qk_matmul_desc* descs, int count, const uint16_t* gamma_f16, float eps,
                                         qk_stream_t stream) {
  if (count < 0) return QK_ERR_SHAPE;
  if (count == 0) return QK_OK;
  if (!descs) return QK_ERR_NULL;
  int64_t need = 0;
  for (int i = 0; i < count; ++i) {
    if (descs[i].qtype != QK_Q4_K && descs[i].qtype != QK_Q6_K) return QK_ERR_SHAPE;
    if (descs[i].M < 0 || descs[i].N < 0 || descs[i].K <= 0 || descs[i].K % qk::kQK != 0 ||
        descs[i].M > kMaxM || descs[i].N >= kMaxDim || descs[i].K >= kMaxDim)
      return QK_ERR_SHAPE;
    need = std::max(need, norm_scratch_bytes(descs[i]));
  }
  if (need > (int64_t)qk::kStaticScratchBytes) return QK_ERR_SCRATCH;
  void* scratch = nullptr;
  if (need > 0) {
    const qk_status st = check_device();
    if (st != QK_OK) return st;
    if (qk::static_scratch_address(&scratch) != cudaSuccess) {
      cudaGetLastError();
      return QK_ERR_CUDA;
    }
  }
  return rmsnorm_matmul_batch(descs, count, gamma_f16, eps, scratch, reinterpret_cast<cudaStream_t>(stream));
}

int64_t qk_rmsnorm_scratch_bytes(int qtype, int gateup, int64_t M, int64_t K) {
  if ((qtype != QK_Q4_K && qtype != QK_Q6_K) || (gateup && qtype != QK_Q4_K)) return -1;
  if (K <= 0 || K % qk::kQK != 0 || K >= kMaxDim || M < 0 || M > kMaxM) return -1;
  const void* up = gateup ? reinterpret_cast<const void*>(uintptr_t(16)) : nullptr;
  const qk_matmul_desc d{qtype, nullptr, up, nullptr, nullptr, M, 1, K};
  return norm_scratch_bytes(d);
}

qk_status qk_debug_wait_timeout(int64_t limit_ns, qk_stream_t stream) {
  qk_status st = check_device();
  if (st != QK_OK) return st;
  if (limit_ns < 1000) limit_ns = 1000;
  if (limit_ns > 1000000000) limit_ns = 1000000000;
  return map_cuda(qk::launch_wait_probe((uint64_t)limit_ns, reinterpret_cast<cudaStream_t>(stream)));
}

qk_status qk_gqa_attention(const uint16_t* q_f16, const uint16_t* k_cache, const uint16_t* v_cache, float* out,
                           int64_t M, int64_t H, int64_t H_kv, int64_t D, int64_t pos0, int64_t L_max, float scale,
                           qk_stream_t stream) {
  if (M < 0 || H <= 0 || H_kv <= 0 || H % H_kv != 0 || H / H_kv > 8 || D != 128 || pos0 < 0 || L_max <= 0 ||
      M > L_max - pos0 || H > 1024 || L_max >= ((int64_t)1 << 31))
    return QK_ERR_SHAPE;
  if (M == 0) return QK_OK;
  if (!q_f16 || !k_cache || !v_cache || !out) return QK_ERR_NULL;
  if (!aligned16(q_f16) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out)) return QK_ERR_ALIGN;
  int64_t q_elems, c_elems, q_bytes, c_bytes, o_bytes;
  if (!mul_ok(M * H, D, &q_elems) || !mul_ok(q_elems, 2, &q_bytes) || !mul_ok(q_elems, 4, &o_bytes) ||
      !mul_ok(H_kv * L_max, D, &c_elems) || !mul_ok(c_elems, 2, &c_bytes))
    return QK_ERR_SHAPE;
  qk_status st = check_device();
  if (st != QK_OK) return st;
  if ((st = check_pointer(q_f16)) != QK_OK || (st = check_pointer(k_cache)) != QK_OK ||
      (st = check_pointer(v_cache)) != QK_OK || (st = check_pointer(out)) != QK_OK)
    return st;
  if (overlaps(out, o_bytes, q_f16, q_bytes) || overlaps(out, o_bytes, k_cache, c_bytes) ||
      overlaps(out, o_bytes, v_cache, c_bytes))
    return QK_ERR_ALIAS;
  return map_cuda(qk::launch_gqa_attention(q_f16, k_cache, v_cache, out, M, (int)H, (int)H_kv, pos0, L_max, scale,
                                           reinterpret_cast<cudaStream_t>(stream)));
}

qk_status qk_get_device_status(qk_stream_t stream) {
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return QK_ERR_CUDA;
  const uint32_t v =
      qk::dequant_take_status() | qk::gemv_take_status() | qk::gemm_take_status() | qk::attn_take_status();
  if (v & QK_DEV_BAD_COPY) return QK_ERR_BAD_COPY;
  return v ? QK_ERR_TIMEOUT : QK_OK;
}

int qk_uses_gemv(int qtype, int gateup, int64_t M, int64_t K) {
  if ((qtype != QK_Q4_K && qtype != QK_Q6_K) || (gateup && qtype != QK_Q4_K)) return -1;
  if (K <= 0 || K % qk::kQK != 0 || K >= kMaxDim || M <= 0 || M > kMaxM) return -1;
  // The weight and activation pointers are not dereferenced by the plan; the
  // up pointer only marks the problem as gate/up.
  const void* up = gateup ? reinterpret_cast<const void*>(uintptr_t(16)) : nullptr;
  const qk::GemvDesc d{qtype == QK_Q4_K ? qk::kQ4K : qk::kQ6K, nullptr, up, nullptr, nullptr, M, 1, K, nullptr, 0.f};
  return use_gemv(d) ? 1 : 0;
}

int qk_decode_uses_gemv(int qtype, int gateup, int64_t K) { return qk_uses_gemv(qtype, gateup, 1, K); }

qk_status qk_gemm_plan(int qtype, int gateup, int64_t M, int64_t N, int64_t K, qk_gemm_plan_info* out) {
  if (!out) return QK_ERR_NULL;
  if ((qtype != QK_Q4_K && qtype != QK_Q6_K) || (gateup && qtype != QK_Q4_K)) return QK_ERR_SHAPE;
  if (M <= 0 || N <= 0 || K <= 0 || K % qk::kQK != 0 || M > kMaxM || N >= kMaxDim || K >= kMaxDim)
    return QK_ERR_SHAPE;
  qk::GemmPlanInfo g;
  if (!qk::gemm_plan(qtype == QK_Q4_K ? qk::kQ4K : qk::kQ6K, gateup != 0, M, N, &g)) return QK_ERR_SHAPE;
  out->token_tile = g.token_tile;
  out->x_stages = g.x_stages;
  out->a_stages = g.a_stages;
  out->packed_stages = g.packed_stages;
  out->a_in_tmem = g.a_in_tmem;
  out->tmem_cols = g.tmem_cols;
  out->smem_bytes = g.smem_bytes;
  out->max_ctas_per_sm = g.max_ctas_per_sm;
  return QK_OK;
}

const char* qk_status_string(qk_status status) {
  switch (status) {
    case QK_OK: return "QK_OK";
    case QK_ERR_NULL: return "QK_ERR_NULL: a required pointer is NULL";
    case QK_ERR_ALIGN: return "QK_ERR_ALIGN: a pointer is not 16-byte aligned";
    case QK_ERR_SHAPE: return "QK_ERR_SHAPE: K must be a positive multiple of 256 and sizes non-negative";
    case QK_ERR_CUDA: return "QK_ERR_CUDA: a CUDA call or kernel launch failed";
    case QK_ERR_TIMEOUT: return "QK_ERR_TIMEOUT: a kernel gave up on a bounded wait";
    case QK_ERR_BAD_COPY: return "QK_ERR_BAD_COPY: a debug build skipped a copy that failed its check";
    case QK_ERR_UNSUPPORTED_DEVICE: return "QK_ERR_UNSUPPORTED_DEVICE: the current device is not sm_103";
    case QK_ERR_ALIAS: return "QK_ERR_ALIAS: the output overlaps an input";
    case QK_ERR_POINTER: return "QK_ERR_POINTER: a pointer is not accessible from the current device";
    case QK_ERR_SCRATCH: return "QK_ERR_SCRATCH: the problems need more than the library's 8 MiB built-in scratch";
    default: return "unknown qk_status";
  }
}

int qk_version(void) { return 100; }

}  // extern "C"
