// qk_device.cuh -- device-side helpers for the sm_103a kernels: inline PTX for
// mbarriers, TMA, tcgen05 (UMMA + tensor memory), and bounded waits.
//
// Every wait on an mbarrier is bounded.  When the bound is hit the waiting
// thread records QK_DEV_TIMEOUT in the translation unit's device status word
// and in a CTA-wide abort flag, and returns false; callers then stop issuing
// work, drain what they already issued and leave.  No path uses __trap, an
// assert or an unbounded spin.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

#define QK_DEV_OK 0u
#define QK_DEV_TIMEOUT 1u
#define QK_DEV_BAD_ARG 2u
#ifndef QK_DEV_BAD_COPY
#define QK_DEV_BAD_COPY 4u
#endif

// Wall-clock bound of one mbarrier wait, in nanoseconds of %globaltimer.  A
// healthy wait lasts at most one tile's worth of work (well under a
// millisecond); the bound only ends waits that can never complete.
#ifndef QK_WAIT_LIMIT_NS
#define QK_WAIT_LIMIT_NS 2000000000ull
#endif

namespace qk {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Debug builds (-DQK_DEBUG) check every bulk and tensor copy before it is
// issued: shared-memory destination and mbarrier aligned (16 and 8 bytes) and
// inside the CTA's shared memory, global source and byte count of a plain
// bulk copy 16-byte aligned, byte count not zero.  A copy that fails is not
// issued; QK_DEV_BAD_COPY goes to a status word of the translation unit,
// which its take_status function reports (the waits on that copy's barrier
// then time out).  Release builds compile the checks away.
#ifdef QK_DEBUG
static __device__ uint32_t g_debug_status;

extern __shared__ uint8_t qk_debug_dyn_smem[];

// End of the CTA's shared memory in the shared window: the dynamic region
// follows the static one, so its base plus its size bounds both.
__device__ __forceinline__ uint32_t smem_end() {
  uint32_t v;
  asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(v));
  return smem_u32(qk_debug_dyn_smem) + v;
}

__device__ __forceinline__ bool copy_ok(uint32_t dst, uint32_t dst_bytes, uint32_t bar, uint64_t src, uint32_t src_align) {
  const uint64_t end = smem_end();
  const bool ok = (dst & 15u) == 0u && (bar & 7u) == 0u && (src & (uint64_t)(src_align - 1u)) == 0u &&
                  dst_bytes > 0u && (uint64_t)dst + dst_bytes <= end && (uint64_t)bar + 8u <= end;
  if (!ok) atomicOr(&g_debug_status, QK_DEV_BAD_COPY);
  return ok;
}

// Reads and clears this translation unit's debug status word.
static inline uint32_t take_debug_status() {
  uint32_t v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_debug_status, sizeof(v)) != cudaSuccess) return 0;
  cudaMemcpyToSymbol(g_debug_status, &zero, sizeof(zero));
  return v;
}
#define QK_COPY_CHECK(dst, bytes, bar, src, align) \
  if (!::qk::copy_ok((dst), (bytes), (bar), (uint64_t)(src), (align))) return
#else
static inline uint32_t take_debug_status() { return 0; }
#define QK_COPY_CHECK(dst, bytes, bar, src, align) (void)0
#endif

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
                   smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait for phase `parity` of `bar`.  Returns false (and raises the
// abort flag and the device status word) once QK_WAIT_LIMIT_NS has passed,
// or early if another thread of the CTA already aborted (unless
// `ignore_abort`, used when draining copies that are still in flight).
// kSleepNs > 0 sleeps that long between polls after the first miss, for
// waits whose latency is hidden anyway, so that the polling warp leaves
// issue slots to the warps sharing its scheduler.
template <uint32_t kSleepNs = 0>
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile uint32_t* abort_flag,
                                          uint32_t* dev_status, bool ignore_abort = false,
                                          uint64_t limit_ns = QK_WAIT_LIMIT_NS) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 1;; ++i) {
    if constexpr (kSleepNs > 0) __nanosleep(kSleepNs);
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0u) {
      if (!ignore_abort && *abort_flag) return false;
      if (global_ns() - t0 > limit_ns) break;
    }
  }
  *abort_flag = 1u;
  atomicOr(dev_status, QK_DEV_TIMEOUT);
  return false;
}

// ---------------------------------------------------------------------------
// TMA (bulk tensor copies) and proxy fences
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_1d(void* dst, const void* tmap, int32_t x, uint64_t* bar) {
  QK_COPY_CHECK(smem_u32(dst), 16u, smem_u32(bar), tmap, 64u);
  asm volatile(
      "cp.async.bulk.tensor.1d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2}], [%3];" ::"r"(
          smem_u32(dst)),
      "l"(tmap), "r"(x), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tma_load_2d(void* dst, const void* tmap, int32_t x, int32_t y, uint64_t* bar) {
  QK_COPY_CHECK(smem_u32(dst), 16u, smem_u32(bar), tmap, 64u);
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(smem_u32(dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* dst, const void* tmap, int32_t x, int32_t y, int32_t z,
                                            uint64_t* bar) {
  QK_COPY_CHECK(smem_u32(dst), 16u, smem_u32(bar), tmap, 64u);
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(smem_u32(dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

// Plain (non-tensor) bulk copy global -> shared: both addresses 16-byte
// aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  QK_COPY_CHECK(smem_u32(dst), (bytes & 15u) ? 0u : bytes, smem_u32(bar), src, 16u);
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// The same with shared-window addresses for the destination and the mbarrier.
__device__ __forceinline__ void bulk_copy_g2s_u32(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  QK_COPY_CHECK(dst, (bytes & 15u) ? 0u : bytes, bar, src, 16u);
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

// Make this thread's generic-proxy shared-memory writes visible to the async
// proxy (the tensor core reads UMMA operands through it).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Thread-block clusters and distributed shared memory
// ---------------------------------------------------------------------------
// Every thread of every CTA of the cluster arrives and waits (release /
// acquire): shared-memory writes before it, including remote ones, are
// visible to every thread after it.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The shared::cluster address of shared-memory address `a` (of this CTA's
// window) in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t a, uint32_t rank) {
  uint32_t d;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(rank));
  return d;
}

// Hardware tanh approximation (one special-function op, relative error
// about 2^-11).
__device__ __forceinline__ float tanh_approx(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void sts128_u(uint32_t a, uint32_t x, uint32_t y, uint32_t z, uint32_t w) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(x), "r"(y), "r"(z), "r"(w) : "memory");
}

// Bulk copy from this CTA's shared memory to another CTA's of the cluster
// (dst and mbar are shared::cluster addresses from mapa): 16-byte aligned
// addresses, size a multiple of 16; completes tx bytes on mbar.
__device__ __forceinline__ void bulk_copy_s2cluster(uint32_t dst, uint32_t src, uint32_t bytes, uint32_t mbar) {
  // dst and mbar are cluster-window addresses of a peer CTA: checked for
  // alignment only; the local source also for its extent.
  QK_COPY_CHECK(src, (bytes & 15u) || (dst & 15u) || (mbar & 7u) ? 0u : bytes, 0u, 0u, 16u);
  asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   dst),
               "r"(src), "r"(bytes), "r"(mbar)
               : "memory");
}

// Named barrier over `count` threads (whole warps).
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ uint4 lds128_u(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a)
               : "memory");
  return v;
}

// ---------------------------------------------------------------------------
// tcgen05: tensor memory and UMMA
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]^T, kind::f16, fp32 accumulate.
__device__ __forceinline__ void umma_f16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem desc]^T, kind::f16, fp32 accumulate.  A is
// 128 lanes (rows) x K/2 columns, two fp16 per 32-bit column (even k low).
__device__ __forceinline__ void umma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Thread i of the warp writes 16 consecutive 32-bit columns of TMEM lane
// (quarter*32 + i) starting at taddr.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Arrive once on `bar` when every UMMA issued so far by this thread completes.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 32 lanes x 32 bit, 16 consecutive columns: thread i of the warp gets lane
// (quarter*32 + i), columns [col, col+16).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

// UMMA shared-memory matrix descriptor for a K-major operand stored in the
// 128-byte-swizzle canonical layout: rows of 64 fp16 (128 B), 8-row atoms of
// 1024 B, atoms stacked along M/N at 1024 B.  Start address in 16 B units.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= (uint64_t)((smem_addr & 0x3FFFFu) >> 4);  // start address
  d |= (uint64_t)1u << 16;                         // leading byte offset (unused for swizzled K-major)
  d |= (uint64_t)(1024u >> 4) << 32;               // stride byte offset: next 8-row atom
  d |= (uint64_t)1u << 46;                         // descriptor version (tcgen05)
  d |= (uint64_t)2u << 61;                         // swizzle mode: 128 B
  return d;
}

// The same for the 64-byte-swizzle canonical layout: rows of 32 fp16 (64 B),
// 8-row atoms of 512 B stacked at 512 B.
__device__ __forceinline__ uint64_t umma_desc_sw64(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= (uint64_t)((smem_addr & 0x3FFFFu) >> 4);  // start address
  d |= (uint64_t)1u << 16;                         // leading byte offset (unused for swizzled K-major)
  d |= (uint64_t)(512u >> 4) << 32;                // stride byte offset: next 8-row atom
  d |= (uint64_t)1u << 46;                         // descriptor version (tcgen05)
  d |= (uint64_t)4u << 61;                         // swizzle mode: 64 B
  return d;
}

// Instruction descriptor, kind::f16: A = B = fp16, D = fp32, both K-major.
__host__ __device__ constexpr uint32_t umma_idesc_f16(uint32_t M, uint32_t N) {
  return (1u << 4)                // D format: fp32
         | (0u << 7)              // A format: fp16
         | (0u << 10)             // B format: fp16
         | (0u << 15)             // A K-major
         | (0u << 16)             // B K-major
         | ((N >> 3) << 17)       // N / 8
         | ((M >> 4) << 24);      // M / 16
}

// ---------------------------------------------------------------------------
// Loads
// ---------------------------------------------------------------------------
// Streaming 16-byte load that bypasses L1 allocation (weights are read once).
__device__ __forceinline__ uint4 ldg_stream16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint2 ldg_stream8(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t ldg_stream4(const void* p) {
  uint32_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// (a & MASK) | orv in one LOP3 (orv held in a register): written out because
// the compiler otherwise splits the two 32-bit constants into two logic ops.
template <uint32_t MASK>
__device__ __forceinline__ uint32_t lop_and_or(uint32_t a, uint32_t orv) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "n"(MASK), "r"(orv));
  return d;
}

}  // namespace qk
