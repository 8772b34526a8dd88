/*
 * qk.h -- C ABI of libqk: fused dequantize-and-multiply of GGUF Q4_K / Q6_K
 * weights with fp16 activations on NVIDIA GB300 (sm_103a).
 *
 * What the library computes (DAMASCUS project overview, "[01] the thesis",
 * "[04] one decode step"; "Building DAMASCUS", "Read the model, then
 * reproduce its operations" and "Prefill and decode need different
 * performance questions"):
 *   every linear layer of a Llama-3.2-3B decoder (QKV, O, SwiGLU gate/up,
 *   down, tied LM head) as y = x . W^T with W stored as quantized Q4_K / Q6_K
 *   super-blocks and dequantized on the fly; decode is the M = 1 case (a
 *   bandwidth-bound GEMV), prefill the M > 1 case (a compute-bound GEMM).
 *
 * Block formats (public GGUF definitions; the pages name them but do not print
 * their layout):
 *   Q4_K, 144 bytes per 256 weights: fp16 d, fp16 dmin, 12 bytes of packed
 *     6-bit scales/mins for 8 sub-blocks of 32, 128 bytes of 4-bit quants;
 *     w = (d * sc) * q - (dmin * m).
 *   Q6_K, 210 bytes per 256 weights: 128 bytes low 4 bits, 64 bytes high 2
 *     bits, 16 int8 scales (one per 16 weights), fp16 d;
 *     w = (d * sc) * (q - 32).
 *
 * Conventions for every entry point:
 *   - Weights W: N rows of K/256 consecutive blocks (row n = output feature n),
 *     rows packed back to back (row stride = K/256 * block bytes).
 *   - x: [M][K] fp16 (IEEE binary16 bit patterns), row-major, dense.
 *   - y: [M][N] row-major, dense (fp32, or fp16 for the SwiGLU entry point).
 *   - All pointers are DEVICE pointers of the current CUDA device (or mapped
 *     host memory the device can read), 16-byte aligned.  The caller owns every
 *     buffer; the library allocates no device memory on any call.
 *   - K must be a positive multiple of 256 and N, K below 2^31; M is at most
 *     8,388,480 (65535 token tiles of 128).  M = 0 or N = 0 is a no-op.
 *   - y must not overlap x or the weights.
 *   - Work is enqueued asynchronously on `stream` (NULL = legacy default
 *     stream).  The return value reports argument and launch errors only; a
 *     kernel that gives up on a bounded wait sets a device flag that
 *     qk_get_device_status() reports.
 *   - No entry point aborts, exits or traps.
 *   - Results are deterministic: the same inputs give bit-identical outputs.
 */
#ifndef QK_H
#define QK_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int qk_status;

#define QK_OK 0
#define QK_ERR_NULL (-1)               /* a required pointer is NULL */
#define QK_ERR_ALIGN (-2)              /* a pointer is not 16-byte aligned */
#define QK_ERR_SHAPE (-3)              /* K % 256 != 0, a negative size, or a size beyond the limits */
#define QK_ERR_CUDA (-4)               /* a CUDA runtime call or kernel launch failed */
#define QK_ERR_TIMEOUT (-5)            /* a kernel gave up on a bounded wait (see qk_get_device_status) */
#define QK_ERR_UNSUPPORTED_DEVICE (-6) /* the current device is not an sm_103 GPU */
#define QK_ERR_ALIAS (-7)              /* the output overlaps an input */
#define QK_ERR_POINTER (-8)            /* a pointer is not accessible from the current device */
#define QK_ERR_SCRATCH (-9)            /* the built-in scratch of qk_rmsnorm_matmul_batch_static is too small */
#define QK_ERR_BAD_COPY (-10)          /* debug builds (QK_DEBUG) only: a kernel skipped a bulk or tensor copy
                                          whose addresses, size or shared-memory extent failed its check */

/* A cudaStream_t, spelled without CUDA headers. */
typedef struct CUstream_st *qk_stream_t;

/*
 * Dequantize n_blocks consecutive Q4_K blocks (144 B each) into n_blocks*256
 * fp32 weights, out[256*b + i] = weight i of block b.  Bit-exact with the
 * fp32 expression fp32(fp32(d)*sc)*q - fp32(fp32(dmin)*m) evaluated left to
 * right with round-to-nearest and no fused multiply-add ("Building DAMASCUS",
 * "Read the model, then reproduce its operations": the dequantizers are the
 * first correctness boundary).  n_blocks = 0 is a no-op.
 */
qk_status qk_dequant_q4k(const void *blocks, int64_t n_blocks, float *out, qk_stream_t stream);

/* As qk_dequant_q4k for Q6_K blocks (210 B each): w = fp32(fp32(d)*sc)*(q-32). */
qk_status qk_dequant_q6k(const void *blocks, int64_t n_blocks, float *out, qk_stream_t stream);

/*
 * Number range of the two paths.  The GEMV (M <= 8) applies the block scales
 * in fp32.  The tensor-core GEMM forms every weight in fp16: fp16(d*sc),
 * fp16(dmin*m) and fp16(q*d*sc - dmin*m), each rounded from fp32; a block
 * whose |d*sc*q| or |dmin*m| exceeds 65504 gives +-inf weights there (the
 * synthetic and real Llama scales are near 1e-4).  A non-finite d or dmin
 * makes its row's outputs non-finite on every path, as in the fp32 definition.
 */

/*
 * y[m][n] = sum_k x[m][k] * w[n][k] for Q4_K weights W (N x K), fp16 x, fp32 y
 * (DAMASCUS project overview, "[01] the thesis" / "[04] one decode step";
 * "Building DAMASCUS", "Prefill and decode need different performance
 * questions").  M <= 8 runs the GEMV (products of the integer quants with
 * fp16 x are exact, sums fp32, block scales applied per sub-block in fp32)
 * where its shared-memory plan fits (see qk_uses_gemv: the model's K = 3072
 * and K = 8192 up to M = 8); larger M, and problems the GEMV cannot
 * stage, run the tensor-core GEMM (weights dequantized to fp16 in
 * shared or tensor memory, never written to device memory; fp32 accumulation
 * in tensor memory),
 * the overview's prefill plan in which dequantized weights feed the matrix
 * unit directly and no fp16 copy of them is stored.  The two paths agree within rounding; results are not
 * bit-identical across M.  Single-tensor GEMMs keep the dequantized tiles in
 * tensor memory where they fit; QK_A_TMEM=0 in the environment (read once per
 * process) selects shared memory instead, with the same results within
 * rounding.
 */
qk_status qk_matmul_q4k(const void *blocks, const uint16_t *x_f16, float *y, int64_t M, int64_t N, int64_t K,
                        qk_stream_t stream);

/* As qk_matmul_q4k for Q6_K weights. */
qk_status qk_matmul_q6k(const void *blocks, const uint16_t *x_f16, float *y, int64_t M, int64_t N, int64_t K,
                        qk_stream_t stream);

/*
 * Fused SwiGLU feed-forward input projection (DAMASCUS project overview,
 * "[04] one decode step" and "[06] the target": FFN = SwiGLU):
 *   g = x . Wg^T, u = x . Wu^T (both N_ff x K, Q4_K), fp32 accumulation,
 *   y[m][n] = fp16( g / (1 + exp(-g)) * u ), y is [M][N_ff] fp16.
 * Gate and up weights are two separate Q4_K tensors of the same shape.  The
 * tensor-core path (M > 1) evaluates the sigmoid as 0.5 + 0.5 * tanh(g / 2)
 * with the hardware tanh approximation (relative error about 2^-11); the
 * result agrees with the definition within the fp16 output's rounding plus
 * that error.
 */
qk_status qk_gateup_swiglu_q4k(const void *gate_blocks, const void *up_blocks, const uint16_t *x_f16,
                               uint16_t *y_f16, int64_t M, int64_t N_ff, int64_t K, qk_stream_t stream);

/* Weight formats for qk_matmul_desc.qtype. */
#define QK_Q4_K 0
#define QK_Q6_K 1

/*
 * One problem of a grouped call.  up_blocks == NULL: y[M][N] (fp32) = x . W^T
 * with W in format `qtype`.  up_blocks != NULL: the fused gate/up + SwiGLU of
 * qk_gateup_swiglu_q4k (qtype must be QK_Q4_K, blocks = gate, y fp16).
 */
typedef struct qk_matmul_desc {
  int qtype;
  const void *blocks;
  const void *up_blocks;
  const uint16_t *x_f16;
  void *y;
  int64_t M, N, K;
} qk_matmul_desc;

/*
 * Run `count` independent problems (DAMASCUS project overview, "[04] one
 * decode step": the QKV projections share x, gate and up share x, and every
 * decode-step linear is an M = 1 GEMV).  Problems the GEMV runs (M <= 8)
 * share launches, up to 8 per launch, with the problems of the same
 * token-slot class (M = 1; 2..8), so small GEMVs stream their weights
 * concurrently; each keeps its own shared-memory plan and split over warps.
 * Other problems run as in qk_matmul_q4k / qk_matmul_q6k /
 * qk_gateup_swiglu_q4k.  Each entry obeys the rules of its single-problem
 * entry point; in addition no y may overlap any input or output of another
 * entry.  count = 0 is a no-op.  Results are bit-identical to calling the
 * single-problem entry points one by one.
 */
qk_status qk_matmul_batch(const qk_matmul_desc *descs, int count, qk_stream_t stream);

/*
 * int8 activations (the paper has no integer-activation variant: this is a
 * trade of accuracy for arithmetic this library offers beside the fp16
 * path).  Decode only (M = 0 or 1).  Each token's x is quantized per block of
 * 32 to int8 with one fp32 scale: d = amax / 127, q = round(x / d) (IEEE fp32
 * division, ties away from zero; d = 0 gives q = 0); y = sum_k d q w with the
 * products done as integer dot products and the block scales applied in fp32.
 * The result differs from the fp16 path by the quantization of x: per output
 * at most sum over 32-blocks of (d / 2) * sum |w| (finite x).  Problems whose K
 * the decode GEMV cannot stage are refused with QK_ERR_SHAPE (there is no
 * other int8 path).  Descriptors and rules as in qk_matmul_batch (up_blocks:
 * the fused gate/up + SwiGLU); M > 1 is QK_ERR_SHAPE.
 */
qk_status qk_matmul_batch_q8x(const qk_matmul_desc *descs, int count, qk_stream_t stream);
qk_status qk_matmul_q8x_q4k(const void *blocks, const uint16_t *x_f16, float *y, int64_t M, int64_t N, int64_t K,
                            qk_stream_t stream);
qk_status qk_matmul_q8x_q6k(const void *blocks, const uint16_t *x_f16, float *y, int64_t M, int64_t N, int64_t K,
                            qk_stream_t stream);

/*
 * RMSNorm in front of the linears (DAMASCUS project overview, "[04] one decode
 * step": an RMSNorm comes before the QKV projections and before the SwiGLU
 * FFN; "Building DAMASCUS", "Read the model, then reproduce its operations").
 * Every problem's x is replaced by
 *   xhat[m][k] = fp16( x[m][k] / sqrt(mean_k x[m][k]^2 + eps) * gamma[k] )
 * (sum of squares, scale and products in fp32; gamma is fp16[K], the same K
 * for every problem of the call; eps finite and >= 0) and the problems then
 * run as in qk_matmul_batch.  Problems the GEMV runs (M <= 8, see
 * qk_uses_gemv) normalize inside its x staging: no extra pass, no scratch.
 * Problems the tensor-core GEMM runs first have their xhat written to
 * `scratch`, a caller-owned device buffer of at least qk_rmsnorm_scratch_bytes
 * (the largest M * K * 2 over those problems; NULL is allowed when no problem
 * needs it); problems run in order on `stream` and share it.  scratch must
 * not overlap gamma or any input or output; the library cannot check its
 * size.  Returns QK_ERR_NULL (gamma, or scratch when needed), QK_ERR_ALIGN,
 * QK_ERR_SHAPE (eps negative or not finite, problems of different K), and the
 * codes of qk_matmul_batch.
 */
qk_status qk_rmsnorm_matmul_batch(const qk_matmul_desc *descs, int count, const uint16_t *gamma_f16, float eps,
                                  void *scratch, qk_stream_t stream);

/* One problem of qk_rmsnorm_matmul_batch: y = (RMSNorm(x) * gamma) . W^T, Q4_K or Q6_K weights. */
qk_status qk_rmsnorm_matmul_q4k(const void *blocks, const uint16_t *x_f16, const uint16_t *gamma_f16, float eps,
                                void *scratch, float *y, int64_t M, int64_t N, int64_t K, qk_stream_t stream);
qk_status qk_rmsnorm_matmul_q6k(const void *blocks, const uint16_t *x_f16, const uint16_t *gamma_f16, float eps,
                                void *scratch, float *y, int64_t M, int64_t N, int64_t K, qk_stream_t stream);

/* The fused gate/up + SwiGLU of qk_gateup_swiglu_q4k over RMSNorm(x) * gamma. */
qk_status qk_rmsnorm_gateup_swiglu_q4k(const void *gate_blocks, const void *up_blocks, const uint16_t *x_f16,
                                       const uint16_t *gamma_f16, float eps, void *scratch, uint16_t *y_f16,
                                       int64_t M, int64_t N_ff, int64_t K, qk_stream_t stream);

/*
 * qk_rmsnorm_matmul_batch without a scratch argument, for callers that cannot
 * allocate device memory: code running while a CUDA graph is being captured
 * (an allocation there is not recorded into the graph), callers inside a
 * framework whose memory pool owns the GPU's memory, and real-time loops that
 * allocate nothing after start-up because cudaMalloc can block and
 * synchronise the device.  The paper has no counterpart of this entry point:
 * it is a convenience of this library, not part of the method.
 *
 * The normalized activations of problems the tensor-core GEMM runs go to a
 * fixed 8 MiB array inside the library instead (every GPU that loads the
 * library holds it until the process exits): the largest M * K over those
 * problems must be at most 4,194,304 (M * K * 2 bytes <= 8 MiB), else the call
 * returns QK_ERR_SCRATCH and enqueues nothing.  The call allocates nothing and
 * calls no allocating routine.  Every call shares the array and it keeps the
 * last call's contents (each call overwrites what it reads), so calls whose
 * work may overlap on the GPU -- on different streams, or from several host
 * threads -- race on it; serialise them.  The first call on a device that
 * needs the array looks up its device address (cudaGetSymbolAddress, with
 * that device current) and keeps it; make that first call before capturing
 * any stream.  Otherwise as qk_rmsnorm_matmul_batch.
 */
qk_status qk_rmsnorm_matmul_batch_static(const qk_matmul_desc *descs, int count, const uint16_t *gamma_f16, float eps,
                                         qk_stream_t stream);

/*
 * Host-only query: bytes of scratch an M-token problem of this format and K
 * needs under qk_rmsnorm_matmul_batch (0 when the GEMV fuses the norm, else
 * M * K * 2), or -1 for invalid arguments.
 */
int64_t qk_rmsnorm_scratch_bytes(int qtype, int gateup, int64_t M, int64_t K);

/*
 * Grouped-query attention over a KV cache (DAMASCUS project overview, "[02]
 * the pipeline", compartment 06: a decoder layer is GQA with a KV cache; "[04]
 * one decode step": after the QKV projections and RoPE, attention over the
 * cache).  The pages print no formula; this is scaled dot-product attention:
 * for query i (0 <= i < M) at position pos0 + i and query head h, with
 * g = h / (H / H_kv) its key/value head,
 *   s_j = scale * sum_d q[i][h][d] * k_cache[g][j][d]   for j = 0 .. pos0 + i,
 *   out[i][h][d] = sum_j softmax(s)_j * v_cache[g][j][d].
 * q_f16: [M][H][D] fp16 (RoPE already applied); k_cache, v_cache: [H_kv][L_max][D]
 * fp16, positions 0 .. pos0 + M - 1 filled (those of the M queries included);
 * out: [M][H][D] fp32.  D must be 128, H a multiple of H_kv with H / H_kv <= 8,
 * pos0 + M <= L_max; all pointers device memory, 16-byte aligned; out may not
 * overlap an input.  M = 1 (a decode step) splits the cache over a cluster of
 * up to 8 CTAs per key/value head; M >= 2 (prefill, or a chunk of it after
 * pos0 cached positions) runs causal 128-query blocks on tcgen05.  Both score
 * on the tensor cores (fp16 operands, fp32 sums) and round the softmax weights
 * to fp16 for the P.V product: the result is within about 2^-10 * max|v| of
 * the exact value.  M = 0 is a no-op.  Errors: QK_ERR_SHAPE, QK_ERR_NULL, QK_ERR_ALIGN, QK_ERR_ALIAS,
 * QK_ERR_POINTER, QK_ERR_UNSUPPORTED_DEVICE before anything is enqueued;
 * QK_ERR_CUDA if the launch fails.
 */
qk_status qk_gqa_attention(const uint16_t *q_f16, const uint16_t *k_cache, const uint16_t *v_cache, float *out,
                           int64_t M, int64_t H, int64_t H_kv, int64_t D, int64_t pos0, int64_t L_max, float scale,
                           qk_stream_t stream);

/*
 * Synchronise `stream`, then report and clear the device-side status flags
 * that the library's kernels set when a bounded wait expires.  Returns QK_OK,
 * QK_ERR_TIMEOUT, or QK_ERR_CUDA if the synchronisation itself failed.  A
 * library built with -DQK_DEBUG also checks each bulk and tensor copy before
 * issuing it (shared-memory destination and mbarrier aligned and inside the
 * CTA's shared memory; source and size of a plain bulk copy 16-byte aligned)
 * and returns QK_ERR_BAD_COPY, ahead of QK_ERR_TIMEOUT, when one failed.
 * The flags belong to the current device, not to a stream: every stream of
 * the process on that device sets the same flags.  A timeout raised by a
 * kernel on another stream that has already finished is therefore reported
 * (and cleared) by whichever call reads the flags first, and a kernel still
 * running on another stream is not waited for.  Callers that run the library
 * on several streams and need to attribute a timeout synchronise those
 * streams before calling this, or call it from one thread after all of them.
 */
qk_status qk_get_device_status(qk_stream_t stream);

/*
 * Diagnostic for the failure path: enqueue on `stream` a kernel whose only
 * wait can never complete (an mbarrier nothing arrives on).  Like every wait
 * in the library's kernels it gives up after a wall-clock limit, here
 * `limit_ns` (clamped to 1 us .. 1 s), raises the device status word and
 * returns, so the next qk_get_device_status() reports QK_ERR_TIMEOUT and the
 * CUDA context stays usable.  No fault, trap or unbounded wait is involved.
 * Returns QK_ERR_UNSUPPORTED_DEVICE or QK_ERR_CUDA on launch problems.
 */
qk_status qk_debug_wait_timeout(int64_t limit_ns, qk_stream_t stream);

/*
 * Host-only query (no CUDA call): 1 if an M = 1 problem in format `qtype`
 * (QK_Q4_K / QK_Q6_K; with gateup != 0 the fused gate/up + SwiGLU, Q4_K only)
 * and inner size K runs on the decode GEMV, 0 if it runs on the tensor-core
 * GEMM because the GEMV cannot stage it (the x table of K plus two weight
 * stages must fit in shared memory: K <= 35840 for Q4_K, 35072 for gate/up;
 * Q6_K up to K = 26624 when K / 256 is a multiple of 8, else up to 6912),
 * -1 for an invalid qtype or K.  The answer depends only on these arguments.
 */
int qk_decode_uses_gemv(int qtype, int gateup, int64_t K);

/*
 * Host-only query (no CUDA call), for any M: 1 if an M x N x K problem in
 * format `qtype` (gateup != 0: the fused gate/up + SwiGLU) runs on the
 * CUDA-core-fed GEMV (M <= 8: M = 1 in the decode layout, 2..8 with the
 * tokens in the MMA columns; the x table of M tokens plus two weight stages
 * must fit in shared memory), 0 if it runs on the tensor-core GEMM, -1 for
 * invalid arguments.  qk_decode_uses_gemv(q, g, K) is qk_uses_gemv(q, g, 1, K).
 */
int qk_uses_gemv(int qtype, int gateup, int64_t M, int64_t K);

/*
 * Host-only query: the launch plan the tensor-core GEMM (M > 1, and M = 1
 * problems the GEMV cannot stage) uses for an M x N problem of format
 * `qtype` (gateup != 0: the fused gate/up + SwiGLU, Q4_K only).  Needs no GPU;
 * with one present, the current device's shared-memory limits are used.
 * tcgen05.alloc waits without a time limit until tensor-memory columns are
 * free, so the plan pads a CTA's shared memory until the CTAs that can share
 * an SM fit in its 512 columns together: max_ctas_per_sm * tmem_cols <= 512.
 * Returns QK_ERR_SHAPE for invalid arguments (as qk_matmul_q4k), else QK_OK.
 */
typedef struct qk_gemm_plan_info {
  int token_tile;      /* tokens per CTA tile (the UMMA N dimension), a multiple of 16 */
  int x_stages;        /* activation-tile ring depth */
  int a_stages;        /* dequantized weight-tile ring depth */
  int packed_stages;   /* packed super-block ring depth */
  int a_in_tmem;       /* 1: dequantized weight tiles live in tensor memory, 0: in shared memory */
  int tmem_cols;       /* tensor-memory columns one CTA allocates */
  int smem_bytes;      /* dynamic shared memory per CTA */
  int max_ctas_per_sm; /* CTAs that fit on one SM by shared memory */
} qk_gemm_plan_info;

qk_status qk_gemm_plan(int qtype, int gateup, int64_t M, int64_t N, int64_t K, qk_gemm_plan_info *out);

/* A static, human-readable name for a status code. */
const char *qk_status_string(qk_status status);

/* Library version, major*10000 + minor*100 + patch. */
int qk_version(void);

#ifdef __cplusplus
}
#endif

#endif /* QK_H */
