/*
 * qk_oracle.c -- the CPU oracle for the quantized Q4_K / Q6_K matmul path.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke
 * check and the benchmark's CPU-baseline leg load this file's library.  The
 * CUDA library never links, includes or calls it, and it shares no header,
 * table or helper with the CUDA sources.
 *
 * What it computes (sources):
 *  - DAMASCUS project overview, "[01] the thesis" and "[04] one decode step":
 *    every linear of a Llama-3.2-3B decoder layer (QKV, O, SwiGLU gate/up,
 *    down, tied LM head) is a matrix product of the quantized weights with the
 *    activations; decode is the M = 1 case (a GEMV), prefill the M > 1 case.
 *  - "Building DAMASCUS", "Read the model, then reproduce its operations":
 *    the weights are Q4_K and Q6_K blocks that are dequantized before use.
 *  - "Building DAMASCUS", "A same-weights oracle makes the comparison useful":
 *    the reference dequantizes the very same quantized blocks.
 *  The pages do not print the block layouts.  The layouts below are the public
 *  GGUF Q4_K / Q6_K super-block definitions (256 weights per block; 144 bytes
 *  and 210 bytes), which is the reading this project takes.
 *
 * Precision rules (the reading taken where the pages are silent):
 *  - fp16 scale fields are widened to fp32 exactly (IEEE binary16 -> binary32).
 *  - Q4_K weight:  w = fp32(fp32(d) * sc) * q  -  fp32(fp32(dmin) * m),
 *    Q6_K weight:  w = fp32(fp32(d) * sc) * q,
 *    each operation a separate fp32 round-to-nearest step (built with
 *    -ffp-contract=off so no multiply-add is fused).
 *  - matmul: y[m][n] = sum_k x[m][k] * w[n][k], summed in fp64 in k order;
 *    x is fp16 widened exactly, w is the fp32 dequantized weight.
 *  - SwiGLU: out = g / (1 + exp(-g)) * u with g, u the fp64 sums above.
 *  - RMSNorm in front of a linear: xhat = x / sqrt(mean(x^2) + eps) * gamma
 *    in fp64, then the matmul above over xhat (not rounded to fp16).
 *  - Q8 activations (no counterpart in the pages): x quantized to int8 per
 *    block of 32 with one fp32 scale, then the matmul above over d * q.
 *  - GQA attention over a KV cache (project overview, "[02] the pipeline",
 *    compartment 06, and "[04] one decode step"; no formula is printed):
 *    scaled dot-product attention, query head h reading key/value head
 *    h / (H / H_kv), softmax over the causally visible positions, in fp64
 *    from fp16 inputs widened exactly.
 *
 * Parity pins live in the test suite (hand-built blocks with closed forms,
 * bit-placement tables, an independent bit-level decoder, one-hot and all-ones
 * activations, a float64 library matmul, linearity and permutation).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_Q4K_BYTES 144
#define ORACLE_Q6K_BYTES 210
#define ORACLE_QK 256

/* ------------------------------------------------------------------------ */
/* IEEE 754 binary16 -> binary32, exact (binary32 holds every binary16).     */
/* ------------------------------------------------------------------------ */
float oracle_half_to_float(uint16_t h)
{
    const int sign = (h >> 15) & 1;
    const int expo = (h >> 10) & 0x1F;
    const int frac = h & 0x3FF;
    float v;
    if (expo == 31 && frac) {
        /* NaN: keep its sign and payload (the payload moves up 13 bits) */
        uint32_t bits = ((uint32_t)sign << 31) | 0x7F800000u | ((uint32_t)frac << 13);
        memcpy(&v, &bits, 4);
        return v;
    }
    if (expo == 31)
        v = INFINITY;
    else if (expo == 0)
        v = ldexpf((float)frac, -24); /* zero or subnormal: frac * 2^-24 */
    else
        v = ldexpf((float)(1024 + frac), expo - 25); /* normal: 1.frac * 2^(expo-15) */
    return sign ? -v : v;
}

static uint16_t rd16(const uint8_t *p) { return (uint16_t)(p[0] | (p[1] << 8)); }

/* ------------------------------------------------------------------------ */
/* Q4_K: bytes 0-1 d (fp16), 2-3 dmin (fp16), 4-15 packed 6-bit scales and    */
/* mins of the 8 sub-blocks of 32 weights, 16-143 the 256 4-bit quants.       */
/* ------------------------------------------------------------------------ */

/* Scale and min of sub-block j (0..7) from the 12 packed bytes s[0..11]:
 *  j < 4 : the low 6 bits of s[j] (scale) and of s[j+4] (min);
 *  j >= 4: low 4 bits from the low / high nibble of s[j+4], the top 2 bits
 *          from bits 6-7 of s[j-4] (scale) and of s[j] (min). */
static void q4k_scale_min(const uint8_t *s, int j, int *sc, int *mn)
{
    if (j < 4) {
        *sc = s[j] & 63;
        *mn = s[j + 4] & 63;
    } else {
        *sc = (s[j + 4] & 0x0F) | ((s[j - 4] >> 6) << 4);
        *mn = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
    }
}

/* 4-bit quant of weight i (0..255): 64-weight group g = i/64 uses bytes
 * qs[32g .. 32g+31]; its first 32 weights are the low nibbles, the next 32
 * the high nibbles. */
static int q4k_quant(const uint8_t *qs, int i)
{
    const uint8_t byte = qs[32 * (i / 64) + (i % 32)];
    return (i % 64) < 32 ? (byte & 0x0F) : (byte >> 4);
}

static void dequant_q4k_block(const uint8_t *blk, float *out)
{
    const float d = oracle_half_to_float(rd16(blk));
    const float dmin = oracle_half_to_float(rd16(blk + 2));
    const uint8_t *s = blk + 4;
    const uint8_t *qs = blk + 16;
    for (int i = 0; i < ORACLE_QK; ++i) {
        int sc, mn;
        q4k_scale_min(s, i / 32, &sc, &mn);
        const float dsc = d * (float)sc;
        const float dmn = dmin * (float)mn;
        const float t = dsc * (float)q4k_quant(qs, i);
        out[i] = t - dmn;
    }
}

/* ------------------------------------------------------------------------ */
/* Q6_K: bytes 0-127 ql (low 4 bits), 128-191 qh (high 2 bits), 192-207 the  */
/* 16 int8 scales (one per 16 weights), 208-209 d (fp16).                     */
/* ------------------------------------------------------------------------ */

/* 6-bit quant of weight i, minus 32.  i = 128h + 32g + l (h 0..1, g 0..3,
 * l 0..31): low 4 bits are the low nibble (g < 2) or high nibble (g >= 2) of
 * ql[64h + 32(g & 1) + l]; the high 2 bits are bits 2g..2g+1 of qh[32h + l]. */
static int q6k_quant(const uint8_t *ql, const uint8_t *qh, int i)
{
    const int h = i / 128, g = (i % 128) / 32, l = i % 32;
    const uint8_t lb = ql[64 * h + 32 * (g & 1) + l];
    const int lo = g < 2 ? (lb & 0x0F) : (lb >> 4);
    const int hi = (qh[32 * h + l] >> (2 * g)) & 3;
    return (lo | (hi << 4)) - 32;
}

static void dequant_q6k_block(const uint8_t *blk, float *out)
{
    const uint8_t *ql = blk;
    const uint8_t *qh = blk + 128;
    const int8_t *sc = (const int8_t *)(blk + 192);
    const float d = oracle_half_to_float(rd16(blk + 208));
    for (int i = 0; i < ORACLE_QK; ++i) {
        const float dsc = d * (float)sc[i / 16];
        out[i] = dsc * (float)q6k_quant(ql, qh, i);
    }
}

/* qtype: 0 = Q4_K, 1 = Q6_K.  Returns bytes per block, or 0 if unknown. */
static int64_t block_bytes(int qtype)
{
    return qtype == 0 ? ORACLE_Q4K_BYTES : qtype == 1 ? ORACLE_Q6K_BYTES : 0;
}

static void dequant_block(int qtype, const uint8_t *blk, float *out)
{
    if (qtype == 0)
        dequant_q4k_block(blk, out);
    else
        dequant_q6k_block(blk, out);
}

/* Dequantize n_blocks consecutive blocks into n_blocks*256 fp32 values. */
int oracle_dequant(int qtype, const uint8_t *blocks, int64_t n_blocks, float *out)
{
    const int64_t bb = block_bytes(qtype);
    if (!bb || n_blocks < 0)
        return -1;
#pragma omp parallel for schedule(static)
    for (int64_t b = 0; b < n_blocks; ++b)
        dequant_block(qtype, blocks + b * bb, out + b * ORACLE_QK);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Matmul: W holds N rows of K/256 blocks (row n = output feature n), x is    */
/* [M][K] fp16 row-major.  The oracle evaluates only the requested rows:      */
/* y[m][r] = sum_k x[m][k] * w[rows[r]][k] in fp64, y being [M][n_rows].      */
/* ------------------------------------------------------------------------ */
static double *widen_x(const uint16_t *x, int64_t M, int64_t K)
{
    double *xd = (double *)malloc((size_t)(M * K) * sizeof(double));
    if (!xd)
        return NULL;
    for (int64_t i = 0; i < M * K; ++i)
        xd[i] = (double)oracle_half_to_float(x[i]);
    return xd;
}

static void dequant_row(int qtype, const uint8_t *W, int64_t n, int64_t K, float *w)
{
    const int64_t bb = block_bytes(qtype);
    const int64_t nb = K / ORACLE_QK;
    for (int64_t b = 0; b < nb; ++b)
        dequant_block(qtype, W + (n * nb + b) * bb, w + b * ORACLE_QK);
}

/* The matmul over activations already widened to fp64 (xd is [M][K]). */
static int matmul_core(int qtype, const uint8_t *W, const double *xd, int64_t M, int64_t K,
                       const int64_t *rows, int64_t n_rows, double *y)
{
    int failed = 0;
#pragma omp parallel
    {
        float *w = (float *)malloc((size_t)K * sizeof(float));
        if (!w) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 4)
        for (int64_t r = 0; r < n_rows; ++r) {
            if (!w)
                continue;
            dequant_row(qtype, W, rows[r], K, w);
            for (int64_t m = 0; m < M; ++m) {
                const double *xm = xd + m * K;
                double acc = 0.0;
                for (int64_t k = 0; k < K; ++k)
                    acc += xm[k] * (double)w[k];
                y[m * n_rows + r] = acc;
            }
        }
        free(w);
    }
    return failed ? -2 : 0;
}

int oracle_matmul_rows(int qtype, const uint8_t *W, const uint16_t *x, int64_t M, int64_t K,
                       const int64_t *rows, int64_t n_rows, double *y)
{
    if (!block_bytes(qtype) || M < 0 || K <= 0 || K % ORACLE_QK || n_rows < 0)
        return -1;
    double *xd = widen_x(x, M, K);
    if (!xd)
        return -2;
    const int rc = matmul_core(qtype, W, xd, M, K, rows, n_rows, y);
    free(xd);
    return rc;
}

/* SwiGLU over two Q4_K weight sets with the same x:
 * out[m][r] = silu(g) * u, g = x[m] . wg[rows[r]], u = x[m] . wu[rows[r]],
 * silu(g) = g / (1 + exp(-g)), all in fp64.  Optionally also returns g and u. */
static int gateup_core(const uint8_t *Wg, const uint8_t *Wu, const double *xd, int64_t M, int64_t K,
                       const int64_t *rows, int64_t n_rows, double *out, double *g_out, double *u_out)
{
    int failed = 0;
#pragma omp parallel
    {
        float *wg = (float *)malloc((size_t)K * sizeof(float));
        float *wu = (float *)malloc((size_t)K * sizeof(float));
        if (!wg || !wu) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 4)
        for (int64_t r = 0; r < n_rows; ++r) {
            if (!wg || !wu)
                continue;
            dequant_row(0, Wg, rows[r], K, wg);
            dequant_row(0, Wu, rows[r], K, wu);
            for (int64_t m = 0; m < M; ++m) {
                const double *xm = xd + m * K;
                double g = 0.0, u = 0.0;
                for (int64_t k = 0; k < K; ++k) {
                    g += xm[k] * (double)wg[k];
                    u += xm[k] * (double)wu[k];
                }
                const double silu = g / (1.0 + exp(-g));
                out[m * n_rows + r] = silu * u;
                if (g_out)
                    g_out[m * n_rows + r] = g;
                if (u_out)
                    u_out[m * n_rows + r] = u;
            }
        }
        free(wg);
        free(wu);
    }
    return failed ? -2 : 0;
}

int oracle_gateup_swiglu_rows(const uint8_t *Wg, const uint8_t *Wu, const uint16_t *x, int64_t M,
                              int64_t K, const int64_t *rows, int64_t n_rows, double *out,
                              double *g_out, double *u_out)
{
    if (M < 0 || K <= 0 || K % ORACLE_QK || n_rows < 0)
        return -1;
    double *xd = widen_x(x, M, K);
    if (!xd)
        return -2;
    const int rc = gateup_core(Wg, Wu, xd, M, K, rows, n_rows, out, g_out, u_out);
    free(xd);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* RMSNorm in front of a linear (DAMASCUS project overview, "[04] one decode  */
/* step": an RMSNorm comes before the QKV projections and before the SwiGLU  */
/* FFN; "Building DAMASCUS", "Read the model, then reproduce its             */
/* operations").  The pages give no formula or epsilon; the reading taken is */
/* the standard RMSNorm of the Llama family:                                  */
/*   xhat[m][k] = x[m][k] / sqrt(mean_k(x[m][k]^2) + eps) * gamma[k],         */
/* all in fp64, with x and gamma fp16 widened exactly.                        */
/* ------------------------------------------------------------------------ */
int oracle_rmsnorm(const uint16_t *x, const uint16_t *gamma, int64_t M, int64_t K, double eps, double *out)
{
    if (M < 0 || K <= 0 || !(eps >= 0.0))
        return -1;
    for (int64_t m = 0; m < M; ++m) {
        const uint16_t *xm = x + m * K;
        double ss = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            const double v = (double)oracle_half_to_float(xm[k]);
            ss += v * v;
        }
        const double inv = 1.0 / sqrt(ss / (double)K + eps);
        for (int64_t k = 0; k < K; ++k)
            out[m * K + k] = (double)oracle_half_to_float(xm[k]) * inv * (double)oracle_half_to_float(gamma[k]);
    }
    return 0;
}

/* y[m][r] = sum_k xhat[m][k] * w[rows[r]][k] with xhat = RMSNorm(x) * gamma. */
int oracle_rmsnorm_matmul_rows(int qtype, const uint8_t *W, const uint16_t *x, const uint16_t *gamma,
                               double eps, int64_t M, int64_t K, const int64_t *rows, int64_t n_rows,
                               double *y)
{
    if (!block_bytes(qtype) || M < 0 || K <= 0 || K % ORACLE_QK || n_rows < 0)
        return -1;
    double *xn = (double *)malloc((size_t)(M * K) * sizeof(double) + 1);
    if (!xn)
        return -2;
    int rc = oracle_rmsnorm(x, gamma, M, K, eps, xn);
    if (rc == 0)
        rc = matmul_core(qtype, W, xn, M, K, rows, n_rows, y);
    free(xn);
    return rc;
}

/* The fused gate/up + SwiGLU of RMSNorm(x) * gamma. */
int oracle_rmsnorm_gateup_swiglu_rows(const uint8_t *Wg, const uint8_t *Wu, const uint16_t *x,
                                      const uint16_t *gamma, double eps, int64_t M, int64_t K,
                                      const int64_t *rows, int64_t n_rows, double *out)
{
    if (M < 0 || K <= 0 || K % ORACLE_QK || n_rows < 0)
        return -1;
    double *xn = (double *)malloc((size_t)(M * K) * sizeof(double) + 1);
    if (!xn)
        return -2;
    int rc = oracle_rmsnorm(x, gamma, M, K, eps, xn);
    if (rc == 0)
        rc = gateup_core(Wg, Wu, xn, M, K, rows, n_rows, out, NULL, NULL);
    free(xn);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* Q8 activations.  The pages do not describe an integer-activation variant;  */
/* this is the reading this project takes (per-32 int8 quantization of x, as  */
/* the GGUF 8-bit activation formats do):                                     */
/*   for each token, each block of 32 consecutive k:                          */
/*     amax = max |x| (fp32; x widened exactly from fp16),                    */
/*     d    = amax / 127            (one fp32 division),                      */
/*     q    = round(x / d)          (fp32 division, ties away from zero),     */
/*            clamped to [-127, 127];  d = 0 (and q = 0) when amax = 0;       */
/*   x~ = d * q, and the matmul is the one above over x~ (fp64 sums).         */
/* Finite x only.                                                             */
/* ------------------------------------------------------------------------ */
int oracle_quantize_q8(const uint16_t *x, int64_t M, int64_t K, int8_t *q, float *d)
{
    if (M < 0 || K <= 0 || K % 32)
        return -1;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t b = 0; b < K / 32; ++b) {
            const uint16_t *xb = x + m * K + 32 * b;
            float amax = 0.0f;
            for (int i = 0; i < 32; ++i) {
                const float v = fabsf(oracle_half_to_float(xb[i]));
                if (v > amax)
                    amax = v;
            }
            volatile float db = amax / 127.0f;
            d[m * (K / 32) + b] = db;
            for (int i = 0; i < 32; ++i) {
                int qi = 0;
                if (db != 0.0f) {
                    volatile float r = oracle_half_to_float(xb[i]) / db;
                    const float t = roundf(r);
                    qi = t > 127.0f ? 127 : t < -127.0f ? -127 : (int)t;
                }
                q[m * K + 32 * b + i] = (int8_t)qi;
            }
        }
    return 0;
}

/* d * q in fp64 (exact) for every element, or NULL. */
static double *q8_values(const uint16_t *x, int64_t M, int64_t K)
{
    int8_t *q = (int8_t *)malloc((size_t)(M * K) + 1);
    float *d = (float *)malloc((size_t)(M * (K / 32)) * sizeof(float) + 1);
    double *xq = (double *)malloc((size_t)(M * K) * sizeof(double) + 1);
    int ok = q && d && xq && oracle_quantize_q8(x, M, K, q, d) == 0;
    for (int64_t i = 0; ok && i < M * K; ++i)
        xq[i] = (double)d[(i / K) * (K / 32) + (i % K) / 32] * (double)q[i];
    free(q);
    free(d);
    if (!ok) {
        free(xq);
        return NULL;
    }
    return xq;
}

int oracle_q8_matmul_rows(int qtype, const uint8_t *W, const uint16_t *x, int64_t M, int64_t K,
                          const int64_t *rows, int64_t n_rows, double *y)
{
    if (!block_bytes(qtype) || M < 0 || K <= 0 || K % ORACLE_QK || n_rows < 0)
        return -1;
    double *xq = q8_values(x, M, K);
    if (!xq)
        return -2;
    const int rc = matmul_core(qtype, W, xq, M, K, rows, n_rows, y);
    free(xq);
    return rc;
}

int oracle_q8_gateup_swiglu_rows(const uint8_t *Wg, const uint8_t *Wu, const uint16_t *x, int64_t M, int64_t K,
                                 const int64_t *rows, int64_t n_rows, double *out)
{
    if (M < 0 || K <= 0 || K % ORACLE_QK || n_rows < 0)
        return -1;
    double *xq = q8_values(x, M, K);
    if (!xq)
        return -2;
    const int rc = gateup_core(Wg, Wu, xq, M, K, rows, n_rows, out, NULL, NULL);
    free(xq);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* GQA attention over a KV cache.                                             */
/* q: [M][H][D] fp16; query i sits at position pos0 + i and sees positions    */
/* 0 .. pos0 + i.  kc, vc: the caches, [H_kv][L_max][D] fp16 (head-major).    */
/* For each selected query i (qrows, or all M if NULL) and head h, with       */
/* g = h / (H / H_kv):                                                        */
/*   s_j = scale * sum_d q[i][h][d] * k[g][j][d]                              */
/*   p_j = exp(s_j - max s) / sum_j' exp(s_j' - max s)                        */
/*   out[r][h][d] = sum_j p_j * v[g][j][d]                                    */
/* every sum in fp64 in index order.                                          */
/* ------------------------------------------------------------------------ */
int oracle_gqa_attention(const uint16_t *q, const uint16_t *kc, const uint16_t *vc, int64_t M, int64_t H,
                         int64_t Hkv, int64_t D, int64_t pos0, int64_t Lmax, double scale, const int64_t *qrows,
                         int64_t n_qrows, double *out)
{
    if (M < 0 || H <= 0 || Hkv <= 0 || H % Hkv || D <= 0 || pos0 < 0 || pos0 + M > Lmax || n_qrows < 0)
        return -1;
    for (int64_t r = 0; qrows && r < n_qrows; ++r)
        if (qrows[r] < 0 || qrows[r] >= M)
            return -1;
    const int64_t group = H / Hkv;
    const int64_t nq = qrows ? n_qrows : M;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t rh = 0; rh < nq * H; ++rh) {
        const int64_t r = rh / H, h = rh % H;
        const int64_t i = qrows ? qrows[r] : r;
        const int64_t g = h / group;
        const int64_t n = pos0 + i + 1;
        const uint16_t *qv = q + (i * H + h) * D;
        double *s = (double *)malloc((size_t)n * sizeof(double));
        if (!s) {
            bad = 1;
            continue;
        }
        double smax = -INFINITY;
        for (int64_t j = 0; j < n; ++j) {
            const uint16_t *kj = kc + (g * Lmax + j) * D;
            double dot = 0.0;
            for (int64_t d = 0; d < D; ++d)
                dot += (double)oracle_half_to_float(qv[d]) * (double)oracle_half_to_float(kj[d]);
            s[j] = scale * dot;
            if (s[j] > smax)
                smax = s[j];
        }
        double denom = 0.0;
        for (int64_t j = 0; j < n; ++j) {
            s[j] = exp(s[j] - smax);
            denom += s[j];
        }
        double *o = out + (r * H + h) * D;
        for (int64_t d = 0; d < D; ++d)
            o[d] = 0.0;
        for (int64_t j = 0; j < n; ++j) {
            const uint16_t *vj = vc + (g * Lmax + j) * D;
            const double p = s[j] / denom;
            for (int64_t d = 0; d < D; ++d)
                o[d] += p * (double)oracle_half_to_float(vj[d]);
        }
        free(s);
    }
    return bad ? -2 : 0;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}
