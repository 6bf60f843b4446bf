/*
 * qz_oracle.c -- the CPU oracle for the quantizers and quantized GEMMs.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the bench's
 * CPU-baseline leg may load this code. The product path (the CUDA library)
 * shares nothing with it: no header, helper, table or constant.
 *
 * Plain, slow, single-threaded C. Every encoder is written as the definition
 * the pages give (nearest representable value; the fake-quant steps in the
 * pages' order) rather than as a fast bit trick. Build with
 * -ffp-contract=off so that every float operation rounds once (IEEE RNE),
 * as the torch CPU float32 ops of the pages do.
 *
 * Sources (page title, section):
 *  [P1] "量化部署实战" (anrans.github.io ai-infra-handbooks), section 伪量化实现:
 *       the fake-quant functions fp8, fp8_per_tensor, fp8_per_row,
 *       fp8_blockwise, fp4, mxfp4, nvfp4 and the FP8 KV cache class; section
 *       格式速查 (format table); 练习 2 (block-scaled FP8 GEMM accumulation).
 *  [P2] "量化：让每一步搬更少的字节" (niuwancheng.cn), section 量化在做什么
 *       (q = round(x / s), x^ = q * s; 4-bit + 2-byte scale per 128) and
 *       新一代低位格式 (E4M3 / E2M1 / MXFP4 / NVFP4 bit budgets).
 *  [P3] "LLM 推理优化 · 量化学习笔记" (zzszmyf.github.io), section 5.1
 *       (symmetric quantization q = clamp(round(x / s), qmin, qmax)).
 *
 * Readings where the pages are silent or ambiguous (each also listed in the
 * design notes):
 *  - bf16 inputs are widened exactly to fp32 before any formula (the pages run
 *    the formulas on fp32 tensors).
 *  - The clamp constant 1e-12 becomes the fp32 value nearest 1e-12, as a
 *    Python scalar does when torch applies it to an fp32 tensor.
 *  - E4M3 conversion saturates to +-448 (values beyond 448 only arise in the
 *    NVFP4 block scale, where they are a few ulp above 448 and round to 448).
 *  - E2M1 rounding: the first index of the minimum distance, so a value
 *    exactly between two grid points goes to the smaller magnitude; the sign
 *    bit is (y < 0), so -0.0 encodes as +0 and a small negative value that
 *    rounds to zero encodes as -0 (code 0x8), as V[idx] * sign(y) does.
 *  - MXFP4 exponent: floor(log2(amax)) taken exactly from the fp32 exponent
 *    field (torch's float log2 rounds up just below a power of two).
 *  - INT4 g128 (the INT4 fake-quant function itself is not on the pages):
 *    symmetric, s = bf16(max(amax, 1e-12) / 7), q = clamp(rint(x / s), -8, 7),
 *    rint = round half to even (torch.round). Divisor 7 = 2^(b-1) - 1, the
 *    INT8 "amax / 127" rule of [P2] carried to 4 bits.
 *  - GEMMs: y = sum over k of the exactly dequantized operands, in double.
 *
 * The variants of the "next" rows, with their readings:
 *  - FP8 KV per head [P1 KV Cache 量化, per_head]: one scale per (batch, head)
 *    over that head's T x D values, otherwise the per-tensor FP8 steps.
 *  - K per channel with a zero point [P1 KV Cache 量化: K as "a constant bias
 *    per channel plus a small variation"; per channel, with a zero point that
 *    absorbs the bias; P3 5.1: asymmetric quantization adds a zero point z].
 *    The cache stays FP8, so the zero point lives in value space: per channel
 *    (b, h, d) over the T tokens, z = fl(0.5 * fl(max + min)) (the midpoint of
 *    the channel's range, so the residual is symmetric), r = fl(x - z),
 *    s = max(max|r|, 1e-12) / 448, code = E4M3(clamp(fl(r / s), +-448)),
 *    dequant = fl(fl(v * s) + z). V is quantized per token (one scale per
 *    (b, h, t) over D), the partner of per-channel K in the KIVI split the
 *    pages cite.
 *  - INT4 with a zero point [P1 格式速查 W4A16 row "+ 零点"; P3 5.1
 *    q = clamp(round(x / s) + z, ...)]: unsigned codes 0..15 per group of 128
 *    along K; the range is widened to include 0 (lo = min(min, 0),
 *    hi = max(max, 0)), s = bf16(max(hi - lo, 1e-12) / 15),
 *    z = clamp(rint(-lo / s), 0, 15), q = clamp(rint(x / s) + z, 0, 15),
 *    dequant = (q - z) * s.
 *  - Weight-only FP4 (W4A16 MXFP4 / NVFP4) [P1 精度比较]: bf16 activations
 *    times weights dequantized exactly from their E2M1 codes and scales.
 *  - SmoothQuant [P2 路线二]: s_j = max|X_j|^a / max|W_j|^(1-a) with a = 0.5,
 *    each amax floored at 1e-12 like every other amax here, computed as
 *    fl(fl(sqrt(ax)) / fl(sqrt(aw))). X' = X / s (per input channel),
 *    W' = W * s.
 *  - INT8 per token / per output channel [P1 格式速查 W8A8 INT8 row, integers
 *    -128..127; P2 量化在做什么: symmetric s = amax / 127]:
 *    s = max(amax_row, 1e-12) / 127, q = clamp(rint(x / s), -128, 127).
 *  - INT8 GEMM: y = sA[i] * sB[j] * sum_k qA[i,k] qB[j,k]; the integer sum is
 *    exact (int64).
 *  - Fused FP8 1x128 output quantization [P1 练习 2: the activation's (1, 128)
 *    scales are computed at the end of the previous kernel]: the producer's
 *    output rounded to bf16 (what the producer would have stored), then the
 *    1x128 FP8 steps of or_quant_fp8; the tests compose the two.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#include <stdlib.h>

#define OR_FP8_MAX 448.0f
#define OR_FP4_MAX 6.0f

/* The clamp floor of the fake-quant functions: 1e-12 as an fp32 value. */
static float or_amax_min(void) { return (float)1e-12; }

/* The eight non-negative E2M1 values, in code order [P1 FP4_VALUES, 格式速查]. */
static const double OR_FP4_VALUES[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

/* ------------------------------------------------------------------ E4M3 */

/* Value of an FP8 E4M3 ("fn": no infinities, one NaN pattern per sign) code:
 * 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits [P1 格式速查; P3 4.2].
 * Codes 0x7F and 0xFF are NaN. */
double or_e4m3_decode(uint8_t c)
{
    int s = (c >> 7) & 1, e = (c >> 3) & 0xF, m = c & 7;
    double v;
    if (e == 0xF && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m / 8.0, -6);          /* subnormal */
    else v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

/* Nearest finite E4M3 value to y, ties to the even code (round to nearest
 * even), magnitudes beyond 448 saturated to 448. The sign bit copies the sign
 * of y (so -0.0 and tiny negatives give 0x80, like torch's cast).
 * Written as the definition: scan every non-negative finite code. */
uint8_t or_e4m3_encode(float y)
{
    double a = fabs((double)y);
    int best = 0;
    double bestd = INFINITY;
    for (int c = 0; c <= 0x7E; c++) {
        double d = fabs(a - or_e4m3_decode((uint8_t)c));
        if (d < bestd || (d == bestd && (c & 1) == 0 && (best & 1) == 1)) {
            bestd = d;
            best = c;
        }
    }
    if (signbit(y)) best |= 0x80;
    return (uint8_t)best;
}

/* ------------------------------------------------------------------ E2M1 */

/* Value of an FP4 E2M1 code: bit 3 = sign, bits 0..2 index FP4_VALUES. */
double or_e2m1_decode(uint8_t c)
{
    double v = OR_FP4_VALUES[c & 7];
    return (c & 8) ? -v : v;
}

/* [P1 fp4]: argmin over |(|y|) - V[i]|, the first index winning a tie, then
 * the sign of y. Distances in double are exact. */
uint8_t or_e2m1_encode(float y)
{
    double a = fabs((double)y);
    int best = 0;
    double bestd = fabs(a - OR_FP4_VALUES[0]);
    for (int i = 1; i < 8; i++) {
        double d = fabs(a - OR_FP4_VALUES[i]);
        if (d < bestd) { bestd = d; best = i; }
    }
    if (y < 0.0f) best |= 8;
    return (uint8_t)best;
}

/* ------------------------------------------------------------------ bf16 */

float or_bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* Nearest bf16 to a finite fp32 value, ties to the even bf16 pattern. */
uint16_t or_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    uint16_t lo = (uint16_t)(u >> 16);           /* truncation toward zero */
    uint16_t hi = (uint16_t)(lo + 1);            /* next bf16 away from zero */
    double dlo = fabs((double)f - (double)or_bf16_to_f32(lo));
    double dhi = fabs((double)f - (double)or_bf16_to_f32(hi));
    if (dlo < dhi) return lo;
    if (dhi < dlo) return hi;
    return (lo & 1) ? hi : lo;
}

/* --------------------------------------------------------------- helpers */

static float or_elem(const void* x, int is_bf16, int64_t i)
{
    if (is_bf16) return or_bf16_to_f32(((const uint16_t*)x)[i]);
    return ((const float*)x)[i];
}

static float or_clampf(float v, float lo, float hi)
{
    /* torch.clamp(min=lo, max=hi) = min(max(v, lo), hi) */
    if (v < lo) v = lo;
    if (v > hi) v = hi;
    return v;
}

/* [P1 fp8]: y = x / scale, clamp to +-448, cast to E4M3; dequant = v * scale.
 * Returns the code; writes the dequantized fp32 value to *deq. */
static uint8_t or_fp8_one(float x, float scale, float* deq)
{
    float y = x / scale;
    y = or_clampf(y, -OR_FP8_MAX, OR_FP8_MAX);
    uint8_t c = or_e4m3_encode(y);
    *deq = (float)or_e4m3_decode(c) * scale;
    return c;
}

/* [P1 fp4]: y = x / scale, clamp to +-6, nearest E2M1 (ties down), dequant
 * = FP4_VALUES[idx] * sign(y) * scale. */
static uint8_t or_fp4_one(float x, float scale, float* deq)
{
    float y = x / scale;
    y = or_clampf(y, -OR_FP4_MAX, OR_FP4_MAX);
    uint8_t c = or_e2m1_encode(y);
    *deq = (float)or_e2m1_decode(c) * scale;
    return c;
}

/* ------------------------------------------------------------ FP8 paths */

enum { OR_TENSOR = 0, OR_ROW = 1, OR_BLOCK128 = 2, OR_GROUP128 = 3 };

/* FP8 E4M3 fake-quant of a row-major [rows, cols] tensor (leading dim ldx),
 * [P1 fp8_per_tensor / fp8_per_row / fp8_blockwise].
 *   gran 0 per tensor:  one scale;            scales[1]
 *   gran 1 per row:     one scale per row;    scales[rows]
 *   gran 2 128x128:     block (br, 128), br = min(128, rows); scales[rows/br][cols/128]
 *   gran 3 1x128:       scales[rows][cols/128]
 * scale = max(amax, 1e-12) / 448. codes[rows*cols], deq[rows*cols] (nullable).
 * Returns 0, or -1 for a shape the page's reshape would reject. */
int or_quant_fp8(const void* x, int is_bf16, int64_t rows, int64_t cols, int64_t ldx,
                 int gran, uint8_t* codes, float* scales, float* deq)
{
    int64_t ur, uc;                     /* unit extent in rows, cols */
    if (rows <= 0 || cols <= 0) return -1;
    switch (gran) {
    case OR_TENSOR: ur = rows; uc = cols; break;
    case OR_ROW: ur = 1; uc = cols; break;
    case OR_BLOCK128: ur = rows < 128 ? rows : 128; uc = 128; break;
    case OR_GROUP128: ur = 1; uc = 128; break;
    default: return -1;
    }
    if (rows % ur || cols % uc) return -1;
    int64_t nbr = rows / ur, nbc = cols / uc;
    for (int64_t br = 0; br < nbr; br++) {
        for (int64_t bc = 0; bc < nbc; bc++) {
            float amax = 0.0f;
            for (int64_t r = br * ur; r < (br + 1) * ur; r++)
                for (int64_t c = bc * uc; c < (bc + 1) * uc; c++) {
                    float a = fabsf(or_elem(x, is_bf16, r * ldx + c));
                    if (a > amax) amax = a;
                }
            float scale = (amax > or_amax_min() ? amax : or_amax_min()) / OR_FP8_MAX;
            scales[br * nbc + bc] = scale;
            for (int64_t r = br * ur; r < (br + 1) * ur; r++)
                for (int64_t c = bc * uc; c < (bc + 1) * uc; c++) {
                    float d;
                    codes[r * cols + c] = or_fp8_one(or_elem(x, is_bf16, r * ldx + c), scale, &d);
                    if (deq) deq[r * cols + c] = d;
                }
        }
    }
    return 0;
}

/* Per-tensor FP8 with a caller-given scale (the calibrated-scale KV mode of
 * [P1 KV Cache 量化, 实际部署时]): codes and dequant only. */
void or_quant_fp8_given(const void* x, int is_bf16, int64_t n, float scale,
                        uint8_t* codes, float* deq)
{
    for (int64_t i = 0; i < n; i++) {
        float d;
        codes[i] = or_fp8_one(or_elem(x, is_bf16, i), scale, &d);
        if (deq) deq[i] = d;
    }
}

/* FP8 KV-cache write [P1 FP8KVCache.update]: fp8_per_tensor(k) and
 * fp8_per_tensor(v), each with its own scale. k, v: bf16 of n elements. */
void or_kv_write_fp8(const uint16_t* k, const uint16_t* v, int64_t n,
                     uint8_t* k_codes, uint8_t* v_codes, float* k_scale, float* v_scale,
                     float* k_deq, float* v_deq)
{
    or_quant_fp8(k, 1, 1, n, n, OR_TENSOR, k_codes, k_scale, k_deq);
    or_quant_fp8(v, 1, 1, n, n, OR_TENSOR, v_codes, v_scale, v_deq);
}

/* ----------------------------------------------------------------- MXFP4 */

/* floor(log2(a)) for a normal positive fp32, from its exponent (exact). */
static int or_floor_log2(float a)
{
    int e;
    frexpf(a, &e);                       /* a = m * 2^e, m in [0.5, 1) */
    return e - 1;
}

/* [P1 mxfp4], block 32 along the last dim: amax = max(|block|, 1e-12),
 * scale = 2^(floor(log2 amax) - 2), then fp4(x, scale). The E8M0 code of the
 * scale is floor(log2 amax) - 2 + 127. codes are packed two per byte, the
 * even element in the low nibble: codes[rows][cols/2]; e8m0[rows][cols/32]. */
int or_quant_mxfp4(const void* x, int is_bf16, int64_t rows, int64_t cols, int64_t ldx,
                   uint8_t* codes, uint8_t* e8m0, float* deq)
{
    if (rows <= 0 || cols <= 0 || cols % 32) return -1;
    for (int64_t r = 0; r < rows; r++) {
        for (int64_t b = 0; b < cols / 32; b++) {
            float amax = 0.0f;
            for (int64_t c = b * 32; c < b * 32 + 32; c++) {
                float a = fabsf(or_elem(x, is_bf16, r * ldx + c));
                if (a > amax) amax = a;
            }
            if (amax < or_amax_min()) amax = or_amax_min();
            int E = or_floor_log2(amax) - 2;
            float scale = ldexpf(1.0f, E);
            e8m0[r * (cols / 32) + b] = (uint8_t)(E + 127);
            for (int64_t c = b * 32; c < b * 32 + 32; c++) {
                float d;
                uint8_t q = or_fp4_one(or_elem(x, is_bf16, r * ldx + c), scale, &d);
                uint8_t* p = &codes[r * (cols / 2) + c / 2];
                if (c % 2 == 0) *p = q; else *p = (uint8_t)(*p | (q << 4));
                if (deq) deq[r * cols + c] = d;
            }
        }
    }
    return 0;
}

/* ----------------------------------------------------------------- NVFP4 */

/* max |x| over the whole tensor. */
float or_amax(const void* x, int is_bf16, int64_t rows, int64_t cols, int64_t ldx)
{
    float amax = 0.0f;
    for (int64_t r = 0; r < rows; r++)
        for (int64_t c = 0; c < cols; c++) {
            float a = fabsf(or_elem(x, is_bf16, r * ldx + c));
            if (a > amax) amax = a;
        }
    return amax;
}

/* [P1 nvfp4], block 16 along the last dim, in the page's order:
 *   g  = max(amax_tensor, 1e-12) / (448 * 6)
 *   b  = E4M3(block_amax / 6 / g)           (stored block scale)
 *   s  = max(b, 1e-12) * g                  (effective scale)
 *   fp4(x, s)
 * amax_tensor is computed unless amax_in is non-null. Outputs:
 * codes[rows][cols/2] (even element low nibble), sb[rows][cols/16] E4M3 bytes,
 * *g_out = g. */
int or_quant_nvfp4(const void* x, int is_bf16, int64_t rows, int64_t cols, int64_t ldx,
                   const float* amax_in, uint8_t* codes, uint8_t* sb, float* g_out, float* deq)
{
    if (rows <= 0 || cols <= 0 || cols % 16) return -1;
    float amax_t = amax_in ? *amax_in : or_amax(x, is_bf16, rows, cols, ldx);
    float g = (amax_t > or_amax_min() ? amax_t : or_amax_min()) / (OR_FP8_MAX * OR_FP4_MAX);
    *g_out = g;
    for (int64_t r = 0; r < rows; r++) {
        for (int64_t b = 0; b < cols / 16; b++) {
            float bamax = 0.0f;
            for (int64_t c = b * 16; c < b * 16 + 16; c++) {
                float a = fabsf(or_elem(x, is_bf16, r * ldx + c));
                if (a > bamax) bamax = a;
            }
            float t = bamax / OR_FP4_MAX / g;
            uint8_t bc = or_e4m3_encode(t);
            sb[r * (cols / 16) + b] = bc;
            float bv = (float)or_e4m3_decode(bc);
            float s = (bv > or_amax_min() ? bv : or_amax_min()) * g;
            for (int64_t c = b * 16; c < b * 16 + 16; c++) {
                float d;
                uint8_t q = or_fp4_one(or_elem(x, is_bf16, r * ldx + c), s, &d);
                uint8_t* p = &codes[r * (cols / 2) + c / 2];
                if (c % 2 == 0) *p = q; else *p = (uint8_t)(*p | (q << 4));
                if (deq) deq[r * cols + c] = d;
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------ INT4 g128 */

/* Uniform symmetric quantization of one value with a given scale
 * [P2 量化在做什么: q = round(x / s); P3 5.1: clamp to [qmin, qmax]].
 * round = rint (half to even, as torch.round). Returns q; *deq = q * s. */
int or_int_quant_one(float x, float s, int qmin, int qmax, float* deq)
{
    float y = x / s;
    float r = rintf(y);
    if (r < (float)qmin) r = (float)qmin;
    if (r > (float)qmax) r = (float)qmax;
    *deq = r * s;
    return (int)r;
}

/* INT4, one bf16 scale per group of 128 along K, of a row-major weight
 * w[K][N] (leading dim ldw) [P1 格式速查 W4A16 row; P2 粒度 table, 每组].
 *   s = bf16(max(amax_group, 1e-12) / 7);  q = clamp(rint(w / s), -8, 7)
 * qweight[K/8][N] int32: element k of a column sits in bits 4*(k%8)..+3,
 * two's complement. scale[K/128][N] bf16 bits. deq[K][N] nullable. */
int or_quant_int4_g128(const void* w, int is_bf16, int64_t K, int64_t N, int64_t ldw,
                       int32_t* qweight, uint16_t* scale, float* deq)
{
    if (K <= 0 || N <= 0 || K % 128) return -1;
    for (int64_t n = 0; n < N; n++) {
        for (int64_t g = 0; g < K / 128; g++) {
            float amax = 0.0f;
            for (int64_t k = g * 128; k < g * 128 + 128; k++) {
                float a = fabsf(or_elem(w, is_bf16, k * ldw + n));
                if (a > amax) amax = a;
            }
            float sf = (amax > or_amax_min() ? amax : or_amax_min()) / 7.0f;
            uint16_t sbits = or_f32_to_bf16(sf);
            scale[g * N + n] = sbits;
            float s = or_bf16_to_f32(sbits);
            for (int64_t k = g * 128; k < g * 128 + 128; k++) {
                float d;
                int q = or_int_quant_one(or_elem(w, is_bf16, k * ldw + n), s, -8, 7, &d);
                uint32_t* p = (uint32_t*)&qweight[(k / 8) * N + n];
                if (k % 8 == 0) *p = 0;
                *p |= ((uint32_t)q & 0xFu) << (4 * (k % 8));
                if (deq) deq[k * N + n] = d;
            }
        }
    }
    return 0;
}

/* --------------------------------------------------------------- GEMMs */

/* Each GEMM reference computes, for the listed output coordinates (i, j),
 *   y[i,j]     = sum_k a[i,k] * b[k,j]        (double)
 *   bound[i,j] = sum_k |a[i,k] * b[k,j]|      (double)
 * on the exactly dequantized operands. Every product of a code value and its
 * scales is exact in double. The acceptance test is
 * |y_gpu - y| <= 1e-3 * bound. */

/* W4A16: a = A[i,k] (bf16), b = q[k,j] * s[k/128, j] (INT4 code, bf16 scale). */
void or_gemm_w4a16(const uint16_t* A, const int32_t* qweight, const uint16_t* scale,
                   int64_t M, int64_t N, int64_t K, const int64_t* ii, const int64_t* jj,
                   int64_t npts, double* y, double* bound)
{
    (void)M;
    for (int64_t p = 0; p < npts; p++) {
        int64_t i = ii[p], j = jj[p];
        double acc = 0.0, mag = 0.0;
        for (int64_t k = 0; k < K; k++) {
            uint32_t word = (uint32_t)qweight[(k / 8) * N + j];
            int q = (int)((word >> (4 * (k % 8))) & 0xF);
            if (q >= 8) q -= 16;
            double b = (double)q * (double)or_bf16_to_f32(scale[(k / 128) * N + j]);
            double a = (double)or_bf16_to_f32(A[i * K + k]);
            acc += a * b;
            mag += fabs(a * b);
        }
        y[p] = acc;
        bound[p] = mag;
    }
}

/* FP8 block GEMM [P1 练习 2]: a = e4m3(qA[i,k]) * sA[i, k/128] (1x128 groups),
 * b = e4m3(qB[j,k]) * sB[j/128, k/128] (128x128 blocks of B^T, [N, K]). */
void or_gemm_fp8_block(const uint8_t* qA, const float* sA, const uint8_t* qB, const float* sB,
                       int64_t M, int64_t N, int64_t K, const int64_t* ii, const int64_t* jj,
                       int64_t npts, double* y, double* bound)
{
    (void)M; (void)N;
    int64_t kb = K / 128;
    for (int64_t p = 0; p < npts; p++) {
        int64_t i = ii[p], j = jj[p];
        double acc = 0.0, mag = 0.0;
        for (int64_t k = 0; k < K; k++) {
            double a = or_e4m3_decode(qA[i * K + k]) * (double)sA[i * kb + k / 128];
            double b = or_e4m3_decode(qB[j * K + k]) * (double)sB[(j / 128) * kb + k / 128];
            acc += a * b;
            mag += fabs(a * b);
        }
        y[p] = acc;
        bound[p] = mag;
    }
}

static double or_fp4_at(const uint8_t* q, int64_t row, int64_t K, int64_t k)
{
    uint8_t byte = q[row * (K / 2) + k / 2];
    return or_e2m1_decode((k % 2 == 0) ? (byte & 0xF) : (byte >> 4));
}

/* NVFP4 GEMM: a = e2m1(qA[i,k]) * e4m3(sA[i, k/16]) * gA, b likewise with
 * B^T [N, K]. */
void or_gemm_nvfp4(const uint8_t* qA, const uint8_t* sA, float gA,
                   const uint8_t* qB, const uint8_t* sB, float gB,
                   int64_t M, int64_t N, int64_t K, const int64_t* ii, const int64_t* jj,
                   int64_t npts, double* y, double* bound)
{
    (void)M; (void)N;
    for (int64_t p = 0; p < npts; p++) {
        int64_t i = ii[p], j = jj[p];
        double acc = 0.0, mag = 0.0;
        for (int64_t k = 0; k < K; k++) {
            double a = or_fp4_at(qA, i, K, k) * or_e4m3_decode(sA[i * (K / 16) + k / 16]) * (double)gA;
            double b = or_fp4_at(qB, j, K, k) * or_e4m3_decode(sB[j * (K / 16) + k / 16]) * (double)gB;
            acc += a * b;
            mag += fabs(a * b);
        }
        y[p] = acc;
        bound[p] = mag;
    }
}

/* MXFP4 GEMM: a = e2m1(qA[i,k]) * 2^(eA[i, k/32] - 127), b likewise. */
void or_gemm_mxfp4(const uint8_t* qA, const uint8_t* eA, const uint8_t* qB, const uint8_t* eB,
                   int64_t M, int64_t N, int64_t K, const int64_t* ii, const int64_t* jj,
                   int64_t npts, double* y, double* bound)
{
    (void)M; (void)N;
    for (int64_t p = 0; p < npts; p++) {
        int64_t i = ii[p], j = jj[p];
        double acc = 0.0, mag = 0.0;
        for (int64_t k = 0; k < K; k++) {
            double a = ldexp(or_fp4_at(qA, i, K, k), (int)eA[i * (K / 32) + k / 32] - 127);
            double b = ldexp(or_fp4_at(qB, j, K, k), (int)eB[j * (K / 32) + k / 32] - 127);
            acc += a * b;
            mag += fabs(a * b);
        }
        y[p] = acc;
        bound[p] = mag;
    }
}

/* ----------------------------------------------------- FP8 KV variants */

/* FP8 KV write with one scale per (batch, head) [P1 KV Cache 量化, per_head:
 * amax over the last two dims (T, D)]. k, v: bf16 [B*H][T*D]. Scales
 * [B*H] each. Each head's slice is quantized by the per-tensor FP8 steps. */
void or_kv_write_fp8_per_head(const uint16_t* k, const uint16_t* v, int64_t BH, int64_t TD,
                              uint8_t* k_codes, uint8_t* v_codes, float* k_scale, float* v_scale,
                              float* k_deq, float* v_deq)
{
    for (int64_t h = 0; h < BH; h++) {
        or_quant_fp8(k + h * TD, 1, 1, TD, TD, OR_TENSOR, k_codes + h * TD, k_scale + h,
                     k_deq ? k_deq + h * TD : NULL);
        or_quant_fp8(v + h * TD, 1, 1, TD, TD, OR_TENSOR, v_codes + h * TD, v_scale + h,
                     v_deq ? v_deq + h * TD : NULL);
    }
}

/* Per-head FP8 with caller-given scales (calibrated, [P1 KV Cache 量化,
 * 实际部署时]): x bf16 [BH][TD], scale[BH]. */
void or_kv_fp8_per_head_given(const uint16_t* x, int64_t BH, int64_t TD, const float* scale,
                              uint8_t* codes, float* deq)
{
    for (int64_t h = 0; h < BH; h++)
        or_quant_fp8_given(x + h * TD, 1, TD, scale[h], codes + h * TD, deq ? deq + h * TD : NULL);
}

/* K per channel with a zero point (FP8 residual), over the T tokens of each
 * channel (b, h, d) of k bf16 [BH][T][D]:
 *   z = fl(0.5 * fl(max + min));  r = fl(x - z)
 *   s = max(max_t |r|, 1e-12) / 448;  code = E4M3(clamp(fl(r / s), +-448))
 *   dequant = fl(fl(E4M3value(code) * s) + z)
 * scale, zero: [BH][D]. */
void or_kv_k_channel_zp(const uint16_t* k, int64_t BH, int64_t T, int64_t D,
                        uint8_t* codes, float* scale, float* zero, float* deq)
{
    for (int64_t h = 0; h < BH; h++) {
        const uint16_t* x = k + h * T * D;
        for (int64_t d = 0; d < D; d++) {
            float mn = or_bf16_to_f32(x[d]), mx = mn;
            for (int64_t t = 1; t < T; t++) {
                float a = or_bf16_to_f32(x[t * D + d]);
                if (a < mn) mn = a;
                if (a > mx) mx = a;
            }
            float z = 0.5f * (mx + mn);
            float ramax = 0.0f;
            for (int64_t t = 0; t < T; t++) {
                float r = fabsf(or_bf16_to_f32(x[t * D + d]) - z);
                if (r > ramax) ramax = r;
            }
            float s = (ramax > or_amax_min() ? ramax : or_amax_min()) / OR_FP8_MAX;
            scale[h * D + d] = s;
            zero[h * D + d] = z;
            for (int64_t t = 0; t < T; t++) {
                float r = or_bf16_to_f32(x[t * D + d]) - z;
                float dq;
                codes[h * T * D + t * D + d] = or_fp8_one(r, s, &dq);
                if (deq) deq[h * T * D + t * D + d] = dq + z;
            }
        }
    }
}

/* ------------------------------------------------- INT4 with a zero point */

/* INT4, unsigned codes 0..15, one bf16 scale and one integer zero point per
 * group of 128 along K, of a row-major weight w[K][N] [P1 格式速查 W4A16
 * "+ 零点"; P3 5.1 asymmetric]:
 *   lo = min(min_group, 0), hi = max(max_group, 0)
 *   s = bf16(max(hi - lo, 1e-12) / 15);  z = clamp(rint(-lo / s), 0, 15)
 *   q = clamp(rint(w / s) + z, 0, 15);    dequant = (q - z) * s
 * qweight[K/8][N] int32: element k in bits 4*(k%8)..+3 (unsigned).
 * scale[K/128][N] bf16 bits; zero[K/128][N] bytes. */
int or_quant_int4_g128_zp(const void* w, int is_bf16, int64_t K, int64_t N, int64_t ldw,
                          int32_t* qweight, uint16_t* scale, uint8_t* zero, float* deq)
{
    if (K <= 0 || N <= 0 || K % 128) return -1;
    for (int64_t n = 0; n < N; n++) {
        for (int64_t g = 0; g < K / 128; g++) {
            float lo = 0.0f, hi = 0.0f;
            for (int64_t k = g * 128; k < g * 128 + 128; k++) {
                float a = or_elem(w, is_bf16, k * ldw + n);
                if (a < lo) lo = a;
                if (a > hi) hi = a;
            }
            float range = hi - lo;
            float sf = (range > or_amax_min() ? range : or_amax_min()) / 15.0f;
            uint16_t sbits = or_f32_to_bf16(sf);
            float sq = or_bf16_to_f32(sbits);
            float zr = rintf(-lo / sq);
            if (zr < 0.0f) zr = 0.0f;
            if (zr > 15.0f) zr = 15.0f;
            int z = (int)zr;
            scale[g * N + n] = sbits;
            zero[g * N + n] = (uint8_t)z;
            for (int64_t k = g * 128; k < g * 128 + 128; k++) {
                float y = or_elem(w, is_bf16, k * ldw + n) / sq;
                float r = rintf(y) + (float)z;
                if (r < 0.0f) r = 0.0f;
                if (r > 15.0f) r = 15.0f;
                int q = (int)r;
                uint32_t* p = (uint32_t*)&qweight[(k / 8) * N + n];
                if (k % 8 == 0) *p = 0;
                *p |= ((uint32_t)q & 0xFu) << (4 * (int)(k % 8));
                if (deq) deq[k * N + n] = (float)(q - z) * sq;
            }
        }
    }
    return 0;
}

/* W4A16 with a zero point: b = (q[k,j] - z[k/128, j]) * s[k/128, j]. */
void or_gemm_w4a16_zp(const uint16_t* A, const int32_t* qweight, const uint16_t* scale,
                      const uint8_t* zero, int64_t M, int64_t N, int64_t K, const int64_t* ii,
                      const int64_t* jj, int64_t npts, double* y, double* bound)
{
    (void)M;
    for (int64_t p = 0; p < npts; p++) {
        int64_t i = ii[p], j = jj[p];
        double acc = 0.0, mag = 0.0;
        const uint16_t* arow = A + i * K;
        for (int64_t k = 0; k < K; ++k) {
            uint32_t word = (uint32_t)qweight[(k / 8) * N + j];
            int q = (int)((word >> (4 * (k % 8))) & 0xF);
            int z = zero[(k / 128) * N + j];
            double b = (double)(q - z) * (double)or_bf16_to_f32(scale[(k >> 7) * N + j]);
            double a = (double)or_bf16_to_f32(arow[k]);
            acc += a * b;
            mag += fabs(a * b);
        }
        y[p] = acc;
        bound[p] = mag;
    }
}

/* ------------------------------------------- weight-only FP4 (W4A16 FP4) */

/* a = A[i,k] (bf16); b = e2m1(qB[j,k]) * e4m3(sB[j, k/16]) * gB, B^T [N, K]. */
void or_gemm_w4a16_nvfp4(const uint16_t* A, const uint8_t* qB, const uint8_t* sB, float gB,
                         int64_t M, int64_t N, int64_t K, const int64_t* ii, const int64_t* jj,
                         int64_t npts, double* y, double* bound)
{
    (void)M; (void)N;
    for (int64_t p = 0; p < npts; p++) {
        int64_t i = ii[p], j = jj[p];
        double acc = 0.0, mag = 0.0;
        const uint16_t* arow = A + i * K;
        const uint8_t* srow = sB + j * (K / 16);
        for (int64_t k = 0; k < K; k++) {
            double a = (double)or_bf16_to_f32(arow[k]);
            double b = or_fp4_at(qB, j, K, k) * or_e4m3_decode(srow[k / 16]) * (double)gB;
            acc += a * b;
            mag += fabs(a * b);
        }
        y[p] = acc;
        bound[p] = mag;
    }
}

/* a = A[i,k] (bf16); b = e2m1(qB[j,k]) * 2^(eB[j, k/32] - 127). */
void or_gemm_w4a16_mxfp4(const uint16_t* A, const uint8_t* qB, const uint8_t* eB,
                         int64_t M, int64_t N, int64_t K, const int64_t* ii, const int64_t* jj,
                         int64_t npts, double* y, double* bound)
{
    (void)M; (void)N;
    for (int64_t p = 0; p < npts; p++) {
        int64_t i = ii[p], j = jj[p];
        double acc = 0.0, mag = 0.0;
        const uint16_t* arow = A + i * K;
        const uint8_t* erow = eB + j * (K / 32);
        for (int64_t k = 0; k < K; k++) {
            double a = (double)or_bf16_to_f32(arow[k]);
            double b = ldexp(or_fp4_at(qB, j, K, k), (int)erow[k / 32] - 127);
            acc += a * b;
            mag += fabs(a * b);
        }
        y[p] = acc;
        bound[p] = mag;
    }
}

/* ----------------------------------------------- SmoothQuant + INT8 W8A8 */

/* max |x[r, c]| over the rows r of each column c (the per-channel statistic
 * of SmoothQuant [P2 路线二]): out[cols]. */
void or_col_amax(const void* x, int is_bf16, int64_t rows, int64_t cols, float* out)
{
    for (int64_t c = 0; c < cols; c++) out[c] = 0.0f;
    for (int64_t r = 0; r < rows; r++)
        for (int64_t c = 0; c < cols; c++) {
            float a = fabsf(or_elem(x, is_bf16, r * cols + c));
            if (a > out[c]) out[c] = a;
        }
}

/* s_j = max|X_j|^0.5 / max|W_j|^0.5 [P2 路线二, alpha = 0.5], each amax
 * floored at 1e-12: s = fl(fl(sqrt(ax)) / fl(sqrt(aw))). */
void or_smooth_factors(const float* xmax, const float* wmax, int64_t n, float* s)
{
    for (int64_t j = 0; j < n; j++) {
        float ax = xmax[j] > or_amax_min() ? xmax[j] : or_amax_min();
        float aw = wmax[j] > or_amax_min() ? wmax[j] : or_amax_min();
        s[j] = sqrtf(ax) / sqrtf(aw);
    }
}

/* INT8 per row of x[rows][cols] (tokens of an activation, or output channels
 * of a weight stored as B^T), after the optional per-column smoothing factor:
 *   x' = fl(x / f[c]) (smooth = 1, activations) or fl(x * f[c]) (smooth = 2,
 *   weights); smooth = 0: x' = x.
 *   s = max(amax_row(x'), 1e-12) / 127;  q = clamp(rint(fl(x' / s)), -128, 127)
 * codes[rows][cols] int8, scales[rows], deq = q * s (nullable). */
int or_quant_int8_rows(const void* x, int is_bf16, int64_t rows, int64_t cols, const float* f, int smooth,
                       int8_t* codes, float* scales, float* deq)
{
    if (rows <= 0 || cols <= 0 || smooth < 0 || smooth > 2 || (smooth && !f)) return -1;
    for (int64_t r = 0; r < rows; r++) {
        float amax = 0.0f;
        for (int64_t c = 0; c < cols; c++) {
            float v = or_elem(x, is_bf16, r * cols + c);
            if (smooth == 1) v = v / f[c];
            else if (smooth == 2) v = v * f[c];
            if (fabsf(v) > amax) amax = fabsf(v);
        }
        float s = (amax > or_amax_min() ? amax : or_amax_min()) / 127.0f;
        scales[r] = s;
        for (int64_t c = 0; c < cols; c++) {
            float v = or_elem(x, is_bf16, r * cols + c);
            if (smooth == 1) v = v / f[c];
            else if (smooth == 2) v = v * f[c];
            float d;
            int q = or_int_quant_one(v, s, -128, 127, &d);
            codes[r * cols + c] = (int8_t)q;
            if (deq) deq[r * cols + c] = d;
        }
    }
    return 0;
}

/* INT8 GEMM: y[i,j] = sA[i] * sB[j] * sum_k qA[i,k] * qB[j,k] (B^T [N, K]),
 * the integer sum exact in int64; bound = sum_k |a * b| of the dequantized
 * operands. */
void or_gemm_int8(const int8_t* qA, const float* sA, const int8_t* qB, const float* sB,
                  int64_t M, int64_t N, int64_t K, const int64_t* ii, const int64_t* jj,
                  int64_t npts, double* y, double* bound)
{
    (void)M; (void)N;
    for (int64_t p = 0; p < npts; p++) {
        int64_t i = ii[p], j = jj[p];
        int64_t acc = 0, mag = 0;
        for (int64_t k = 0; k < K; k++) {
            int64_t t = (int64_t)qA[i * K + k] * (int64_t)qB[j * K + k];
            acc += t;
            mag += t < 0 ? -t : t;
        }
        double sc = (double)sA[i] * (double)sB[j];
        y[p] = (double)acc * sc;
        bound[p] = (double)mag * fabs(sc);
    }
}
