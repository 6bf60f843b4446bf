/*
 * qz.h -- C ABI of libqz: low-bit quantizers and quantized linear layers for
 * one GB300 (sm_103a) GPU.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Ownership: every data pointer is a DEVICE pointer owned by the caller. The
 *   library never allocates or frees device memory. Scratch that a call needs
 *   comes from a caller buffer `ws` of at least qz_workspace_size(...) bytes.
 * Streams: `stream` is a cudaStream_t passed as void* (NULL = the legacy
 *   default stream). Every call only enqueues work on that stream and returns
 *   without synchronising; outputs are valid in stream order. A workspace must
 *   not be shared by calls that may run concurrently.
 * Early start: most calls launch under programmatic dependent launch, so their
 *   kernels may begin while the previous kernel on the stream is still running.
 *   Each waits for that kernel before it reads or writes anything, with one
 *   exception. The INT4 W4A16 GEMMs (qz_gemm_w4a16, _grouped, _zp) read qweight,
 *   scale_bf16 and zero BEFORE that wait, so the weight stream overlaps the
 *   previous kernel's tail. The library tracks the outputs of its own INT4
 *   quantizers per device and stream. A W4A16 call whose weights such a call may
 *   still be writing is launched only after the stream's earlier work. Weights
 *   written by other code must not come from the kernel enqueued directly
 *   before the W4A16 call on its stream. Any synchronisation, copy or other
 *   kernel between the two is enough.
 * Layout: row-major, leading dimension in elements. Packed 4-bit codes put
 *   the even-index element in the low nibble of each byte. bf16 data is passed
 *   as uint16_t bit patterns. Scales use the row-major layouts given per call.
 * Errors: every call returns a qz_status. Arguments are validated on the host
 *   before anything is enqueued, so a rejected call launches nothing and
 *   leaves every output untouched. No call aborts, throws or prints.
 *   QZ_ERR_CUDA reports a launch or runtime error seen right after enqueueing.
 * Numerics: the codes and scales of every quantizer are defined by the fake-
 *   quant functions of "量化部署实战" (anrans.github.io), section 伪量化实现,
 *   computed in IEEE fp32 (bf16 inputs are widened exactly to fp32 first):
 *   E4M3 rounds to nearest even and saturates at +-448; E2M1 rounds to the
 *   nearest of +-{0, .5, 1, 1.5, 2, 3, 4, 6} with exact ties going to the
 *   smaller magnitude; the clamp floor 1e-12 is the fp32 value nearest 1e-12.
 *   NaN or infinite inputs are outside the contract (no fault, undefined codes).
 */
#ifndef QZ_H
#define QZ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum qz_status {
    QZ_OK = 0,
    QZ_ERR_INVALID_ARG = 1,   /* null pointer, unknown enum value, negative size */
    QZ_ERR_SHAPE = 2,         /* size not divisible as required, or out of the supported range */
    QZ_ERR_ALIGNMENT = 3,     /* pointer or leading dimension not aligned as required */
    QZ_ERR_UNSUPPORTED = 4,   /* no usable sm_103 device, or the path is not available */
    QZ_ERR_CUDA = 5,          /* a CUDA runtime call or kernel launch failed */
    QZ_ERR_TIMEOUT = 6,       /* a bounded device-side wait gave up (see qz_device_error) */
    QZ_ERR_WORKSPACE = 7      /* ws is NULL or smaller than qz_workspace_size() */
} qz_status;

typedef enum qz_dtype { QZ_F32 = 0, QZ_BF16 = 1 } qz_dtype;

typedef enum qz_fp8_gran {
    QZ_FP8_PER_TENSOR = 0,    /* one scale for the tensor                      scales[1]             */
    QZ_FP8_PER_ROW = 1,       /* one scale per row (output channel / token)    scales[rows]          */
    QZ_FP8_BLOCK_128x128 = 2, /* one scale per (br x 128) block, br=min(128,rows) scales[rows/br][cols/128] */
    QZ_FP8_GROUP_1x128 = 3    /* one scale per row per 128 columns             scales[rows][cols/128] */
} qz_fp8_gran;

typedef enum qz_scale_mode {
    QZ_SCALE_COMPUTE = 0,     /* scale = max(amax, 1e-12) / 448 from the data written   */
    QZ_SCALE_GIVEN = 1        /* use the caller's (calibrated) scale, read from device  */
} qz_scale_mode;

typedef enum qz_op {
    QZ_OP_QUANTIZE_FP8 = 0,   /* d0 = rows, d1 = cols, d2 = granularity   */
    QZ_OP_QUANTIZE_NVFP4 = 1, /* d0 = rows, d1 = cols                      */
    QZ_OP_KV_WRITE_FP8 = 2,   /* d0 = elements per tensor (B*H*T*D)        */
    QZ_OP_GEMM_W4A16 = 3,     /* d0 = M, d1 = N, d2 = K                    */
    QZ_OP_GEMM_FP8_BLOCK = 4, /* d0 = M, d1 = N, d2 = K                    */
    QZ_OP_GEMM_NVFP4 = 5,     /* d0 = M, d1 = N, d2 = K                    */
    QZ_OP_GEMM_MXFP4 = 6,     /* d0 = M, d1 = N, d2 = K                    */
    QZ_OP_GEMM_NVFP4_GROUPED = 7, /* d0 = problem count, d1 = largest K    */
    QZ_OP_PREPARE_FP4_SCALES = 8, /* d0 = rows, d1 = K, d2 = 1 NVFP4 / 0 MXFP4:
                                     bytes of the prepared output (not scratch) */
    QZ_OP_QUANTIZE_NVFP4_GROUPED = 9, /* d0 = tensor count                   */
    QZ_OP_KV_WRITE_FP8_PER_HEAD = 10, /* d0 = B*H, d1 = T*D                   */
    QZ_OP_KV_WRITE_FP8_CHANNEL_ZP = 11, /* d0 = B*H, d1 = T, d2 = D           */
    QZ_OP_COL_AMAX = 12                 /* d0 = rows, d1 = cols               */
} qz_op;

typedef enum qz_smooth_op {
    QZ_SMOOTH_NONE = 0,       /* x' = x                                          */
    QZ_SMOOTH_DIVIDE = 1,     /* x' = x / f[col]  (activations, SmoothQuant)     */
    QZ_SMOOTH_MULTIPLY = 2    /* x' = x * f[col]  (weights as B^T, SmoothQuant)  */
} qz_smooth_op;

/* Bytes of workspace the call `op` needs for the given sizes (0 if none).
 * Returns 0 for an unknown op. Sizes that the call itself would reject still
 * return a (harmless) value. Workspace contents need no initialisation. */
size_t qz_workspace_size(qz_op op, int64_t d0, int64_t d1, int64_t d2);

/* Human-readable name of a status (static string, never NULL). */
const char* qz_status_string(qz_status s);

/* Reads and clears the library's device-side error word on the current
 * device (set when a bounded wait inside a GEMM kernel gives up). Returns
 * QZ_ERR_TIMEOUT if it was set, QZ_OK if not, QZ_ERR_CUDA if the read failed.
 * Synchronises with the legacy default stream. */
qz_status qz_device_error(void);

/* Self-test of the failure detection (the pages have no counterpart; this is
 * a property of this library's kernels). Launches one CTA on `stream` that
 * waits on an mbarrier nothing ever completes, using the same bounded wait as
 * every GEMM kernel but giving up after `polls` polls (1 <= polls <= 2^20,
 * each poll suspends for at most tens of nanoseconds). The wait runs out,
 * records QZ_ERR_TIMEOUT in the device error word and the kernel returns, so
 * the next qz_device_error() reports QZ_ERR_TIMEOUT and the CUDA context stays
 * usable. Returns QZ_ERR_INVALID_ARG for polls out of range. */
qz_status qz_selftest_bounded_wait(uint32_t polls, void* stream);

/* ------------------------------------------------------------ quantizers */

/* FP8 E4M3 quantization of x[rows, cols] (leading dim ldx >= cols) at one of
 * four scale granularities ("量化部署实战", 伪量化实现: fp8_per_tensor,
 * fp8_per_row, fp8_blockwise with (128,128) for weights and (1,128) for
 * activations; 格式速查: FP8 E4M3 row):
 *   scale = max(amax_unit, 1e-12) / 448;  code = E4M3(clamp(x / scale, +-448))
 *   dequant = E4M3value(code) * scale    (fp32, one rounding)
 * codes:   [rows, cols] bytes, dense.
 * scales:  fp32, shape per qz_fp8_gran.
 * dequant: nullable; fp32 [rows, cols], dense.
 * ws:      PER_TENSOR needs qz_workspace_size(QZ_OP_QUANTIZE_FP8, rows, cols, 0)
 *          bytes; the other granularities need none (ws may be NULL).
 * Shapes:  BLOCK_128x128 needs cols % 128 == 0 and rows % min(128, rows) == 0;
 *          GROUP_1x128 needs cols % 128 == 0. rows == 0 or cols == 0 is a no-op
 *          returning QZ_OK, except PER_TENSOR (amax undefined) -> QZ_ERR_SHAPE.
 * Alignment: x 16-byte aligned with ldx*elemsize % 16 == 0 and cols % 8 == 0
 *          give the vector path; PER_TENSOR and PER_ROW also accept any other
 *          x/ldx/cols (scalar path). BLOCK/GROUP require the vector conditions
 *          (QZ_ERR_ALIGNMENT), and codes/dequant must then be 8/16-byte aligned. */
qz_status qz_quantize_fp8(const void* x, qz_dtype xt, int64_t rows, int64_t cols, int64_t ldx,
                          qz_fp8_gran gran, uint8_t* codes, float* scales, float* dequant,
                          void* ws, size_t ws_bytes, void* stream);

/* MXFP4 quantization, one power-of-two (E8M0) scale per 32 consecutive
 * elements of a row ("量化部署实战", 伪量化实现: mxfp4; "量化：让每一步搬更少的
 * 字节", 新一代低位格式: MXFP4):
 *   E = floor(log2(max(amax32, 1e-12))) (exact, from the exponent field)
 *   scale = 2^(E-2); scale_e8m0 = E - 2 + 127
 *   code = E2M1(clamp(x / scale, +-6));  dequant = E2M1value(code) * scale
 * codes: [rows, cols/2] bytes (even element in the low nibble).
 * scale_e8m0: [rows, cols/32] bytes. dequant: nullable fp32 [rows, cols].
 * Shapes: cols % 32 == 0. Alignment: x 16 B, ldx*elemsize % 16 == 0, codes 4 B,
 * dequant 16 B. rows == 0 is a no-op. No workspace. */
qz_status qz_quantize_mxfp4(const void* x, qz_dtype xt, int64_t rows, int64_t cols, int64_t ldx,
                            uint8_t* codes, uint8_t* scale_e8m0, float* dequant, void* stream);

/* NVFP4 quantization, one E4M3 scale per 16 consecutive elements of a row
 * plus one fp32 scale per tensor ("量化部署实战", 伪量化实现: nvfp4;
 * 格式速查: NVFP4 row), in the page's order:
 *   g = max(amax_tensor, 1e-12) / (448 * 6)         -> *global_scale
 *   b = E4M3(amax16 / 6 / g)                         -> scale_e4m3
 *   s = max(E4M3value(b), 1e-12) * g
 *   code = E2M1(clamp(x / s, +-6));  dequant = E2M1value(code) * s
 * global_amax_in: nullable device pointer; when given, its value replaces the
 *   computed tensor amax (calibrated or shared across slices) and no
 *   workspace is needed.
 * codes: [rows, cols/2]; scale_e4m3: [rows, cols/16]; global_scale: 1 fp32.
 * ws: qz_workspace_size(QZ_OP_QUANTIZE_NVFP4, rows, cols, 0) bytes when
 *   global_amax_in is NULL. Shapes: cols % 16 == 0; rows == 0 -> QZ_ERR_SHAPE
 *   unless global_amax_in is given (then a no-op). Alignment as MXFP4. */
qz_status qz_quantize_nvfp4(const void* x, qz_dtype xt, int64_t rows, int64_t cols, int64_t ldx,
                            uint8_t* codes, uint8_t* scale_e4m3, float* global_scale,
                            const float* global_amax_in, float* dequant,
                            void* ws, size_t ws_bytes, void* stream);

/* One tensor of qz_quantize_nvfp4_grouped: contiguous x [rows, cols] (cols %
 * 16 == 0) and its outputs, laid out as qz_quantize_nvfp4 writes them. */
typedef struct qz_nvfp4_tensor {
    const void* x;
    int64_t rows, cols;
    uint8_t* codes;
    uint8_t* scale_e4m3;
    float* global_scale;
} qz_nvfp4_tensor;

/* NVFP4 quantization of `count` independent tensors (the activations of a
 * decoder step's linears, "量化部署实战", 精度比较: each linear quantizes its
 * input) in two launches: the same computation as one qz_quantize_nvfp4 call
 * with a computed tensor amax per tensor, bit for bit. All tensors share the
 * dtype xt. count <= 256. Alignment: x 16 B, codes 4 B. ws:
 * qz_workspace_size(QZ_OP_QUANTIZE_NVFP4_GROUPED, count, 0, 0) bytes. */
qz_status qz_quantize_nvfp4_grouped(const qz_nvfp4_tensor* tensors, int count, qz_dtype xt,
                                    void* ws, size_t ws_bytes, void* stream);

/* Symmetric INT4 weight quantization with one bf16 scale per group of 128
 * along K, for a row-major weight w[K, N] (leading dim ldw >= N)
 * ("量化部署实战", 格式速查: W4A16 row, integers -8..7 with a scale per 128;
 * "量化：让每一步搬更少的字节", 量化在做什么: q = round(x / s), x^ = q * s;
 * "LLM 推理优化 · 量化学习笔记" 5.1: q = clamp(round(x / s), qmin, qmax)):
 *   s = bf16_rne(max(amax_group, 1e-12) / 7);  q = clamp(rint(w / s), -8, 7)
 * qweight: int32 [K/8, N]; element k of column n sits in bits 4*(k%8)..+3 of
 *   qweight[k/8][n], two's complement.
 * scale_bf16: [K/128, N] bf16 bits. dequant: nullable fp32 [K, N] = q * s.
 * Shapes: K % 128 == 0, N % 64 == 0. Alignment: w 16 B, ldw*elemsize % 16 == 0,
 * qweight and dequant 16 B, scale_bf16 16 B. K == 0 or N == 0 is a no-op. */
qz_status qz_quantize_int4_g128(const void* w, qz_dtype wt, int64_t K, int64_t N, int64_t ldw,
                                int32_t* qweight, uint16_t* scale_bf16, float* dequant,
                                void* stream);

/* FP8 KV-cache write: per-tensor E4M3 quantization of K and of V, each with
 * its own scale ("量化部署实战", 伪量化实现: FP8KVCache.update applies
 * fp8_per_tensor to k and to v; KV Cache 量化: calibrated offline scales).
 * k, v: bf16 [B, H, T, D] contiguous (n = B*H*T*D elements each).
 * k_codes, v_codes: n bytes each. k_scale, v_scale: one fp32 each (device).
 * mode COMPUTE: scales = max(amax, 1e-12) / 448 written to k_scale/v_scale;
 *   needs qz_workspace_size(QZ_OP_KV_WRITE_FP8, n, 0, 0) bytes.
 * mode GIVEN: k_scale/v_scale are read (must be finite and > 0); no workspace.
 * Alignment: k, v 16 B; codes 8 B. n == 0 -> QZ_ERR_SHAPE (COMPUTE), no-op (GIVEN). */
qz_status qz_kv_write_fp8(const uint16_t* k, const uint16_t* v, int B, int H, int T, int D,
                          uint8_t* k_codes, uint8_t* v_codes, float* k_scale, float* v_scale,
                          qz_scale_mode mode, void* ws, size_t ws_bytes, void* stream);

/* ----------------------------------------------------------------- GEMMs */

/* W4A16 GEMM ("量化：让每一步搬更少的字节", 路线一: one kernel that fuses the
 * INT4 unpack, the dequantization and the matrix product):
 *   Y[m, n] = bf16_rne( sum_g s[g, n] * sum_{k in g} A[m, k] * q[k, n] )
 * accumulated in fp32. A: bf16 [M, K] row-major. qweight, scale_bf16: the
 * layouts written by qz_quantize_int4_g128. Y: bf16 [M, N].
 * Shapes: 1 <= M <= 64, K % 128 == 0, N % 64 == 0.
 * Alignment: all pointers 16 B. ws: qz_workspace_size(QZ_OP_GEMM_W4A16, M, N, K). */
qz_status qz_gemm_w4a16(const uint16_t* A, const int32_t* qweight, const uint16_t* scale_bf16,
                        uint16_t* Y, int M, int N, int K, void* ws, size_t ws_bytes, void* stream);

/* One W4A16 problem of a grouped launch (all pointers device, layouts as in
 * qz_gemm_w4a16). */
typedef struct qz_w4a16_problem {
    const uint16_t* A;
    const int32_t* qweight;
    const uint16_t* scale_bf16;
    uint16_t* Y;
    int M, N, K;
} qz_w4a16_problem;

/* Runs `count` independent W4A16 problems (a decoder step's linears, whose
 * inputs are all ready) in as few launches as the kernel parameter space
 * allows (per launch: up to 120 problems of at most 8 tokens and K <= 8192,
 * 256 for deeper K, 56 at 9-16 tokens, 80 at 17-64), split into equal
 * shares. The kernel is chosen by the largest M of the group. Each problem
 * obeys the rules of qz_gemm_w4a16; outputs must not overlap. count <= 256.
 * ws: qz_workspace_size(QZ_OP_GEMM_W4A16, Mmax, sum of N, Kmax) bytes
 * suffices. */
qz_status qz_gemm_w4a16_grouped(const qz_w4a16_problem* problems, int count,
                                void* ws, size_t ws_bytes, void* stream);

/* FP8 block-scaled GEMM ("量化部署实战", 练习 2: inside each 128-wide K block
 * the tensor cores multiply-accumulate FP8, then the partial sum is multiplied
 * by that block's activation and weight scales and added into the fp32 result):
 *   Y[i, j] = bf16_rne( sum_kb sA[i, kb] * sB[j/128, kb] * sum_{k in kb} qA[i,k] * qB[j,k] )
 * qA: E4M3 [M, K] (1x128 groups, as written by qz_quantize_fp8 GROUP_1x128);
 * sA: fp32 [M, K/128]. qB: E4M3 [N, K] = B^T, K-major (128x128 blocks, as
 * written by qz_quantize_fp8 BLOCK_128x128 on B^T); sB: fp32 [N/128, K/128].
 * Y: bf16 [M, N]. Shapes: M % 128 == 0, N % 256 == 0, K % 128 == 0, K >= 128.
 * Alignment: all pointers 16 B. */
qz_status qz_gemm_fp8_block(const uint8_t* qA, const float* sA, const uint8_t* qB, const float* sB,
                            uint16_t* Y, int M, int N, int K, void* ws, size_t ws_bytes, void* stream);

/* NVFP4 GEMM (Blackwell FP4 tensor cores; "量化部署实战", 格式速查: NVFP4):
 *   Y[i, j] = bf16_rne( gA * gB * sum_b sA[i,b] * sB[j,b] * sum_{k in b} qA[i,k] * qB[j,k] )
 * qA: [M, K/2] packed E2M1, sA: E4M3 [M, K/16], gA: fp32 device scalar;
 * qB, sB, gB likewise for B^T [N, K]; layouts as written by qz_quantize_nvfp4.
 * Y: bf16 [M, N]. Shapes: M % 128 == 0, N % 256 == 0, K % 256 == 0.
 * Alignment: all pointers 16 B. */
qz_status qz_gemm_nvfp4(const uint8_t* qA, const uint8_t* sA, const float* gA,
                        const uint8_t* qB, const uint8_t* sB, const float* gB,
                        uint16_t* Y, int M, int N, int K, void* ws, size_t ws_bytes, void* stream);

/* MXFP4 GEMM: Y[i, j] = bf16_rne( sum_b 2^(eA[i,b]-127) * 2^(eB[j,b]-127) *
 * sum_{k in b} qA[i,k] * qB[j,k] ), blocks of 32 along K. Layouts as written by
 * qz_quantize_mxfp4 on A [M, K] and B^T [N, K]. Shapes and alignment as NVFP4. */
qz_status qz_gemm_mxfp4(const uint8_t* qA, const uint8_t* eA, const uint8_t* qB, const uint8_t* eB,
                        uint16_t* Y, int M, int N, int K, void* ws, size_t ws_bytes, void* stream);

/* Re-lays a row-major block-scale matrix, as the FP4 quantizers write it
 * (NVFP4: E4M3 [rows, K/16], nv = 1; MXFP4: E8M0 [rows, K/32], nv = 0), into the
 * order the FP4 tensor cores read scale factors in: per 128 rows and 4
 * consecutive scales, a 512-byte block where byte (m%32)*16 + (m/32)*4 + k holds
 * the scale k of row m (rows beyond `rows` up to a multiple of 128 are 0).
 * Weights are static, so their scales are re-laid once and handed to
 * qz_gemm_nvfp4_grouped; the single-problem GEMMs do this per call in their
 * workspace. This is a layout step of this library; the pages define no
 * layout for the scales beyond the row-major block order.
 * out: qz_workspace_size(QZ_OP_PREPARE_FP4_SCALES, rows, K, nv) bytes, 16 B
 * aligned, caller-owned. Shapes: rows >= 1, K % 256 == 0. */
qz_status qz_prepare_fp4_scales(const uint8_t* scales, int rows, int K, int nv, uint8_t* out, void* stream);

/* One problem of qz_gemm_nvfp4_grouped: Y = A B with A NVFP4 codes [M, K/2],
 * row-major E4M3 scales [M, K/16] and tensor scale gA (as qz_quantize_nvfp4
 * writes them), B^T NVFP4 codes [N, K/2] with its scales already re-laid by
 * qz_prepare_fp4_scales(nv = 1) and tensor scale gB, Y bf16 [M, N]. */
typedef struct qz_nvfp4_problem {
    const uint8_t* qA;
    const uint8_t* sA;
    const float* gA;
    const uint8_t* qB;
    const uint8_t* sB_prepared;
    const float* gB;
    uint16_t* Y;
    int M, N, K;
} qz_nvfp4_problem;

/* Runs `count` independent NVFP4 GEMMs of decode shape (the linears of a
 * decoder step, "量化部署实战", 精度比较: every linear of the block quantized)
 * with one scale re-layout launch for all A operands and one GEMM launch per
 * 72 problems, the problems' 128 x 256 output tiles shared out over the SMs.
 * Same arithmetic as qz_gemm_nvfp4. Shapes per problem: 1 <= M <= 128,
 * N % 256 == 0, K % 256 == 0. count <= 256. Alignment: codes, prepared scales
 * and Y 16 B, sA 4 B. ws: qz_workspace_size(QZ_OP_GEMM_NVFP4_GROUPED, count,
 * largest K, 0) bytes. */
qz_status qz_gemm_nvfp4_grouped(const qz_nvfp4_problem* problems, int count, void* ws, size_t ws_bytes,
                                void* stream);

/* -------------------------------------------- variants (zero points, KV, INT8) */

/* FP8 KV-cache write with one scale per (batch, head) for K and for V
 * ("量化部署实战", KV Cache 量化: per_head, the amax over the head's T x D
 * values; calibrated scales per 实际部署时):
 *   scale[b, h] = max(amax over k[b, h, :, :], 1e-12) / 448; code = E4M3(x / scale)
 * k, v: bf16 [B, H, T, D] contiguous; codes: n bytes each; k_scale, v_scale:
 * fp32 [B, H] (device). mode COMPUTE writes the scales and needs
 * qz_workspace_size(QZ_OP_KV_WRITE_FP8_PER_HEAD, B*H, T*D, 0) bytes of ws; mode
 * GIVEN reads them (finite, > 0) and needs no workspace.
 * Shapes: B, H, T >= 1, D % 8 == 0. Alignment: k, v 16 B; codes 8 B. */
qz_status qz_kv_write_fp8_per_head(const uint16_t* k, const uint16_t* v, int B, int H, int T, int D,
                                   uint8_t* k_codes, uint8_t* v_codes, float* k_scale, float* v_scale,
                                   qz_scale_mode mode, void* ws, size_t ws_bytes, void* stream);

/* FP8 KV-cache write with K per channel and a zero point, V per token
 * ("量化部署实战", KV Cache 量化: K carries a constant bias per channel plus a
 * small variation; quantizing K per channel with a zero point absorbs the bias,
 * and the KIVI split quantizes K per channel and V per token; "LLM 推理优化 ·
 * 量化学习笔记" 5.1: asymmetric quantization adds a zero point). The codes stay
 * E4M3, so the zero point lives in value space. For each channel (b, h, d), over
 * its T tokens:
 *   z = fl(0.5 * fl(max + min));  s = max(max_t |fl(x - z)|, 1e-12) / 448
 *   k_code = E4M3(clamp(fl(x - z) / s, +-448)); dequant = fl(fl(value * s) + z)
 * and for each token (b, h, t): v_scale = max(amax over its D values, 1e-12) / 448,
 * v_code = E4M3(v / v_scale).
 * k_scale, k_zero: fp32 [B, H, D]; v_scale: fp32 [B, H, T]; codes [B, H, T, D].
 * ws: qz_workspace_size(QZ_OP_KV_WRITE_FP8_CHANNEL_ZP, B*H, T, D) bytes.
 * Shapes: B, H, T >= 1, D one of 8, 16, 32, 64, 128, 256. Alignment: k, v 16 B,
 * codes 8 B. */
qz_status qz_kv_write_fp8_channel_zp(const uint16_t* k, const uint16_t* v, int B, int H, int T, int D,
                                     uint8_t* k_codes, uint8_t* v_codes, float* k_scale, float* k_zero,
                                     float* v_scale, void* ws, size_t ws_bytes, void* stream);

/* INT4 weight quantization with a zero point: unsigned codes 0..15, one bf16
 * scale and one integer zero point per group of 128 along K ("量化部署实战",
 * 格式速查: W4A16, a scale per 128 "+ 零点"; "LLM 推理优化 · 量化学习笔记" 5.1:
 * q = clamp(round(x / s) + z, ...)). Per group and column the range is widened
 * to include 0 (lo = min(min, 0), hi = max(max, 0)):
 *   s = bf16_rne(max(hi - lo, 1e-12) / 15);  z = clamp(rint(-lo / s), 0, 15)
 *   q = clamp(rint(w / s) + z, 0, 15);         dequant = (q - z) * s
 * qweight: int32 [K/8, N], element k in bits 4*(k%8)..+3 (unsigned);
 * scale_bf16: [K/128, N]; zero: uint8 [K/128, N]; dequant nullable fp32 [K, N].
 * Shapes: K % 128 == 0, N % 64 == 0. Alignment as qz_quantize_int4_g128. */
qz_status qz_quantize_int4_g128_zp(const void* w, qz_dtype wt, int64_t K, int64_t N, int64_t ldw,
                                   int32_t* qweight, uint16_t* scale_bf16, uint8_t* zero, float* dequant,
                                   void* stream);

/* W4A16 GEMM with zero points (the fused unpack + dequant + matmul of
 * "量化：让每一步搬更少的字节", 路线一, on the codes of qz_quantize_int4_g128_zp):
 *   Y[m, n] = bf16_rne( sum_g s[g, n] * sum_{k in g} A[m, k] * (q[k, n] - z[g, n]) )
 * fp32 accumulation. Shapes: 1 <= M <= 16, K % 128 == 0, N % 64 == 0.
 * Alignment: A, qweight, scale, Y 16 B; zero 4 B. */
qz_status qz_gemm_w4a16_zp(const uint16_t* A, const int32_t* qweight, const uint16_t* scale_bf16,
                           const uint8_t* zero, uint16_t* Y, int M, int N, int K, void* stream);

/* Weight-only FP4 GEMMs ("量化部署实战", 精度比较: W4A16 NVFP4 and W4A16
 * MXFP4): bf16 activations times FP4 weights given as B^T [N, K] exactly as the
 * FP4 quantizers write them, fp32 accumulation, bf16 output:
 *   NVFP4: Y[m, n] = bf16_rne( gB * sum_k A[m, k] * e2m1(q[n, k]) * e4m3(s[n, k/16]) )
 *   MXFP4: Y[m, n] = bf16_rne( sum_k A[m, k] * e2m1(q[n, k]) * 2^(e[n, k/32] - 127) )
 * qB: [N, K/2]; sB: E4M3 [N, K/16]; gB: fp32 device scalar; eB: E8M0 [N, K/32].
 * MXFP4 scale codes must lie in 66..192 (scales 2^-61 .. 2^65).
 * Shapes: 1 <= M <= 16, K % 128 == 0, N % 32 == 0. Alignment: A, qB, Y 16 B;
 * sB 2 B. */
qz_status qz_gemm_w4a16_nvfp4(const uint16_t* A, const uint8_t* qB, const uint8_t* sB, const float* gB,
                              uint16_t* Y, int M, int N, int K, void* stream);
qz_status qz_gemm_w4a16_mxfp4(const uint16_t* A, const uint8_t* qB, const uint8_t* eB,
                              uint16_t* Y, int M, int N, int K, void* stream);

/* Per-column amax of x[rows, cols] (the per-channel statistic of SmoothQuant,
 * "量化：让每一步搬更少的字节", 路线二: max|X_j| over the tokens, max|W_j| over
 * the output channels of a weight stored as B^T): out[c] = max_r |x[r, c]|.
 * ws: qz_workspace_size(QZ_OP_COL_AMAX, rows, cols, 0) bytes.
 * Shapes: rows >= 1, cols % 8 == 0. Alignment: x, out 16 B. */
qz_status qz_col_amax(const void* x, qz_dtype xt, int64_t rows, int64_t cols, float* out, void* ws,
                      size_t ws_bytes, void* stream);

/* SmoothQuant migration factors ("量化：让每一步搬更少的字节", 路线二:
 * s_j = max|X_j|^a / max|W_j|^(1-a), a = 0.5 for most models):
 *   s[j] = fl(sqrt(max(x_amax[j], 1e-12))) / fl(sqrt(max(w_amax[j], 1e-12)))
 * alpha must be 0.5 (QZ_ERR_UNSUPPORTED otherwise). n >= 1. */
qz_status qz_smooth_factors(const float* x_amax, const float* w_amax, int64_t n, float alpha, float* s,
                            void* stream);

/* INT8 quantization per row ("量化部署实战", 格式速查: W8A8 INT8, integers
 * -128..127, per token for activations and per output channel for weights;
 * "量化：让每一步搬更少的字节", 量化在做什么: s = amax / 127), after the optional
 * SmoothQuant factor of each column (op DIVIDE for activations, MULTIPLY for
 * a weight stored as B^T [N, K]; factors nullable for op NONE):
 *   x' = fl(x / f[c]) or fl(x * f[c]);  s = max(amax_row(x'), 1e-12) / 127
 *   q = clamp(rint(x' / s), -128, 127);  dequant = q * s
 * codes int8 [rows, cols]; scales fp32 [rows]; dequant nullable fp32.
 * Shapes: cols % 8 == 0. Alignment: x, factors, dequant 16 B; codes 8 B. */
qz_status qz_quantize_int8_rows(const void* x, qz_dtype xt, int64_t rows, int64_t cols, const float* factors,
                                qz_smooth_op op, int8_t* codes, float* scales, float* dequant, void* stream);

/* INT8 W8A8 GEMM ("量化：让每一步搬更少的字节", 路线二):
 *   Y[i, j] = bf16_rne( sA[i] * sB[j] * sum_k qA[i, k] * qB[j, k] )
 * qA int8 [M, K], qB int8 [N, K] (B^T), sA fp32 [M], sB fp32 [N]; the integer
 * products are summed exactly while |sum| < 2^24 (fp16 tensor cores on the
 * widened codes, fp32 accumulation). Shapes: M % 128 == 0, N % 256 == 0,
 * K % 64 == 0. Alignment: all pointers 16 B. */
qz_status qz_gemm_int8(const int8_t* qA, const float* sA, const int8_t* qB, const float* sB, uint16_t* Y,
                       int M, int N, int K, void* stream);

/* FP8 block-scaled GEMM whose epilogue also quantizes its output for the next
 * layer ("量化部署实战", 练习 2: the activation's (1, 128) scales are computed at
 * the end of the previous kernel, avoiding another read and write): the same
 * arithmetic as qz_gemm_fp8_block, then each row's 128-column groups of the
 * bf16 output y are quantized exactly as qz_quantize_fp8(GROUP_1x128) would:
 *   y_scale = max(amax(y_group), 1e-12) / 448;  y_code = E4M3(y / y_scale)
 * y_codes: [M, N] bytes; y_scales: fp32 [M, N/128]; Y (bf16 [M, N]) nullable:
 * stored too when given. Shapes, layouts and alignment as qz_gemm_fp8_block. */
qz_status qz_gemm_fp8_block_quant(const uint8_t* qA, const float* sA, const uint8_t* qB, const float* sB,
                                  uint16_t* Y, uint8_t* y_codes, float* y_scales, int M, int N, int K,
                                  void* stream);

/* NVFP4 GEMM whose epilogue quantizes its output to NVFP4 for the next layer
 * ("量化部署实战", 练习 2: activation scales computed at the end of the previous
 * kernel; 格式速查: NVFP4, E2M1 + E4M3 per 16 + fp32 per tensor). The same
 * arithmetic as qz_gemm_nvfp4 up to the bf16 output y, which is then encoded
 * exactly as qz_quantize_nvfp4(y, global_amax_in = y_amax) would:
 *   g = max(*y_amax, 1e-12) / 2688 (written to y_global);
 *   per 16 columns: s_code = E4M3(amax16 / 6 / g), s = max(e4m3(s_code), 1e-12) * g,
 *   codes = E2M1(y / s).
 * The tensor amax is the caller's (a calibrated or previous-step value): the
 * kernel cannot know the output's own amax before every tile is done. Blocks
 * whose amax exceeds it saturate as in the quantizer.
 * y_codes: [M, N/2] bytes (16 B aligned); y_scales: E4M3 [M, N/16] (8 B aligned);
 * y_amax, y_global: one fp32 each (device). No bf16 output is written. Other
 * shapes, layouts, workspace and alignment as qz_gemm_nvfp4. */
qz_status qz_gemm_nvfp4_quant(const uint8_t* qA, const uint8_t* sA, const float* gA,
                              const uint8_t* qB, const uint8_t* sB, const float* gB,
                              const float* y_amax, uint8_t* y_codes, uint8_t* y_scales, float* y_global,
                              int M, int N, int K, void* ws, size_t ws_bytes, void* stream);

/* MXFP4 GEMM whose epilogue quantizes its output to MXFP4 for the next layer
 * (as qz_gemm_nvfp4_quant; 格式速查: MXFP4, E2M1 + an E8M0 scale per 32). The
 * same arithmetic as qz_gemm_mxfp4 up to the bf16 output y, then encoded
 * exactly as qz_quantize_mxfp4(y) would: per 32 columns,
 * scale = 2^(floor(log2 max(amax32, 1e-12)) - 2), codes = E2M1(y / scale).
 * No tensor amax is needed. y_codes: [M, N/2] bytes (16 B aligned); y_e8m0:
 * [M, N/32] (4 B aligned). No bf16 output is written. Other shapes, layouts,
 * workspace and alignment as qz_gemm_mxfp4. */
qz_status qz_gemm_mxfp4_quant(const uint8_t* qA, const uint8_t* eA, const uint8_t* qB, const uint8_t* eB,
                              uint8_t* y_codes, uint8_t* y_e8m0, int M, int N, int K,
                              void* ws, size_t ws_bytes, void* stream);

/* NVFP4 GEMM that allocates nothing and takes no workspace. (The quantization
 * pages have no counterpart: this is an interface convenience of this library.)
 * Some callers cannot call cudaMalloc or hand this library a workspace: runtimes
 * whose device memory is planned once at start-up and parcelled out by their own
 * arena (plug-ins get no allocator), and latency-critical loops that must not
 * risk cudaMalloc/cudaFree synchronising the device or failing mid-step. This
 * call computes exactly what qz_gemm_nvfp4 computes, with the same arguments
 * minus ws/ws_bytes; its scratch (the scale factors re-laid for the tensor
 * cores) lives in a fixed device array of QZ_NVFP4_NOALLOC_SCRATCH_BYTES that
 * the library defines, which every GPU that loads the library holds until the
 * process exits.
 * Limit: round_up(M*K/16, 1024) + round_up(N*K/16, 1024) must not exceed
 *   QZ_NVFP4_NOALLOC_SCRATCH_BYTES (4 MiB: e.g. M + N <= 16384 at K = 4096);
 *   larger sizes return QZ_ERR_SHAPE and launch nothing.
 * Set-up: the first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current; make that first call
 *   before any stream capture on the device. The address belongs to the
 *   device's primary context (the CUDA runtime's); it is not looked up again,
 *   so it is stale after cudaDeviceReset or under another context.
 * Sharing: every call uses the same array and leaves its last contents there;
 *   nothing in it needs to start at zero (each call writes every byte it later
 *   reads). Calls whose executions overlap on the GPU (different streams, no
 *   ordering between them) race on the array and must be serialised by the
 *   caller. Other rules, layouts and errors: as qz_gemm_nvfp4. */
#define QZ_NVFP4_NOALLOC_SCRATCH_BYTES ((size_t)4 << 20)
qz_status qz_gemm_nvfp4_noalloc(const uint8_t* qA, const uint8_t* sA, const float* gA,
                                const uint8_t* qB, const uint8_t* sB, const float* gB,
                                uint16_t* Y, int M, int N, int K, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* QZ_H */
