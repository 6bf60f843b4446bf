// qz_api_next.cu -- extern "C" entry points of the variants (zero points,
// per-head and per-channel KV scales, weight-only FP4, SmoothQuant INT8, the
// fused FP8 output quantization): host-side validation, workspace checks and
// dispatch. Nothing here allocates; a rejected call launches nothing.
#include "qz_internal.cuh"
#include "qz_gemm.cuh"
#include "qz_next.cuh"

using namespace qz;

static bool dtype_ok(qz_dtype t) { return t == QZ_F32 || t == QZ_BF16; }
static size_t elem_size(qz_dtype t) { return t == QZ_F32 ? 4 : 2; }
static qz_status ws_ok(void* ws, size_t ws_bytes, size_t need) {
    if (need && (!ws || ws_bytes < need || !is_aligned(ws, 16))) return QZ_ERR_WORKSPACE;
    return QZ_OK;
}

extern "C" {

qz_status qz_kv_write_fp8_per_head(const uint16_t* k, const uint16_t* v, int B, int H, int T, int D,
                                   uint8_t* k_codes, uint8_t* v_codes, float* k_scale, float* v_scale,
                                   qz_scale_mode mode, void* ws, size_t ws_bytes, void* stream) {
    if (!k || !v || !k_codes || !v_codes || !k_scale || !v_scale) return QZ_ERR_INVALID_ARG;
    if (mode != QZ_SCALE_COMPUTE && mode != QZ_SCALE_GIVEN) return QZ_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || T < 1 || D < 1) return QZ_ERR_INVALID_ARG;
    if (D % 8) return QZ_ERR_SHAPE;
    if (!is_aligned(k, 16) || !is_aligned(v, 16) || !is_aligned(k_codes, 8) || !is_aligned(v_codes, 8) ||
        !is_aligned(k_scale, 4) || !is_aligned(v_scale, 4))
        return QZ_ERR_ALIGNMENT;
    const int64_t BH = (int64_t)B * H, L = (int64_t)T * D;
    if (mode == QZ_SCALE_COMPUTE) QZ_TRY(ws_ok(ws, ws_bytes, ws_kv_per_head(BH, L)));
    QZ_TRY(device_check());
    return kv_per_head_launch(k, v, BH, L, k_codes, v_codes, k_scale, v_scale, mode, ws, (cudaStream_t)stream);
}

qz_status qz_kv_write_fp8_channel_zp(const uint16_t* k, const uint16_t* v, int B, int H, int T, int D,
                                     uint8_t* k_codes, uint8_t* v_codes, float* k_scale, float* k_zero,
                                     float* v_scale, void* ws, size_t ws_bytes, void* stream) {
    if (!k || !v || !k_codes || !v_codes || !k_scale || !k_zero || !v_scale) return QZ_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || T < 1 || D < 1) return QZ_ERR_INVALID_ARG;
    if (D != 8 && D != 16 && D != 32 && D != 64 && D != 128 && D != 256) return QZ_ERR_SHAPE;
    if (!is_aligned(k, 16) || !is_aligned(v, 16) || !is_aligned(k_codes, 8) || !is_aligned(v_codes, 8) ||
        !is_aligned(k_scale, 4) || !is_aligned(k_zero, 4) || !is_aligned(v_scale, 4))
        return QZ_ERR_ALIGNMENT;
    const int64_t BH = (int64_t)B * H;
    QZ_TRY(ws_ok(ws, ws_bytes, ws_kv_channel_zp(BH, T, D)));
    QZ_TRY(device_check());
    return kv_channel_zp_launch(k, v, B, H, T, D, k_codes, v_codes, k_scale, k_zero, v_scale, ws,
                                (cudaStream_t)stream);
}

qz_status qz_quantize_int4_g128_zp(const void* w, qz_dtype wt, int64_t K, int64_t N, int64_t ldw,
                                   int32_t* qweight, uint16_t* scale_bf16, uint8_t* zero, float* dequant,
                                   void* stream) {
    if (!dtype_ok(wt) || K < 0 || N < 0 || ldw < N) return QZ_ERR_INVALID_ARG;
    if (K == 0 || N == 0) return QZ_OK;
    if (!w || !qweight || !scale_bf16 || !zero) return QZ_ERR_INVALID_ARG;
    if (K % 128 || N % 64) return QZ_ERR_SHAPE;
    if (!is_aligned(w, 16) || ((size_t)ldw * elem_size(wt)) % 16 || !is_aligned(qweight, 16) ||
        !is_aligned(scale_bf16, 16) || !is_aligned(zero, 16) || (dequant && !is_aligned(dequant, 16)))
        return QZ_ERR_ALIGNMENT;
    QZ_TRY(device_check());
    QZ_TRY(int4_zp_launch(w, wt, K, N, ldw, qweight, scale_bf16, zero, dequant, (cudaStream_t)stream));
    const Span out[3] = {{qweight, (size_t)K * N / 2}, {scale_bf16, (size_t)K * N / 64}, {zero, (size_t)K * N / 128}};
    note_int4_writes((cudaStream_t)stream, out, 3);
    return QZ_OK;
}

qz_status qz_gemm_w4a16_zp(const uint16_t* A, const int32_t* qweight, const uint16_t* scale_bf16,
                           const uint8_t* zero, uint16_t* Y, int M, int N, int K, void* stream) {
    if (!A || !qweight || !scale_bf16 || !zero || !Y) return QZ_ERR_INVALID_ARG;
    if (M < 1 || N < 1 || K < 1) return QZ_ERR_INVALID_ARG;
    if (M > 16 || K % 128 || N % 64) return QZ_ERR_SHAPE;
    if (!is_aligned(A, 16) || !is_aligned(qweight, 16) || !is_aligned(scale_bf16, 16) || !is_aligned(Y, 16) ||
        !is_aligned(zero, 4))
        return QZ_ERR_ALIGNMENT;
    QZ_TRY(device_check());
    // as qz_gemm_w4a16_grouped: weights still in flight -> no dependent launch
    const Int4Writes rec = int4_writes((cudaStream_t)stream);
    const bool early = !w4a16_reads_in_flight(rec, qweight, scale_bf16, zero, N, K);
    QZ_TRY(gemm_w4a16_zp_launch(A, qweight, scale_bf16, zero, Y, M, N, K, (cudaStream_t)stream, early));
    if (!early) clear_int4_writes((cudaStream_t)stream, rec.gen);
    return QZ_OK;
}

static qz_status w4a16_fp4_checks(const uint16_t* A, const uint8_t* qB, const uint8_t* sB, const uint16_t* Y,
                                  int M, int N, int K) {
    if (!A || !qB || !sB || !Y) return QZ_ERR_INVALID_ARG;
    if (M < 1 || N < 1 || K < 1) return QZ_ERR_INVALID_ARG;
    if (M > 16 || K % 128 || N % 32) return QZ_ERR_SHAPE;
    if (!is_aligned(A, 16) || !is_aligned(qB, 16) || !is_aligned(Y, 16) || !is_aligned(sB, 2))
        return QZ_ERR_ALIGNMENT;
    return QZ_OK;
}

qz_status qz_gemm_w4a16_nvfp4(const uint16_t* A, const uint8_t* qB, const uint8_t* sB, const float* gB,
                              uint16_t* Y, int M, int N, int K, void* stream) {
    if (!gB) return QZ_ERR_INVALID_ARG;
    QZ_TRY(w4a16_fp4_checks(A, qB, sB, Y, M, N, K));
    QZ_TRY(device_check());
    return gemm_w4a16_fp4_launch(true, A, qB, sB, gB, Y, M, N, K, (cudaStream_t)stream);
}

qz_status qz_gemm_w4a16_mxfp4(const uint16_t* A, const uint8_t* qB, const uint8_t* eB,
                              uint16_t* Y, int M, int N, int K, void* stream) {
    QZ_TRY(w4a16_fp4_checks(A, qB, eB, Y, M, N, K));
    QZ_TRY(device_check());
    return gemm_w4a16_fp4_launch(false, A, qB, eB, nullptr, Y, M, N, K, (cudaStream_t)stream);
}

qz_status qz_col_amax(const void* x, qz_dtype xt, int64_t rows, int64_t cols, float* out, void* ws,
                      size_t ws_bytes, void* stream) {
    if (!x || !out || !dtype_ok(xt) || rows < 1 || cols < 1) return QZ_ERR_INVALID_ARG;
    if (cols % 8) return QZ_ERR_SHAPE;
    if (!is_aligned(x, 16) || !is_aligned(out, 16)) return QZ_ERR_ALIGNMENT;
    QZ_TRY(ws_ok(ws, ws_bytes, ws_col_amax(rows, cols)));
    QZ_TRY(device_check());
    return col_amax_launch(x, xt, rows, cols, out, ws, (cudaStream_t)stream);
}

qz_status qz_smooth_factors(const float* x_amax, const float* w_amax, int64_t n, float alpha, float* s,
                            void* stream) {
    if (!x_amax || !w_amax || !s || n < 1) return QZ_ERR_INVALID_ARG;
    if (alpha != 0.5f) return QZ_ERR_UNSUPPORTED;
    QZ_TRY(device_check());
    return smooth_factors_launch(x_amax, w_amax, n, s, (cudaStream_t)stream);
}

qz_status qz_quantize_int8_rows(const void* x, qz_dtype xt, int64_t rows, int64_t cols, const float* factors,
                                qz_smooth_op op, int8_t* codes, float* scales, float* dequant, void* stream) {
    if (!dtype_ok(xt) || rows < 0 || cols < 0) return QZ_ERR_INVALID_ARG;
    if (op != QZ_SMOOTH_NONE && op != QZ_SMOOTH_DIVIDE && op != QZ_SMOOTH_MULTIPLY) return QZ_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0) return QZ_OK;
    if (!x || !codes || !scales || (op != QZ_SMOOTH_NONE && !factors)) return QZ_ERR_INVALID_ARG;
    if (cols % 8) return QZ_ERR_SHAPE;
    if (!is_aligned(x, 16) || !is_aligned(codes, 8) || (factors && !is_aligned(factors, 16)) ||
        (dequant && !is_aligned(dequant, 16)))
        return QZ_ERR_ALIGNMENT;
    QZ_TRY(device_check());
    return int8_rows_launch(x, xt, rows, cols, factors, (int)op, codes, scales, dequant, (cudaStream_t)stream);
}

qz_status qz_gemm_int8(const int8_t* qA, const float* sA, const int8_t* qB, const float* sB, uint16_t* Y,
                       int M, int N, int K, void* stream) {
    if (!qA || !sA || !qB || !sB || !Y) return QZ_ERR_INVALID_ARG;
    if (M < 1 || N < 1 || K < 1) return QZ_ERR_INVALID_ARG;
    if (M % 128 || N % 256 || K % 64) return QZ_ERR_SHAPE;
    if (!is_aligned(qA, 16) || !is_aligned(qB, 16) || !is_aligned(sA, 16) || !is_aligned(sB, 16) ||
        !is_aligned(Y, 16))
        return QZ_ERR_ALIGNMENT;
    QZ_TRY(device_check());
    return gemm_int8_launch(qA, sA, qB, sB, Y, M, N, K, (cudaStream_t)stream);
}

qz_status qz_gemm_fp8_block_quant(const uint8_t* qA, const float* sA, const uint8_t* qB, const float* sB,
                                  uint16_t* Y, uint8_t* y_codes, float* y_scales, int M, int N, int K,
                                  void* stream) {
    if (!qA || !sA || !qB || !sB || !y_codes || !y_scales) return QZ_ERR_INVALID_ARG;
    if (M < 1 || N < 1 || K < 1) return QZ_ERR_INVALID_ARG;
    if (M % kFp8BlockM || N % kFp8BlockN || K % 128) return QZ_ERR_SHAPE;
    if (!is_aligned(qA, 16) || !is_aligned(qB, 16) || !is_aligned(sA, 16) || !is_aligned(sB, 16) ||
        (Y && !is_aligned(Y, 16)) || !is_aligned(y_codes, 16) || !is_aligned(y_scales, 4))
        return QZ_ERR_ALIGNMENT;
    QZ_TRY(device_check());
    return gemm_fp8_block_quant_launch(qA, sA, qB, sB, Y, y_codes, y_scales, M, N, K, (cudaStream_t)stream);
}

} // extern "C"
