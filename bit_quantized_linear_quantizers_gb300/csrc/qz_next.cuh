// qz_next.cuh -- launchers of the quantizer and GEMM variants beyond the four
// base formats (zero points, per-head and per-channel KV scales, weight-only
// FP4, SmoothQuant INT8 W8A8, the fused FP8 output quantization).
#pragma once

#include "qz_internal.cuh"

namespace qz {

size_t ws_kv_per_head(int64_t BH, int64_t L);
size_t ws_kv_channel_zp(int64_t BH, int64_t T, int64_t D);
size_t ws_col_amax(int64_t rows, int64_t cols);

qz_status int4_zp_launch(const void* w, qz_dtype wt, int64_t K, int64_t N, int64_t ldw, int32_t* qweight,
                         uint16_t* scale, uint8_t* zero, float* deq, cudaStream_t st);
qz_status kv_per_head_launch(const uint16_t* k, const uint16_t* v, int64_t BH, int64_t L, uint8_t* kc, uint8_t* vc,
                             float* ks, float* vs, qz_scale_mode mode, void* ws, cudaStream_t st);
qz_status kv_channel_zp_launch(const uint16_t* k, const uint16_t* v, int64_t B, int64_t H, int64_t T, int64_t D,
                               uint8_t* kc, uint8_t* vc, float* k_scale, float* k_zero, float* v_scale, void* ws,
                               cudaStream_t st);
qz_status col_amax_launch(const void* x, qz_dtype xt, int64_t rows, int64_t cols, float* out, void* ws,
                          cudaStream_t st);
qz_status smooth_factors_launch(const float* xm, const float* wm, int64_t n, float* s, cudaStream_t st);
qz_status int8_rows_launch(const void* x, qz_dtype xt, int64_t rows, int64_t cols, const float* f, int op,
                           int8_t* codes, float* scales, float* deq, cudaStream_t st);

qz_status gemm_w4a16_zp_launch(const uint16_t* A, const int32_t* qweight, const uint16_t* scale, const uint8_t* zero,
                               uint16_t* Y, int M, int N, int K, cudaStream_t st, bool early);
qz_status gemm_w4a16_fp4_launch(bool nv, const uint16_t* A, const uint8_t* qB, const uint8_t* sB, const float* gB,
                                uint16_t* Y, int M, int N, int K, cudaStream_t st);
qz_status gemm_int8_launch(const int8_t* qA, const float* sA, const int8_t* qB, const float* sB, uint16_t* Y, int M,
                           int N, int K, cudaStream_t st);
qz_status int8_error_read_and_clear();
qz_status gemm_fp8_block_quant_launch(const uint8_t* qA, const float* sA, const uint8_t* qB, const float* sB,
                                      uint16_t* Y, uint8_t* Yq, float* Yqs, int M, int N, int K, cudaStream_t st);

} // namespace qz
