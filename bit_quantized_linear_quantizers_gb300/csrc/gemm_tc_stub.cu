// Placeholder translation unit for the tcgen05 GEMMs until their kernels land.
#include "qz_gemm.cuh"
namespace qz {
size_t ws_gemm_fp8_block(int, int, int) { return 0; }
size_t ws_gemm_fp4(int, int, int) { return 0; }
qz_status gemm_fp8_block_launch(const uint8_t*, const float*, const uint8_t*, const float*, uint16_t*, int, int,
                                int, void*, size_t, cudaStream_t) { return QZ_ERR_UNSUPPORTED; }
qz_status gemm_fp4_launch(bool, const uint8_t*, const uint8_t*, const float*, const uint8_t*, const uint8_t*,
                          const float*, uint16_t*, int, int, int, void*, size_t, cudaStream_t) { return QZ_ERR_UNSUPPORTED; }
qz_status fp8_block_error_read_and_clear() { return QZ_OK; }
qz_status fp4_error_read_and_clear() { return QZ_OK; }
qz_status device_error_read_and_clear() {
    qz_status s = w4a16_error_read_and_clear();
    if (s != QZ_OK) return s;
    s = fp8_block_error_read_and_clear();
    if (s != QZ_OK) return s;
    return fp4_error_read_and_clear();
}
}
