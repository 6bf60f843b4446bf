// qz_gemm.cuh -- GEMM launchers and the PTX helpers they share (mbarrier,
// bulk copies, bounded waits).
#pragma once

#include "qz_internal.cuh"

namespace qz {

constexpr int kW4A16MaxProblems = 256;
constexpr int kFp8BlockM = 128, kFp8BlockN = 256;
constexpr int kFp4BlockM = 128, kFp4BlockN = 256, kFp4BlockK = 256;

size_t ws_gemm_w4a16(int M, int N, int K);
size_t ws_gemm_fp8_block(int M, int N, int K);
size_t ws_gemm_fp4(int M, int N, int K);

// early: launch under programmatic dependent launch (the kernels read their
// weights before waiting for the previous kernel on the stream); false: after
// all earlier work on the stream.
qz_status gemm_w4a16_launch(const qz_w4a16_problem* problems, int count, void* ws, size_t ws_bytes,
                            cudaStream_t st, bool early);
qz_status gemm_fp8_block_launch(const uint8_t* qA, const float* sA, const uint8_t* qB, const float* sB,
                                uint16_t* Y, int M, int N, int K, void* ws, size_t ws_bytes, cudaStream_t st);
qz_status gemm_fp8_block_quant_launch(const uint8_t* qA, const float* sA, const uint8_t* qB, const float* sB,
                                      uint16_t* Y, uint8_t* Yq, float* Yqs, int M, int N, int K, cudaStream_t st);
size_t ws_gemm_nvfp4_grouped(int count, int kmax);
size_t prepared_fp4_scale_bytes(int rows, int K, bool nv);
qz_status gemm_nvfp4_grouped_launch(const qz_nvfp4_problem* problems, int count, void* ws, size_t ws_bytes,
                                    cudaStream_t st);
qz_status prepare_fp4_scales_launch(const uint8_t* scales, int rows, int K, bool nv, uint8_t* out,
                                    cudaStream_t st);
constexpr int kNvfp4MaxProblems = 256;
qz_status gemm_fp4_launch(bool nv, const uint8_t* qA, const uint8_t* sA, const float* gA,
                          const uint8_t* qB, const uint8_t* sB, const float* gB, uint16_t* Y,
                          int M, int N, int K, void* ws, size_t ws_bytes, cudaStream_t st);
// FP4 output of qz_gemm_nvfp4_quant / qz_gemm_mxfp4_quant: codes [M, N/2];
// scales E4M3 [M, N/16] (NVFP4) or E8M0 [M, N/32] (MXFP4); NVFP4 only: the
// caller's tensor amax and the tensor scale g computed from it.
struct qz_fp4_out {
    uint8_t* codes;
    uint8_t* scales;
    const float* amax;
    float* g;
};
// As gemm_fp4_launch; with yq the output is quantized, in the GEMM's own
// format, instead of written as bf16 (Y unused).
qz_status gemm_fp4_launch_q(bool nv, const uint8_t* qA, const uint8_t* sA, const float* gA,
                            const uint8_t* qB, const uint8_t* sB, const float* gB, uint16_t* Y,
                            const qz_fp4_out* yq, int M, int N, int K, void* ws, size_t ws_bytes,
                            cudaStream_t st);

// Device error words of the GEMM translation units (read and cleared by
// qz_device_error). Each returns QZ_OK, QZ_ERR_TIMEOUT or QZ_ERR_CUDA.
qz_status w4a16_error_read_and_clear();
qz_status w4a16_tc_error_read_and_clear();
// tcgen05 W4A16 for 17..64 tokens (mt = 32 or 64: the token count padded)
qz_status w4a16_tc_launch(const qz_w4a16_problem* problems, int count, int mt, cudaStream_t st, bool early);
qz_status fp8_block_error_read_and_clear();
qz_status fp4_error_read_and_clear();
qz_status selftest_error_read_and_clear();
qz_status device_error_read_and_clear();
qz_status device_check();

// Device address of the fixed scratch array of qz_gemm_nvfp4_noalloc on the
// current device (looked up on first use per device).
qz_status nvfp4_noalloc_scratch(void** out);

// ------------------------------------------------------------ PTX helpers

// A bounded spin-wait gives up after this many polls (seconds of waiting),
// records QZ_ERR_TIMEOUT in the translation unit's error word and returns
// false, so no kernel can hang the GPU on a lost arrival.
constexpr uint32_t kWaitLimit = 1u << 24;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("{ .reg .b64 st; mbarrier.arrive.shared::cta.b64 st, [%0]; }" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("{ .reg .b64 st; mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1; }"
                 ::"r"(bar), "r"(bytes) : "memory");
}

// One potentially blocking test of the phase. The explicit suspend-time hint
// (in ns) replaces the system-dependent limit: measured, every hint from 5 to
// 1000 ns woke the waiting threads sooner than the default (the tcgen05 W4A16
// kernel at 64 tokens: 24.4 -> 22.1 us; its hand-off skeleton 14.6 -> 10.0 us).
constexpr uint32_t kSuspendHintNs = 20;
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3; selp.u32 %0, 1, 0, p; }"
                 : "=r"(ok) : "r"(bar), "r"(parity), "r"(kSuspendHintNs) : "memory");
    return ok != 0;
}

// The same test with the system-dependent time limit (measured slightly faster
// for warps that wait on TMA bytes rather than on another warp's hand-off).
__device__ __forceinline__ bool mbar_try_wait_default(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
                 : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}

// Waits for phase `parity` of the mbarrier for at most `limit` polls; false (and
// *err set to QZ_ERR_TIMEOUT) when the limit runs out.
template <bool HINT = true>
__device__ __forceinline__ bool mbar_wait_n(uint32_t bar, uint32_t parity, unsigned int* err, uint32_t limit) {
    for (uint32_t i = 0; i < limit; i++)
        if (HINT ? mbar_try_wait(bar, parity) : mbar_try_wait_default(bar, parity)) return true;
    atomicExch(err, (unsigned int)QZ_ERR_TIMEOUT);
    return false;
}

// Waits for phase `parity` of the mbarrier; false (and *err set) on timeout.
template <bool HINT = true>
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, unsigned int* err) {
    return mbar_wait_n<HINT>(bar, parity, err, kWaitLimit);
}

// 1-D bulk copy global -> shared through the TMA unit, completing on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

} // namespace qz
