// qz_api.cu -- the extern "C" entry points of libqz: host-side validation,
// workspace sizing and dispatch to the kernels. Nothing here allocates device
// memory; a call that fails validation enqueues nothing.
#include "qz_internal.cuh"
#include "qz_gemm.cuh"
#include "qz_next.cuh"

#include <algorithm>
#include <mutex>
#include <vector>

namespace qz {

namespace {
constexpr int kMaxDevices = 64;
int g_sms[kMaxDevices];
int g_arch_ok[kMaxDevices];   // 0 unknown, 1 sm_103, -1 other
std::mutex g_mu;

int current_device() {
    int d = 0;
    if (cudaGetDevice(&d) != cudaSuccess) return -1;
    return (d >= 0 && d < kMaxDevices) ? d : -1;
}
} // namespace

int num_sms() {
    const int d = current_device();
    if (d < 0) return 1;
    if (g_sms[d] == 0) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d);
        g_sms[d] = n > 0 ? n : 1;
    }
    return g_sms[d];
}

// The library carries sm_103a code only: refuse other devices up front.
qz_status device_check() {
    const int d = current_device();
    if (d < 0) return QZ_ERR_UNSUPPORTED;
    if (g_arch_ok[d] == 0) {
        std::lock_guard<std::mutex> lk(g_mu);
        int ma = 0, mi = 0;
        if (cudaDeviceGetAttribute(&ma, cudaDevAttrComputeCapabilityMajor, d) != cudaSuccess ||
            cudaDeviceGetAttribute(&mi, cudaDevAttrComputeCapabilityMinor, d) != cudaSuccess) {
            cudaGetLastError();
            return QZ_ERR_UNSUPPORTED;
        }
        g_arch_ok[d] = (ma == 10 && mi == 3) ? 1 : -1;
    }
    return g_arch_ok[d] == 1 ? QZ_OK : QZ_ERR_UNSUPPORTED;
}

// Bounded-wait self-test: one CTA waits on an mbarrier that nothing ever
// completes, with the same bounded wait every GEMM kernel uses but a short
// limit, so the wait runs out, records QZ_ERR_TIMEOUT in this word and the
// kernel returns normally.
__device__ unsigned int g_selftest_err;

__global__ void selftest_wait_kernel(uint32_t polls) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait_n(smem_u32(&bar), 0, &g_selftest_err, polls);
}

qz_status selftest_error_read_and_clear() {
    unsigned int v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_selftest_err, sizeof(v)) != cudaSuccess) return QZ_ERR_CUDA;
    if (v && cudaMemcpyToSymbol(g_selftest_err, &z, sizeof(z)) != cudaSuccess) return QZ_ERR_CUDA;
    return v ? QZ_ERR_TIMEOUT : QZ_OK;
}

qz_status device_error_read_and_clear() {
    // read and clear every word, report the first error found
    const qz_status s[6] = {w4a16_error_read_and_clear(), w4a16_tc_error_read_and_clear(),
                            fp8_block_error_read_and_clear(), fp4_error_read_and_clear(),
                            int8_error_read_and_clear(), selftest_error_read_and_clear()};
    for (qz_status v : s)
        if (v != QZ_OK) return v;
    return QZ_OK;
}

qz_status launch_status() {
    return cudaGetLastError() == cudaSuccess ? QZ_OK : QZ_ERR_CUDA;
}

bool is_aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

// Raises a kernel's dynamic shared-memory limit on the current device to at
// least `bytes`. One lock covers every kernel and device, so concurrent host
// threads neither race on the record nor lower a limit another thread raised.
qz_status opt_in_smem(const void* fn, int bytes) {
    struct Entry { const void* fn; int dev; int bytes; };
    static Entry done[256];
    static int ndone = 0;
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return QZ_ERR_CUDA;
    std::lock_guard<std::mutex> lk(mu);
    Entry* e = nullptr;
    for (int i = 0; i < ndone; i++)
        if (done[i].fn == fn && done[i].dev == dev) e = &done[i];
    if (e && e->bytes >= bytes) return QZ_OK;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) {
        cudaGetLastError();
        return QZ_ERR_CUDA;
    }
    if (!e) {
        if (ndone == 256) return QZ_OK;          // record full: the attribute is set, just not cached
        e = &done[ndone++];
        e->fn = fn;
        e->dev = dev;
    }
    e->bytes = bytes;
    return QZ_OK;
}

namespace {
struct StreamInt4 {
    int dev;
    cudaStream_t st;
    Int4Writes w;
};
std::mutex g_int4_mu;
std::vector<StreamInt4> g_int4;         // one entry per device and stream an INT4 quantizer ran on
uint64_t g_int4_gen;

StreamInt4* find_int4(int dev, cudaStream_t st) {
    if (st == cudaStreamLegacy) st = nullptr;   // two handles of the legacy default stream, one key
    for (StreamInt4& e : g_int4)
        if (e.dev == dev && e.st == st) return &e;
    return nullptr;
}
} // namespace

void note_int4_writes(cudaStream_t st, const Span* w, int n) {
    const int dev = current_device();
    std::lock_guard<std::mutex> lk(g_int4_mu);
    StreamInt4* e = find_int4(dev, st);
    if (!e) {
        g_int4.push_back(StreamInt4{dev, st == cudaStreamLegacy ? nullptr : st, {}});
        e = &g_int4.back();
    }
    e->w.gen = ++g_int4_gen;
    e->w.n = std::min(n, 3);
    for (int i = 0; i < e->w.n; i++) e->w.s[i] = w[i];
}

Int4Writes int4_writes(cudaStream_t st) {
    const int dev = current_device();
    std::lock_guard<std::mutex> lk(g_int4_mu);
    const StreamInt4* e = find_int4(dev, st);
    return e ? e->w : Int4Writes{0, 0, {}};
}

void clear_int4_writes(cudaStream_t st, uint64_t gen) {
    const int dev = current_device();
    std::lock_guard<std::mutex> lk(g_int4_mu);
    StreamInt4* e = find_int4(dev, st);
    if (e && e->w.gen == gen) e->w.n = 0;
}

} // namespace qz

using namespace qz;

static size_t elem_size(qz_dtype t) { return t == QZ_F32 ? 4 : 2; }
static bool dtype_ok(qz_dtype t) { return t == QZ_F32 || t == QZ_BF16; }

extern "C" {

const char* qz_status_string(qz_status s) {
    switch (s) {
    case QZ_OK: return "QZ_OK";
    case QZ_ERR_INVALID_ARG: return "QZ_ERR_INVALID_ARG: null pointer, bad enum or negative size";
    case QZ_ERR_SHAPE: return "QZ_ERR_SHAPE: size not divisible as required or out of range";
    case QZ_ERR_ALIGNMENT: return "QZ_ERR_ALIGNMENT: pointer or leading dimension misaligned";
    case QZ_ERR_UNSUPPORTED: return "QZ_ERR_UNSUPPORTED: no sm_103 device or path unavailable";
    case QZ_ERR_CUDA: return "QZ_ERR_CUDA: CUDA runtime or launch error";
    case QZ_ERR_TIMEOUT: return "QZ_ERR_TIMEOUT: a bounded device wait gave up";
    case QZ_ERR_WORKSPACE: return "QZ_ERR_WORKSPACE: workspace missing or too small";
    }
    return "QZ_ERR_UNKNOWN";
}

size_t qz_workspace_size(qz_op op, int64_t d0, int64_t d1, int64_t d2) {
    switch (op) {
    case QZ_OP_QUANTIZE_FP8: return d2 == QZ_FP8_PER_TENSOR ? ws_quantize_fp8_tensor(d0, d1) : 0;
    case QZ_OP_QUANTIZE_NVFP4: return ws_quantize_nvfp4(d0, d1);
    case QZ_OP_KV_WRITE_FP8: return ws_kv_write(d0);
    case QZ_OP_GEMM_W4A16: return ws_gemm_w4a16((int)d0, (int)d1, (int)d2);
    case QZ_OP_GEMM_FP8_BLOCK: return ws_gemm_fp8_block((int)d0, (int)d1, (int)d2);
    case QZ_OP_GEMM_NVFP4: return ws_gemm_fp4((int)d0, (int)d1, (int)d2);
    case QZ_OP_GEMM_MXFP4: return ws_gemm_fp4((int)d0, (int)d1, (int)d2);
    case QZ_OP_GEMM_NVFP4_GROUPED:
        return d0 >= 1 && d0 <= kNvfp4MaxProblems && d1 >= 1 && d1 <= (1 << 24) ? ws_gemm_nvfp4_grouped((int)d0, (int)d1)
                                                                                 : 0;
    case QZ_OP_QUANTIZE_NVFP4_GROUPED:
        return d0 >= 1 && d0 <= kNvfp4GroupMax ? ws_quantize_nvfp4_grouped((int)d0) : 0;
    case QZ_OP_KV_WRITE_FP8_PER_HEAD: return d0 >= 1 && d1 >= 1 ? ws_kv_per_head(d0, d1) : 0;
    case QZ_OP_KV_WRITE_FP8_CHANNEL_ZP: return d0 >= 1 && d1 >= 1 && d2 >= 1 ? ws_kv_channel_zp(d0, d1, d2) : 0;
    case QZ_OP_COL_AMAX: return d0 >= 1 && d1 >= 1 ? ws_col_amax(d0, d1) : 0;
    case QZ_OP_PREPARE_FP4_SCALES:
        return d0 >= 1 && d0 <= (1 << 24) && d1 >= 1 && d1 <= (1 << 24) ? prepared_fp4_scale_bytes((int)d0, (int)d1, d2 != 0)
                                                                         : 0;
    }
    return 0;
}

qz_status qz_device_error(void) { return device_error_read_and_clear(); }

qz_status qz_selftest_bounded_wait(uint32_t polls, void* stream) {
    if (polls < 1 || polls > (1u << 20)) return QZ_ERR_INVALID_ARG;
    QZ_TRY(device_check());
    selftest_wait_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(polls);
    return launch_status();
}

qz_status qz_quantize_fp8(const void* x, qz_dtype xt, int64_t rows, int64_t cols, int64_t ldx,
                          qz_fp8_gran gran, uint8_t* codes, float* scales, float* dequant,
                          void* ws, size_t ws_bytes, void* stream) {
    if (!dtype_ok(xt) || gran < QZ_FP8_PER_TENSOR || gran > QZ_FP8_GROUP_1x128) return QZ_ERR_INVALID_ARG;
    if (rows < 0 || cols < 0 || ldx < cols) return QZ_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0) return gran == QZ_FP8_PER_TENSOR ? QZ_ERR_SHAPE : QZ_OK;
    if (!x || !codes || !scales) return QZ_ERR_INVALID_ARG;
    const bool vec = is_aligned(x, 16) && ((size_t)ldx * elem_size(xt)) % 16 == 0 && cols % 8 == 0;
    if (gran == QZ_FP8_BLOCK_128x128 || gran == QZ_FP8_GROUP_1x128) {
        if (cols % 128) return QZ_ERR_SHAPE;
        if (gran == QZ_FP8_BLOCK_128x128 && rows > 128 && rows % 128) return QZ_ERR_SHAPE;
        if (!vec) return QZ_ERR_ALIGNMENT;
    }
    if (vec && (!is_aligned(codes, 8) || (dequant && !is_aligned(dequant, 16)))) return QZ_ERR_ALIGNMENT;
    if (gran == QZ_FP8_PER_TENSOR) {
        if (!ws) return QZ_ERR_WORKSPACE;
        if (ws_bytes < ws_quantize_fp8_tensor(rows, cols) || !is_aligned(ws, 4)) return QZ_ERR_WORKSPACE;
    }
    QZ_TRY(device_check());
    return quantize_fp8_launch(x, xt, rows, cols, ldx, gran, codes, scales, dequant, ws, ws_bytes,
                               (cudaStream_t)stream);
}

static qz_status fp4_common_checks(const void* x, qz_dtype xt, int64_t rows, int64_t cols, int64_t ldx,
                                   int block, const uint8_t* codes, const void* scales, const float* deq) {
    if (!dtype_ok(xt)) return QZ_ERR_INVALID_ARG;
    if (rows < 0 || cols < 0 || ldx < cols) return QZ_ERR_INVALID_ARG;
    if (cols % block) return QZ_ERR_SHAPE;
    if (rows == 0 || cols == 0) return QZ_OK;
    if (!x || !codes || !scales) return QZ_ERR_INVALID_ARG;
    if (!is_aligned(x, 16) || ((size_t)ldx * elem_size(xt)) % 16) return QZ_ERR_ALIGNMENT;
    if (!is_aligned(codes, 4) || (deq && !is_aligned(deq, 16))) return QZ_ERR_ALIGNMENT;
    return QZ_OK;
}

qz_status qz_quantize_mxfp4(const void* x, qz_dtype xt, int64_t rows, int64_t cols, int64_t ldx,
                            uint8_t* codes, uint8_t* scale_e8m0, float* dequant, void* stream) {
    QZ_TRY(fp4_common_checks(x, xt, rows, cols, ldx, 32, codes, scale_e8m0, dequant));
    if (rows == 0 || cols == 0) return QZ_OK;
    QZ_TRY(device_check());
    return quantize_mxfp4_launch(x, xt, rows, cols, ldx, codes, scale_e8m0, dequant, (cudaStream_t)stream);
}

qz_status qz_quantize_nvfp4(const void* x, qz_dtype xt, int64_t rows, int64_t cols, int64_t ldx,
                            uint8_t* codes, uint8_t* scale_e4m3, float* global_scale,
                            const float* global_amax_in, float* dequant,
                            void* ws, size_t ws_bytes, void* stream) {
    QZ_TRY(fp4_common_checks(x, xt, rows, cols, ldx, 16, codes, scale_e4m3, dequant));
    if (rows == 0 || cols == 0) return global_amax_in ? QZ_OK : QZ_ERR_SHAPE;
    if (!global_scale) return QZ_ERR_INVALID_ARG;
    if (!global_amax_in) {
        if (!ws) return QZ_ERR_WORKSPACE;
        if (ws_bytes < ws_quantize_nvfp4(rows, cols) || !is_aligned(ws, 4)) return QZ_ERR_WORKSPACE;
    }
    QZ_TRY(device_check());
    return quantize_nvfp4_launch(x, xt, rows, cols, ldx, codes, scale_e4m3, global_scale, global_amax_in,
                                 dequant, ws, ws_bytes, (cudaStream_t)stream);
}

qz_status qz_quantize_int4_g128(const void* w, qz_dtype wt, int64_t K, int64_t N, int64_t ldw,
                                int32_t* qweight, uint16_t* scale_bf16, float* dequant, void* stream) {
    if (!dtype_ok(wt)) return QZ_ERR_INVALID_ARG;
    if (K < 0 || N < 0 || ldw < N) return QZ_ERR_INVALID_ARG;
    if (K % 128 || N % 64) return QZ_ERR_SHAPE;
    if (K == 0 || N == 0) return QZ_OK;
    if (!w || !qweight || !scale_bf16) return QZ_ERR_INVALID_ARG;
    if (!is_aligned(w, 16) || ((size_t)ldw * elem_size(wt)) % 16) return QZ_ERR_ALIGNMENT;
    if (!is_aligned(qweight, 16) || !is_aligned(scale_bf16, 16) || (dequant && !is_aligned(dequant, 16)))
        return QZ_ERR_ALIGNMENT;
    QZ_TRY(device_check());
    QZ_TRY(quantize_int4_launch(w, wt, K, N, ldw, qweight, scale_bf16, dequant, (cudaStream_t)stream));
    const Span out[2] = {{qweight, (size_t)K * N / 2}, {scale_bf16, (size_t)K * N / 64}};
    note_int4_writes((cudaStream_t)stream, out, 2);
    return QZ_OK;
}

qz_status qz_kv_write_fp8(const uint16_t* k, const uint16_t* v, int B, int H, int T, int D,
                          uint8_t* k_codes, uint8_t* v_codes, float* k_scale, float* v_scale,
                          qz_scale_mode mode, void* ws, size_t ws_bytes, void* stream) {
    if (mode != QZ_SCALE_COMPUTE && mode != QZ_SCALE_GIVEN) return QZ_ERR_INVALID_ARG;
    if (B < 0 || H < 0 || T < 0 || D < 0) return QZ_ERR_INVALID_ARG;
    const int64_t n = (int64_t)B * H * T * D;
    if (n == 0) return mode == QZ_SCALE_GIVEN ? QZ_OK : QZ_ERR_SHAPE;
    if (!k || !v || !k_codes || !v_codes || !k_scale || !v_scale) return QZ_ERR_INVALID_ARG;
    if (n % 8) return QZ_ERR_SHAPE;
    if (!is_aligned(k, 16) || !is_aligned(v, 16) || !is_aligned(k_codes, 8) || !is_aligned(v_codes, 8))
        return QZ_ERR_ALIGNMENT;
    if (mode == QZ_SCALE_COMPUTE) {
        if (!ws) return QZ_ERR_WORKSPACE;
        if (ws_bytes < ws_kv_write(n) || !is_aligned(ws, 4)) return QZ_ERR_WORKSPACE;
    }
    QZ_TRY(device_check());
    return kv_write_launch(k, v, n, k_codes, v_codes, k_scale, v_scale, mode, ws, ws_bytes,
                           (cudaStream_t)stream);
}

qz_status qz_gemm_w4a16(const uint16_t* A, const int32_t* qweight, const uint16_t* scale_bf16,
                        uint16_t* Y, int M, int N, int K, void* ws, size_t ws_bytes, void* stream) {
    qz_w4a16_problem p{A, qweight, scale_bf16, Y, M, N, K};
    return qz_gemm_w4a16_grouped(&p, 1, ws, ws_bytes, stream);
}

qz_status qz_gemm_w4a16_grouped(const qz_w4a16_problem* problems, int count, void* ws, size_t ws_bytes,
                                void* stream) {
    if (!problems || count < 1 || count > kW4A16MaxProblems) return QZ_ERR_INVALID_ARG;
    int mmax = 0, kmax = 0;
    int64_t nsum = 0;
    for (int i = 0; i < count; i++) {
        const qz_w4a16_problem& p = problems[i];
        if (!p.A || !p.qweight || !p.scale_bf16 || !p.Y) return QZ_ERR_INVALID_ARG;
        if (p.M < 1 || p.N < 1 || p.K < 1) return QZ_ERR_INVALID_ARG;
        if (p.M > 64 || p.K % 128 || p.N % 64) return QZ_ERR_SHAPE;
        if (!is_aligned(p.A, 16) || !is_aligned(p.qweight, 16) || !is_aligned(p.scale_bf16, 16) ||
            !is_aligned(p.Y, 16))
            return QZ_ERR_ALIGNMENT;
        mmax = p.M > mmax ? p.M : mmax;
        kmax = p.K > kmax ? p.K : kmax;
        nsum += p.N;
    }
    const size_t need = ws_gemm_w4a16(mmax, (int)nsum, kmax);
    if (need && (!ws || ws_bytes < need || !is_aligned(ws, 16))) return QZ_ERR_WORKSPACE;
    QZ_TRY(device_check());
    // Weights an INT4 quantizer call may still be writing: launch after all
    // earlier work on the stream instead of under dependent launch.
    const Int4Writes rec = int4_writes((cudaStream_t)stream);
    bool early = true;
    for (int i = 0; i < count && rec.n && early; i++) {
        const qz_w4a16_problem& p = problems[i];
        early = !w4a16_reads_in_flight(rec, p.qweight, p.scale_bf16, nullptr, p.N, p.K);
    }
    QZ_TRY(gemm_w4a16_launch(problems, count, ws, ws_bytes, (cudaStream_t)stream, early));
    if (!early) clear_int4_writes((cudaStream_t)stream, rec.gen);
    return QZ_OK;
}

qz_status qz_gemm_fp8_block(const uint8_t* qA, const float* sA, const uint8_t* qB, const float* sB,
                            uint16_t* Y, int M, int N, int K, void* ws, size_t ws_bytes, void* stream) {
    if (!qA || !sA || !qB || !sB || !Y) return QZ_ERR_INVALID_ARG;
    if (M < 1 || N < 1 || K < 1) return QZ_ERR_INVALID_ARG;
    if (M % kFp8BlockM || N % kFp8BlockN || K % 128) return QZ_ERR_SHAPE;
    if (!is_aligned(qA, 16) || !is_aligned(qB, 16) || !is_aligned(sA, 16) || !is_aligned(sB, 16) ||
        !is_aligned(Y, 16))
        return QZ_ERR_ALIGNMENT;
    const size_t need = ws_gemm_fp8_block(M, N, K);
    if (need && (!ws || ws_bytes < need || !is_aligned(ws, 16))) return QZ_ERR_WORKSPACE;
    QZ_TRY(device_check());
    return gemm_fp8_block_launch(qA, sA, qB, sB, Y, M, N, K, ws, ws_bytes, (cudaStream_t)stream);
}

static qz_status fp4_gemm_checks(const void* qA, const void* sA, const void* qB, const void* sB,
                                 const void* Y, int M, int N, int K, void* ws, size_t ws_bytes) {
    if (!qA || !sA || !qB || !sB || !Y) return QZ_ERR_INVALID_ARG;
    if (M < 1 || N < 1 || K < 1) return QZ_ERR_INVALID_ARG;
    if (M % kFp4BlockM || N % kFp4BlockN || K % kFp4BlockK) return QZ_ERR_SHAPE;
    if (!is_aligned(qA, 16) || !is_aligned(qB, 16) || !is_aligned(sA, 16) || !is_aligned(sB, 16) ||
        !is_aligned(Y, 16))
        return QZ_ERR_ALIGNMENT;
    const size_t need = ws_gemm_fp4(M, N, K);
    if (need && (!ws || ws_bytes < need || !is_aligned(ws, 16))) return QZ_ERR_WORKSPACE;
    return QZ_OK;
}

qz_status qz_gemm_nvfp4(const uint8_t* qA, const uint8_t* sA, const float* gA,
                        const uint8_t* qB, const uint8_t* sB, const float* gB,
                        uint16_t* Y, int M, int N, int K, void* ws, size_t ws_bytes, void* stream) {
    if (!gA || !gB) return QZ_ERR_INVALID_ARG;
    QZ_TRY(fp4_gemm_checks(qA, sA, qB, sB, Y, M, N, K, ws, ws_bytes));
    QZ_TRY(device_check());
    return gemm_fp4_launch(true, qA, sA, gA, qB, sB, gB, Y, M, N, K, ws, ws_bytes, (cudaStream_t)stream);
}

qz_status qz_gemm_nvfp4_quant(const uint8_t* qA, const uint8_t* sA, const float* gA,
                              const uint8_t* qB, const uint8_t* sB, const float* gB,
                              const float* y_amax, uint8_t* y_codes, uint8_t* y_scales, float* y_global,
                              int M, int N, int K, void* ws, size_t ws_bytes, void* stream) {
    if (!gA || !gB || !y_amax || !y_codes || !y_scales || !y_global) return QZ_ERR_INVALID_ARG;
    if (!is_aligned(y_scales, 8) || !is_aligned(y_amax, 4) || !is_aligned(y_global, 4)) return QZ_ERR_ALIGNMENT;
    // the bf16 output is not written: Y's checks run on the codes pointer
    QZ_TRY(fp4_gemm_checks(qA, sA, qB, sB, y_codes, M, N, K, ws, ws_bytes));
    QZ_TRY(device_check());
    const qz_fp4_out yq{y_codes, y_scales, y_amax, y_global};
    return gemm_fp4_launch_q(true, qA, sA, gA, qB, sB, gB, nullptr, &yq, M, N, K, ws, ws_bytes, (cudaStream_t)stream);
}

qz_status qz_gemm_mxfp4_quant(const uint8_t* qA, const uint8_t* eA, const uint8_t* qB, const uint8_t* eB,
                              uint8_t* y_codes, uint8_t* y_e8m0, int M, int N, int K,
                              void* ws, size_t ws_bytes, void* stream) {
    if (!y_codes || !y_e8m0) return QZ_ERR_INVALID_ARG;
    if (!is_aligned(y_e8m0, 4)) return QZ_ERR_ALIGNMENT;
    // the bf16 output is not written: Y's checks run on the codes pointer
    QZ_TRY(fp4_gemm_checks(qA, eA, qB, eB, y_codes, M, N, K, ws, ws_bytes));
    QZ_TRY(device_check());
    const qz_fp4_out yq{y_codes, y_e8m0, nullptr, nullptr};
    return gemm_fp4_launch_q(false, qA, eA, nullptr, qB, eB, nullptr, nullptr, &yq, M, N, K, ws, ws_bytes,
                             (cudaStream_t)stream);
}

qz_status qz_gemm_mxfp4(const uint8_t* qA, const uint8_t* eA, const uint8_t* qB, const uint8_t* eB,
                        uint16_t* Y, int M, int N, int K, void* ws, size_t ws_bytes, void* stream) {
    QZ_TRY(fp4_gemm_checks(qA, eA, qB, eB, Y, M, N, K, ws, ws_bytes));
    QZ_TRY(device_check());
    return gemm_fp4_launch(false, qA, eA, nullptr, qB, eB, nullptr, Y, M, N, K, ws, ws_bytes,
                           (cudaStream_t)stream);
}

qz_status qz_quantize_nvfp4_grouped(const qz_nvfp4_tensor* tensors, int count, qz_dtype xt, void* ws,
                                    size_t ws_bytes, void* stream) {
    if (!tensors || count < 1 || count > kNvfp4GroupMax || !dtype_ok(xt)) return QZ_ERR_INVALID_ARG;
    for (int i = 0; i < count; i++) {
        const qz_nvfp4_tensor& t = tensors[i];
        if (!t.x || !t.codes || !t.scale_e4m3 || !t.global_scale) return QZ_ERR_INVALID_ARG;
        if (t.rows < 1 || t.cols < 1) return QZ_ERR_INVALID_ARG;
        if (t.cols % 16) return QZ_ERR_SHAPE;
        if (!is_aligned(t.x, 16) || !is_aligned(t.codes, 4)) return QZ_ERR_ALIGNMENT;
    }
    if (!ws || ws_bytes < ws_quantize_nvfp4_grouped(count) || !is_aligned(ws, 4)) return QZ_ERR_WORKSPACE;
    QZ_TRY(device_check());
    return quantize_nvfp4_grouped_launch(tensors, count, xt, ws, (cudaStream_t)stream);
}

qz_status qz_prepare_fp4_scales(const uint8_t* scales, int rows, int K, int nv, uint8_t* out, void* stream) {
    if (!scales || !out || (nv != 0 && nv != 1)) return QZ_ERR_INVALID_ARG;
    if (rows < 1 || K < 1) return QZ_ERR_INVALID_ARG;
    if (K % kFp4BlockK) return QZ_ERR_SHAPE;
    if (!is_aligned(scales, 4) || !is_aligned(out, 16)) return QZ_ERR_ALIGNMENT;
    QZ_TRY(device_check());
    return prepare_fp4_scales_launch(scales, rows, K, nv == 1, out, (cudaStream_t)stream);
}

qz_status qz_gemm_nvfp4_grouped(const qz_nvfp4_problem* problems, int count, void* ws, size_t ws_bytes,
                                void* stream) {
    if (!problems || count < 1 || count > kNvfp4MaxProblems) return QZ_ERR_INVALID_ARG;
    int kmax = 0;
    for (int i = 0; i < count; i++) {
        const qz_nvfp4_problem& p = problems[i];
        if (!p.qA || !p.sA || !p.gA || !p.qB || !p.sB_prepared || !p.gB || !p.Y) return QZ_ERR_INVALID_ARG;
        if (p.M < 1 || p.N < 1 || p.K < 1) return QZ_ERR_INVALID_ARG;
        if (p.M > kFp4BlockM || p.N % kFp4BlockN || p.K % kFp4BlockK) return QZ_ERR_SHAPE;
        if (!is_aligned(p.qA, 16) || !is_aligned(p.qB, 16) || !is_aligned(p.sB_prepared, 16) ||
            !is_aligned(p.Y, 16) || !is_aligned(p.sA, 4))
            return QZ_ERR_ALIGNMENT;
        kmax = std::max(kmax, p.K);
    }
    const size_t need = ws_gemm_nvfp4_grouped(count, kmax);
    if (!ws || ws_bytes < need || !is_aligned(ws, 16)) return QZ_ERR_WORKSPACE;
    QZ_TRY(device_check());
    return gemm_nvfp4_grouped_launch(problems, count, ws, ws_bytes, (cudaStream_t)stream);
}

// Same computation as qz_gemm_nvfp4; the scratch is the library's fixed array
// (see nvfp4_noalloc_scratch) instead of a caller workspace. No allocation.
qz_status qz_gemm_nvfp4_noalloc(const uint8_t* qA, const uint8_t* sA, const float* gA,
                                const uint8_t* qB, const uint8_t* sB, const float* gB,
                                uint16_t* Y, int M, int N, int K, void* stream) {
    if (!gA || !gB || !qA || !sA || !qB || !sB || !Y) return QZ_ERR_INVALID_ARG;
    if (M < 1 || N < 1 || K < 1) return QZ_ERR_INVALID_ARG;
    if (M % kFp4BlockM || N % kFp4BlockN || K % kFp4BlockK) return QZ_ERR_SHAPE;
    if (!is_aligned(qA, 16) || !is_aligned(qB, 16) || !is_aligned(sA, 16) || !is_aligned(sB, 16) ||
        !is_aligned(Y, 16))
        return QZ_ERR_ALIGNMENT;
    const size_t need = ws_gemm_fp4(M, N, K);
    if (need > QZ_NVFP4_NOALLOC_SCRATCH_BYTES) return QZ_ERR_SHAPE;   // beyond the fixed scratch
    QZ_TRY(device_check());
    void* scratch = nullptr;
    QZ_TRY(nvfp4_noalloc_scratch(&scratch));
    return gemm_fp4_launch(true, qA, sA, gA, qB, sB, gB, Y, M, N, K, scratch, QZ_NVFP4_NOALLOC_SCRATCH_BYTES,
                           (cudaStream_t)stream);
}

} // extern "C"
