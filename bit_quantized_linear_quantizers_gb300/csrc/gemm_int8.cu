// gemm_int8.cu -- INT8 W8A8 GEMM, per-token activation scales times
// per-output-channel weight scales ("量化部署实战", 格式速查: W8A8 INT8, per
// channel + per token, usually with SmoothQuant; "量化：让每一步搬更少的字节",
// 路线二):
//   Y[i, j] = bf16( sA[i] * sB[j] * sum_k qA[i, k] * qB[j, k] )
// with qA int8 [M, K], qB int8 [N, K] (B^T, K-major), fp32 scales.
//
// This GPU has no INT8 kind of tcgen05.mma, and its legacy INT8 mma.sync path
// runs at a quarter of the bf16 mma.sync rate. Every int8 value is an exact
// fp16 integer and every product of two is exact in fp32, so the kernel
// widens the codes to fp16 on chip and runs the fp16 tensor cores
// (tcgen05.mma kind::f16, fp32 accumulator in TMEM). Each 128 x 256 x 64 step
// sums at most 64 products of magnitude <= 2^14, and the accumulator stays an
// exact integer while |sum| < 2^24; beyond that (far outside realistic
// activations) it rounds like any fp32 accumulation.
//
// Design (one CTA per SM, persistent over 256 x 256 output tiles, M fastest):
// the conversion, not the tensor core, sets the rate, so each converted B
// stage serves two 128-row MMA halves (a third less conversion per product
// than 128-row tiles).
//  warp 0      TMA producer: 64-byte-wide int8 boxes of A (256 rows) and B
//              (256 rows) into a 3-stage ring.
//  warps 2-9   converters: each int8 stage becomes an fp16 operand stage in the
//              128-byte-swizzled K-major layout the tensor core reads (16-byte
//              chunk c of row r at chunk c ^ (r & 7)); 2-stage ring.
//  warp 1      MMA issuer (one thread): per stage 2 x 4 kind::f16 MMAs (M=128,
//              N=256, K=16), one TMEM accumulator per 128-row half.
//  warps 10-17 epilogue: each thread owns one row of each half and 128
//              columns; loads the accumulators (tcgen05.ld), applies sA * sB,
//              rounds to bf16.
#include "qz_tc.cuh"
#include "qz_next.cuh"

#include <algorithm>

namespace qz {

namespace {

__device__ unsigned int g_int8_err;

constexpr int BM = 128, BN = 256, BK = 64;       // one MMA: 128 x 256 x 16
constexpr int MH = 2;                             // 128-row halves per CTA tile
constexpr int TM = MH * BM;                       // CTA tile rows
constexpr int IST = 3;                            // int8 stages
constexpr int HST = 2;                            // fp16 stages
constexpr int IA = TM * BK, IB = BN * BK;         // int8 bytes per stage: 16 KB + 16 KB
constexpr int HA = TM * BK * 2, HB = BN * BK * 2; // fp16 bytes per stage: 32 KB + 32 KB
constexpr int I_STAGE = IA + IB, H_STAGE = HA + HB;
constexpr int CONV_WARPS = 8, EPI_WARPS = 8;
constexpr int THREADS = (2 + CONV_WARPS + EPI_WARPS) * 32;
constexpr int EPI_COLS = BN / (EPI_WARPS / 4);
constexpr uint32_t TMEM_COLS = MH * BN;          // one accumulator per half, one tile in flight
constexpr uint32_t IDESC = idesc_dense(0u, 0u, BM, BN);     // f16 x f16 -> fp32
constexpr int SMEM_BYTES = HST * H_STAGE + IST * I_STAGE + 512 + 1024;

// int8x4 -> two fp16x2: (x + 128) as a byte is the low mantissa of 1024 + u
// (fp16 0x6400 | u); subtracting 1152 leaves x exactly.
__device__ __forceinline__ void i8x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
    const uint32_t u = w ^ 0x80808080u;
    const uint32_t a = __byte_perm(u, 0x64646464u, 0x4140u);
    const uint32_t b = __byte_perm(u, 0x64646464u, 0x4342u);
    const uint32_t bias = 0xE480E480u;            // fp16x2 (-1152, -1152)
    asm("add.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(bias));
    asm("add.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(bias));
}

__global__ void __launch_bounds__(THREADS, 1)
int8_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const float* __restrict__ sA, const float* __restrict__ sB, uint16_t* __restrict__ Y,
                 int M, int N, int K) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t hbase = smem_u32(smem);                          // fp16 ring (1 KB aligned)
    const uint32_t ibase = hbase + HST * H_STAGE;                   // int8 ring
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + HST * H_STAGE + IST * I_STAGE);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * IST + 2 * HST + 2);
    auto ifull = [&](int s) { return smem_u32(bars + s); };
    auto iempty = [&](int s) { return smem_u32(bars + IST + s); };
    auto hfull = [&](int s) { return smem_u32(bars + 2 * IST + s); };
    auto hempty = [&](int s) { return smem_u32(bars + 2 * IST + HST + s); };
    const uint32_t tfull = smem_u32(bars + 2 * IST + 2 * HST), tempty = smem_u32(bars + 2 * IST + 2 * HST + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int mt = (M + TM - 1) / TM, tiles = mt * (N / BN), nks = K / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < IST; s++) {
            mbar_init(ifull(s), 1);
            mbar_init(iempty(s), CONV_WARPS);
        }
        for (int s = 0; s < HST; s++) {
            mbar_init(hfull(s), CONV_WARPS);
            mbar_init(hempty(s), 1);
        }
        mbar_init(tfull, 1);
        mbar_init(tempty, EPI_WARPS);
        fence_barrier_init();
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x) {
                const int m0 = (tile % mt) * TM, n0 = (tile / mt) * BN;
                for (int ks = 0; ks < nks; ks++, it++) {
                    const int s = it % IST;
                    if (!mbar_wait(iempty(s), ((it / IST) & 1) ^ 1, &g_int8_err)) { ok = false; break; }
                    mbar_arrive_expect_tx(ifull(s), I_STAGE);
                    tma_load_2d(ibase + s * I_STAGE, &tmA, ks * BK, m0, ifull(s));
                    tma_load_2d(ibase + s * I_STAGE + IA, &tmB, ks * BK, n0, ifull(s));
                }
            }
            // every copy into this CTA's shared memory has landed before it exits
            for (uint32_t j = it > IST ? it - IST : 0; j < it; j++)
                mbar_wait(iempty(j % IST), (j / IST) & 1, &g_int8_err);
        }
    } else if (warp == 1) {
        // -------------------------------------------------------- MMA issuer
        if (lane == 0) {
            uint32_t it = 0, tc = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x, tc++) {
                if (!mbar_wait(tempty, (tc & 1) ^ 1, &g_int8_err)) break;
                tc_fence_after();
                for (int ks = 0; ks < nks; ks++, it++) {
                    const int s = it % HST;
                    if (!mbar_wait(hfull(s), (it / HST) & 1, &g_int8_err)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t bd = sdesc_k_sw128(hbase + s * H_STAGE + HA);
#pragma unroll
                    for (int mh = 0; mh < MH; mh++) {                // both halves share the stage's B
                        const uint64_t ad = sdesc_k_sw128(hbase + s * H_STAGE + mh * (BM * 128));
#pragma unroll
                        for (int kk = 0; kk < BK / 16; kk++)        // K = 16 fp16 = 32 bytes per MMA
                            mma_f16_ss(tmem_base + mh * BN, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2), IDESC,
                                       (ks | kk) != 0);
                    }
                    tc_commit(hempty(s));
                }
                if (!ok) break;
                tc_commit(tfull);
            }
            if (tc > 0) mbar_wait(tfull, (tc - 1) & 1, &g_int8_err);
        }
        __syncwarp();
    } else if (warp < 2 + CONV_WARPS) {
        // --------------------------------------------------------- converters
        const int ct = threadIdx.x - 64;                            // 0 .. 32 * CONV_WARPS - 1
        uint32_t it = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x) {
            for (int ks = 0; ks < nks; ks++, it++) {
                const int si = it % IST, sh = it % HST;
                if (!mbar_wait(ifull(si), (it / IST) & 1, &g_int8_err)) { ok = false; break; }
                if (!mbar_wait(hempty(sh), ((it / HST) & 1) ^ 1, &g_int8_err)) { ok = false; break; }
                const uint8_t* src = smem + HST * H_STAGE + si * I_STAGE;
                uint8_t* dst = smem + sh * H_STAGE;
                // 512 rows (A's 256, then B's 256) x 4 input chunks of 16 bytes
#pragma unroll 2
                for (int j = ct; j < (TM + BN) * 4; j += CONV_WARPS * 32) {
                    const int row = j >> 2, c = j & 3;
                    const uint4 v = *reinterpret_cast<const uint4*>(src + row * BK + c * 16);
                    uint4 o0, o1;
                    i8x4_to_f16x4(v.x, o0.x, o0.y);
                    i8x4_to_f16x4(v.y, o0.z, o0.w);
                    i8x4_to_f16x4(v.z, o1.x, o1.y);
                    i8x4_to_f16x4(v.w, o1.z, o1.w);
                    // fp16 row of 128 bytes; output chunks 2c, 2c+1, swizzled by the row in its 8-row atom
                    uint8_t* drow = dst + (row < TM ? row * 128 : HA + (row - TM) * 128);
                    const int r7 = row & 7;
                    *reinterpret_cast<uint4*>(drow + (((2 * c) ^ r7) << 4)) = o0;
                    *reinterpret_cast<uint4*>(drow + (((2 * c + 1) ^ r7) << 4)) = o1;
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(iempty(si));
                    mbar_arrive(hfull(sh));
                }
            }
        }
    } else {
        // ------------------------------------------------------------- epilogue
        const int q = warp & 3;                   // TMEM lane quarter
        const int h = (warp - 2 - CONV_WARPS) >> 2;
        const int r = q * 32 + lane;
        uint32_t tc = 0;
        for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x, tc++) {
            const int n0 = (tile / mt) * BN;
            if (!mbar_wait(tfull, tc & 1, &g_int8_err)) break;
            tc_fence_after();
            const float* sbp = sB + n0 + h * EPI_COLS;
#pragma unroll 1
            for (int mh = 0; mh < MH; mh++) {
                const int m0 = (tile % mt) * TM + mh * BM;
                if (m0 >= M) break;                   // M % 128 == 0: a half lies wholly inside or outside
                const float sa = __ldg(sA + m0 + r);
                uint4* yrow = reinterpret_cast<uint4*>(Y + (size_t)(m0 + r) * N + n0 + h * EPI_COLS);
                const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + mh * BN + h * EPI_COLS;
#pragma unroll 1
                for (int c = 0; c < EPI_COLS / 32; c++) {
                    uint32_t v[32];
                    tmem_ld32(taddr + c * 32, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 4; j++) {
                        const float4 s0 = __ldg(reinterpret_cast<const float4*>(sbp + c * 32 + j * 8));
                        const float4 s1 = __ldg(reinterpret_cast<const float4*>(sbp + c * 32 + j * 8) + 1);
                        const float sb[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
                        uint4 o;
                        uint32_t* w = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
                        for (int e = 0; e < 4; e++) {
                            const float y0 = __fmul_rn(__fmul_rn(__uint_as_float(v[j * 8 + 2 * e]), sa), sb[2 * e]);
                            const float y1 = __fmul_rn(__fmul_rn(__uint_as_float(v[j * 8 + 2 * e + 1]), sa), sb[2 * e + 1]);
                            const __nv_bfloat162 p = __floats2bfloat162_rn(y0, y1);
                            w[e] = *reinterpret_cast<const uint32_t*>(&p);
                        }
                        yrow[c * 4 + j] = o;
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

} // namespace

qz_status int8_error_read_and_clear() {
    unsigned int v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_int8_err, sizeof(v)) != cudaSuccess) return QZ_ERR_CUDA;
    if (v && cudaMemcpyToSymbol(g_int8_err, &z, sizeof(z)) != cudaSuccess) return QZ_ERR_CUDA;
    return v ? QZ_ERR_TIMEOUT : QZ_OK;
}

qz_status gemm_int8_launch(const int8_t* qA, const float* sA, const int8_t* qB, const float* sB, uint16_t* Y, int M,
                           int N, int K, cudaStream_t st) {
    CUtensorMap ta, tb;
    if (!encode_tmap_2d(&ta, qA, 1, (uint64_t)K, (uint64_t)M, (uint64_t)K, BK, TM, false)) return QZ_ERR_CUDA;
    if (!encode_tmap_2d(&tb, qB, 1, (uint64_t)K, (uint64_t)N, (uint64_t)K, BK, BN, false)) return QZ_ERR_CUDA;
    QZ_TRY(opt_in_smem((const void*)int8_gemm_kernel, SMEM_BYTES));
    const int tiles = ((M + TM - 1) / TM) * (N / BN);
    int8_gemm_kernel<<<std::min(tiles, num_sms()), THREADS, SMEM_BYTES, st>>>(ta, tb, sA, sB, Y, M, N, K);
    return launch_status();
}

} // namespace qz
