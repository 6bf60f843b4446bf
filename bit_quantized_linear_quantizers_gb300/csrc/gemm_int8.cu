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
// (tcgen05.mma kind::f16, fp32 accumulator in TMEM). Each 128 x 192 x 64 step
// sums at most 64 products of magnitude <= 2^14, and the accumulator stays an
// exact integer while |sum| < 2^24; beyond that (far outside realistic
// activations) it rounds like any fp32 accumulation.
//
// What sets the rate is the SM's L1 data stage, which carries both the
// converters' shared-memory loads and stores and the tensor core's operand
// reads from shared memory (about one 128-byte wavefront per cycle between
// them). So the widened A operand never touches shared memory: the
// converters write it straight into tensor memory (tcgen05.st), where the MMA
// reads it, and only B goes through shared memory as fp16. TMEM then holds two
// 128 x 192 fp32 accumulators (384 columns) and two A buffers (2 x 64 columns).
//
// Design (one CTA per SM, persistent over 256 x 192 output tiles, M fastest):
//  warp 0      TMA producer: per stage the int8 A box (256 rows x 64 bytes,
//              64-byte swizzle) and B box (192 rows x 64 bytes) into a 5-stage
//              ring.
//  warps 2-9   converters: thread = one A row of one half (warp w serves TMEM
//              lanes 32*(w%4) .. +31 of half (w-2)/4); its 64 codes become 32
//              fp16 pairs written to the stage's TMEM A buffer. Then the 192 B
//              rows, 16-byte chunks in turn, become fp16 rows in the
//              128-byte-swizzled K-major layout (chunk c of row r at c ^ (r & 7))
//              of a 2-stage ring.
//  warp 1      MMA issuer (one thread): per stage 2 halves x 4 kind::f16 MMAs
//              (M = 128, N = 192, K = 16), A from TMEM, B from shared memory.
//  warps 10-17 epilogue: each thread owns one row of each half and 96 columns;
//              loads the accumulators (tcgen05.ld), applies sA * sB, rounds to
//              bf16 into a 32-row x 32-column staging tile (64-byte swizzle, so
//              the row-per-lane writes are conflict-free) that one TMA tensor
//              store writes out (clipped at N).
#include "qz_tc.cuh"
#include "qz_next.cuh"

#include <algorithm>

namespace qz {

namespace {

__device__ unsigned int g_int8_err;

constexpr int BM = 128, BN = 192, BK = 64;       // one MMA: 128 x 192 x 16
constexpr int MH = 2;                             // 128-row halves per CTA tile
constexpr int TM = MH * BM;                       // CTA tile rows
constexpr int IST = 5;                            // int8 stages
constexpr int HST = 2;                            // fp16 B stages = TMEM A buffers
constexpr int IA = TM * BK, IB = BN * BK;         // int8 bytes per stage: 16 KB + 12 KB
constexpr int I_STAGE = IA + IB;
constexpr int H_STAGE = BN * BK * 2;              // fp16 B bytes per stage: 24 KB
constexpr int CONV_WARPS = 8, EPI_WARPS = 8;
constexpr int THREADS = (2 + CONV_WARPS + EPI_WARPS) * 32;
constexpr int EPI_COLS = BN / (EPI_WARPS / 4);    // 96 columns per epilogue thread
constexpr uint32_t ACC_COLS = MH * BN;            // accumulators: half h at column h * BN
constexpr uint32_t A_COLS = MH * BK / 2;          // one stage of A in TMEM: 2 halves x 32 columns
constexpr uint32_t TMEM_COLS = 512;
static_assert(ACC_COLS + HST * A_COLS <= TMEM_COLS, "accumulators and A buffers fit in TMEM");
constexpr uint32_t IDESC = idesc_dense(0u, 0u, BM, BN);     // f16 x f16 -> fp32
constexpr int STG_WARP = 32 * 64;                 // epilogue staging: 32 rows x 32 bf16
constexpr int H_OFF = IST * I_STAGE;              // fp16 ring after the int8 ring (1 KB aligned)
constexpr int STG_OFF = H_OFF + HST * H_STAGE;
constexpr int SMEM_BYTES = STG_OFF + EPI_WARPS * STG_WARP + 256 + 1024;
static_assert(I_STAGE % 1024 == 0 && H_OFF % 1024 == 0 && STG_OFF % 1024 == 0, "swizzled buffers 1 KB aligned");

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
                 const __grid_constant__ CUtensorMap tmY, const float* __restrict__ sA,
                 const float* __restrict__ sB, int M, int N, int K) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t ibase = smem_u32(smem);                          // int8 ring
    const uint32_t hbase = ibase + H_OFF;                           // fp16 B ring
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STG_OFF + EPI_WARPS * STG_WARP);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * IST + 2 * HST + 2);
    auto ifull = [&](int s) { return smem_u32(bars + s); };
    auto iempty = [&](int s) { return smem_u32(bars + IST + s); };
    auto hfull = [&](int s) { return smem_u32(bars + 2 * IST + s); };
    auto hempty = [&](int s) { return smem_u32(bars + 2 * IST + HST + s); };
    const uint32_t tfull = smem_u32(bars + 2 * IST + 2 * HST), tempty = smem_u32(bars + 2 * IST + 2 * HST + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int mt = (M + TM - 1) / TM, tiles = mt * ((N + BN - 1) / BN), nks = K / BK;

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
        prefetch_tmap(&tmY);
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
                    const uint64_t bd = sdesc_k_sw128(hbase + s * H_STAGE);
#pragma unroll
                    for (int mh = 0; mh < MH; mh++) {                // both halves share the stage's B
                        const uint32_t at = tmem_base + ACC_COLS + s * A_COLS + mh * (BK / 2);
#pragma unroll
                        for (int kk = 0; kk < BK / 16; kk++)        // K = 16: 8 TMEM columns of A, 32 bytes of B
                            mma_f16_ts(tmem_base + mh * BN, at + kk * 8, bd + (uint64_t)(kk * 2), IDESC,
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
        const int q = warp & 3, h = (warp - 2) >> 2;                // TMEM lane quarter; A half
        const int ra = h * BM + q * 32 + lane;                      // this thread's A row in the tile
        const int sw = (ra >> 1) & 3;                               // its 64-byte swizzle phase
        constexpr int BPER = BN * 4 / (CONV_WARPS * 32);            // B chunks per thread
        static_assert(BPER * CONV_WARPS * 32 == BN * 4, "B chunks divide evenly over the converter threads");
        uint32_t it = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x) {
            for (int ks = 0; ks < nks; ks++, it++) {
                const int si = it % IST, sh = it % HST;
                if (!mbar_wait(ifull(si), (it / IST) & 1, &g_int8_err)) { ok = false; break; }
                const uint8_t* src = smem + si * I_STAGE;
                // every load first: a shared store may alias a later load, so the compiler keeps the order
                uint4 a[4], b[BPER];
#pragma unroll
                for (int c = 0; c < 4; c++)
                    a[c] = *reinterpret_cast<const uint4*>(src + ra * BK + ((c ^ sw) << 4));
#pragma unroll
                for (int i = 0; i < BPER; i++) {
                    const int j = ct + i * CONV_WARPS * 32;
                    b[i] = *reinterpret_cast<const uint4*>(src + IA + (j >> 2) * BK + (j & 3) * 16);
                }
                if (!mbar_wait(hempty(sh), ((it / HST) & 1) ^ 1, &g_int8_err)) { ok = false; break; }
                tc_fence_after();
                // A row -> 32 TMEM columns of fp16 pairs (column c holds k = 2c, 2c + 1)
                uint32_t o[32];
#pragma unroll
                for (int c = 0; c < 4; c++) {
                    i8x4_to_f16x4(a[c].x, o[c * 8 + 0], o[c * 8 + 1]);
                    i8x4_to_f16x4(a[c].y, o[c * 8 + 2], o[c * 8 + 3]);
                    i8x4_to_f16x4(a[c].z, o[c * 8 + 4], o[c * 8 + 5]);
                    i8x4_to_f16x4(a[c].w, o[c * 8 + 6], o[c * 8 + 7]);
                }
                tmem_st32(tmem_base + ((uint32_t)(q * 32) << 16) + ACC_COLS + sh * A_COLS + h * (BK / 2), o);
                // B rows -> fp16 rows of 128 bytes, 128-byte swizzle
                uint8_t* dst = smem + H_OFF + sh * H_STAGE;
#pragma unroll
                for (int i = 0; i < BPER; i++) {
                    const int j = ct + i * CONV_WARPS * 32, row = j >> 2, c = j & 3, r7 = row & 7;
                    uint4 o0, o1;
                    i8x4_to_f16x4(b[i].x, o0.x, o0.y);
                    i8x4_to_f16x4(b[i].y, o0.z, o0.w);
                    i8x4_to_f16x4(b[i].z, o1.x, o1.y);
                    i8x4_to_f16x4(b[i].w, o1.z, o1.w);
                    *reinterpret_cast<uint4*>(dst + row * 128 + (((2 * c) ^ r7) << 4)) = o0;
                    *reinterpret_cast<uint4*>(dst + row * 128 + (((2 * c + 1) ^ r7) << 4)) = o1;
                }
                tmem_wait_st();
                fence_proxy_async_smem();
                tc_fence_before();
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
        const int ch = (warp - 2 - CONV_WARPS) >> 2;
        const int r = q * 32 + lane;
        uint8_t* stg = smem + STG_OFF + (warp - 2 - CONV_WARPS) * STG_WARP;
        const uint32_t stg_s = smem_u32(stg);
        uint32_t tc = 0;
        for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x, tc++) {
            const int nc = (tile / mt) * BN + ch * EPI_COLS;        // this thread's first column
            // the tile's scales are fetched while its accumulators fill: sA of this thread's two
            // rows, sB of column nc + 32 c + lane (shared across the warp by shuffles)
            float sav[MH], sbv[EPI_COLS / 32];
#pragma unroll
            for (int mh = 0; mh < MH; mh++) {
                const int m = (tile % mt) * TM + mh * BM + r;
                sav[mh] = m < M ? __ldg(sA + m) : 0.f;
            }
#pragma unroll
            for (int c = 0; c < EPI_COLS / 32; c++) sbv[c] = nc + c * 32 < N ? __ldg(sB + nc + c * 32 + lane) : 0.f;
            if (!mbar_wait(tfull, tc & 1, &g_int8_err)) break;
            tc_fence_after();
#pragma unroll
            for (int mh = 0; mh < MH; mh++) {
                const int m0 = (tile % mt) * TM + mh * BM;
                if (m0 >= M) break;                   // M % 128 == 0: a half lies wholly inside or outside
                const float sa = sav[mh];
                const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + mh * BN + ch * EPI_COLS;
#pragma unroll
                for (int c = 0; c < EPI_COLS / 32; c++) {
                    const int n = nc + c * 32;
                    if (n >= N) break;                // the last column tile is ragged; N % 32 == 0
                    uint32_t v[32];
                    tmem_ld32(taddr + c * 32, v);
                    tmem_wait_ld();
                    if (lane == 0) bulk_wait_read0(); // the staging tile's previous store has read it
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < 4; j++) {
                        float sb[8];
#pragma unroll
                        for (int e = 0; e < 8; e++) sb[e] = __shfl_sync(0xffffffffu, sbv[c], j * 8 + e);
                        uint4 o;
                        uint32_t* w = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
                        for (int e = 0; e < 4; e++) {
                            const float y0 = __fmul_rn(__fmul_rn(__uint_as_float(v[j * 8 + 2 * e]), sa), sb[2 * e]);
                            const float y1 = __fmul_rn(__fmul_rn(__uint_as_float(v[j * 8 + 2 * e + 1]), sa), sb[2 * e + 1]);
                            const __nv_bfloat162 p = __floats2bfloat162_rn(y0, y1);
                            w[e] = *reinterpret_cast<const uint32_t*>(&p);
                        }
                        // 16-byte chunk j of the 64-byte staging row, 64-byte swizzle
                        *reinterpret_cast<uint4*>(stg + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4)) = o;
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) tma_store_2d(&tmY, stg_s, n, m0 + q * 32);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty);
        }
        if (lane == 0) bulk_wait_all0();          // stores complete before the CTA exits
        __syncwarp();
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
    CUtensorMap ta, tb, ty;
    if (!encode_tmap_2d_swz(&ta, qA, 1, (uint64_t)K, (uint64_t)M, (uint64_t)K, BK, TM, 64)) return QZ_ERR_CUDA;
    if (!encode_tmap_2d(&tb, qB, 1, (uint64_t)K, (uint64_t)N, (uint64_t)K, BK, BN, false)) return QZ_ERR_CUDA;
    if (!encode_tmap_2d_swz(&ty, Y, 2, (uint64_t)N, (uint64_t)M, (uint64_t)N * 2, 32, 32, 64)) return QZ_ERR_CUDA;
    QZ_TRY(opt_in_smem((const void*)int8_gemm_kernel, SMEM_BYTES));
    const int tiles = ((M + TM - 1) / TM) * ((N + BN - 1) / BN);
    int8_gemm_kernel<<<std::min(tiles, num_sms()), THREADS, SMEM_BYTES, st>>>(ta, tb, ty, sA, sB, M, N, K);
    return launch_status();
}

} // namespace qz
