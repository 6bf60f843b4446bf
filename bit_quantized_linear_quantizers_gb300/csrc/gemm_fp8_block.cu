// gemm_fp8_block.cu -- block-scaled FP8 GEMM for prefill on tcgen05:
//   Y[i, j] = bf16( sum_kb sA[i, kb] * sB[j/128, kb] * sum_{k in kb} qA[i,k] qB[j,k] )
// with E4M3 operands, 1x128 activation scales and 128x128 weight scales
// ("量化部署实战", 练习 2: inside each 128-deep K block the tensor cores
// multiply-accumulate FP8, the partial sum is then multiplied by that block's
// activation and weight scales and added into the fp32 result).
//
// The fp32 block scales are not powers of two, so they cannot ride in the
// tensor core's own block-scale path (E8M0 / UE4M3). Instead each 128-deep K
// block is an independent tcgen05 MMA chain into a TMEM accumulator, and the
// epilogue warps promote it on the CUDA cores: acc += P_kb * (sA * sB).
//
// Design (one CTA per SM, persistent over 128 x 256 output tiles):
//  warp 0      TMA producer: 128x128 A and 256x128 B boxes (128-byte swizzle)
//              into a 4-stage shared-memory ring, mbarrier complete_tx.
//  warp 1      MMA issuer (one thread): 4 x tcgen05.mma kind::f8f6f4
//              (M=128, N=256, K=32) per K block into one of two TMEM
//              accumulators (2 x 256 columns), committed to the stage's
//              "empty" barrier and the accumulator's "full" barrier.
//  warps 2-9   promotion + epilogue: each thread owns one output row and 128
//              columns; per K block it loads its partial sums from TMEM
//              (tcgen05.ld), multiplies by sA*sB and adds into fp32 registers,
//              then frees the accumulator; at the end of the tile it rounds
//              to bf16 and stores.
// The MMA of K block kb+1 runs while block kb is being promoted.
//
#include "qz_tc.cuh"

#include <algorithm>
#include <cstring>

namespace qz {

namespace {

__device__ unsigned int g_fp8_err;

constexpr int BM = 128, BN = 256, BK = 128, STAGES = 4;
constexpr int A_BYTES = BM * BK;                  // 16 KB
constexpr int B_BYTES = BN * BK;                  // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int EPI_WARPS = 8;
constexpr int EPI_COLS = BN / (EPI_WARPS / 4);   // columns per promotion thread
constexpr int SD = 1;                            // K blocks of scales kept in flight
constexpr int THREADS = 64 + EPI_WARPS * 32;
constexpr uint32_t TMEM_COLS = 2 * BN;
constexpr uint32_t IDESC = idesc_dense(0u, 0u, BM, BN);   // E4M3 x E4M3 -> fp32
// Each epilogue warp stages 32 rows x 128 bytes of its bf16 output in its own
// slice of shared memory (16-byte chunk j of row r at chunk j ^ (r & 7): the
// TMA 128-byte swizzle) and one TMA store writes the block. Stored a row per
// lane, each store instruction touched 32 lines (110.3 us at 2048 x 14336 x
// 4096); read back row-wise and stored by the warp, 107.7 us, but those loads
// and stores crowd the L1 data stage, which the MMA's operand reads keep busy.
constexpr int STG_OFF = STAGES * STAGE_BYTES + 1024;
constexpr int STG_WARP = 32 * 128;
constexpr int SMEM_BYTES = STG_OFF + EPI_WARPS * STG_WARP + 1024;
constexpr int SMEM_BYTES_Q = STAGES * STAGE_BYTES + 256 + 1024;   // quantized output: no staging

// acc (two fp32 lanes) += v * s per lane, each lane one correctly rounded fma
// (the paired fp32 FMA of sm_100+: half the instructions of two fmaf).
__device__ __forceinline__ void fma2(uint64_t& acc, uint32_t v0, uint32_t v1, uint64_t s2) {
    asm("{ .reg .b64 t; mov.b64 t, {%1, %2}; fma.rn.f32x2 %0, t, %3, %0; }" : "+l"(acc) : "r"(v0), "r"(v1), "l"(s2));
}

// 16-byte chunk j of the lane's row in a warp's staged 32 x 128-byte block.
__device__ __forceinline__ void stage_put(uint8_t* stg, int lane, int j, uint4 v) {
    *reinterpret_cast<uint4*>(stg + lane * 128 + ((j ^ (lane & 7)) << 4)) = v;
}

// QOUT: the epilogue also quantizes its output for the next layer, FP8 E4M3
// with one scale per row and 128 columns ("量化部署实战", 练习 2: the
// activation's (1, 128) scales are computed at the end of the previous
// kernel): each thread's 128 bf16 outputs are exactly one such group. Y (bf16)
// is then stored only when non-null.
template <bool QOUT>
__global__ void __launch_bounds__(THREADS, 1)
fp8_block_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const __grid_constant__ CUtensorMap tmY, const float* __restrict__ sA, const float* __restrict__ sB, uint16_t* __restrict__ Y,
                      uint8_t* __restrict__ Yq, float* __restrict__ Yqs, int M, int N, int K) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 4);
    auto full = [&](int s) { return smem_u32(bars + s); };
    auto empty = [&](int s) { return smem_u32(bars + STAGES + s); };
    auto tfull = [&](int b) { return smem_u32(bars + 2 * STAGES + b); };
    auto tempty = [&](int b) { return smem_u32(bars + 2 * STAGES + 2 + b); };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Tiles M-fastest: the CTAs working at one time share few B tiles (L2 reuse).
    const int mt = M / BM, tiles = mt * (N / BN), nkb = K / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; s++) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 1);
        }
        for (int b = 0; b < 2; b++) {
            mbar_init(tfull(b), 1);
            mbar_init(tempty(b), EPI_WARPS);
        }
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
                const int m0 = (tile % mt) * BM, n0 = (tile / mt) * BN;
                for (int kb = 0; kb < nkb; kb++, it++) {
                    const int s = it % STAGES;
                    const uint32_t ph = (it / STAGES) & 1;
                    if (!mbar_wait(empty(s), ph ^ 1, &g_fp8_err)) { ok = false; break; }
                    mbar_arrive_expect_tx(full(s), STAGE_BYTES);
                    tma_load_2d(sbase + s * STAGE_BYTES, &tmA, kb * BK, m0, full(s));
                    tma_load_2d(sbase + s * STAGE_BYTES + A_BYTES, &tmB, kb * BK, n0, full(s));
                }
            }
            // Before the CTA may exit, every stage it filled has been released
            // by the MMAs of both CTAs: all copies into its shared memory have
            // landed and no peer's commit is still on its way to these barriers.
            for (uint32_t j = it > STAGES ? it - STAGES : 0; j < it; j++)
                mbar_wait(empty(j % STAGES), (j / STAGES) & 1, &g_fp8_err);
        }
    } else if (warp == 1) {
        // -------------------------------------------------------- MMA issuer
        if (lane == 0) {
            uint32_t it = 0, ac = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x) {
                for (int kb = 0; kb < nkb; kb++, it++, ac++) {
                    const int b = ac & 1;
                    if (!mbar_wait(tempty(b), ((ac >> 1) & 1) ^ 1, &g_fp8_err)) { ok = false; break; }
                    tc_fence_after();
                    const int s = it % STAGES;
                    if (!mbar_wait(full(s), (it / STAGES) & 1, &g_fp8_err)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t ad = sdesc_k_sw128(sbase + s * STAGE_BYTES);
                    const uint64_t bd = sdesc_k_sw128(sbase + s * STAGE_BYTES + A_BYTES);
                    const uint32_t d = tmem_base + b * BN;
#pragma unroll
                    for (int ks = 0; ks < BK / 32; ks++)                 // K = 32 bytes per MMA
                        mma_f8f6f4(d, ad + (uint64_t)(ks * 2), bd + (uint64_t)(ks * 2), IDESC, ks > 0);
                    tc_commit(empty(s));
                    tc_commit(tfull(b));
                }
            }
            // the last accumulators are complete before TMEM is released
            if (ac > 0) mbar_wait(tfull((ac - 1) & 1), ((ac - 1) >> 1) & 1, &g_fp8_err);
        }
        __syncwarp();
    } else {
        // ------------------------------------------ promotion + epilogue warps
        const int q = warp & 3;                   // TMEM lane quarter of this warp
        const int h = (warp - 2) >> 2;            // column slice of the 256-wide tile
        const int r = q * 32 + lane;              // row within the tile
        uint32_t ac = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x) {
            const int m0 = (tile % mt) * BM, n0 = (tile / mt) * BN;
            const float* sa_row = sA + (size_t)(m0 + r) * nkb;
            const float* sb_row = sB + (size_t)((n0 + h * EPI_COLS) / 128) * nkb;
            // plain output: columns 2i, 2i+1 as one fp32 pair (paired FMAs, 106.9 -> 104.2 us);
            // the output-quantizing instance keeps scalar FMAs (its epilogue needs the registers)
            uint64_t acc2[QOUT ? 1 : EPI_COLS / 2];
            float accf[QOUT ? EPI_COLS : 1];
#pragma unroll
            for (int i = 0; i < (QOUT ? 1 : EPI_COLS / 2); i++) acc2[i] = 0ull;
#pragma unroll
            for (int i = 0; i < (QOUT ? EPI_COLS : 1); i++) accf[i] = 0.0f;
            // Scales of the next SD K blocks stay in flight as raw loads (an L2
            // round trip is longer than one block's MMAs); each is multiplied out
            // only when its block is promoted, so no load is waited on early.
            float ra[SD], rb[SD];
#pragma unroll
            for (int u = 0; u < SD; u++) {
                ra[u] = u < nkb ? __ldg(sa_row + u) : 0.0f;
                rb[u] = u < nkb ? __ldg(sb_row + u) : 0.0f;
            }
            for (int kb0 = 0; kb0 < nkb && ok; kb0 += SD) {
#pragma unroll
                for (int u = 0; u < SD; u++) {
                    const int kb = kb0 + u;
                    if (kb >= nkb || !ok) break;
                    const float scale = ra[u] * rb[u];
                    const uint64_t s2 = ((uint64_t)__float_as_uint(scale) << 32) | __float_as_uint(scale);
                    if (kb + SD < nkb) {
                        ra[u] = __ldg(sa_row + kb + SD);
                        rb[u] = __ldg(sb_row + kb + SD);
                    }
                    const int b = ac & 1;
                    if (!mbar_wait(tfull(b), (ac >> 1) & 1, &g_fp8_err)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + b * BN + h * EPI_COLS;
#pragma unroll
                    for (int c = 0; c < EPI_COLS / 16; c++) {
                        uint32_t v[16];
                        tmem_ld16(taddr + c * 16, v);
                        tmem_wait_ld();
                        if constexpr (QOUT) {
#pragma unroll
                            for (int i = 0; i < 16; i++)
                                accf[c * 16 + i] = fmaf(__uint_as_float(v[i]), scale, accf[c * 16 + i]);
                        } else {
#pragma unroll
                            for (int i = 0; i < 8; i++) fma2(acc2[c * 8 + i], v[2 * i], v[2 * i + 1], s2);
                        }
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(tempty(b));
                    ac++;
                }
            }
            if (!ok) break;
            float acc[EPI_COLS];
            if constexpr (QOUT) {
#pragma unroll
                for (int i = 0; i < EPI_COLS; i++) acc[i] = accf[i];
            } else {
#pragma unroll
                for (int i = 0; i < EPI_COLS / 2; i++) {
                    acc[2 * i] = __uint_as_float((uint32_t)acc2[i]);
                    acc[2 * i + 1] = __uint_as_float((uint32_t)(acc2[i] >> 32));
                }
            }
            if (QOUT) {
                // the bf16 output (what this kernel would store), then its 1x128 FP8 group:
                // s = max(amax, 1e-12) / 448, code = E4M3(y / s), quotients correctly rounded
                float am = 0.0f;
#pragma unroll
                for (int i = 0; i < EPI_COLS; i++) {
                    acc[i] = __bfloat162float(__float2bfloat16_rn(acc[i]));
                    am = fmaxf(am, fabsf(acc[i]));
                }
                const float sq = div1(fmaxf(am, kAmaxMin), Recip(kFp8Max));
                const Recip dq(sq);
                uint4* qrow = reinterpret_cast<uint4*>(Yq + (size_t)(m0 + r) * N + n0 + h * EPI_COLS);
#pragma unroll
                for (int j = 0; j < EPI_COLS / 16; j++) {
                    uint32_t p[8];
#pragma unroll
                    for (int e = 0; e < 8; e++) {
                        const float a = acc[j * 16 + 2 * e], b = acc[j * 16 + 2 * e + 1];
                        p[e] = e4m3x2(sign_of(div1(a, dq), a), sign_of(div1(b, dq), b));
                    }
                    qrow[j] = make_uint4(__byte_perm(p[0], p[1], 0x5410), __byte_perm(p[2], p[3], 0x5410),
                                         __byte_perm(p[4], p[5], 0x5410), __byte_perm(p[6], p[7], 0x5410));
                }
                Yqs[(size_t)(m0 + r) * (N / 128) + (n0 + h * EPI_COLS) / 128] = sq;
                if (Y == nullptr) continue;
            }
            if constexpr (!QOUT) {
                // re-derived here: keeping the aligned base live through the
                // promotion loop costs registers (spills at the 168-register cap)
                uint8_t* stg = smem_raw + (STG_OFF + (warp - 2) * STG_WARP + (smem - smem_raw));
                #pragma unroll
                for (int hf = 0; hf < EPI_COLS / 64; hf++) {          // 64 bf16 columns = 128 bytes a row
                    if (lane == 0) bulk_wait_read0();                 // the previous store has read the block
                    __syncwarp();
                    #pragma unroll
                    for (int j = 0; j < 8; j++) {
                        uint4 o;
                        uint32_t* w = reinterpret_cast<uint32_t*>(&o);
                        #pragma unroll
                        for (int e = 0; e < 4; e++) {
                            const int c = hf * 64 + j * 8 + 2 * e;
                            __nv_bfloat162 p = __floats2bfloat162_rn(acc[c], acc[c + 1]);
                            w[e] = *reinterpret_cast<uint32_t*>(&p);
                        }
                        stage_put(stg, lane, j, o);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) tma_store_2d(&tmY, smem_u32(stg), n0 + h * EPI_COLS + hf * 64, m0 + q * 32);
                }
            } else {
                uint4* yrow = reinterpret_cast<uint4*>(Y + (size_t)(m0 + r) * N + n0 + h * EPI_COLS);
#pragma unroll
                for (int j = 0; j < EPI_COLS / 8; j++) {
                    uint4 o;
                    uint32_t* w = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
                    for (int e = 0; e < 4; e++) {
                        __nv_bfloat162 p = __floats2bfloat162_rn(acc[j * 8 + 2 * e], acc[j * 8 + 2 * e + 1]);
                        w[e] = *reinterpret_cast<uint32_t*>(&p);
                    }
                    yrow[j] = o;
                }
            }
        }
        if (!QOUT && lane == 0) bulk_wait_all0();            // stores complete before the CTA exits
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

size_t ws_gemm_fp8_block(int, int, int) { return 0; }

qz_status fp8_block_error_read_and_clear() {
    unsigned int v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_fp8_err, sizeof(v)) != cudaSuccess) return QZ_ERR_CUDA;
    if (v && cudaMemcpyToSymbol(g_fp8_err, &z, sizeof(z)) != cudaSuccess) return QZ_ERR_CUDA;
    return v ? QZ_ERR_TIMEOUT : QZ_OK;
}

qz_status gemm_fp8_block_launch(const uint8_t* qA, const float* sA, const uint8_t* qB, const float* sB,
                                uint16_t* Y, int M, int N, int K, void*, size_t, cudaStream_t st) {
    return gemm_fp8_block_quant_launch(qA, sA, qB, sB, Y, nullptr, nullptr, M, N, K, st);
}

qz_status gemm_fp8_block_quant_launch(const uint8_t* qA, const float* sA, const uint8_t* qB, const float* sB,
                                      uint16_t* Y, uint8_t* Yq, float* Yqs, int M, int N, int K, cudaStream_t st) {
    CUtensorMap ta, tb, ty;
    if (!encode_tmap_2d_u8(&ta, qA, (uint64_t)K, (uint64_t)M, (uint64_t)K, BK, BM)) return QZ_ERR_CUDA;
    if (!encode_tmap_2d_u8(&tb, qB, (uint64_t)K, (uint64_t)N, (uint64_t)K, BK, BN)) return QZ_ERR_CUDA;
    memset(&ty, 0, sizeof(ty));                   // the output-quantizing instance stores without TMA
    if (!Yq && !encode_tmap_2d_swz(&ty, Y, 2, (uint64_t)N, (uint64_t)M, (uint64_t)N * 2, 64, 32, 128))
        return QZ_ERR_CUDA;
    const int tiles = (M / BM) * (N / BN);
    const int grid = std::min(tiles, num_sms());
    if (Yq) {
        QZ_TRY(opt_in_smem((const void*)fp8_block_gemm_kernel<true>, SMEM_BYTES_Q));
        fp8_block_gemm_kernel<true><<<grid, THREADS, SMEM_BYTES_Q, st>>>(ta, tb, ty, sA, sB, Y, Yq, Yqs, M, N, K);
    } else {
        QZ_TRY(opt_in_smem((const void*)fp8_block_gemm_kernel<false>, SMEM_BYTES));
        fp8_block_gemm_kernel<false><<<grid, THREADS, SMEM_BYTES, st>>>(ta, tb, ty, sA, sB, Y, nullptr, nullptr, M, N, K);
    }
    return launch_status();
}

} // namespace qz
