// gemm_fp4.cu -- NVFP4 and MXFP4 GEMMs on the Blackwell FP4 tensor cores
// ("量化部署实战", 格式速查: MXFP4 and NVFP4 rows -- Blackwell computes in
// FP4 natively; "量化：让每一步搬更少的字节", 新一代低位格式):
//   NVFP4: Y = bf16( gA * gB * sum_b sA[i,b] sB[j,b] sum_{k in b} qA[i,k] qB[j,k] ),
//          blocks of 16, UE4M3 block scales, fp32 tensor scales gA, gB;
//   MXFP4: Y = bf16( sum_b 2^eA[i,b] 2^eB[j,b] sum_{k in b} qA[i,k] qB[j,k] ),
//          blocks of 32, UE8M0 block scales.
// The block scales ride in the tensor core's own block-scale path
// (tcgen05.mma kind::mxf4nvf4 scale_vec::4X, kind::mxf4 scale_vec::2X); the
// NVFP4 tensor scales are applied in the epilogue.
//
// Scale factors: the MMA reads them from tensor memory, where a 128-row x
// 4-scale block sits in 32 lanes x 4 columns (row m of the block at lane
// m % 32, column m / 32, byte = scale index; replicated into the four lane
// quarters). A pre-pass (sf_relayout_kernel) rewrites the row-major scales
// written by the quantizers into 512-byte atoms of exactly that order, in the
// caller's workspace; per pipeline stage the producer bulk-copies the atoms
// next to the operand tiles and the MMA thread moves them into TMEM with
// tcgen05.cp (32x128b, warpx4) right before the MMAs that use them.
//
// CTA (one per SM, persistent over 128 x 256 output tiles, K in 256-element
// stages of 128 bytes per row):
//  warp 0      TMA: A 128x128 B and B 256x128 B boxes (128-byte swizzle) plus
//              the stage's scale atoms (bulk copies), 4-stage ring.
//  warp 1      MMA issuer: tcgen05.cp of the scale atoms, 4 MMAs (K = 64 each)
//              per stage into one 256-column fp32 accumulator.
//  warps 2-9   epilogue: drain the accumulator into registers (then release it
//              so the next tile's MMAs start), apply gA*gB, round to bf16, store.
#include "qz_tc.cuh"

#include <algorithm>
#include <mutex>

namespace qz {

namespace {

__device__ unsigned int g_fp4_err;

constexpr int BM = 128, BN = 256;
constexpr int BKB = 128;                          // K bytes per stage (256 E2M1 values)
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BKB;                 // 16 KB
constexpr int B_BYTES = BN * BKB;                 // 32 KB
constexpr int ATOM = 512;                         // 128 rows x 4 scales
constexpr int SF_BYTES = 12 * ATOM;               // NVFP4: 4 atoms for A + 2 x 4 for B (MXFP4 uses half)
constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SF_BYTES;
constexpr int EPI_WARPS = 8;
constexpr int THREADS = 64 + EPI_WARPS * 32;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t SF_COL = 256;                  // scale-factor ring after the accumulator
constexpr uint32_t SF_COLS_PER_STAGE = 48;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 256 + 1024;

// Row-major scales sf[R][KS] -> atoms[R/128][KS/4][512]: byte (m%32)*16 +
// (m/32)*4 + k of atom (rb, kg) holds sf[rb*128 + m][kg*4 + k].
__global__ void sf_relayout_kernel(const uint8_t* __restrict__ sf, int R, int KS, uint8_t* __restrict__ out) {
    const int64_t words = (int64_t)(R / 128) * (KS / 4) * 128;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < words; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t a = i >> 7;
        const int p = (int)(i & 127);
        const int64_t rb = a / (KS / 4), kg = a % (KS / 4);
        const int64_t m = rb * 128 + (p >> 2) + 32 * (p & 3);
        const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(sf + m * KS + kg * 4));
        reinterpret_cast<uint32_t*>(out)[i] = w;
    }
}

template <bool NV>
__global__ void __launch_bounds__(THREADS, 1)
fp4_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const uint8_t* __restrict__ sfA, const uint8_t* __restrict__ sfB,
                const float* __restrict__ gA, const float* __restrict__ gB, uint16_t* __restrict__ Y,
                int M, int N, int K) {
    constexpr int G = NV ? 4 : 2;                 // scale atoms per row block per stage
    constexpr uint32_t SFA_COLS = 4 * G;          // TMEM columns of A's scales per stage
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 2);
    auto full = [&](int s) { return smem_u32(bars + s); };
    auto empty = [&](int s) { return smem_u32(bars + STAGES + s); };
    const uint32_t tfull = smem_u32(bars + 2 * STAGES), tempty = smem_u32(bars + 2 * STAGES + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int mt = M / BM, tiles = mt * (N / BN), nks = K / (2 * BKB);
    const int ksa = K / (NV ? 16 : 32);           // scales per row
    const int atoms_per_rb = ksa / 4;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; s++) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 1);
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
            const uint32_t sf_bytes = 3u * G * ATOM;
            uint32_t it = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x) {
                const int m0 = (tile % mt) * BM, n0 = (tile / mt) * BN;
                const uint8_t* sa = sfA + ((size_t)(m0 / 128) * atoms_per_rb) * ATOM;
                const uint8_t* sb0 = sfB + ((size_t)(n0 / 128) * atoms_per_rb) * ATOM;
                const uint8_t* sb1 = sb0 + (size_t)atoms_per_rb * ATOM;
                for (int c = 0; c < nks; c++, it++) {
                    const int s = it % STAGES;
                    if (!mbar_wait(empty(s), ((it / STAGES) & 1) ^ 1, &g_fp4_err)) { ok = false; break; }
                    const uint32_t st = sbase + s * STAGE_BYTES;
                    mbar_arrive_expect_tx(full(s), A_BYTES + B_BYTES + sf_bytes);
                    tma_load_2d(st, &tmA, c * BKB, m0, full(s));
                    tma_load_2d(st + A_BYTES, &tmB, c * BKB, n0, full(s));
                    const size_t off = (size_t)c * G * ATOM;
                    bulk_g2s(st + A_BYTES + B_BYTES, sa + off, G * ATOM, full(s));
                    bulk_g2s(st + A_BYTES + B_BYTES + G * ATOM, sb0 + off, G * ATOM, full(s));
                    bulk_g2s(st + A_BYTES + B_BYTES + 2 * G * ATOM, sb1 + off, G * ATOM, full(s));
                }
            }
            for (uint32_t j = it > STAGES ? it - STAGES : 0; j < it; j++)
                mbar_wait(full(j % STAGES), (j / STAGES) & 1, &g_fp4_err);
        }
    } else if (warp == 1) {
        // -------------------------------------------------------- MMA issuer
        if (lane == 0) {
            uint32_t it = 0, tcount = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x, tcount++) {
                if (!mbar_wait(tempty, (tcount & 1) ^ 1, &g_fp4_err)) { ok = false; break; }
                tc_fence_after();
                for (int c = 0; c < nks; c++, it++) {
                    const int s = it % STAGES;
                    if (!mbar_wait(full(s), (it / STAGES) & 1, &g_fp4_err)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t st = sbase + s * STAGE_BYTES;
                    const uint32_t sfa_t = tmem_base + SF_COL + s * SF_COLS_PER_STAGE;
                    const uint32_t sfb_t = sfa_t + SFA_COLS;
                    const uint32_t sfa_s = st + A_BYTES + B_BYTES;
#pragma unroll
                    for (int g = 0; g < G; g++) {
                        tmem_cp_32x128b_x4(sfa_t + 4 * g, sdesc_plain(sfa_s + g * ATOM));
                        tmem_cp_32x128b_x4(sfb_t + 8 * g, sdesc_plain(sfa_s + (G + g) * ATOM));
                        tmem_cp_32x128b_x4(sfb_t + 8 * g + 4, sdesc_plain(sfa_s + (2 * G + g) * ATOM));
                    }
                    const uint64_t ad = sdesc_k_sw128(st);
                    const uint64_t bd = sdesc_k_sw128(st + A_BYTES);
#pragma unroll
                    for (int j = 0; j < 4; j++) {                         // K = 64 values (32 bytes) each
                        const uint32_t acc = (c > 0 || j > 0) ? 1u : 0u;
                        if (NV) {
                            mma_nvf4(tmem_base, ad + (uint64_t)(j * 2), bd + (uint64_t)(j * 2),
                                     idesc_fp4(false, BM, BN, 0, 0), sfa_t + 4 * j, sfb_t + 8 * j, acc);
                        } else {
                            const uint32_t id = (uint32_t)(j & 1) * 2;    // which scale pair of the atom word
                            mma_mxf4(tmem_base, ad + (uint64_t)(j * 2), bd + (uint64_t)(j * 2),
                                     idesc_fp4(true, BM, BN, id, id), sfa_t + 4 * (j >> 1), sfb_t + 8 * (j >> 1), acc);
                        }
                    }
                    tc_commit(empty(s));
                }
                if (!ok) break;
                tc_commit(tfull);
            }
            if (tcount > 0) mbar_wait(tfull, (tcount - 1) & 1, &g_fp4_err);
        }
        __syncwarp();
    } else {
        // --------------------------------------------------------- epilogue
        const int q = warp & 3, h = (warp - 2) >> 2, r = q * 32 + lane;
        const float gscale = NV ? __ldg(gA) * __ldg(gB) : 1.0f;
        uint32_t tcount = 0;
        for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x, tcount++) {
            const int m0 = (tile % mt) * BM, n0 = (tile / mt) * BN;
            if (!mbar_wait(tfull, tcount & 1, &g_fp4_err)) break;
            tc_fence_after();
            float acc[128];
            const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + h * 128;
#pragma unroll
            for (int c = 0; c < 4; c++) {
                uint32_t v[32];
                tmem_ld32(taddr + c * 32, v);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; i++) acc[c * 32 + i] = __uint_as_float(v[i]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty);
            uint4* yrow = reinterpret_cast<uint4*>(Y + (size_t)(m0 + r) * N + n0 + h * 128);
#pragma unroll
            for (int j = 0; j < 16; j++) {
                uint4 o;
                uint32_t* w = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
                for (int e = 0; e < 4; e++) {
                    __nv_bfloat162 p = __floats2bfloat162_rn(acc[j * 8 + 2 * e] * gscale, acc[j * 8 + 2 * e + 1] * gscale);
                    w[e] = *reinterpret_cast<uint32_t*>(&p);
                }
                yrow[j] = o;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

size_t sf_bytes(bool nv, int R, int K) { return (size_t)R * (K / (nv ? 16 : 32)); }

} // namespace

size_t ws_gemm_fp4(int M, int N, int K) {
    // re-laid scales of A and B (NVFP4 size; MXFP4 uses half)
    return ((sf_bytes(true, M, K) + 1023) & ~size_t(1023)) + ((sf_bytes(true, N, K) + 1023) & ~size_t(1023));
}

qz_status fp4_error_read_and_clear() {
    unsigned int v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_fp4_err, sizeof(v)) != cudaSuccess) return QZ_ERR_CUDA;
    if (v && cudaMemcpyToSymbol(g_fp4_err, &z, sizeof(z)) != cudaSuccess) return QZ_ERR_CUDA;
    return v ? QZ_ERR_TIMEOUT : QZ_OK;
}

qz_status gemm_fp4_launch(bool nv, const uint8_t* qA, const uint8_t* sA, const float* gA,
                          const uint8_t* qB, const uint8_t* sB, const float* gB, uint16_t* Y,
                          int M, int N, int K, void* ws, size_t, cudaStream_t st) {
    uint8_t* wsA = static_cast<uint8_t*>(ws);
    uint8_t* wsB = wsA + ((sf_bytes(true, M, K) + 1023) & ~size_t(1023));
    const int ks = K / (nv ? 16 : 32);
    {
        const int64_t wa = (int64_t)M * ks / 4, wb = (int64_t)N * ks / 4;
        const int ga = (int)std::min<int64_t>((wa + 255) / 256, (int64_t)num_sms() * 8);
        const int gb = (int)std::min<int64_t>((wb + 255) / 256, (int64_t)num_sms() * 8);
        sf_relayout_kernel<<<ga, 256, 0, st>>>(sA, M, ks, wsA);
        sf_relayout_kernel<<<gb, 256, 0, st>>>(sB, N, ks, wsB);
    }
    CUtensorMap ta, tb;
    if (!encode_tmap_2d_u8(&ta, qA, (uint64_t)K / 2, (uint64_t)M, (uint64_t)K / 2, BKB, BM)) return QZ_ERR_CUDA;
    if (!encode_tmap_2d_u8(&tb, qB, (uint64_t)K / 2, (uint64_t)N, (uint64_t)K / 2, BKB, BN)) return QZ_ERR_CUDA;
    static int attr_set[64][2];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return QZ_ERR_UNSUPPORTED;
    const void* fn = nv ? (const void*)fp4_gemm_kernel<true> : (const void*)fp4_gemm_kernel<false>;
    if (!attr_set[dev][nv]) {
        if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES) != cudaSuccess)
            return QZ_ERR_CUDA;
        attr_set[dev][nv] = 1;
    }
    const int tiles = (M / BM) * (N / BN);
    const int grid = std::min(tiles, num_sms());
    if (nv)
        fp4_gemm_kernel<true><<<grid, THREADS, SMEM_BYTES, st>>>(ta, tb, wsA, wsB, gA, gB, Y, M, N, K);
    else
        fp4_gemm_kernel<false><<<grid, THREADS, SMEM_BYTES, st>>>(ta, tb, wsA, wsB, gA, gB, Y, M, N, K);
    return launch_status();
}

} // namespace qz

// ------------------------------------------------ allocation-free NVFP4 GEMM
//
// Scratch of qz_gemm_nvfp4_noalloc: a fixed device array defined here, so
// callers that cannot allocate still get the re-laid scale factors somewhere.
// In host code the symbol is only a host-side stand-in; its device address is
// looked up once per device (with that device current) and cached.
static __device__ __align__(256) uint8_t qz_nvfp4_noalloc_scratch[QZ_NVFP4_NOALLOC_SCRATCH_BYTES];

namespace qz {

namespace {
void* g_noalloc_ptr[64];
std::mutex g_noalloc_mu;
} // namespace

qz_status nvfp4_noalloc_scratch(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return QZ_ERR_CUDA;
    if (dev < 0 || dev >= 64) return QZ_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, qz_nvfp4_noalloc_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return QZ_ERR_CUDA;
        }
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return QZ_OK;
}

} // namespace qz
