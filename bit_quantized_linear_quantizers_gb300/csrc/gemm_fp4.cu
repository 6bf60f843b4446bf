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
// next to the operand tiles and a warp of its own moves them into TMEM with
// tcgen05.cp (32x128b, warpx4) once the stage has landed: issued by the MMA
// thread between its MMAs, the copies made every stage wait on their issue
// (NVFP4 8192 x 4096 x 4096: 78.9 -> 73.0 us).
//
// CTA (one per SM, persistent over 128 x 256 output tiles, K in 256-element
// stages of 128 bytes per row):
//  warp 0      TMA: A 128x128 B and B 256x128 B boxes (128-byte swizzle) plus
//              the stage's scale atoms (bulk copies), 4-stage ring.
//  warp 10     scale copies: per stage tcgen05.cp of the atoms into the
//              stage's TMEM scale slot, then a commit the MMA thread waits on.
//  warp 1      MMA issuer: 4 MMAs (K = 64 each) per stage into one
//              256-column fp32 accumulator.
//  warps 2-9   epilogue: drain the accumulator into registers (then release it
//              so the next tile's MMAs start), apply gA*gB, round to bf16, and
//              write 32-row x 16-column chunks through a 1 KB staging tile
//              (32-byte swizzle: the row-per-lane writes are conflict-free)
//              with one TMA store each. Stored straight from registers, a lane
//              per row made every store instruction touch 32 lines, and those
//              wavefronts competed with the tensor core's operand reads in
//              the L1 data stage.
//
// The CTAs walk a table of problems (one entry for qz_gemm_nvfp4/mxfp4, a
// decoder step's linears for the grouped call): tile t belongs to the last
// problem whose first tile is <= t. Rows of A beyond M (a decode batch is one
// partial 128-row tile) are read as zeros by TMA, their scales re-laid as
// zeros, and never stored.
#include "qz_tc.cuh"

#include <algorithm>
#include <cstring>
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
constexpr int SF_WARP = 2 + EPI_WARPS;            // issues the stage's scale copies into TMEM
constexpr int THREADS = 64 + EPI_WARPS * 32 + 32;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t SF_COL = 256;                  // scale-factor ring after the accumulator
constexpr uint32_t SF_COLS_PER_STAGE = 48;
constexpr int STG_WARP = 32 * 32;                 // epilogue staging: 32 rows x 16 bf16 (32-byte swizzle)
constexpr int STG_OFF = STAGES * STAGE_BYTES;     // after the stages (1 KB aligned)
constexpr int BAR_OFF = STG_OFF + EPI_WARPS * STG_WARP;
constexpr int SMEM_BYTES = BAR_OFF + 256 + 1024;
static_assert((3 * STAGES + 2) * 8 + 4 <= 256, "barriers and the TMEM slot fit their region");

// Row-major scales sf[R][KS] -> atoms[ceil(R/128)][KS/4][512]: byte
// (m%32)*16 + (m/32)*4 + k of atom (rb, kg) holds sf[rb*128 + m][kg*4 + k]
// (0 for rows >= R). One launch re-lays every job of the table.
constexpr int RELAY_MAX = 256;

struct RelayJob {
    const uint8_t* src;
    uint8_t* dst;
    long long word_begin;             // first 32-bit word of this job in the launch
    int R, KS;
};

struct RelayParams {
    RelayJob j[RELAY_MAX];
    int count;
    long long total_words;
};

// CTA (x, y) re-lays atoms x, x + gridDim.x, ... of job y; thread p of an atom
// writes its word p (row m = rb*128 + p/4 + 32*(p%4), the four scales of group kg).
__global__ void __launch_bounds__(128) sf_relayout_kernel(const __grid_constant__ RelayParams P) {
    const RelayJob& jb = P.j[blockIdx.y];
    const int kgn = jb.KS / 4;                                // 4-scale groups per row
    const int atoms = ((jb.R + 127) / 128) * kgn;
    const int p = threadIdx.x;
    const int r_in = (p >> 2) + 32 * (p & 3);
    for (int a = blockIdx.x; a < atoms; a += gridDim.x) {
        const int rb = a / kgn, kg = a - rb * kgn;
        const int m = rb * 128 + r_in;
        const uint32_t v = m < jb.R ? __ldg(reinterpret_cast<const uint32_t*>(jb.src + (size_t)m * jb.KS + kg * 4)) : 0u;
        reinterpret_cast<uint32_t*>(jb.dst)[(size_t)a * 128 + p] = v;
    }
}

long long relay_words(int R, int KS) { return (long long)((R + 127) / 128) * (KS / 4) * 128; }

qz_status relayout(const RelayParams& P, cudaStream_t st) {
    if (P.total_words == 0) return QZ_OK;
    int amax = 0;
    for (int i = 0; i < P.count; i++) amax = std::max(amax, ((P.j[i].R + 127) / 128) * (P.j[i].KS / 4));
    const int gx = std::max(1, std::min(amax, num_sms() * 16 / P.count + 1));
    sf_relayout_kernel<<<dim3(gx, P.count), 128, 0, st>>>(P);
    return launch_status();
}

// One GEMM problem of a launch: its tensor maps and its other fields, kept in
// two arrays (a tensor map is 128-byte aligned, so one struct of both would pad
// each entry to 512 bytes; as two arrays 72 problems fit the kernel parameter space).
struct Fp4Maps {
    CUtensorMap tmA;                  // A codes [M, K/2] u8, box 128 B x 128 rows
    CUtensorMap tmB;                  // B^T codes [N, K/2] u8, box 128 B x 256 rows
    CUtensorMap tmY;                  // Y bf16 [M, N], box 16 x 32, 32-byte swizzle (stores)
};
struct Fp4Prob {
    const uint8_t* sfA;               // A scales, tensor-core atoms, rows padded to 128
    const uint8_t* sfB;               // B scales, tensor-core atoms
    const float* gA;                  // NVFP4 tensor scales (unused for MXFP4)
    const float* gB;
    uint16_t* Y;
    int M, N, K;
    int mt;                           // 128-row tiles of M
    int tile_begin;                   // first tile of this problem in the launch
};

constexpr int FP4_PER_LAUNCH = 72;
static_assert(sizeof(Fp4Maps) == 384 && sizeof(Fp4Prob) == 64, "problem table layout");

// NVFP4 output of a single-problem launch (QOUT): codes [M, N/2], E4M3 block
// scales [M, N/16], the tensor scale g from the caller's amax.
struct Fp4Qout {
    uint8_t* codes;
    uint8_t* scales;
    const float* amax;
    float* g;
};

struct Fp4Params {
    Fp4Maps m[FP4_PER_LAUNCH];
    Fp4Prob p[FP4_PER_LAUNCH];
    Fp4Qout q;
    int count;
    int total_tiles;
};

// QOUT: instead of bf16 Y the epilogue writes Y quantized for the next layer:
// each value rounded to bf16 as the plain epilogue rounds it, then, in the
// GEMM's own format, NVFP4 with the caller's tensor amax (exactly as
// qz_quantize_nvfp4 with a given amax encodes that bf16 tensor) or MXFP4
// (exactly as qz_quantize_mxfp4 encodes it). One thread per row: 16-byte code
// stores, the row's scale bytes of the tile in one store.
template <bool NV, bool QOUT = false>
__global__ void __launch_bounds__(THREADS, 1)
fp4_gemm_kernel(const __grid_constant__ Fp4Params P) {
    constexpr int G = NV ? 4 : 2;                 // scale atoms per row block per stage
    constexpr uint32_t SFA_COLS = 4 * G;          // TMEM columns of A's scales per stage
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + BAR_OFF);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 3 * STAGES + 2);
    auto full = [&](int s) { return smem_u32(bars + s); };
    auto empty = [&](int s) { return smem_u32(bars + STAGES + s); };
    auto sfready = [&](int s) { return smem_u32(bars + 2 * STAGES + 2 + s); };
    const uint32_t tfull = smem_u32(bars + 2 * STAGES), tempty = smem_u32(bars + 2 * STAGES + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tiles = P.total_tiles;
    auto find = [&](int tile) {                   // last problem with tile_begin <= tile
        int lo = 0, hi = P.count - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (P.p[mid].tile_begin <= tile) lo = mid; else hi = mid - 1;
        }
        return lo;
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; s++) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 1);
            mbar_init(sfready(s), 1);
        }
        mbar_init(tfull, 1);
        mbar_init(tempty, EPI_WARPS);
        fence_barrier_init();
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
                const int pi = find(tile);
                const Fp4Prob& pr = P.p[pi];
                const Fp4Maps& mp = P.m[pi];
                const int local = tile - pr.tile_begin;
                const int m0 = (local % pr.mt) * BM, n0 = (local / pr.mt) * BN;
                const int nks = pr.K / (2 * BKB);
                const int atoms_per_rb = pr.K / (NV ? 16 : 32) / 4;
                const uint8_t* sa = pr.sfA + ((size_t)(m0 / 128) * atoms_per_rb) * ATOM;
                const uint8_t* sb0 = pr.sfB + ((size_t)(n0 / 128) * atoms_per_rb) * ATOM;
                const uint8_t* sb1 = sb0 + (size_t)atoms_per_rb * ATOM;
                prefetch_tmap(&mp.tmA);
                prefetch_tmap(&mp.tmB);
                for (int c = 0; c < nks; c++, it++) {
                    const int s = it % STAGES;
                    if (!mbar_wait(empty(s), ((it / STAGES) & 1) ^ 1, &g_fp4_err)) { ok = false; break; }
                    const uint32_t st = sbase + s * STAGE_BYTES;
                    mbar_arrive_expect_tx(full(s), A_BYTES + B_BYTES + sf_bytes);
                    tma_load_2d(st, &mp.tmA, c * BKB, m0, full(s));     // rows >= M read as zeros
                    tma_load_2d(st + A_BYTES, &mp.tmB, c * BKB, n0, full(s));
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
                const int nks = P.p[find(tile)].K / (2 * BKB);
                if (!mbar_wait(tempty, (tcount & 1) ^ 1, &g_fp4_err)) { ok = false; break; }
                tc_fence_after();
                for (int c = 0; c < nks; c++, it++) {
                    const int s = it % STAGES;
                    // the scale copies' completion implies the stage's operands have landed
                    if (!mbar_wait(sfready(s), (it / STAGES) & 1, &g_fp4_err)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t st = sbase + s * STAGE_BYTES;
                    const uint32_t sfa_t = tmem_base + SF_COL + s * SF_COLS_PER_STAGE;
                    const uint32_t sfb_t = sfa_t + SFA_COLS;
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
    } else if (warp == SF_WARP) {
        // -------------------------------------------------- scale-copy issuer
        // The copies of stage s go into its own TMEM slot, which the MMAs of
        // stage s - STAGES have finished reading before the producer refilled
        // the stage (it waits for their commit).
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x) {
                const int nks = P.p[find(tile)].K / (2 * BKB);
                for (int c = 0; c < nks; c++, it++) {
                    const int s = it % STAGES;
                    if (!mbar_wait(full(s), (it / STAGES) & 1, &g_fp4_err)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t sfa_t = tmem_base + SF_COL + s * SF_COLS_PER_STAGE;
                    const uint32_t sfb_t = sfa_t + SFA_COLS;
                    const uint32_t sfa_s = sbase + s * STAGE_BYTES + A_BYTES + B_BYTES;
#pragma unroll
                    for (int g = 0; g < G; g++) {
                        tmem_cp_32x128b_x4(sfa_t + 4 * g, sdesc_plain(sfa_s + g * ATOM));
                        tmem_cp_32x128b_x4(sfb_t + 8 * g, sdesc_plain(sfa_s + (G + g) * ATOM));
                        tmem_cp_32x128b_x4(sfb_t + 8 * g + 4, sdesc_plain(sfa_s + (2 * G + g) * ATOM));
                    }
                    tc_commit(sfready(s));
                }
            }
        }
        __syncwarp();
    } else {
        // --------------------------------------------------------- epilogue
        const int q = warp & 3, h = (warp - 2) >> 2;
        uint8_t* stg = smem + STG_OFF + (warp - 2) * STG_WARP;
        const uint32_t stg_s = smem_u32(stg);
        uint32_t tcount = 0;
        for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x, tcount++) {
            const int pi = find(tile);
            const Fp4Prob& pr = P.p[pi];
            const int local = tile - pr.tile_begin;
            const int m0 = (local % pr.mt) * BM, n0 = (local / pr.mt) * BN;
            const float gscale = NV ? __ldg(pr.gA) * __ldg(pr.gB) : 1.0f;
            if (!mbar_wait(tfull, tcount & 1, &g_fp4_err)) break;
            tc_fence_after();
            uint32_t v[4][32];                           // all four loads in flight, one wait
            const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + h * 128;
#pragma unroll
            for (int c = 0; c < 4; c++) tmem_ld32(taddr + c * 32, v[c]);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty);          // the next tile's MMAs may start
            if constexpr (QOUT && !NV) {
                const int row = m0 + q * 32 + lane;
                if (row < pr.M) {
                    const int c0 = n0 + h * 128;         // this thread's 128 columns: 4 blocks of 32
                    uint8_t* crow = P.q.codes + (size_t)row * (pr.N / 2) + c0 / 2;
                    uint32_t e4 = 0u;
#pragma unroll
                    for (int b = 0; b < 4; b++) {
                        float y[32];
                        float m = 0.0f;
#pragma unroll
                        for (int e = 0; e < 32; e++) {
                            y[e] = __bfloat162float(__float2bfloat16_rn(__uint_as_float(v[b][e])));
                            m = fmaxf(m, fabsf(y[e]));
                        }
                        m = fmaxf(m, kAmaxMin);
                        const int E = (int)((__float_as_uint(m) >> 23) & 0xFF) - 127;   // m is normal
                        const float inv = __uint_as_float((uint32_t)(127 + 2 - E) << 23);
                        uint32_t w[4];
#pragma unroll
                        for (int o = 0; o < 4; o++) w[o] = mxfp4_encode8<true>(y + 8 * o, inv);
                        *reinterpret_cast<uint4*>(crow + 16 * b) = make_uint4(w[0], w[1], w[2], w[3]);
                        e4 |= (uint32_t)(E - 2 + 127) << (8 * b);
                    }
                    *reinterpret_cast<uint32_t*>(P.q.scales + (size_t)row * (pr.N / 32) + c0 / 32) = e4;
                }
                continue;
            }
            if constexpr (QOUT) {
                const float g = div_rn(fmaxf(__ldg(P.q.amax), kAmaxMin), kFp8Max * kFp4Max);
                if (tcount == 0 && blockIdx.x == 0 && warp == 2 && lane == 0) *P.q.g = g;
                const Recip dg(g), d6(kFp4Max);
                const int row = m0 + q * 32 + lane;
                if (row < pr.M) {
                    const int c0 = n0 + h * 128;         // this thread's 128 columns
                    uint8_t* crow = P.q.codes + (size_t)row * (pr.N / 2) + c0 / 2;
                    uint32_t sc[2] = {0u, 0u};
#pragma unroll
                    for (int b2 = 0; b2 < 4; b2++) {     // two 16-column blocks per 16-byte store
                        uint2 pk[2];
#pragma unroll
                        for (int u = 0; u < 2; u++) {
                            const int b = 2 * b2 + u;
                            float y[16];
#pragma unroll
                            for (int e = 0; e < 16; e++)
                                y[e] = __bfloat162float(__float2bfloat16_rn(
                                    __uint_as_float(v[b >> 1][(b & 1) * 16 + e]) * gscale));
                            uint32_t bcode;
                            pk[u] = nvfp4_block16(y, g, dg, d6, bcode);
                            sc[b >> 2] |= bcode << (8 * (b & 3));
                        }
                        *reinterpret_cast<uint4*>(crow + 16 * b2) = make_uint4(pk[0].x, pk[0].y, pk[1].x, pk[1].y);
                    }
                    *reinterpret_cast<uint2*>(P.q.scales + (size_t)row * (pr.N / 16) + c0 / 16) = make_uint2(sc[0], sc[1]);
                }
                continue;
            }
            // 16-column chunks through the staging tile, each written by one TMA store
            // (rows past M fall outside the tensor and are not written)
#pragma unroll
            for (int j = 0; j < 8; j++) {
                uint32_t w[8];
#pragma unroll
                for (int e = 0; e < 8; e++) {
                    const __nv_bfloat162 p = __floats2bfloat162_rn(__uint_as_float(v[j >> 1][(j & 1) * 16 + 2 * e]) * gscale,
                                                                   __uint_as_float(v[j >> 1][(j & 1) * 16 + 2 * e + 1]) * gscale);
                    w[e] = *reinterpret_cast<const uint32_t*>(&p);
                }
                if (lane == 0) bulk_wait_read0();        // the previous store has read the staging tile
                __syncwarp();
                const int sw = (lane >> 2) & 1;          // 32-byte swizzle: chunk c of row r at c ^ ((r >> 2) & 1)
                *reinterpret_cast<uint4*>(stg + lane * 32 + ((0 ^ sw) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
                *reinterpret_cast<uint4*>(stg + lane * 32 + ((1 ^ sw) << 4)) = make_uint4(w[4], w[5], w[6], w[7]);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) tma_store_2d(&P.m[pi].tmY, stg_s, n0 + h * 128 + j * 16, m0 + q * 32);
            }
        }
        if (lane == 0) bulk_wait_all0();                 // stores complete before the CTA exits
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

size_t sf_bytes(bool nv, int R, int K) { return (size_t)R * (K / (nv ? 16 : 32)); }
size_t round1k(size_t b) { return (b + 1023) & ~size_t(1023); }

// Fills problem slot `p` (tensor maps and tile bookkeeping); false if a
// tensor map cannot be encoded.
bool fill_problem(Fp4Maps& mp, Fp4Prob& p, const uint8_t* qA, const uint8_t* sfA, const float* gA, const uint8_t* qB,
                  const uint8_t* sfB, const float* gB, uint16_t* Y, int M, int N, int K, int& tiles) {
    if (!encode_tmap_2d_u8(&mp.tmA, qA, (uint64_t)K / 2, (uint64_t)M, (uint64_t)K / 2, BKB, BM) ||
        !encode_tmap_2d_u8(&mp.tmB, qB, (uint64_t)K / 2, (uint64_t)N, (uint64_t)K / 2, BKB, BN))
        return false;
    if (Y && !encode_tmap_2d_swz(&mp.tmY, Y, 2, (uint64_t)N, (uint64_t)M, (uint64_t)N * 2, 16, 32, 32)) return false;
    if (!Y) memset(&mp.tmY, 0, sizeof(mp.tmY));                 // QOUT: no bf16 output
    p.sfA = sfA; p.sfB = sfB; p.gA = gA; p.gB = gB; p.Y = Y;
    p.M = M; p.N = N; p.K = K;
    p.mt = (M + BM - 1) / BM;
    p.tile_begin = tiles;
    tiles += p.mt * (N / BN);
    return true;
}

qz_status launch_table(bool nv, const Fp4Params& P, cudaStream_t st, bool qout = false) {
    const void* fn = qout ? (nv ? (const void*)fp4_gemm_kernel<true, true> : (const void*)fp4_gemm_kernel<false, true>)
                          : nv ? (const void*)fp4_gemm_kernel<true> : (const void*)fp4_gemm_kernel<false>;
    QZ_TRY(opt_in_smem(fn, SMEM_BYTES));
    const int grid = std::min(P.total_tiles, num_sms());
    if (qout && nv)
        fp4_gemm_kernel<true, true><<<grid, THREADS, SMEM_BYTES, st>>>(P);
    else if (qout)
        fp4_gemm_kernel<false, true><<<grid, THREADS, SMEM_BYTES, st>>>(P);
    else if (nv)
        fp4_gemm_kernel<true><<<grid, THREADS, SMEM_BYTES, st>>>(P);
    else
        fp4_gemm_kernel<false><<<grid, THREADS, SMEM_BYTES, st>>>(P);
    return launch_status();
}

} // namespace

size_t ws_gemm_fp4(int M, int N, int K) {
    // re-laid scales of A and B (NVFP4 size; MXFP4 uses half)
    return round1k(sf_bytes(true, M, K)) + round1k(sf_bytes(true, N, K));
}

size_t ws_gemm_nvfp4_grouped(int count, int kmax) {
    // re-laid scales of each problem's A (at most 128 rows)
    return (size_t)count * round1k(sf_bytes(true, 128, kmax));
}

size_t prepared_fp4_scale_bytes(int rows, int K, bool nv) { return sf_bytes(nv, (rows + 127) / 128 * 128, K); }

qz_status fp4_error_read_and_clear() {
    unsigned int v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_fp4_err, sizeof(v)) != cudaSuccess) return QZ_ERR_CUDA;
    if (v && cudaMemcpyToSymbol(g_fp4_err, &z, sizeof(z)) != cudaSuccess) return QZ_ERR_CUDA;
    return v ? QZ_ERR_TIMEOUT : QZ_OK;
}

qz_status gemm_fp4_launch(bool nv, const uint8_t* qA, const uint8_t* sA, const float* gA,
                          const uint8_t* qB, const uint8_t* sB, const float* gB, uint16_t* Y,
                          int M, int N, int K, void* ws, size_t ws_bytes, cudaStream_t st) {
    return gemm_fp4_launch_q(nv, qA, sA, gA, qB, sB, gB, Y, nullptr, M, N, K, ws, ws_bytes, st);
}

qz_status gemm_fp4_launch_q(bool nv, const uint8_t* qA, const uint8_t* sA, const float* gA,
                            const uint8_t* qB, const uint8_t* sB, const float* gB, uint16_t* Y,
                            const qz_fp4_out* yq, int M, int N, int K, void* ws, size_t, cudaStream_t st) {
    uint8_t* wsA = static_cast<uint8_t*>(ws);
    uint8_t* wsB = wsA + round1k(sf_bytes(true, M, K));
    const int ks = K / (nv ? 16 : 32);
    RelayParams R;
    R.count = 2;
    R.j[0] = RelayJob{sA, wsA, 0, M, ks};
    R.j[1] = RelayJob{sB, wsB, relay_words(M, ks), N, ks};
    R.total_words = relay_words(M, ks) + relay_words(N, ks);
    QZ_TRY(relayout(R, st));
    Fp4Params P;
    int tiles = 0;
    if (!fill_problem(P.m[0], P.p[0], qA, wsA, gA, qB, wsB, gB, Y, M, N, K, tiles)) return QZ_ERR_CUDA;
    P.q = yq ? Fp4Qout{yq->codes, yq->scales, yq->amax, yq->g} : Fp4Qout{nullptr, nullptr, nullptr, nullptr};
    P.count = 1;
    P.total_tiles = tiles;
    return launch_table(nv, P, st, yq != nullptr);
}

qz_status gemm_nvfp4_grouped_launch(const qz_nvfp4_problem* problems, int count, void* ws, size_t,
                                    cudaStream_t st) {
    // every problem's A scales re-laid in one launch (B's come prepared)
    int kmax = 0;
    for (int i = 0; i < count; i++) kmax = std::max(kmax, problems[i].K);
    const size_t slot = round1k(sf_bytes(true, 128, kmax));
    uint8_t* wsb = static_cast<uint8_t*>(ws);
    RelayParams R;
    R.count = count;
    R.total_words = 0;
    for (int i = 0; i < count; i++) {
        const qz_nvfp4_problem& q = problems[i];
        R.j[i] = RelayJob{q.sA, wsb + (size_t)i * slot, R.total_words, q.M, q.K / 16};
        R.total_words += relay_words(q.M, q.K / 16);
    }
    QZ_TRY(relayout(R, st));
    // as few launches as the parameter space allows, with equal shares of problems
    const int launches = (count + FP4_PER_LAUNCH - 1) / FP4_PER_LAUNCH;
    const int share = (count + launches - 1) / launches;
    for (int i0 = 0; i0 < count; i0 += share) {
        Fp4Params P;
        int tiles = 0;
        P.count = std::min(share, count - i0);
        for (int i = 0; i < P.count; i++) {
            const qz_nvfp4_problem& q = problems[i0 + i];
            if (!fill_problem(P.m[i], P.p[i], q.qA, wsb + (size_t)(i0 + i) * slot, q.gA, q.qB, q.sB_prepared, q.gB, q.Y,
                              q.M, q.N, q.K, tiles))
                return QZ_ERR_CUDA;
        }
        P.total_tiles = tiles;
        QZ_TRY(launch_table(true, P, st));
    }
    return QZ_OK;
}

qz_status prepare_fp4_scales_launch(const uint8_t* scales, int rows, int K, bool nv, uint8_t* out,
                                    cudaStream_t st) {
    RelayParams R;
    R.count = 1;
    R.j[0] = RelayJob{scales, out, 0, rows, K / (nv ? 16 : 32)};
    R.total_words = relay_words(rows, K / (nv ? 16 : 32));
    return relayout(R, st);
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
