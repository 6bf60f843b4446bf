// gemm_w4a16_tc.cu -- W4A16 GEMM for 17 to 64 tokens on the tcgen05 tensor
// cores: Y[M, N] = A[M, K] (bf16) times an INT4 weight with one bf16 scale per
// 128 rows of K, fp32 accumulation, bf16 output ("量化：让每一步搬更少的字节",
// 路线一: one kernel that unpacks, dequantizes and multiplies, so the packed
// weights cross HBM once).
//
// The MMA computes Y^T = W^T A^T: the 128 weight columns of a tile are the
// MMA's M side, the tokens its N side (N = MT = 32 or 64), so one staged
// activation slice serves 128 weight columns. Per CTA (one per SM, persistent
// over tiles of 128 weight columns x all of K, several problems per launch):
//  The pipeline moves in units of GU = 2 groups of 128 K (one stage, one TMEM
//  weight buffer, one hand-off between the warps per unit): each hand-off
//  costs a few hundred ns of mbarrier wake-up whatever the work behind it.
//  warp 0       TMA producer: per unit, for each of its 128-deep K groups the
//               packed weights (16 k-octet rows x 128 columns of int32, 8 KB)
//               and the activations (two 64-element x MT boxes, 128-byte
//               swizzle) into a ring.
//  warps 2-9    unpack: thread = one weight column (its TMEM lane); each of
//               its packed words (8 consecutive k) becomes 8 exact bf16
//               integers q in [-8, 7], and the 64 K of the thread's half of
//               each group go straight from registers into tensor memory
//               (tcgen05.st), which is where the MMA reads its A operand from
//               (double-buffered, 64 TMEM columns per group).
//  warp 1       MMA issuer (one thread): per group 8 x tcgen05.mma kind::f16
//               with A in TMEM and the activations from shared memory
//               (M = 128, N = MT, K = 16) into the group's own TMEM
//               accumulator (two units of accumulators in flight).
//  warps 10-13  promotion + epilogue: thread = one weight column (its TMEM
//               lane); per group it loads the MT partial sums, multiplies them
//               by the group's bf16 scale and adds them into fp32 registers
//               (the scale is not folded into bf16 weights, which would round);
//               at the end of the tile it rounds to bf16 into a shared-memory
//               tile [MT][128], from which each promotion warp's lane 0 writes
//               its rows to Y with bulk asynchronous stores (one 256-byte row
//               each), so the warps return to the accumulators at once.
// Every wait is bounded; on expiry the kernel records QZ_ERR_TIMEOUT and winds
// down.
#include "qz_tc.cuh"

#include <cuda_bf16.h>
#include <algorithm>

namespace qz {

namespace {

__device__ unsigned int g_w4tc_err;

constexpr int TN = 128;                           // weight columns per tile (MMA M)
constexpr int GK = 128;                           // K per group (one bf16 scale per column)
constexpr int GU = 2;                             // groups per pipeline unit
constexpr int W_BYTES = (GK / 8) * TN * 4;        // packed weights of one group: 8 KB
constexpr int NWT = 2;                            // unpacked weight units (in TMEM) in flight
constexpr int NAU = 2;                            // accumulator units in flight (GU accumulators each)
constexpr int UNPACK_WARPS = 8, PROMO_WARPS = 4;
constexpr int THREADS = (2 + UNPACK_WARPS + PROMO_WARPS) * 32;
constexpr int TC_PER_LAUNCH = 80;                 // problems per launch (kernel parameter space)

struct TcProb {
    CUtensorMap tmW;                              // qweight [K/8][N] int32, box 128 x 16, no swizzle
    CUtensorMap tmA;                              // A [M][K] bf16, box 64 x MT, 128-byte swizzle
    const uint16_t* S;                            // scale bf16 [K/128][N]
    uint16_t* Y;                                  // bf16 [M][N]
    int M, N, K;
    int tile_begin;
};

struct TcParams {
    TcProb p[TC_PER_LAUNCH];
    int count;
    int total_tiles;
};

template <int MT>
struct TcLayout {
    static constexpr int A_BYTES = MT * GK * 2;                       // two 64 x MT boxes per group
    static constexpr int A_OFF = GU * W_BYTES;                        // activations after the weights
    static constexpr int STAGE = (GU * (W_BYTES + A_BYTES) + 1023) / 1024 * 1024;
    static constexpr int STAGES = MT == 64 ? 4 : 6;       // 192 KB of ring
    static constexpr int YT_OFF = STAGES * STAGE + 1024;                // output tile after the barriers
    static constexpr int YT_BYTES = MT * TN * 2;
    static constexpr int SMEM = YT_OFF + YT_BYTES + 1024;
    static constexpr uint32_t ACC_COLS = NAU * GU * MT;                 // accumulators first
    static constexpr uint32_t WCOLS = GU * 64;                          // TMEM columns of one weight unit
    static constexpr uint32_t TMEM_COLS = ACC_COLS + NWT * WCOLS <= 128 ? 128
                                        : ACC_COLS + NWT * WCOLS <= 256 ? 256 : 512;
    static constexpr uint32_t IDESC = idesc_dense(1u, 1u, TN, MT);   // bf16 x bf16 -> fp32
};

// Packed word -> 8 exact bf16 integers (element 2B in the low nibble of byte B,
// two's complement). One byte-permute brings the even code of byte B (from w)
// and the odd one (from w >> 4) into the low nibbles of the two halves; one
// lop3 keeps the nibbles, flips their sign bit (u = q + 8) and sets the
// exponent of 128, so each half holds 128 + u exactly; one bf16x2 fma
// (x * 1 - 136) leaves q.
template <int B>
__device__ __forceinline__ uint32_t unpack_pair(uint32_t w, uint32_t w4) {
    const uint32_t r = __byte_perm(w, w4, (uint32_t)B | ((uint32_t)(4 + B) << 8));
    uint32_t v, out;
    asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(v) : "r"(r), "r"(0x000F000Fu), "r"(0x43084308u));
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(out) : "r"(v), "r"(0x3F803F80u), "r"(0xC308C308u));
    return out;
}

template <int MT>
__global__ void __launch_bounds__(THREADS, 1)
w4a16_tc_kernel(const __grid_constant__ TcParams P) {
    using L = TcLayout<MT>;
    constexpr int S = L::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * L::STAGE);
    auto full = [&](int s) { return smem_u32(bars + s); };
    auto empty = [&](int s) { return smem_u32(bars + S + s); };
    auto wfull = [&](int b) { return smem_u32(bars + 2 * S + b); };
    auto wempty = [&](int b) { return smem_u32(bars + 2 * S + NWT + b); };
    auto afull = [&](int b) { return smem_u32(bars + 2 * S + 2 * NWT + b); };
    auto aempty = [&](int b) { return smem_u32(bars + 2 * S + 2 * NWT + NAU + b); };
    auto ep_free = [&]() { return smem_u32(bars + 2 * S + 2 * NWT + 2 * NAU); };      // output tile free
    auto ep_full = [&]() { return smem_u32(bars + 2 * S + 2 * NWT + 2 * NAU + 1); };  // output tile written
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 2 * NWT + 2 * NAU + 2);
    uint16_t* ytile = reinterpret_cast<uint16_t*>(smem + L::YT_OFF);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    auto find = [&](int tile) {                   // last problem with tile_begin <= tile
        int lo = 0, hi = P.count - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (P.p[mid].tile_begin <= tile) lo = mid; else hi = mid - 1;
        }
        return lo;
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; s++) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 1);
        }
        for (int b = 0; b < NWT; b++) {
            mbar_init(wfull(b), UNPACK_WARPS);
            mbar_init(wempty(b), 1);
        }
        for (int b = 0; b < NAU; b++) {
            mbar_init(afull(b), 1);
            mbar_init(aempty(b), PROMO_WARPS);
        }
        mbar_init(ep_free(), PROMO_WARPS);
        mbar_init(ep_full(), PROMO_WARPS);
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), L::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // Programmatic dependent launch: the next kernel may start launching now;
    // this one waits for the previous kernel only before loading activations.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true, waited = false;
            for (int tile = blockIdx.x; tile < P.total_tiles && ok; tile += gridDim.x) {
                const TcProb& pr = P.p[find(tile)];
                const int n0 = (tile - pr.tile_begin) * TN;
                const int ng = pr.K / GK;
                prefetch_tmap(&pr.tmW);
                prefetch_tmap(&pr.tmA);
                for (int g0 = 0; g0 < ng; g0 += GU, it++) {
                    const int s = it % S, gu = min(GU, ng - g0);
                    if (!mbar_wait(empty(s), ((it / S) & 1) ^ 1, &g_w4tc_err)) { ok = false; break; }
                    const uint32_t st = sbase + s * L::STAGE;
                    mbar_arrive_expect_tx(full(s), (uint32_t)gu * (W_BYTES + L::A_BYTES));
                    for (int j = 0; j < gu; j++)                                    // columns past N: zeros
                        tma_load_2d(st + j * W_BYTES, &pr.tmW, n0, (g0 + j) * (GK / 8), full(s));
                    if (!waited) {
                        asm volatile("griddepcontrol.wait;" ::: "memory");
                        waited = true;
                    }
                    for (int j = 0; j < gu; j++) {                                  // tokens past M: zeros
                        const uint32_t sa = st + L::A_OFF + j * L::A_BYTES;
                        tma_load_2d(sa, &pr.tmA, (g0 + j) * GK, 0, full(s));
                        tma_load_2d(sa + MT * 128, &pr.tmA, (g0 + j) * GK + 64, 0, full(s));
                    }
                }
            }
            for (uint32_t j = it > (uint32_t)S ? it - S : 0; j < it; j++)
                mbar_wait(empty(j % S), (j / S) & 1, &g_w4tc_err);
        }
    } else if (warp == 1) {
        // -------------------------------------------------------- MMA issuer
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < P.total_tiles && ok; tile += gridDim.x) {
                const int ng = P.p[find(tile)].K / GK;
                for (int g0 = 0; g0 < ng; g0 += GU, it++) {
                    const int s = it % S, wb = it % NWT, ab = it % NAU, gu = min(GU, ng - g0);
                    if (!mbar_wait(aempty(ab), ((it / NAU) & 1) ^ 1, &g_w4tc_err)) { ok = false; break; }
                    if (!mbar_wait(full(s), (it / S) & 1, &g_w4tc_err)) { ok = false; break; }
                    if (!mbar_wait(wfull(wb), (it / NWT) & 1, &g_w4tc_err)) { ok = false; break; }
                    tc_fence_after();
                    for (int j = 0; j < gu; j++) {
                        const uint32_t d = tmem_base + (uint32_t)(ab * GU + j) * MT;
                        const uint32_t sa = sbase + s * L::STAGE + L::A_OFF + j * L::A_BYTES;
#pragma unroll
                        for (int ks = 0; ks < GK / 16; ks++) {           // K = 16 per MMA = 8 TMEM columns
                            const int slab = ks >> 2, kk = ks & 3;       // 64-element slab, 32-byte step
                            const uint32_t at = tmem_base + L::ACC_COLS + wb * L::WCOLS + j * 64 + ks * 8;
                            const uint64_t bd = sdesc_k_sw128(sa + slab * (MT * 128)) + kk * 2;
                            mma_f16_ts(d, at, bd, L::IDESC, ks > 0);
                        }
                    }
                    tc_commit(empty(s));
                    tc_commit(wempty(wb));
                    tc_commit(afull(ab));
                }
            }
            if (it > 0) mbar_wait(afull((it - 1) % NAU), ((it - 1) / NAU) & 1, &g_w4tc_err);
        }
        __syncwarp();
    } else if (warp < 2 + UNPACK_WARPS) {
        // ------------------------------------------------------------ unpack
        const int q = warp & 3, h = (warp - 2) >> 2;     // TMEM lane quarter; half of the group's K
        const int n = q * 32 + lane;                     // weight column = TMEM lane
        uint32_t it = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < P.total_tiles && ok; tile += gridDim.x) {
            const int ng = P.p[find(tile)].K / GK;
            for (int g0 = 0; g0 < ng; g0 += GU, it++) {
                const int s = it % S, wb = it % NWT, gu = min(GU, ng - g0);
                if (!mbar_wait(full(s), (it / S) & 1, &g_w4tc_err)) { ok = false; break; }
                if (!mbar_wait(wempty(wb), ((it / NWT) & 1) ^ 1, &g_w4tc_err)) { ok = false; break; }
                tc_fence_after();
                for (int j = 0; j < gu; j++) {
                    const uint32_t* wsrc = reinterpret_cast<const uint32_t*>(smem + s * L::STAGE + j * W_BYTES);
                    uint32_t o[32];
#pragma unroll
                    for (int i = 0; i < 8; i++) {                // k-octet rows 8h .. 8h+7
                        const uint32_t w = wsrc[(8 * h + i) * TN + n], w4 = w >> 4;
                        o[4 * i + 0] = unpack_pair<0>(w, w4);
                        o[4 * i + 1] = unpack_pair<1>(w, w4);
                        o[4 * i + 2] = unpack_pair<2>(w, w4);
                        o[4 * i + 3] = unpack_pair<3>(w, w4);
                    }
                    tmem_st32(tmem_base + ((uint32_t)(q * 32) << 16) + L::ACC_COLS + wb * L::WCOLS + j * 64 + h * 32, o);
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(wfull(wb));
            }
        }
    } else {
        // ------------------------------------------------ promotion + epilogue
        const int q = warp & 3;                          // TMEM lane quarter
        const int n = q * 32 + lane;                     // weight column within the tile
        uint32_t it = 0, tcount = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < P.total_tiles && ok; tile += gridDim.x) {
            const TcProb& pr = P.p[find(tile)];
            const int n0 = (tile - pr.tile_begin) * TN;
            const int ng = pr.K / GK;
            const bool col_ok = n0 + n < pr.N;
            const uint16_t* srow = pr.S + n0 + (col_ok ? n : 0);
            float acc[MT];
#pragma unroll
            for (int i = 0; i < MT; i++) acc[i] = 0.0f;
            uint32_t sraw[GU];                            // scales of the unit's groups, one unit ahead
#pragma unroll
            for (int j = 0; j < GU; j++) sraw[j] = j < ng ? __ldg(srow + (size_t)j * pr.N) : 0u;
            for (int g0 = 0; g0 < ng; g0 += GU, it++) {
                const int gu = min(GU, ng - g0);
                float sc[GU];
#pragma unroll
                for (int j = 0; j < GU; j++) {
                    sc[j] = bf16_bits_to_f32(sraw[j]);
                    const int gn = g0 + GU + j;
                    if (gn < ng) sraw[j] = __ldg(srow + (size_t)gn * pr.N);
                }
                const int ab = it % NAU;
                if (!mbar_wait(afull(ab), (it / NAU) & 1, &g_w4tc_err)) { ok = false; break; }
                tc_fence_after();
                for (int j = 0; j < gu; j++) {
                    const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(ab * GU + j) * MT;
#pragma unroll
                    for (int c = 0; c < MT / 16; c++) {
                        uint32_t v[16];
                        tmem_ld16(taddr + c * 16, v);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 16; i++) acc[c * 16 + i] = fmaf(__uint_as_float(v[i]), sc[j], acc[c * 16 + i]);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(aempty(ab));
            }
            if (!ok) break;
            // the output tile: free (this warp's stores of the last tile have read
            // it), written by all four warps, then stored row by row
            const uint32_t tp = tcount & 1;
            if (lane == 0) {
                asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
                mbar_arrive(ep_free());
            }
            if (!mbar_wait(ep_free(), tp, &g_w4tc_err)) break;
#pragma unroll
            for (int m = 0; m < MT; m++) ytile[m * TN + n] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[m]));
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(ep_full());
                if (!mbar_wait(ep_full(), tp, &g_w4tc_err)) { ok = false; }
                else {
                    const int mrows = min(pr.M, MT);
                    const uint32_t rb = (uint32_t)min(TN, pr.N - n0) * 2;           // bytes of a row in Y
                    for (int m = q; m < mrows; m += PROMO_WARPS) {
                        const uint32_t src = smem_u32(ytile + m * TN);
                        uint16_t* dst = pr.Y + (size_t)m * pr.N + n0;
                        asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                                     ::"l"(dst), "r"(src), "r"(rb) : "memory");
                    }
                    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
                }
            }
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            tcount++;
        }
        if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, L::TMEM_COLS);
    }
}

template <int MT>
qz_status launch_tc(const TcParams& P, cudaStream_t st, bool early) {
    using L = TcLayout<MT>;
    QZ_TRY(opt_in_smem((const void*)w4a16_tc_kernel<MT>, L::SMEM));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(std::min(P.total_tiles, num_sms()));
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = (size_t)L::SMEM;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = early ? 1 : 0;                 // without it: after all earlier work on the stream
    if (cudaLaunchKernelEx(&cfg, w4a16_tc_kernel<MT>, P) != cudaSuccess) return QZ_ERR_CUDA;
    return launch_status();
}

} // namespace

qz_status w4a16_tc_error_read_and_clear() {
    unsigned int v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_w4tc_err, sizeof(v)) != cudaSuccess) return QZ_ERR_CUDA;
    if (v && cudaMemcpyToSymbol(g_w4tc_err, &z, sizeof(z)) != cudaSuccess) return QZ_ERR_CUDA;
    return v ? QZ_ERR_TIMEOUT : QZ_OK;
}

// Problems with 17..64 tokens (mt = 32 or 64 padded rows), up to 80 per launch.
qz_status w4a16_tc_launch(const qz_w4a16_problem* problems, int count, int mt, cudaStream_t st, bool early) {
    // as few launches as the parameter space allows, with equal shares of problems
    const int launches = (count + TC_PER_LAUNCH - 1) / TC_PER_LAUNCH;
    const int share = (count + launches - 1) / launches;
    for (int i0 = 0; i0 < count; i0 += share) {
        TcParams P;
        int tiles = 0;
        P.count = std::min(share, count - i0);
        // deepest K first: the CTAs take tiles round-robin, so the long tiles
        // spread over the SMs and the launch ends on short ones
        int order[TC_PER_LAUNCH];
        for (int i = 0; i < P.count; i++) order[i] = i0 + i;
        std::stable_sort(order, order + P.count, [&](int a, int b) { return problems[a].K > problems[b].K; });
        for (int i = 0; i < P.count; i++) {
            const qz_w4a16_problem& q = problems[order[i]];
            TcProb& p = P.p[i];
            if (!encode_tmap_2d(&p.tmW, q.qweight, 4, (uint64_t)q.N, (uint64_t)q.K / 8, (uint64_t)q.N * 4, TN,
                                GK / 8, false) ||
                !encode_tmap_2d(&p.tmA, q.A, 2, (uint64_t)q.K, (uint64_t)q.M, (uint64_t)q.K * 2, 64, (uint32_t)mt,
                                true))
                return QZ_ERR_CUDA;
            p.S = q.scale_bf16;
            p.Y = q.Y;
            p.M = q.M; p.N = q.N; p.K = q.K;
            p.tile_begin = tiles;
            tiles += (q.N + TN - 1) / TN;
        }
        P.total_tiles = tiles;
        const qz_status s = mt == 32 ? launch_tc<32>(P, st, early) : launch_tc<64>(P, st, early);
        if (s != QZ_OK) return s;
    }
    return QZ_OK;
}

} // namespace qz
