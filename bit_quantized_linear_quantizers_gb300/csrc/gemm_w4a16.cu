// gemm_w4a16.cu -- W4A16 GEMM for decode: Y[M, N] = A[M, K] (bf16) times an
// INT4 weight with one bf16 scale per 128 rows of K, fp32 accumulation, bf16
// output. This is the fused unpack + dequant + matmul kernel that
// "量化：让每一步搬更少的字节" (路线一) calls for: at decode sizes the time
// is the weight bytes read from HBM, so the kernel streams the packed
// weights exactly once and does the rest on chip.
//
// Design (one GB300, sm_103a):
//  * swap A and B: the MMA computes Y^T = W^T A^T, so 16 weight columns fill
//    the MMA's 16-row side and up to 8 tokens its 8-wide side; M <= 64 tokens
//    take MT/8 MMAs per weight fragment (mma.m16n8k16, bf16 in, fp32 out).
//  * one CTA per tile of NT weight columns and the whole K range: NT is
//    chosen so that the tile count is about the SM count (no split-K and no
//    scratch memory); grouped launches run many problems' tiles in one grid.
//  * a producer warp stages 256-deep K slices of the weights, the
//    activations and the scales into shared memory with TMA bulk copies
//    (cp.async.bulk) completing on mbarriers; NT/16 MMA warps consume them.
//  * the INT4 codes are exact integers in bf16, so each 128-deep group is
//    multiplied exactly and the fp32 group sum is scaled by its bf16 scale
//    (folding the scale into bf16 weights would round).
//  * k inside a 32-deep chunk is permuted consistently for both operands:
//    thread (g, t) takes the whole packed word of k-octet t, so one 32-bit
//    shared load feeds two MMA k-steps, and the matching activations are 8
//    consecutive bf16 (one 16-byte load).
#include "qz_gemm.cuh"

#include <cuda_bf16.h>
#include <algorithm>

namespace qz {

namespace {

__device__ unsigned int g_w4a16_err;

constexpr int KT = 256;                 // K per pipeline stage (two scale groups)
constexpr int WPAD = 8;                 // words of padding per weight row (bank spread)
constexpr int AROW = KT * 2 + 64;       // bytes per activation row in shared memory
constexpr int NTMAX = 128;

struct Prob {
    const uint16_t* A;
    const uint32_t* q;
    const uint16_t* s;
    uint16_t* Y;
    int M, N, K;
    int nt;          // tile width (columns), multiple of 16
    int cta_begin;   // first CTA index of this problem
};

struct Params {
    int count;
    Prob p[kW4A16MaxProblems];
};

struct Layout {
    int nt, mt, ns;
    uint32_t w_bytes, a_bytes, s_bytes, stage_bytes;
    __host__ __device__ Layout(int nt_, int mt_, int ns_) : nt(nt_), mt(mt_), ns(ns_) {
        w_bytes = 32u * (uint32_t)(nt + WPAD) * 4u;
        a_bytes = (uint32_t)mt * AROW;
        s_bytes = 2u * NTMAX * 2u;
        stage_bytes = w_bytes + a_bytes + s_bytes;
    }
    __host__ __device__ uint32_t smem_bytes() const { return (uint32_t)ns * stage_bytes + 2u * ns * 8u; }
};

__device__ __forceinline__ void mma_bf16(float c[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
                 "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Byte B of an offset-binary word u (two 4-bit codes u = q + 8 per byte) ->
// bf16x2 (q_even, q_odd). The even code comes from byte B of u, the odd code
// from byte B of u >> 4 (u4); each lands in mantissa bits 0-3 of its bf16
// half (value 128 + u), and one fma (x * 1 - 136) gives q exactly.
template <int B>
__device__ __forceinline__ uint32_t nib_pair(uint32_t u, uint32_t u4) {
    const uint32_t r = __byte_perm(u, u4, (uint32_t)B | ((uint32_t)(4 + B) << 8));
    uint32_t v;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(v) : "r"(r), "r"(0x000F000Fu), "r"(0x43004300u));
    uint32_t out;
    const uint32_t one = 0x3F803F80u;    // bf16x2 (1.0, 1.0)
    const uint32_t add = 0xC308C308u;    // bf16x2 (-136.0, -136.0)
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(out) : "r"(v), "r"(one), "r"(add));
    return out;
}

template <int MT>
__global__ void __launch_bounds__((NTMAX / 16 + 1) * 32)
w4a16_kernel(const __grid_constant__ Params P, int nt_max, int ns) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int MB = MT / 8;                       // 8-token MMA blocks
    const int nwarps_c = nt_max / 16;                // consumer warps
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // ---- locate problem and tile
    int lo = 0, hi = P.count - 1;
    while (lo < hi) {                                // last problem with cta_begin <= blockIdx.x
        const int mid = (lo + hi + 1) >> 1;
        if (P.p[mid].cta_begin <= (int)blockIdx.x) lo = mid; else hi = mid - 1;
    }
    const Prob& pr = P.p[lo];
    const int tile = blockIdx.x - pr.cta_begin;
    const int n0 = tile * pr.nt;
    const int ntv = min(pr.nt, pr.N - n0);           // valid columns (multiple of 16)
    const int nstage = (pr.K + KT - 1) / KT;
    const Layout L(nt_max, MT, ns);

    uint8_t* sW = smem;
    uint8_t* sA = smem + L.w_bytes;
    uint8_t* sS = sA + L.a_bytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)ns * L.stage_bytes);
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + ns);

    if (threadIdx.x == 0) {
        for (int i = 0; i < ns; i++) {
            mbar_init(full0 + 8 * i, 1);
            mbar_init(empty0 + 8 * i, nwarps_c);
        }
        fence_barrier_init();
    }
    __syncthreads();

    bool ok = true;
    if (warp == nwarps_c) {
        // ------------------------------------------------ producer warp
        const uint32_t wrow = (uint32_t)ntv * 4u, srow = (uint32_t)ntv * 2u;
        const int mrows = min(pr.M, MT);
        for (int s = 0; s < nstage && ok; s++) {
            const int k0 = s * KT;
            const int kl = min(KT, pr.K - k0);               // 256, or 128 for the last stage
            const uint32_t bytes = (uint32_t)(kl / 8) * wrow + (uint32_t)mrows * kl * 2u + (uint32_t)(kl / 128) * srow;
            const int slot = s % ns;
            if (s >= ns) ok = mbar_wait(empty0 + 8 * slot, ((s / ns) - 1) & 1, &g_w4a16_err);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            const uint32_t full = full0 + 8 * slot;
            if (lane == 0) mbar_arrive_expect_tx(full, bytes);
            __syncwarp();
            const uint32_t st = smem_u32(smem) + slot * L.stage_bytes;
            if (lane < kl / 8)
                bulk_g2s(st + lane * (uint32_t)(nt_max + WPAD) * 4u,
                         pr.q + (size_t)(k0 / 8 + lane) * pr.N + n0, wrow, full);
            for (int r = lane; r < mrows; r += 32)
                bulk_g2s(st + L.w_bytes + r * AROW, pr.A + (size_t)r * pr.K + k0, (uint32_t)kl * 2u, full);
            if (lane < kl / 128)
                bulk_g2s(st + L.w_bytes + L.a_bytes + lane * NTMAX * 2u,
                         pr.s + (size_t)(k0 / 128 + lane) * pr.N + n0, srow, full);
        }
    } else {
        // ------------------------------------------------- MMA warps
        const int g = lane >> 2, t = lane & 3;
        const bool active = warp * 16 < ntv;
        float acc[MB][4];
#pragma unroll
        for (int mb = 0; mb < MB; mb++) acc[mb][0] = acc[mb][1] = acc[mb][2] = acc[mb][3] = 0.0f;

        for (int s = 0; s < nstage; s++) {
            const int slot = s % ns;
            if (!mbar_wait(full0 + 8 * slot, (s / ns) & 1, &g_w4a16_err)) { ok = false; break; }
            const int ngrp = min(KT, pr.K - s * KT) / 128;
            if (active) {
                const uint32_t* w = reinterpret_cast<const uint32_t*>(sW + (size_t)slot * L.stage_bytes);
                const uint8_t* a = sA + (size_t)slot * L.stage_bytes;
                const uint16_t* sc = reinterpret_cast<const uint16_t*>(sS + (size_t)slot * L.stage_bytes);
#pragma unroll
                for (int grp = 0; grp < 2; grp++) {
                    if (grp >= ngrp) break;
                    float ag[MB][4];
#pragma unroll
                    for (int mb = 0; mb < MB; mb++) ag[mb][0] = ag[mb][1] = ag[mb][2] = ag[mb][3] = 0.0f;
#pragma unroll
                    for (int c = 0; c < 4; c++) {
                        const int j = grp * 4 + c;                       // 32-deep chunk in the stage
                        const uint32_t* wr = w + (size_t)(4 * j + t) * (nt_max + WPAD) + warp * 16 + g;
                        const uint32_t u0 = wr[0] ^ 0x88888888u;         // column n
                        const uint32_t u1 = wr[8] ^ 0x88888888u;         // column n + 8
                        const uint32_t v0 = u0 >> 4, v1 = u1 >> 4;
                        const uint32_t f0[4] = {nib_pair<0>(u0, v0), nib_pair<0>(u1, v1), nib_pair<1>(u0, v0),
                                                nib_pair<1>(u1, v1)};
                        const uint32_t f1[4] = {nib_pair<2>(u0, v0), nib_pair<2>(u1, v1), nib_pair<3>(u0, v0),
                                                nib_pair<3>(u1, v1)};
#pragma unroll
                        for (int mb = 0; mb < MB; mb++) {
                            const uint4 b = *reinterpret_cast<const uint4*>(a + (mb * 8 + g) * AROW + (32 * j + 8 * t) * 2);
                            mma_bf16(ag[mb], f0, b.x, b.y);
                            mma_bf16(ag[mb], f1, b.z, b.w);
                        }
                    }
                    const float s0 = bf16_bits_to_f32(sc[grp * NTMAX + warp * 16 + g]);
                    const float s1 = bf16_bits_to_f32(sc[grp * NTMAX + warp * 16 + g + 8]);
#pragma unroll
                    for (int mb = 0; mb < MB; mb++) {
                        acc[mb][0] = fmaf(s0, ag[mb][0], acc[mb][0]);
                        acc[mb][1] = fmaf(s0, ag[mb][1], acc[mb][1]);
                        acc[mb][2] = fmaf(s1, ag[mb][2], acc[mb][2]);
                        acc[mb][3] = fmaf(s1, ag[mb][3], acc[mb][3]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8 * slot);
        }
        // ---- epilogue: stage the tile as bf16 [MT][NT] in shared memory (stage 0)
        // after every warp has finished reading the pipeline buffers.
        asm volatile("bar.sync 1, %0;" ::"r"(nwarps_c * 32) : "memory");
        if (active && ok) {
            __nv_bfloat16* ys = reinterpret_cast<__nv_bfloat16*>(smem);
            const int n = warp * 16 + g;
#pragma unroll
            for (int mb = 0; mb < MB; mb++) {
                const int m = mb * 8 + 2 * t;
                ys[m * nt_max + n] = __float2bfloat16_rn(acc[mb][0]);
                ys[(m + 1) * nt_max + n] = __float2bfloat16_rn(acc[mb][1]);
                ys[m * nt_max + n + 8] = __float2bfloat16_rn(acc[mb][2]);
                ys[(m + 1) * nt_max + n + 8] = __float2bfloat16_rn(acc[mb][3]);
            }
        }
        asm volatile("bar.sync 1, %0;" ::"r"(nwarps_c * 32) : "memory");
        if (ok) {
            const int vec_per_row = ntv / 8;                 // 16-byte vectors per output row
            const int mrows = min(pr.M, MT);
            for (int i = threadIdx.x; i < mrows * vec_per_row; i += nwarps_c * 32) {
                const int m = i / vec_per_row, v = i - m * vec_per_row;
                const uint4 val = *reinterpret_cast<const uint4*>(smem + ((size_t)m * nt_max + v * 8) * 2);
                *reinterpret_cast<uint4*>(pr.Y + (size_t)m * pr.N + n0 + v * 8) = val;
            }
        }
    }
}

int choose_mt(int m) { return m <= 8 ? 8 : m <= 16 ? 16 : m <= 32 ? 32 : 64; }

template <int MT>
qz_status launch_mt(const Params& P, int total_ctas, int nt_max, cudaStream_t st) {
    const int sms = num_sms();
    // Few large tiles (about one per SM): deep pipeline, one CTA per SM.
    // Many tiles: two CTAs per SM so one CTA's epilogue overlaps another's loads.
    const int budget = total_ctas <= sms ? 200 * 1024 : 110 * 1024;
    int ns = (int)(budget / Layout(nt_max, MT, 1).stage_bytes);
    ns = std::max(2, std::min(ns, 8));
    const Layout L(nt_max, MT, ns);
    const int smem = (int)L.smem_bytes();
    static int smem_set[64];                       // per device: largest size opted in so far
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return QZ_ERR_UNSUPPORTED;
    if (smem > smem_set[dev]) {
        if (cudaFuncSetAttribute(w4a16_kernel<MT>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
            return QZ_ERR_CUDA;
        smem_set[dev] = smem;
    }
    const int threads = (nt_max / 16 + 1) * 32;
    w4a16_kernel<MT><<<total_ctas, threads, smem, st>>>(P, nt_max, ns);
    return launch_status();
}

} // namespace

size_t ws_gemm_w4a16(int, int, int) { return 0; }

qz_status w4a16_error_read_and_clear() {
    unsigned int v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_w4a16_err, sizeof(v)) != cudaSuccess) return QZ_ERR_CUDA;
    if (v && cudaMemcpyToSymbol(g_w4a16_err, &z, sizeof(z)) != cudaSuccess) return QZ_ERR_CUDA;
    return v ? QZ_ERR_TIMEOUT : QZ_OK;
}

qz_status gemm_w4a16_launch(const qz_w4a16_problem* problems, int count, void*, size_t, cudaStream_t st) {
    Params P;          // the kernel parameter block (copied at launch)
    const int sms = num_sms();
    int mmax = 0;
    for (int i = 0; i < count; i++) mmax = std::max(mmax, problems[i].M);
    // Tile width: with one problem, the smallest multiple of 16 giving at
    // most one tile per SM (capped at 128 columns); grouped problems use 128.
    int nt_max = NTMAX;
    if (count == 1) {
        const int N = problems[0].N;
        nt_max = std::min(NTMAX, 16 * (int)((N + 16LL * sms - 1) / (16LL * sms)));
    }
    int total = 0;
    P.count = count;
    for (int i = 0; i < count; i++) {
        const qz_w4a16_problem& q = problems[i];
        Prob& p = P.p[i];
        p.A = q.A;
        p.q = reinterpret_cast<const uint32_t*>(q.qweight);
        p.s = q.scale_bf16;
        p.Y = q.Y;
        p.M = q.M; p.N = q.N; p.K = q.K;
        p.nt = nt_max;
        p.cta_begin = total;
        total += (q.N + nt_max - 1) / nt_max;
    }
    switch (choose_mt(mmax)) {
    case 8: return launch_mt<8>(P, total, nt_max, st);
    case 16: return launch_mt<16>(P, total, nt_max, st);
    case 32: return launch_mt<32>(P, total, nt_max, st);
    default: return launch_mt<64>(P, total, nt_max, st);
    }
}

} // namespace qz
