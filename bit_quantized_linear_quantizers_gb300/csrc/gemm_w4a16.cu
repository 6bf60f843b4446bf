// gemm_w4a16.cu -- W4A16 GEMM for decode: Y[M, N] = A[M, K] (bf16) times an
// INT4 weight with one bf16 scale per 128 rows of K, fp32 accumulation, bf16
// output. This is the fused unpack + dequant + matmul kernel that
// "量化：让每一步搬更少的字节" (路线一) calls for: at decode sizes the time
// is the weight bytes read from HBM, so the kernel streams the packed
// weights exactly once and does the rest on chip.
//
// Kernels by token count:
//  * up to 8 tokens with K <= 8192: w4a16_bulk_kernel, the register-direct
//    kernel's arithmetic with the CTA's whole weight range staged in shared
//    memory by TMA boxes requested at once (see its section below).
//  * up to 8 tokens, deeper K: w4a16_rd_kernel, register-direct. A CTA owns 32
//    weight columns; its 8 warps split K by 128-deep scale groups. Each lane
//    loads the packed weights with one coalesced 16-byte load per k-octet row
//    (4 consecutive columns) straight into registers, after an L2 prefetch
//    of the CTA's whole weight range has been issued: no shared-memory
//    staging, so several small CTAs share each SM, their loads overlap, and
//    the next launch's CTAs start as soon as any of these finish. The warps' partial sums meet in shared memory and are
//    added in a fixed order.
//  * 9 to 16 tokens: w4a16_kernel, persistent CTAs (at most one per SM) walking
//    tiles of NT weight columns x the whole K range, fed by a producer thread
//    that stages 256-deep K slices through an mbarrier ring with 2-D tensor TMA
//    (weights as 32-column x 32-row boxes with the 128-byte swizzle,
//    activations as one 256 x MT box, scales as one NT x 2 box). Two MMA
//    warps share each 16-column slice, one per 128-deep scale group of every
//    stage. Grouped launches (a decoder step's linears) stream all problems'
//    tiles through one pipeline.
//  * 17 to 64 tokens: the tcgen05 kernel of gemm_w4a16_tc.cu.
// Common to the mma.sync kernels:
//  * swap A and B: the MMA computes Y^T = W^T A^T, so 16 weight columns fill
//    the MMA's 16-row side and up to 8 tokens its 8-wide side (mma.m16n8k16,
//    bf16 in, fp32 out; MT/8 MMAs per weight fragment).
//  * the INT4 codes are exact integers in bf16, so each 128-deep group is
//    multiplied exactly and the fp32 group sum is scaled by its bf16 scale
//    (folding the scale into bf16 weights would round).
//  * in the register-direct kernel the unpack stops at the biased code v = q + 136
//    (exact in bf16) and the MMA sums a*v; a second MMA of the activations
//    against a fragment of ones gives sum(a) over the same k, and the group
//    sum is sum(a*v) - 136*sum(a). That drops one bf16x2 FMA per code pair.
//  * k inside a 32-deep chunk is permuted consistently for both operands:
//    thread (g, t) takes the whole packed word of k-octet t, so one word feeds
//    two MMA k-steps, and the matching activations are 8 consecutive bf16
//    (one 16-byte load).
#include "qz_tc.cuh"

#include <cuda_bf16.h>
#include <algorithm>
#include <mutex>

namespace qz {

namespace {

__device__ unsigned int g_w4a16_err;

constexpr int KT = 256;                 // K per pipeline stage (two scale groups)

// Widest tile of the TMA-staged kernel (9 to 16 tokens): 128 columns, 16 MMA warps.
__host__ __device__ constexpr int ntmax_for(int) { return 128; }
constexpr int PER_LAUNCH = 56;          // problems per launch (kernel parameter space: 32 KB)
constexpr int WBOX = 4096;              // one 32-column x 32-row weight box

struct Prob {
    CUtensorMap tmW;                    // qweight [K/8][N] int32, box 32 x 32, 128-byte swizzle
    CUtensorMap tmA;                    // A [M][K] bf16, box 256 x MT
    CUtensorMap tmS;                    // scale [K/128][N] bf16, box NT x 2
    uint16_t* Y;
    int M, N, K;
    int tile_begin;                     // first tile index of this problem
};

// Kernel parameter block of NP problems: a single call passes a one-problem
// block, so its launch does not copy a table sized for a whole group.
template <int NP>
struct ParamsN {
    Prob p[NP];
    int count;
    int total_tiles;
};

struct Layout {
    uint32_t w_bytes, a_bytes, s_bytes, stage_bytes, y_pitch, y_bytes;
    __host__ __device__ Layout(int nt, int mt) {
        w_bytes = (uint32_t)(nt / 32) * WBOX;
        a_bytes = (uint32_t)mt * KT * 2u;
        s_bytes = ((uint32_t)nt * 4u + 127u) & ~127u;
        stage_bytes = (w_bytes + a_bytes + s_bytes + 1023u) & ~1023u;
        y_pitch = (uint32_t)nt + 4u;                      // fp32 words per staged output row
        y_bytes = ((uint32_t)mt * y_pitch * 4u + 1023u) & ~1023u;
    }
    __host__ __device__ uint32_t smem_bytes(int ns) const {
        return (uint32_t)ns * stage_bytes + y_bytes + 2u * ns * 8u + 1024u;
    }
};

__device__ __forceinline__ void mma_bf16(float c[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
                 "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Byte B of a packed word w (two's-complement 4-bit codes, element 2B in
// the low nibble of byte B) -> bf16x2 (q_even, q_odd). The even code comes
// from byte B of w, the odd one from byte B of w4 = w >> 4; one lop3 keeps
// each code in mantissa bits 0-3 of its half, flips its sign bit (u = q + 8)
// and sets the exponent of 128, so the half holds 128 + u exactly; one fma
// (x * 1 - 136) leaves q.
template <int B>
__device__ __forceinline__ uint32_t nib_pair(uint32_t w, uint32_t w4) {
    const uint32_t r = __byte_perm(w, w4, (uint32_t)B | ((uint32_t)(4 + B) << 8));
    uint32_t v;
    asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(v) : "r"(r), "r"(0x000F000Fu), "r"(0x43084308u));
    uint32_t out;
    const uint32_t one = 0x3F803F80u;    // bf16x2 (1.0, 1.0)
    const uint32_t add = 0xC308C308u;    // bf16x2 (-136.0, -136.0)
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(out) : "r"(v), "r"(one), "r"(add));
    return out;
}

// ------------------------------------------------ register-direct kernel

constexpr int RD_COLS = 32;             // weight columns per CTA
constexpr int RD_WARPS = 8;             // warps per CTA, taking 128-deep groups round-robin
constexpr int RD_MAX_PROBLEMS = 256;    // problems per launch (kernel parameter space: 32 KB)

struct RdProb {
    const uint16_t* A;                  // bf16 [M, K]
    const uint4* W;                     // qweight [K/8, N] int32, as 16-byte quads of columns
    const uint16_t* S;                  // bf16 [K/128, N]
    const uint8_t* Z;                   // zero points [K/128, N] (unsigned codes only)
    uint16_t* Y;                        // bf16 [M, N]
    int M, N, K;
    int cta_begin;                      // first CTA of this problem
};

template <int NP>                       // NP = 1 for a single call, RD_MAX_PROBLEMS for a group
struct RdParamsN {
    RdProb p[NP];
    int count;
};

// Biased unpack: bf16x2 (q_even + 136, q_odd + 136) of byte B of w (w4 = w >> 4)
// for two's-complement codes; with UNSIGNED codes (0..15, used with a zero
// point) the sign flip is left out and the halves hold u + 128.
template <int B, bool UNSIGNED = false>
__device__ __forceinline__ uint32_t nib_pair_biased(uint32_t w, uint32_t w4) {
    const uint32_t r = __byte_perm(w, w4, (uint32_t)B | ((uint32_t)(4 + B) << 8));
    uint32_t v;
    if (UNSIGNED)
        asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(v) : "r"(r), "r"(0x000F000Fu), "r"(0x43004300u));
    else
        asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(v) : "r"(r), "r"(0x000F000Fu), "r"(0x43084308u));
    return v;
}

// Weights of one 128-deep group for one lane: k-octet rows 4c + t (c = 0..3),
// columns 4g .. 4g+3 of the CTA's 32, and the group's 4 scales of those columns.
struct RdGroup {
    uint4 w[4];
    uint2 s;
    uint32_t z;                         // the 4 columns' zero points (unsigned codes only)
};

template <bool ZP = false>
__device__ __forceinline__ void rd_load(RdGroup& G, const RdProb& pr, int n0, int grp, int g, int t) {
    const int nq = pr.N >> 2;                                     // 16-byte quads per row
    const uint4* base = pr.W + (size_t)(grp * 16 + t) * nq + ((n0 >> 2) + g);
#pragma unroll
    for (int c = 0; c < 4; c++) {                                  // streamed once: no L1 allocation
        const uint4* q = base + (size_t)(4 * c) * nq;
        asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(G.w[c].x), "=r"(G.w[c].y), "=r"(G.w[c].z), "=r"(G.w[c].w) : "l"(q));
    }
    G.s = __ldg(reinterpret_cast<const uint2*>(pr.S + (size_t)grp * pr.N + n0 + 4 * g));
    if (ZP) G.z = __ldg(reinterpret_cast<const uint32_t*>(pr.Z + (size_t)grp * pr.N + n0 + 4 * g));
}

// ZP: unsigned codes with one zero point per group and column; the group sum
// is sum(a * (u + 128)) - (128 + z) * sum(a).
template <int MT, bool ZP, int NP>
__global__ void __launch_bounds__(RD_WARPS * 32, MT <= 8 ? 3 : 2)
w4a16_rd_kernel(const __grid_constant__ RdParamsN<NP> P) {
    constexpr int MB = MT / 8;
    __shared__ float red[RD_WARPS][MT][RD_COLS + 1];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    int lo = 0, hi = P.count - 1;                                  // last problem with cta_begin <= blockIdx.x
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (P.p[mid].cta_begin <= (int)blockIdx.x) lo = mid; else hi = mid - 1;
    }
    const RdProb& pr = P.p[lo];
    const int n0 = ((int)blockIdx.x - pr.cta_begin) * RD_COLS;
    const int ngroups = pr.K >> 7;
    // Programmatic dependent launch: the next kernel may start as SMs free up;
    // this one loads its first weights before waiting for the previous kernel
    // (whose output may be this kernel's activations).
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    // Ask L2 for the CTA's whole weight and scale range at once (one 128-byte
    // line per k-octet row, one 64-byte segment per scale row): HBM then streams
    // at full rate while the register loads below find their lines in flight
    // or already in L2.
    {
        const int nq = pr.N >> 2;
        const int rows = pr.K >> 3;
        for (int r = threadIdx.x; r < rows; r += RD_WARPS * 32)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(pr.W + (size_t)r * nq + (n0 >> 2)));
        for (int r = threadIdx.x; r < ngroups; r += RD_WARPS * 32) {
            asm volatile("prefetch.global.L2 [%0];" ::"l"(pr.S + (size_t)r * pr.N + n0));
            if (ZP) asm volatile("prefetch.global.L2 [%0];" ::"l"(pr.Z + (size_t)r * pr.N + n0));
        }
    }

    float acc[2][MB][4];
#pragma unroll
    for (int sl = 0; sl < 2; sl++)
#pragma unroll
        for (int mb = 0; mb < MB; mb++) acc[sl][mb][0] = acc[sl][mb][1] = acc[sl][mb][2] = acc[sl][mb][3] = 0.0f;

    RdGroup cur;
    int grp = warp;
    if (grp < ngroups) rd_load<ZP>(cur, pr, n0, grp, g, t);
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const uint16_t* arow[MB];
    bool live[MB];
#pragma unroll
    for (int mb = 0; mb < MB; mb++) {
        live[mb] = mb * 8 + g < pr.M;
        arow[mb] = pr.A + (size_t)(live[mb] ? mb * 8 + g : 0) * pr.K + 8 * t;
    }
    const uint32_t ones[4] = {0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u};
    for (; grp < ngroups; grp += RD_WARPS) {
        float ag[2][MB][4], sg[MB][4];
#pragma unroll
        for (int mb = 0; mb < MB; mb++) {
            sg[mb][0] = sg[mb][1] = sg[mb][2] = sg[mb][3] = 0.0f;
#pragma unroll
            for (int sl = 0; sl < 2; sl++) ag[sl][mb][0] = ag[sl][mb][1] = ag[sl][mb][2] = ag[sl][mb][3] = 0.0f;
        }
#pragma unroll
        for (int c = 0; c < 4; c++) {                             // 32-deep chunks of the group
            uint4 bv[MB];
#pragma unroll
            for (int mb = 0; mb < MB; mb++) {                      // 8 activations of token mb*8+g
                bv[mb] = live[mb] ? __ldg(reinterpret_cast<const uint4*>(arow[mb] + grp * 128 + 32 * c))
                                  : make_uint4(0u, 0u, 0u, 0u);
            }
            const uint32_t wq[4] = {cur.w[c].x, cur.w[c].y, cur.w[c].z, cur.w[c].w};
#pragma unroll
            for (int sl = 0; sl < 2; sl++) {                       // MMA rows g, g+8 = columns 4g+2sl, 4g+2sl+1
                const uint32_t w0 = wq[2 * sl], w1 = wq[2 * sl + 1];
                const uint32_t x0 = w0 >> 4, x1 = w1 >> 4;
                const uint32_t f0[4] = {nib_pair_biased<0, ZP>(w0, x0), nib_pair_biased<0, ZP>(w1, x1),
                                        nib_pair_biased<1, ZP>(w0, x0), nib_pair_biased<1, ZP>(w1, x1)};
                const uint32_t f1[4] = {nib_pair_biased<2, ZP>(w0, x0), nib_pair_biased<2, ZP>(w1, x1),
                                        nib_pair_biased<3, ZP>(w0, x0), nib_pair_biased<3, ZP>(w1, x1)};
#pragma unroll
                for (int mb = 0; mb < MB; mb++) {
                    mma_bf16(ag[sl][mb], f0, bv[mb].x, bv[mb].y);
                    mma_bf16(ag[sl][mb], f1, bv[mb].z, bv[mb].w);
                }
            }
#pragma unroll
            for (int mb = 0; mb < MB; mb++) {                      // sum(a) of tokens 2t, 2t+1
                mma_bf16(sg[mb], ones, bv[mb].x, bv[mb].y);
                mma_bf16(sg[mb], ones, bv[mb].z, bv[mb].w);
            }
        }
        const float sc[4] = {bf16_bits_to_f32(cur.s.x & 0xFFFFu), bf16_bits_to_f32(cur.s.x >> 16),
                             bf16_bits_to_f32(cur.s.y & 0xFFFFu), bf16_bits_to_f32(cur.s.y >> 16)};
        float nb[4] = {-136.0f, -136.0f, -136.0f, -136.0f};       // minus the bias of each column
        if (ZP) {
#pragma unroll
            for (int c = 0; c < 4; c++) nb[c] = -(128.0f + (float)((cur.z >> (8 * c)) & 0xFFu));
        }
#pragma unroll
        for (int sl = 0; sl < 2; sl++)
#pragma unroll
            for (int mb = 0; mb < MB; mb++) {                      // remove the bias, scale, accumulate
                acc[sl][mb][0] = fmaf(sc[2 * sl], fmaf(nb[2 * sl], sg[mb][0], ag[sl][mb][0]), acc[sl][mb][0]);
                acc[sl][mb][1] = fmaf(sc[2 * sl], fmaf(nb[2 * sl], sg[mb][1], ag[sl][mb][1]), acc[sl][mb][1]);
                acc[sl][mb][2] = fmaf(sc[2 * sl + 1], fmaf(nb[2 * sl + 1], sg[mb][0], ag[sl][mb][2]), acc[sl][mb][2]);
                acc[sl][mb][3] = fmaf(sc[2 * sl + 1], fmaf(nb[2 * sl + 1], sg[mb][1], ag[sl][mb][3]), acc[sl][mb][3]);
            }
        // the next group's loads (already requested from L2 by the prefetch above)
        if (grp + RD_WARPS < ngroups) rd_load<ZP>(cur, pr, n0, grp + RD_WARPS, g, t);
    }
    // partial sums of this warp -> shared memory; fixed-order sum over warps
#pragma unroll
    for (int sl = 0; sl < 2; sl++)
#pragma unroll
        for (int mb = 0; mb < MB; mb++) {
            const int m = mb * 8 + 2 * t, col = 4 * g + 2 * sl;
            red[warp][m][col] = acc[sl][mb][0];
            red[warp][m + 1][col] = acc[sl][mb][1];
            red[warp][m][col + 1] = acc[sl][mb][2];
            red[warp][m + 1][col + 1] = acc[sl][mb][3];
        }
    __syncthreads();
    const int mrows = min(pr.M, MT);
    for (int i = threadIdx.x; i < mrows * (RD_COLS / 2); i += RD_WARPS * 32) {
        const int m = i / (RD_COLS / 2), col = 2 * (i % (RD_COLS / 2));
        float y0 = red[0][m][col], y1 = red[0][m][col + 1];
#pragma unroll
        for (int w = 1; w < RD_WARPS; w++) {
            y0 += red[w][m][col];
            y1 += red[w][m][col + 1];
        }
        const __nv_bfloat162 o = __floats2bfloat162_rn(y0, y1);
        *reinterpret_cast<__nv_bfloat162*>(pr.Y + (size_t)m * pr.N + n0 + col) = o;
    }
}

// ------------------------------------------------ bulk-staged kernel

// Up to 8 tokens with K <= SA_KMAX: the arithmetic of the register-direct
// kernel, but the CTA's whole weight and scale range is requested at once by
// the TMA unit (one 2-D box of 16*SA_GPB k-octet rows x 32 columns plus the
// matching 64-byte scale rows per mbarrier) into shared memory. The memory
// system then holds the whole launch in flight from its first microsecond and
// each warp only waits for the box of the group it is about to use; no
// registers are spent on loads in flight. With a single token, sum(a) of a
// group comes from one MMA whose 8 columns are 16-deep slices of the token's
// activations (the ones fragment sums each column), instead of eight.
constexpr int SA_GPB = 2;               // 128-deep scale groups per box and mbarrier
constexpr int SA_MAX_PROBLEMS = 120;    // problems per launch (kernel parameter space: 32 KB)
constexpr int SA_KMAX = 8192;           // deepest K staged whole (132 KB of weights per CTA)
constexpr uint32_t SA_RED_BYTES = RD_WARPS * 8 * (RD_COLS + 1) * 4;

struct SaProb {
    CUtensorMap tmW;                    // qweight [K/8][N] int32, box 32 x 16*SA_GPB, no swizzle
    const uint16_t* A;                  // bf16 [M, K]
    const uint16_t* S;                  // bf16 [K/128, N]
    uint16_t* Y;                        // bf16 [M, N]
    int M, N, K;
    int cta_begin;                      // first CTA of this problem
};

template <int NP>                       // NP = 1 for a single call, SA_MAX_PROBLEMS for a group
struct SaParamsN {
    SaProb p[NP];
    int count;
};

// Shared memory: whole boxes of weights (a partial last box is zero-filled
// past K; the region later holds the cross-warp sums), the scale rows, the
// mbarriers; 1 KB of slack to align the base.
__host__ __device__ inline uint32_t sa_wregion(int K) {
    const uint32_t nb = (uint32_t)((K / 128 + SA_GPB - 1) / SA_GPB);
    const uint32_t w = nb * SA_GPB * 2048u;
    return w > SA_RED_BYTES ? w : ((SA_RED_BYTES + 127u) & ~127u);
}
__host__ __device__ inline uint32_t sa_smem_bytes(int K) {
    const int ng = K / 128, nb = (ng + SA_GPB - 1) / SA_GPB;
    return 1024u + sa_wregion(K) + (uint32_t)ng * 64u + (uint32_t)nb * 8u;
}

// mma.m16n8k16 with a zero accumulator in.
__device__ __forceinline__ void mma_bf16_z(float c[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
                 "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
                 : "=f"(c[0]), "=f"(c[1]), "=f"(c[2]), "=f"(c[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.0f));
}

// ONE: every problem of the launch has a single token.
template <bool ONE, int NP>
__global__ void __launch_bounds__(RD_WARPS * 32, 3)
w4a16_bulk_kernel(const __grid_constant__ SaParamsN<NP> P) {
    extern __shared__ uint8_t sa_dyn[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(sa_dyn) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    int lo = 0, hi = P.count - 1;                                  // last problem with cta_begin <= blockIdx.x
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (P.p[mid].cta_begin <= (int)blockIdx.x) lo = mid; else hi = mid - 1;
    }
    const SaProb& pr = P.p[lo];
    const int n0 = ((int)blockIdx.x - pr.cta_begin) * RD_COLS;
    const int ngroups = pr.K >> 7;
    const int nbars = (ngroups + SA_GPB - 1) / SA_GPB;
    uint8_t* sW = sm;
    uint8_t* sS = sm + sa_wregion(pr.K);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sS + ngroups * 64);
    if (threadIdx.x == 0) {
        for (int b = 0; b < nbars; b++) mbar_init(smem_u32(bars + b), 1);
        fence_barrier_init();
        prefetch_tmap(&pr.tmW);
    }
    __syncthreads();
    // Programmatic dependent launch: the next kernel may start as SMs free up;
    // the weight copies go out before waiting for the previous kernel (whose
    // output may be this kernel's activations).
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (warp == 0) {
        for (int b = lane; b < nbars; b += 32) {
            const int gs = min(SA_GPB, ngroups - b * SA_GPB);
            const uint32_t bar = smem_u32(bars + b);
            mbar_arrive_expect_tx(bar, SA_GPB * 2048u + (uint32_t)gs * 64u);   // a box always lands whole
            tma_load_2d(smem_u32(sW + (size_t)b * SA_GPB * 2048), &pr.tmW, n0, b * SA_GPB * 16, bar);
            for (int j = 0; j < gs; j++) {
                const int grp = b * SA_GPB + j;
                bulk_g2s(smem_u32(sS + grp * 64), pr.S + (size_t)grp * pr.N + n0, 64u, bar);
            }
        }
    }
    float acc[2][4];
#pragma unroll
    for (int sl = 0; sl < 2; sl++) acc[sl][0] = acc[sl][1] = acc[sl][2] = acc[sl][3] = 0.0f;

    asm volatile("griddepcontrol.wait;" ::: "memory");
    const bool live = g < pr.M;                                    // token g of the lane's MMA column
    const uint16_t* arow = pr.A + (size_t)(live ? g : 0) * pr.K + 8 * t;
    const uint16_t* srow = pr.A + 16 * g + 4 * t;                   // ONE: slice g of the token's group
    const uint32_t ones[4] = {0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u};
    uint4 an[4];                                                   // the next group's activations
    uint2 sn = make_uint2(0u, 0u);
    if (warp < ngroups) {
#pragma unroll
        for (int c = 0; c < 4; c++)
            an[c] = live ? __ldg(reinterpret_cast<const uint4*>(arow + warp * 128 + 32 * c)) : make_uint4(0u, 0u, 0u, 0u);
        if (ONE) sn = __ldg(reinterpret_cast<const uint2*>(srow + warp * 128));
    }
    bool ok = true;
    for (int grp = warp; grp < ngroups; grp += RD_WARPS) {
        uint4 av[4];
#pragma unroll
        for (int c = 0; c < 4; c++) av[c] = an[c];
        const uint2 sv = sn;
        if (grp + RD_WARPS < ngroups) {
#pragma unroll
            for (int c = 0; c < 4; c++)
                an[c] = live ? __ldg(reinterpret_cast<const uint4*>(arow + (grp + RD_WARPS) * 128 + 32 * c))
                             : make_uint4(0u, 0u, 0u, 0u);
            if (ONE) sn = __ldg(reinterpret_cast<const uint2*>(srow + (grp + RD_WARPS) * 128));
        }
        if (!mbar_wait<false>(smem_u32(bars + grp / SA_GPB), 0, &g_w4a16_err)) { ok = false; break; }
        float ag[2][4], sg[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        const uint8_t* wg = sW + (size_t)grp * 2048 + t * 128 + g * 16;     // k-octet row 4c + t, columns 4g..4g+3
#pragma unroll
        for (int c = 0; c < 4; c++) {
            const uint4 wv = *reinterpret_cast<const uint4*>(wg + c * 512);
            const uint32_t wq[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
            for (int sl = 0; sl < 2; sl++) {                       // MMA rows g, g+8 = columns 4g+2sl, 4g+2sl+1
                const uint32_t w0 = wq[2 * sl], w1 = wq[2 * sl + 1];
                const uint32_t x0 = w0 >> 4, x1 = w1 >> 4;
                const uint32_t f0[4] = {nib_pair_biased<0>(w0, x0), nib_pair_biased<0>(w1, x1),
                                        nib_pair_biased<1>(w0, x0), nib_pair_biased<1>(w1, x1)};
                const uint32_t f1[4] = {nib_pair_biased<2>(w0, x0), nib_pair_biased<2>(w1, x1),
                                        nib_pair_biased<3>(w0, x0), nib_pair_biased<3>(w1, x1)};
                if (c == 0) mma_bf16_z(ag[sl], f0, av[c].x, av[c].y);
                else mma_bf16(ag[sl], f0, av[c].x, av[c].y);
                mma_bf16(ag[sl], f1, av[c].z, av[c].w);
            }
            if (!ONE) {                                            // sum(a) of tokens 2t, 2t+1
                mma_bf16(sg, ones, av[c].x, av[c].y);
                mma_bf16(sg, ones, av[c].z, av[c].w);
            }
        }
        if (ONE) {                                                 // columns hold 16-deep slices: add them all
            float sd[4];
            mma_bf16_z(sd, ones, sv.x, sv.y);
            float v = sd[0] + sd[1];
            v += __shfl_xor_sync(0xFFFFFFFFu, v, 1);
            v += __shfl_xor_sync(0xFFFFFFFFu, v, 2);
            sg[0] = v;                                             // token 0 (lanes with t = 0 keep it)
        }
        const uint2 sc2 = *reinterpret_cast<const uint2*>(sS + grp * 64 + g * 8);
        const float sc[4] = {bf16_bits_to_f32(sc2.x & 0xFFFFu), bf16_bits_to_f32(sc2.x >> 16),
                             bf16_bits_to_f32(sc2.y & 0xFFFFu), bf16_bits_to_f32(sc2.y >> 16)};
#pragma unroll
        for (int sl = 0; sl < 2; sl++) {                           // remove the bias, scale, accumulate
            acc[sl][0] = fmaf(sc[2 * sl], fmaf(-136.0f, sg[0], ag[sl][0]), acc[sl][0]);
            acc[sl][1] = fmaf(sc[2 * sl], fmaf(-136.0f, sg[1], ag[sl][1]), acc[sl][1]);
            acc[sl][2] = fmaf(sc[2 * sl + 1], fmaf(-136.0f, sg[0], ag[sl][2]), acc[sl][2]);
            acc[sl][3] = fmaf(sc[2 * sl + 1], fmaf(-136.0f, sg[1], ag[sl][3]), acc[sl][3]);
        }
    }
    // Every box must have landed before its region is reused for the sums; a
    // warp that gave up on a wait checks the others with the same bound.
    if (!ok)
        for (int b = 0; b < nbars; b++) mbar_wait<false>(smem_u32(bars + b), 0, &g_w4a16_err);
    __syncthreads();
    float (*red)[8][RD_COLS + 1] = reinterpret_cast<float (*)[8][RD_COLS + 1]>(sm);
#pragma unroll
    for (int sl = 0; sl < 2; sl++) {
        const int m = 2 * t, col = 4 * g + 2 * sl;
        red[warp][m][col] = acc[sl][0];
        red[warp][m + 1][col] = acc[sl][1];
        red[warp][m][col + 1] = acc[sl][2];
        red[warp][m + 1][col + 1] = acc[sl][3];
    }
    __syncthreads();
    const int mrows = min(pr.M, 8);
    for (int i = threadIdx.x; i < mrows * (RD_COLS / 2); i += RD_WARPS * 32) {
        const int m = i / (RD_COLS / 2), col = 2 * (i % (RD_COLS / 2));
        float y0 = red[0][m][col], y1 = red[0][m][col + 1];
#pragma unroll
        for (int w = 1; w < RD_WARPS; w++) {
            y0 += red[w][m][col];
            y1 += red[w][m][col + 1];
        }
        const __nv_bfloat162 o = __floats2bfloat162_rn(y0, y1);
        *reinterpret_cast<__nv_bfloat162*>(pr.Y + (size_t)m * pr.N + n0 + col) = o;
    }
}

// ------------------------------------------------ TMA-staged kernel

template <int MT, int NP>
__global__ void __launch_bounds__((2 * ntmax_for(MT) / 16 + 1) * 32, 1)
w4a16_kernel(const __grid_constant__ ParamsN<NP> P, int nt, int ns) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    constexpr int MB = MT / 8;                       // 8-token MMA blocks
    const int nslice = nt / 16;                      // 16-column MMA slices
    const int nwarps_c = 2 * nslice;                 // MMA warps: one per slice and scale group
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Layout L(nt, MT);

    float* ybuf = reinterpret_cast<float*>(smem + (size_t)ns * L.stage_bytes);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)ns * L.stage_bytes + L.y_bytes);
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + ns);

    if (threadIdx.x == 0) {
        for (int i = 0; i < ns; i++) {
            mbar_init(full0 + 8 * i, 1);
            mbar_init(empty0 + 8 * i, nwarps_c);
        }
        fence_barrier_init();
    }
    __syncthreads();
    // Programmatic dependent launch: the next kernel on the stream may start as
    // soon as SMs free up; this kernel waits for the previous one (griddepcontrol
    // .wait, producer below) only before loading activations, so its first weight
    // stages stream in while the previous kernel finishes.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    auto find = [&](int tile) {                      // last problem with tile_begin <= tile
        int lo = 0, hi = P.count - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (P.p[mid].tile_begin <= tile) lo = mid; else hi = mid - 1;
        }
        return lo;
    };

    if (warp == nwarps_c) {
        // ------------------------------------------------ producer (one thread)
        if (lane == 0) {
            const uint32_t bytes = L.w_bytes + L.a_bytes + (uint32_t)nt * 4u;
            uint32_t it = 0;
            bool ok = true, waited = false;
            for (int tile = blockIdx.x; tile < P.total_tiles && ok; tile += gridDim.x) {
                const Prob& pr = P.p[find(tile)];
                const int n0 = (tile - pr.tile_begin) * nt;
                const int nstage = (pr.K + KT - 1) / KT;
                prefetch_tmap(&pr.tmW);
                prefetch_tmap(&pr.tmA);
                prefetch_tmap(&pr.tmS);
                // first tile: weights and scales of the first ring's worth of stages
                // before the dependency wait, activations after it
                const int early = waited ? 0 : min(nstage, ns);
                for (int s = 0; s < early; s++) {
                    const uint32_t full = full0 + 8 * s;
                    const uint32_t st = smem_u32(smem) + s * L.stage_bytes;
                    mbar_arrive_expect_tx(full, bytes);
                    for (int b = 0; b < nt / 32; b++)
                        tma_load_2d(st + b * WBOX, &pr.tmW, n0 + 32 * b, s * (KT / 8), full);
                    tma_load_2d(st + L.w_bytes + L.a_bytes, &pr.tmS, n0, s * (KT / 128), full);
                }
                if (!waited) {
                    asm volatile("griddepcontrol.wait;" ::: "memory");
                    waited = true;
                }
                for (int s = 0; s < early; s++)
                    tma_load_2d(smem_u32(smem) + s * L.stage_bytes + L.w_bytes, &pr.tmA, s * KT, 0, full0 + 8 * s);
                it += early;
                for (int s = early; s < nstage; s++, it++) {
                    const int slot = it % ns;
                    if (it >= (uint32_t)ns && !mbar_wait(empty0 + 8 * slot, ((it / ns) - 1) & 1, &g_w4a16_err)) {
                        ok = false;
                        break;
                    }
                    const uint32_t full = full0 + 8 * slot;
                    const uint32_t st = smem_u32(smem) + slot * L.stage_bytes;
                    mbar_arrive_expect_tx(full, bytes);
                    for (int b = 0; b < nt / 32; b++)
                        tma_load_2d(st + b * WBOX, &pr.tmW, n0 + 32 * b, s * (KT / 8), full);
                    tma_load_2d(st + L.w_bytes, &pr.tmA, s * KT, 0, full);
                    tma_load_2d(st + L.w_bytes + L.a_bytes, &pr.tmS, n0, s * (KT / 128), full);
                }
            }
            // every issued copy has landed before the CTA may exit
            for (uint32_t j = it > (uint32_t)ns ? it - ns : 0; j < it; j++)
                mbar_wait(full0 + 8 * (j % ns), (j / ns) & 1, &g_w4a16_err);
        }
    } else {
        // ------------------------------------------------- MMA warps
        const int g = lane >> 2, t = lane & 3;
        const int slice = warp % nslice, half = warp / nslice;   // half = scale group in each stage
        const int c0 = 16 * (slice & 1) + g;
        // swizzled byte offsets of columns c0 and c0 + 8 in rows with (row & 7) = 4 * par + t
        uint32_t off[2][2];
#pragma unroll
        for (int par = 0; par < 2; par++)
#pragma unroll
            for (int h = 0; h < 2; h++) {
                const int c = c0 + 8 * h;
                off[par][h] = ((((uint32_t)c >> 2) ^ (uint32_t)(4 * par + t)) << 4) | (((uint32_t)c & 3u) << 2);
            }
        const uint32_t wrow = (uint32_t)(slice >> 1) * WBOX + (uint32_t)(16 * half + t) * 128u;
        const uint32_t arow = (uint32_t)g * (KT * 2) + (uint32_t)(128 * half + 8 * t) * 2u;
        uint32_t it = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < P.total_tiles && ok; tile += gridDim.x) {
            const Prob& pr = P.p[find(tile)];
            const int n0 = (tile - pr.tile_begin) * nt;
            const int ntv = min(nt, pr.N - n0);          // valid columns (multiple of 32)
            const bool active = slice * 16 < ntv;
            const int nstage = (pr.K + KT - 1) / KT;
            float acc[MB][4];
#pragma unroll
            for (int mb = 0; mb < MB; mb++) acc[mb][0] = acc[mb][1] = acc[mb][2] = acc[mb][3] = 0.0f;

            for (int s = 0; s < nstage; s++, it++) {
                const int slot = it % ns;
                if (!mbar_wait(full0 + 8 * slot, (it / ns) & 1, &g_w4a16_err)) { ok = false; break; }
                if (active) {
                    const uint8_t* st = smem + (size_t)slot * L.stage_bytes;
                    const uint8_t* wb = st + wrow;
                    const uint8_t* a = st + L.w_bytes + arow;
                    const uint16_t* sc = reinterpret_cast<const uint16_t*>(st + L.w_bytes + L.a_bytes);
                    float ag[MB][4];
#pragma unroll
                    for (int mb = 0; mb < MB; mb++) ag[mb][0] = ag[mb][1] = ag[mb][2] = ag[mb][3] = 0.0f;
#pragma unroll
                    for (int c = 0; c < 4; c++) {                    // 32-deep chunks of this group
                        const uint8_t* rowp = wb + c * 512;          // k-octet row 16*half + 4c + t
                        const uint32_t w0 = *reinterpret_cast<const uint32_t*>(rowp + off[c & 1][0]);
                        const uint32_t w1 = *reinterpret_cast<const uint32_t*>(rowp + off[c & 1][1]);
                        const uint32_t x0 = w0 >> 4, x1 = w1 >> 4;
                        const uint32_t f0[4] = {nib_pair<0>(w0, x0), nib_pair<0>(w1, x1), nib_pair<1>(w0, x0),
                                                nib_pair<1>(w1, x1)};
                        const uint32_t f1[4] = {nib_pair<2>(w0, x0), nib_pair<2>(w1, x1), nib_pair<3>(w0, x0),
                                                nib_pair<3>(w1, x1)};
#pragma unroll
                        for (int mb = 0; mb < MB; mb++) {
                            const uint4 bv = *reinterpret_cast<const uint4*>(a + mb * 8 * (KT * 2) + c * 64);
                            mma_bf16(ag[mb], f0, bv.x, bv.y);
                            mma_bf16(ag[mb], f1, bv.z, bv.w);
                        }
                    }
                    const float s0 = bf16_bits_to_f32(sc[half * nt + slice * 16 + g]);
                    const float s1 = bf16_bits_to_f32(sc[half * nt + slice * 16 + g + 8]);
#pragma unroll
                    for (int mb = 0; mb < MB; mb++) {
                        acc[mb][0] = fmaf(s0, ag[mb][0], acc[mb][0]);
                        acc[mb][1] = fmaf(s0, ag[mb][1], acc[mb][1]);
                        acc[mb][2] = fmaf(s1, ag[mb][2], acc[mb][2]);
                        acc[mb][3] = fmaf(s1, ag[mb][3], acc[mb][3]);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(empty0 + 8 * slot);
            }
            // ---- tile epilogue: group-0 warps store their sums, group-1 warps add
            // theirs, then all MMA warps write the bf16 tile (rows < M, valid columns).
            const int n = slice * 16 + g;
            if (half == 0 && active && ok) {
#pragma unroll
                for (int mb = 0; mb < MB; mb++) {
                    const int m = mb * 8 + 2 * t;
                    ybuf[m * L.y_pitch + n] = acc[mb][0];
                    ybuf[(m + 1) * L.y_pitch + n] = acc[mb][1];
                    ybuf[m * L.y_pitch + n + 8] = acc[mb][2];
                    ybuf[(m + 1) * L.y_pitch + n + 8] = acc[mb][3];
                }
            }
            asm volatile("bar.sync 1, %0;" ::"r"(nwarps_c * 32) : "memory");
            if (half == 1 && active && ok) {
#pragma unroll
                for (int mb = 0; mb < MB; mb++) {
                    const int m = mb * 8 + 2 * t;
                    ybuf[m * L.y_pitch + n] += acc[mb][0];
                    ybuf[(m + 1) * L.y_pitch + n] += acc[mb][1];
                    ybuf[m * L.y_pitch + n + 8] += acc[mb][2];
                    ybuf[(m + 1) * L.y_pitch + n + 8] += acc[mb][3];
                }
            }
            asm volatile("bar.sync 1, %0;" ::"r"(nwarps_c * 32) : "memory");
            if (ok) {
                const int vec_per_row = ntv / 8;             // 16-byte output vectors per row
                const int mrows = min(pr.M, MT);
                for (int i = threadIdx.x; i < mrows * vec_per_row; i += nwarps_c * 32) {
                    const int m = i / vec_per_row, v = i - m * vec_per_row;
                    const float4 lo4 = *reinterpret_cast<const float4*>(ybuf + m * L.y_pitch + v * 8);
                    const float4 hi4 = *reinterpret_cast<const float4*>(ybuf + m * L.y_pitch + v * 8 + 4);
                    uint4 o;
                    __nv_bfloat162 b0 = __floats2bfloat162_rn(lo4.x, lo4.y), b1 = __floats2bfloat162_rn(lo4.z, lo4.w);
                    __nv_bfloat162 b2 = __floats2bfloat162_rn(hi4.x, hi4.y), b3 = __floats2bfloat162_rn(hi4.z, hi4.w);
                    o.x = *reinterpret_cast<uint32_t*>(&b0);
                    o.y = *reinterpret_cast<uint32_t*>(&b1);
                    o.z = *reinterpret_cast<uint32_t*>(&b2);
                    o.w = *reinterpret_cast<uint32_t*>(&b3);
                    *reinterpret_cast<uint4*>(pr.Y + (size_t)m * pr.N + n0 + v * 8) = o;
                }
            }
            asm volatile("bar.sync 1, %0;" ::"r"(nwarps_c * 32) : "memory");
        }
    }
}

int choose_mt(int m) { return m <= 8 ? 8 : m <= 16 ? 16 : m <= 32 ? 32 : 64; }

// Register-direct launch for up to 8 tokens: one CTA per 32 columns of every
// problem, programmatic dependent launch.
template <int MT, bool ZP, int NP>
qz_status launch_rd_n(const qz_w4a16_problem* problems, int count, cudaStream_t st, bool early,
                      const uint8_t* const* zeros) {
    RdParamsN<NP> P;                              // the kernel parameter block (copied at launch)
    int total = 0;
    P.count = count;
    for (int i = 0; i < count; i++) {
        const qz_w4a16_problem& q = problems[i];
        RdProb& p = P.p[i];
        p.A = q.A;
        p.W = reinterpret_cast<const uint4*>(q.qweight);
        p.S = q.scale_bf16;
        p.Z = zeros ? zeros[i] : nullptr;
        p.Y = q.Y;
        p.M = q.M; p.N = q.N; p.K = q.K;
        p.cta_begin = total;
        total += q.N / RD_COLS;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(total);
    cfg.blockDim = dim3(RD_WARPS * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = early ? 1 : 0;                 // without it: after all earlier work on the stream
    if (cudaLaunchKernelEx(&cfg, w4a16_rd_kernel<MT, ZP, NP>, P) != cudaSuccess) return QZ_ERR_CUDA;
    return launch_status();
}

template <int MT, bool ZP = false>
qz_status launch_rd(const qz_w4a16_problem* problems, int count, cudaStream_t st, bool early,
                    const uint8_t* const* zeros = nullptr) {
    return count == 1 ? launch_rd_n<MT, ZP, 1>(problems, count, st, early, zeros)
                      : launch_rd_n<MT, ZP, RD_MAX_PROBLEMS>(problems, count, st, early, zeros);
}

// Bulk-staged launch for up to 8 tokens and K <= SA_KMAX: one CTA per 32
// columns of every problem, programmatic dependent launch.
template <int NP>
qz_status launch_bulk_n(const qz_w4a16_problem* problems, int count, cudaStream_t st, bool early) {
    SaParamsN<NP> P;                              // the kernel parameter block (copied at launch)
    int total = 0, kmax = 0, mmax = 0;
    P.count = count;
    for (int i = 0; i < count; i++) {
        const qz_w4a16_problem& q = problems[i];
        SaProb& p = P.p[i];
        if (!encode_tmap_2d(&p.tmW, q.qweight, 4, (uint64_t)q.N, (uint64_t)q.K / 8, (uint64_t)q.N * 4, 32,
                            16 * SA_GPB, false))
            return QZ_ERR_CUDA;
        p.A = q.A;
        p.S = q.scale_bf16;
        p.Y = q.Y;
        p.M = q.M; p.N = q.N; p.K = q.K;
        p.cta_begin = total;
        total += q.N / RD_COLS;
        kmax = std::max(kmax, q.K);
        mmax = std::max(mmax, q.M);
    }
    const int smem = (int)sa_smem_bytes(kmax);
    static int smem_set[64];                       // per device: largest size opted in so far
    static std::mutex smem_mu;                     // host threads must not lower each other's opt-in
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return QZ_ERR_UNSUPPORTED;
    {
        std::lock_guard<std::mutex> lock(smem_mu);
        if (smem > smem_set[dev]) {
            if (cudaFuncSetAttribute(w4a16_bulk_kernel<true, NP>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
                    cudaSuccess ||
                cudaFuncSetAttribute(w4a16_bulk_kernel<false, NP>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
                    cudaSuccess)
                return QZ_ERR_CUDA;
            smem_set[dev] = smem;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(total);
    cfg.blockDim = dim3(RD_WARPS * 32);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = early ? 1 : 0;                 // without it: after all earlier work on the stream
    const cudaError_t e = mmax == 1 ? cudaLaunchKernelEx(&cfg, w4a16_bulk_kernel<true, NP>, P)
                                    : cudaLaunchKernelEx(&cfg, w4a16_bulk_kernel<false, NP>, P);
    if (e != cudaSuccess) return QZ_ERR_CUDA;
    return launch_status();
}

qz_status launch_bulk(const qz_w4a16_problem* problems, int count, cudaStream_t st, bool early) {
    return count == 1 ? launch_bulk_n<1>(problems, count, st, early)
                      : launch_bulk_n<SA_MAX_PROBLEMS>(problems, count, st, early);
}

template <int MT, int NP>
qz_status launch_mt(const ParamsN<NP>& P, int nt, cudaStream_t st, bool early) {
    // One persistent CTA per SM (or per tile, if fewer), ring as deep as fits.
    const Layout L(nt, MT);
    const uint32_t budget = 200u * 1024u;
    int ns = (int)((budget - 1024u - L.y_bytes) / (L.stage_bytes + 16u));
    ns = std::max(2, std::min(ns, 8));
    const int smem = (int)L.smem_bytes(ns);
    static int smem_set[64];                       // per device: largest size opted in so far
    static std::mutex smem_mu;                     // host threads must not lower each other's opt-in
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return QZ_ERR_UNSUPPORTED;
    {
        std::lock_guard<std::mutex> lock(smem_mu);
        if (smem > smem_set[dev]) {
            if (cudaFuncSetAttribute(w4a16_kernel<MT, NP>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
                    cudaSuccess)
                return QZ_ERR_CUDA;
            smem_set[dev] = smem;
        }
    }
    const int threads = (2 * (nt / 16) + 1) * 32;
    const int grid = std::min(P.total_tiles, num_sms());
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = early ? 1 : 0;                 // without it: after all earlier work on the stream
    if (cudaLaunchKernelEx(&cfg, w4a16_kernel<MT, NP>, P, nt, ns) != cudaSuccess) return QZ_ERR_CUDA;
    return launch_status();
}

template <int NP>
qz_status launch_chunk_n(const qz_w4a16_problem* problems, int count, int nt, int mt, cudaStream_t st,
                         bool early) {
    ParamsN<NP> P;                                // the kernel parameter block (copied at launch)
    int total = 0;
    P.count = count;
    for (int i = 0; i < count; i++) {
        const qz_w4a16_problem& q = problems[i];
        Prob& p = P.p[i];
        if (!encode_tmap_2d(&p.tmW, q.qweight, 4, (uint64_t)q.N, (uint64_t)q.K / 8, (uint64_t)q.N * 4, 32, 32, true) ||
            !encode_tmap_2d(&p.tmA, q.A, 2, (uint64_t)q.K, (uint64_t)q.M, (uint64_t)q.K * 2, KT, (uint32_t)mt, false) ||
            !encode_tmap_2d(&p.tmS, q.scale_bf16, 2, (uint64_t)q.N, (uint64_t)q.K / 128, (uint64_t)q.N * 2,
                            (uint32_t)nt, 2, false))
            return QZ_ERR_CUDA;
        p.Y = q.Y;
        p.M = q.M; p.N = q.N; p.K = q.K;
        p.tile_begin = total;
        total += (q.N + nt - 1) / nt;
    }
    P.total_tiles = total;
    return launch_mt<16, NP>(P, nt, st, early);         // 9..16 tokens (the only width this kernel serves)
}

qz_status launch_chunk(const qz_w4a16_problem* problems, int count, int nt, int mt, cudaStream_t st, bool early) {
    return count == 1 ? launch_chunk_n<1>(problems, count, nt, mt, st, early)
                      : launch_chunk_n<PER_LAUNCH>(problems, count, nt, mt, st, early);
}

} // namespace

size_t ws_gemm_w4a16(int, int, int) { return 0; }

// W4A16 with unsigned codes and a zero point per group and column, up to 16
// tokens: the register-direct kernel.
qz_status gemm_w4a16_zp_launch(const uint16_t* A, const int32_t* qweight, const uint16_t* scale, const uint8_t* zero,
                               uint16_t* Y, int M, int N, int K, cudaStream_t st, bool early) {
    const qz_w4a16_problem p = {A, qweight, scale, Y, M, N, K};
    const uint8_t* z[1] = {zero};
    return M <= 8 ? launch_rd<8, true>(&p, 1, st, early, z) : launch_rd<16, true>(&p, 1, st, early, z);
}

qz_status w4a16_error_read_and_clear() {
    unsigned int v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_w4a16_err, sizeof(v)) != cudaSuccess) return QZ_ERR_CUDA;
    if (v && cudaMemcpyToSymbol(g_w4a16_err, &z, sizeof(z)) != cudaSuccess) return QZ_ERR_CUDA;
    return v ? QZ_ERR_TIMEOUT : QZ_OK;
}

qz_status gemm_w4a16_launch(const qz_w4a16_problem* problems, int count, void*, size_t, cudaStream_t st,
                            bool early) {
    const int sms = num_sms();
    int mmax = 0;
    for (int i = 0; i < count; i++) mmax = std::max(mmax, problems[i].M);
    // Tile width: with one problem, the smallest multiple of 32 giving at most
    // one tile per SM (capped at the widest tile for M); grouped problems use
    // the widest tile.
    const int mt = choose_mt(mmax);
    // as few launches as the parameter space allows (cap per launch), with equal
    // shares of the problems: every launch pays a ramp and a tail
    auto share = [count](int cap) { const int n = (count + cap - 1) / cap; return (count + n - 1) / n; };
    int kmax = 0;
    for (int i = 0; i < count; i++) kmax = std::max(kmax, problems[i].K);
    if (mt == 8 && kmax <= SA_KMAX) {             // up to 8 tokens: bulk-staged kernel
        const int sh = share(SA_MAX_PROBLEMS);
        for (int i = 0; i < count; i += sh) {
            const qz_status s = launch_bulk(problems + i, std::min(sh, count - i), st, early);
            if (s != QZ_OK) return s;
        }
        return QZ_OK;
    }
    if (mt == 8) {                                // deeper K: register-direct kernel
        const int sh = share(RD_MAX_PROBLEMS);
        for (int i = 0; i < count; i += sh) {
            const qz_status s = launch_rd<8>(problems + i, std::min(sh, count - i), st, early);
            if (s != QZ_OK) return s;
        }
        return QZ_OK;
    }
    if (mt >= 32) return w4a16_tc_launch(problems, count, mt, st, early);   // 17..64 tokens: tcgen05
    int nt = ntmax_for(mt);
    if (count == 1) {
        const int N = problems[0].N;
        nt = std::min(nt, 32 * (int)((N + 32LL * sms - 1) / (32LL * sms)));
    }
    const int sh = share(PER_LAUNCH);
    for (int i = 0; i < count; i += sh) {
        const qz_status s = launch_chunk(problems + i, std::min(sh, count - i), nt, mt, st, early);
        if (s != QZ_OK) return s;
    }
    return QZ_OK;
}

} // namespace qz
