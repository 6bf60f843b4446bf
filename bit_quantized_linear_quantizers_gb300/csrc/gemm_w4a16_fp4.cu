// gemm_w4a16_fp4.cu -- weight-only FP4 decode GEMM (W4A16 with MXFP4 or NVFP4
// weights, "量化部署实战", 精度比较: the W4A16 MXFP4 / W4A16 NVFP4 rows):
//   Y[m, n] = bf16( sum_k A[m, k] * e2m1(q[n, k]) * scale(n, k) )
// with bf16 activations A [M, K] (M <= 16), weights as B^T [N, K] exactly as
// the FP4 quantizers write them (codes [N, K/2], the even element in the low
// nibble; NVFP4: E4M3 scales [N, K/16] and one fp32 tensor scale; MXFP4: E8M0
// scales [N, K/32]), fp32 accumulation.
//
// Decode is bound by the weight bytes, so the kernel streams each weight byte
// once, straight into registers. Every E2M1 code times its block scale is
// exact in bf16 (at most 6 significant bits), so the dequantized weight is fed
// to bf16 tensor-core MMAs (mma.m16n8k16, fp32 accumulate) with no rounding:
//  * a code's three magnitude bits go to bf16 bits 6..8 and its sign to bit
//    15; that bit pattern is the code's value times 2^-126 (code 1, the value
//    0.5, is the subnormal 2^-127);
//  * one bf16x2 multiply by F = scale * 2^62 (exact: F has at most 4
//    significant bits and stays a normal bf16) gives value * scale * 2^-64;
//  * the fp32 sums are multiplied back by 2^64 (and by the NVFP4 tensor scale)
//    in the epilogue.
// The MXFP4 scale must lie in [2^-61, 2^65] (E8M0 codes 66..192) for F and
// the products to stay normal bf16; the NVFP4 block scales always do.
//
// Work split (swap AB: the weight rows are the MMA's 16-row side, up to 8
// tokens its 8-wide side, two 8-token blocks for 16): one CTA per 32 weight
// rows, its 8 warps take 128-deep K windows round-robin; lane (g, t) loads,
// per window, the 16 bytes (32 codes, k = 32t..32t+31) of rows g and g + 8 of
// both 16-row slices, and the matching 32 activations of token g. Within a
// window the MMA k order is permuted consistently for both operands: step j
// takes codes 4j..4j+3 of each lane's 32, i.e. bytes 2j and 2j+1.
#include "qz_gemm.cuh"
#include "qz_next.cuh"

#include <algorithm>

namespace qz {

namespace {

constexpr int F4_ROWS = 32;             // weight rows (output columns) per CTA
constexpr int F4_WARPS = 8;

struct F4Prob {
    const uint16_t* A;                  // bf16 [M, K]
    const uint8_t* Q;                   // E2M1 codes [N, K/2]
    const uint8_t* S;                   // NVFP4: E4M3 [N, K/16]; MXFP4: E8M0 [N, K/32]
    const float* g;                     // NVFP4 tensor scale (device scalar), MXFP4: unused
    uint16_t* Y;                        // bf16 [M, N]
    int M, N, K;
};

__device__ __forceinline__ void mma16816(float c[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
                 "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The two codes of byte P of w as bf16x2 bit patterns of value * 2^-126 (low
// half: the even code). w4 = w >> 4, whose top byte has a clear top bit, so
// selector 0xF yields a zero byte.
template <int P>
__device__ __forceinline__ uint32_t e2m1_pair_placed(uint32_t w, uint32_t w4) {
    const uint32_t r = __byte_perm(w, w4, (uint32_t)P | 0xF0u | ((uint32_t)(4 + P) << 8) | 0xF000u);
    const uint32_t a = r << 6, b = (r << 12) & 0x80008000u;
    uint32_t out;
    asm("lop3.b32 %0, %1, %2, %3, 0xEC;" : "=r"(out) : "r"(a), "r"(b), "r"(0x01C001C0u));   // (a & c) | b
    return out;
}

__device__ __forceinline__ uint32_t bmul2(uint32_t x, uint32_t f) {
    uint32_t out;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(out) : "r"(x), "r"(f));
    return out;
}

// F = scale * 2^62 as bf16x2 (both halves). NVFP4: E4M3 byte -> fp32 bits with
// the code at bits 20..27 are scale * 2^-120 (normal or subnormal, exact),
// times 2^91 twice; MXFP4: exponent field E - 127 + 62 + 127.
template <bool NV>
__device__ __forceinline__ uint32_t scale_x2(uint32_t code) {
    uint32_t hi;
    if (NV) {
        const float f = __fmul_rn(__fmul_rn(__uint_as_float((code & 0x7Fu) << 20), 0x1p91f), 0x1p91f);
        hi = (__float_as_uint(f) >> 16) | ((code & 0x80u) << 8);
    } else {
        hi = (code + 62u) << 7;
    }
    return hi | (hi << 16);
}

template <int MT, bool NV>
__global__ void __launch_bounds__(F4_WARPS * 32, MT <= 8 ? 3 : 2)
w4a16_fp4_kernel(const __grid_constant__ F4Prob P) {
    constexpr int MB = MT / 8;
    __shared__ float red[F4_WARPS][MT][F4_ROWS + 1];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const int n0 = blockIdx.x * F4_ROWS;
    const int nwin = P.K >> 7;
    const size_t qpitch = (size_t)P.K / 2, spitch = (size_t)P.K / (NV ? 16 : 32);
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    // rows n0 + 16 sl + g + 8 h of the CTA's 32
    const uint8_t* qrow[2][2];
    const uint8_t* srow[2][2];
#pragma unroll
    for (int sl = 0; sl < 2; sl++)
#pragma unroll
        for (int h = 0; h < 2; h++) {
            const size_t n = (size_t)n0 + 16 * sl + g + 8 * h;
            qrow[sl][h] = P.Q + n * qpitch + 16 * t;
            srow[sl][h] = P.S + n * spitch + (NV ? 2 * t : t);
        }
    float acc[2][MB][4];
#pragma unroll
    for (int sl = 0; sl < 2; sl++)
#pragma unroll
        for (int mb = 0; mb < MB; mb++) acc[sl][mb][0] = acc[sl][mb][1] = acc[sl][mb][2] = acc[sl][mb][3] = 0.0f;

    asm volatile("griddepcontrol.wait;" ::: "memory");
    const uint16_t* arow[MB];
    bool live[MB];
#pragma unroll
    for (int mb = 0; mb < MB; mb++) {
        live[mb] = mb * 8 + g < P.M;
        arow[mb] = P.A + (size_t)(live[mb] ? mb * 8 + g : 0) * P.K + 32 * t;
    }

    for (int win = warp; win < nwin; win += F4_WARPS) {
        uint4 wv[2][2];
        uint32_t sc[2][2];
#pragma unroll
        for (int sl = 0; sl < 2; sl++)
#pragma unroll
            for (int h = 0; h < 2; h++) {
                const uint8_t* q = qrow[sl][h] + (size_t)win * 64;
                asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                             : "=r"(wv[sl][h].x), "=r"(wv[sl][h].y), "=r"(wv[sl][h].z), "=r"(wv[sl][h].w) : "l"(q));
                sc[sl][h] = NV ? (uint32_t)__ldg(reinterpret_cast<const unsigned short*>(srow[sl][h] + (size_t)win * 8))
                               : (uint32_t)__ldg(srow[sl][h] + (size_t)win * 4);
            }
        uint4 av[MB][4];
#pragma unroll
        for (int mb = 0; mb < MB; mb++)
#pragma unroll
            for (int c = 0; c < 4; c++)
                av[mb][c] = live[mb] ? __ldg(reinterpret_cast<const uint4*>(arow[mb] + (size_t)win * 128 + 8 * c))
                                     : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int sl = 0; sl < 2; sl++) {
            // F of each row's block(s): NVFP4 blocks 2t (steps 0-3) and 2t+1 (steps 4-7); MXFP4 block t
            uint32_t f[2][2];
#pragma unroll
            for (int h = 0; h < 2; h++) {
                f[h][0] = scale_x2<NV>(NV ? (sc[sl][h] & 0xFFu) : sc[sl][h]);
                f[h][1] = NV ? scale_x2<NV>(sc[sl][h] >> 8) : f[h][0];
            }
#pragma unroll
            for (int c = 0; c < 4; c++) {                          // word c of each row: steps 2c, 2c+1
                const uint32_t w0 = c == 0 ? wv[sl][0].x : c == 1 ? wv[sl][0].y : c == 2 ? wv[sl][0].z : wv[sl][0].w;
                const uint32_t w1 = c == 0 ? wv[sl][1].x : c == 1 ? wv[sl][1].y : c == 2 ? wv[sl][1].z : wv[sl][1].w;
                const uint32_t x0 = w0 >> 4, x1 = w1 >> 4;
                const int b = c >> 1;                              // scale block of steps 2c, 2c+1
                const uint32_t a00 = bmul2(e2m1_pair_placed<0>(w0, x0), f[0][b]);
                const uint32_t a01 = bmul2(e2m1_pair_placed<1>(w0, x0), f[0][b]);
                const uint32_t a02 = bmul2(e2m1_pair_placed<2>(w0, x0), f[0][b]);
                const uint32_t a03 = bmul2(e2m1_pair_placed<3>(w0, x0), f[0][b]);
                const uint32_t a10 = bmul2(e2m1_pair_placed<0>(w1, x1), f[1][b]);
                const uint32_t a11 = bmul2(e2m1_pair_placed<1>(w1, x1), f[1][b]);
                const uint32_t a12 = bmul2(e2m1_pair_placed<2>(w1, x1), f[1][b]);
                const uint32_t a13 = bmul2(e2m1_pair_placed<3>(w1, x1), f[1][b]);
#pragma unroll
                for (int mb = 0; mb < MB; mb++) {
                    const uint4 bv = av[mb][c];                    // activations 8c .. 8c+7 of the lane's 32
                    mma16816(acc[sl][mb], a00, a10, a01, a11, bv.x, bv.y);     // step 2c: bytes 0, 1
                    mma16816(acc[sl][mb], a02, a12, a03, a13, bv.z, bv.w);     // step 2c+1: bytes 2, 3
                }
            }
        }
    }
    // warp partial sums -> shared memory; fixed-order sum over warps
#pragma unroll
    for (int sl = 0; sl < 2; sl++)
#pragma unroll
        for (int mb = 0; mb < MB; mb++) {
            const int m = mb * 8 + 2 * t, col = 16 * sl + g;
            red[warp][m][col] = acc[sl][mb][0];
            red[warp][m + 1][col] = acc[sl][mb][1];
            red[warp][m][col + 8] = acc[sl][mb][2];
            red[warp][m + 1][col + 8] = acc[sl][mb][3];
        }
    __syncthreads();
    const float back = NV ? __fmul_rn(0x1p64f, __ldg(P.g)) : 0x1p64f;
    const int mrows = min(P.M, MT);
    for (int i = threadIdx.x; i < mrows * (F4_ROWS / 2); i += F4_WARPS * 32) {
        const int m = i / (F4_ROWS / 2), col = 2 * (i % (F4_ROWS / 2));
        float y0 = red[0][m][col], y1 = red[0][m][col + 1];
#pragma unroll
        for (int w = 1; w < F4_WARPS; w++) {
            y0 += red[w][m][col];
            y1 += red[w][m][col + 1];
        }
        const __nv_bfloat162 o = __floats2bfloat162_rn(y0 * back, y1 * back);
        *reinterpret_cast<__nv_bfloat162*>(P.Y + (size_t)m * P.N + n0 + col) = o;
    }
}

template <int MT, bool NV>
qz_status launch_f4(const F4Prob& p, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.N / F4_ROWS);
    cfg.blockDim = dim3(F4_WARPS * 32);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, w4a16_fp4_kernel<MT, NV>, p) != cudaSuccess) return QZ_ERR_CUDA;
    return launch_status();
}

} // namespace

qz_status gemm_w4a16_fp4_launch(bool nv, const uint16_t* A, const uint8_t* qB, const uint8_t* sB, const float* gB,
                                uint16_t* Y, int M, int N, int K, cudaStream_t st) {
    const F4Prob p = {A, qB, sB, gB, Y, M, N, K};
    if (nv) return M <= 8 ? launch_f4<8, true>(p, st) : launch_f4<16, true>(p, st);
    return M <= 8 ? launch_f4<8, false>(p, st) : launch_f4<16, false>(p, st);
}

} // namespace qz
