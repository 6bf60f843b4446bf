// quantize.cu -- quantizer kernels: FP8 E4M3 (per tensor / row / 128x128 /
// 1x128), MXFP4, NVFP4, INT4 g128, and the FP8 KV-cache write.
//
// Each quantizer follows the fake-quant functions of "量化部署实战"
// (anrans.github.io), section 伪量化实现: reduce |x| to an amax per scale
// unit, derive the scale, then encode every element as code(x / scale).
// The kernels emit the codes, the scales and optionally the dequantized fp32
// tensor. They are HBM-bound: every thread moves 8 consecutive elements with
// 16- or 32-byte loads, amax reductions use warp shuffles, and codes leave as
// packed 4- or 8-byte stores.
//
// Per-tensor amax (FP8 per tensor, NVFP4's tensor scale, the KV write) is a
// two-kernel reduction: kernel 1 writes one partial max per CTA into the
// workspace, kernel 2 reduces those partials in every CTA (a few KB, read from
// L2) before encoding. No atomics, no zero-initialised workspace.
#include "qz_internal.cuh"

#include <cuda_fp16.h>
#include <algorithm>

namespace qz {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

// Programmatic dependent launch: the amax kernel lets its dependent (the
// encoder) start once every CTA has stored its partial; the encoder waits for
// the amax kernel's results before reading the partials (a no-op when it was
// launched without a programmatic dependency).
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// CTA-wide max of a per-thread value; every thread gets the result.
__device__ __forceinline__ float block_max(float v, float* red) {
    v = warp_max(v, 32);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    __syncthreads();                       // `red` may still be in use by a previous call
    if (l == 0) red[w] = v;
    __syncthreads();
    float r = red[0];
#pragma unroll
    for (int i = 1; i < kWarps; i++) r = fmaxf(r, red[i]);
    return r;
}

// FP8 encode of one value with scale s (clamp to +-448, E4M3 RNE).
__device__ __forceinline__ uint32_t fp8_code(float x, float s) {
    float y = div_rn(x, s);
    y = fminf(fmaxf(y, -kFp8Max), kFp8Max);
    return e4m3_code(y);
}

__device__ __forceinline__ float fp8_scale(float amax) {
    return div1(fmaxf(amax, kAmaxMin), Recip(kFp8Max));     // max(amax, 1e-12) / 448, correctly rounded
}

// Encode 8 values with scale d.s; write 8 code bytes (and 8 dequantized
// floats). The quotients are correctly rounded (Recip), the E4M3 conversion
// is the hardware's round-to-nearest-even, saturating at +-448 (the clamp).
__device__ __forceinline__ void fp8_encode8(const float v[8], const Recip& d, uint8_t* codes, float* deq) {
    float y[8];
#pragma unroll
    for (int j = 0; j < 8; j++) y[j] = sign_of(div1(v[j], d), v[j]);
    uint32_t p[4];
#pragma unroll
    for (int j = 0; j < 4; j++) p[j] = e4m3x2(y[2 * j], y[2 * j + 1]);
    uint2 out;
    out.x = __byte_perm(p[0], p[1], 0x5410);
    out.y = __byte_perm(p[2], p[3], 0x5410);
    *reinterpret_cast<uint2*>(codes) = out;
    if (deq) {
        float o[8];
#pragma unroll
        for (int j = 0; j < 8; j++) o[j] = __fmul_rn(e4m3_value((j & 1) ? (p[j >> 1] >> 8) : p[j >> 1]), d.s);
        reinterpret_cast<float4*>(deq)[0] = make_float4(o[0], o[1], o[2], o[3]);
        reinterpret_cast<float4*>(deq)[1] = make_float4(o[4], o[5], o[6], o[7]);
    }
}

// Element offset of chunk i (8 elements per chunk when VEC, 1 otherwise).
template <bool VEC>
__device__ __forceinline__ int64_t chunk_offset(int64_t i, bool contig, int64_t cpr, int64_t ldx) {
    constexpr int E = VEC ? 8 : 1;
    if (contig) return i * E;
    int64_t r = i / cpr;
    return r * ldx + (i - r * cpr) * E;
}

// Chunks of 8 elements per lane per iteration: U for the amax pass (loads kept
// in flight), UQ for the warp-uniform encoders (one: those run as many small
// CTAs instead, which measured faster than deeper unrolling).
constexpr int U = 4;
constexpr int UQ = 1;

// ------------------------------------------------------ per-tensor amax

// Kernel 1 of a per-tensor reduction: partial[y * gridDim.x + blockIdx.x] =
// max |x_y| over this CTA's grid-stride share of tensor y (y = blockIdx.y,
// at most two tensors, for K and V). U chunks per thread are loaded before
// any is reduced.
template <typename T, bool VEC>
__global__ void __launch_bounds__(kThreads)
amax_partial_kernel(const T* __restrict__ x0, const T* __restrict__ x1, int64_t rows, int64_t cols,
                    int64_t ldx, bool contig, float* __restrict__ partial) {
    pdl_wait();                                   // the previous kernel on the stream has finished
    __shared__ float red[kWarps];
    const T* x = blockIdx.y ? x1 : x0;
    const int64_t cpr = VEC ? cols / 8 : cols;
    const int64_t total = rows * cpr;
    float m = 0.0f;
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    for (int64_t i0 = (int64_t)blockIdx.x * kThreads + threadIdx.x; i0 < total; i0 += U * stride) {
        if constexpr (VEC && sizeof(T) == 2) {               // bf16: raw words in flight, widened at use
            uint4 r[U];
#pragma unroll
            for (int u = 0; u < U; u++) {
                const int64_t i = i0 + u * stride;
                r[u] = i < total ? __ldg(reinterpret_cast<const uint4*>(x + chunk_offset<true>(i, contig, cpr, ldx)))
                                 : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int u = 0; u < U; u++) {
                const uint32_t w[4] = {r[u].x, r[u].y, r[u].z, r[u].w};
#pragma unroll
                for (int q = 0; q < 4; q++)
                    m = fmaxf(m, fmaxf(fabsf(__uint_as_float(w[q] << 16)), fabsf(__uint_as_float(w[q] & 0xFFFF0000u))));
            }
        } else if constexpr (VEC) {
            float v[U][8];
#pragma unroll
            for (int u = 0; u < U; u++) {
                const int64_t i = i0 + u * stride;
                if (i < total) Load8<T>::run(x + chunk_offset<true>(i, contig, cpr, ldx), v[u]);
                else for (int j = 0; j < 8; j++) v[u][j] = 0.0f;
            }
#pragma unroll
            for (int u = 0; u < U; u++)
#pragma unroll
                for (int j = 0; j < 8; j++) m = fmaxf(m, fabsf(v[u][j]));
        } else {
#pragma unroll
            for (int u = 0; u < U; u++) {
                const int64_t i = i0 + u * stride;
                if (i < total) m = fmaxf(m, fabsf(load1(x + chunk_offset<false>(i, contig, cpr, ldx))));
            }
        }
    }
    m = block_max(m, red);
    if (threadIdx.x == 0) partial[(int64_t)blockIdx.y * gridDim.x + blockIdx.x] = m;
    pdl_trigger();
}

__device__ __forceinline__ float reduce_partials(const float* __restrict__ p, int n, float* red) {
    pdl_wait();
    float m = 0.0f;
    for (int i = threadIdx.x; i < n; i += kThreads) m = fmaxf(m, __ldcg(p + i));
    return block_max(m, red);
}

// Kernel 2 of per-tensor FP8: every CTA reduces the partials to the tensor
// amax (or reads a caller-given scale, GIVEN), then encodes its grid-stride
// share. A given scale may make x / s overflow, so that path divides exactly
// per element and clamps as the fake-quant does.
template <typename T, bool VEC, bool GIVEN>
__global__ void __launch_bounds__(kThreads)
fp8_tensor_encode_kernel(const T* __restrict__ x0, const T* __restrict__ x1, int64_t rows, int64_t cols,
                         int64_t ldx, bool contig, const float* __restrict__ partial, int nparts,
                         const float* given0, const float* given1, uint8_t* __restrict__ c0,
                         uint8_t* __restrict__ c1, float* s0, float* s1, float* __restrict__ d0,
                         float* __restrict__ d1) {
    __shared__ float red[kWarps];
    const int y = blockIdx.y;
    const T* x = y ? x1 : x0;
    uint8_t* codes = y ? c1 : c0;
    float* deq = y ? d1 : d0;
    float s;
    if (!GIVEN) {
        s = fp8_scale(reduce_partials(partial + (int64_t)y * nparts, nparts, red));
        if (blockIdx.x == 0 && threadIdx.x == 0) *(y ? s1 : s0) = s;
    } else {
        s = __ldg(y ? given1 : given0);
    }
    const Recip d(s);
    const int64_t cpr = VEC ? cols / 8 : cols;
    const int64_t total = rows * cpr;
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    for (int64_t i0 = (int64_t)blockIdx.x * kThreads + threadIdx.x; i0 < total; i0 += 2 * stride) {
        if constexpr (VEC) {
            float v[2][8];
#pragma unroll
            for (int u = 0; u < 2; u++) {
                const int64_t i = i0 + u * stride;
                if (i < total) Load8<T>::run(x + chunk_offset<true>(i, contig, cpr, ldx), v[u]);
            }
#pragma unroll
            for (int u = 0; u < 2; u++) {
                const int64_t i = i0 + u * stride;
                if (i >= total) continue;
                if (GIVEN) {
                    uint8_t cb[8];
                    float o[8];
#pragma unroll
                    for (int j = 0; j < 8; j++) {
                        const uint32_t c = fp8_code(v[u][j], s);
                        cb[j] = (uint8_t)c;
                        o[j] = __fmul_rn(e4m3_value(c), s);
                    }
                    uint2 w;
                    w.x = cb[0] | (cb[1] << 8) | (cb[2] << 16) | ((uint32_t)cb[3] << 24);
                    w.y = cb[4] | (cb[5] << 8) | (cb[6] << 16) | ((uint32_t)cb[7] << 24);
                    *reinterpret_cast<uint2*>(codes + i * 8) = w;
                    if (deq) {
                        reinterpret_cast<float4*>(deq + i * 8)[0] = make_float4(o[0], o[1], o[2], o[3]);
                        reinterpret_cast<float4*>(deq + i * 8)[1] = make_float4(o[4], o[5], o[6], o[7]);
                    }
                } else {
                    fp8_encode8(v[u], d, codes + i * 8, deq ? deq + i * 8 : nullptr);
                }
            }
        } else {
#pragma unroll
            for (int u = 0; u < 2; u++) {
                const int64_t i = i0 + u * stride;
                if (i >= total) continue;
                const uint32_t c = fp8_code(load1(x + chunk_offset<false>(i, contig, cpr, ldx)), s);
                codes[i] = (uint8_t)c;
                if (deq) deq[i] = __fmul_rn(e4m3_value(c), s);
            }
        }
    }
    pdl_trigger();                                // the next call may launch as this one drains
}

// ---------------------------------------------------------- per row

// One warp per row: pass 1 reduces the row's amax (U loads in flight per
// lane), pass 2 re-reads the row (from L1/L2) and encodes it.
template <typename T, bool VEC>
__global__ void __launch_bounds__(kThreads)
fp8_row_kernel(const T* __restrict__ x, int64_t rows, int64_t cols, int64_t ldx,
               uint8_t* __restrict__ codes, float* __restrict__ scales, float* __restrict__ deq) {
    pdl_wait();                                   // the previous kernel on the stream has finished
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
    const int64_t nwarps = (int64_t)gridDim.x * kWarps;
    for (int64_t r = warp; r < rows; r += nwarps) {
        const T* xr = x + r * ldx;
        float m = 0.0f;
        if constexpr (VEC) {
            for (int64_t c0 = lane * 8; c0 < cols; c0 += U * 256) {
                float v[U][8];
#pragma unroll
                for (int u = 0; u < U; u++) {
                    if (c0 + u * 256 < cols) Load8<T>::run(xr + c0 + u * 256, v[u]);
                    else for (int j = 0; j < 8; j++) v[u][j] = 0.0f;
                }
#pragma unroll
                for (int u = 0; u < U; u++)
#pragma unroll
                    for (int j = 0; j < 8; j++) m = fmaxf(m, fabsf(v[u][j]));
            }
        } else {
            for (int64_t c = lane; c < cols; c += 32) m = fmaxf(m, fabsf(load1(xr + c)));
        }
        const float s = fp8_scale(warp_max(m, 32));
        if (lane == 0) scales[r] = s;
        uint8_t* cr = codes + r * cols;
        float* dr = deq ? deq + r * cols : nullptr;
        if constexpr (VEC) {
            const Recip d(s);
            for (int64_t c0 = lane * 8; c0 < cols; c0 += 2 * 256) {
                float v[2][8];
#pragma unroll
                for (int u = 0; u < 2; u++)
                    if (c0 + u * 256 < cols) Load8<T>::run(xr + c0 + u * 256, v[u]);
#pragma unroll
                for (int u = 0; u < 2; u++) {
                    const int64_t c = c0 + u * 256;
                    if (c < cols) fp8_encode8(v[u], d, cr + c, dr ? dr + c : nullptr);
                }
            }
        } else {
            for (int64_t c = lane; c < cols; c += 32) {
                const uint32_t code = fp8_code(load1(xr + c), s);
                cr[c] = (uint8_t)code;
                if (dr) dr[c] = __fmul_rn(e4m3_value(code), s);
            }
        }
    }
    pdl_trigger();                                // the next call may launch as this one drains
}

// ------------------------------------------------------- 1 x 128 groups

// 16 threads per 128-element group (8 elements each); a warp covers two
// groups per step and takes two steps at once. Loops run warp-uniformly so
// the shuffles always see 32 lanes.
template <typename T>
__global__ void __launch_bounds__(kThreads)
fp8_group_kernel(const T* __restrict__ x, int64_t rows, int64_t cols, int64_t ldx, bool contig,
                 uint8_t* __restrict__ codes, float* __restrict__ scales, float* __restrict__ deq) {
    pdl_wait();                                   // the previous kernel on the stream has finished
    const int lane = threadIdx.x & 31;
    const int64_t cpr = cols / 8;
    const int64_t total = rows * cpr;
    const int64_t wbase = (((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5) * (32 * UQ);
    const int64_t wstride = (int64_t)gridDim.x * kThreads * UQ;
    for (int64_t base = wbase; base < total; base += wstride) {
        float v[UQ][8];
#pragma unroll
        for (int u = 0; u < UQ; u++) {
            const int64_t i = base + u * 32 + lane;
            if (i < total) Load8<T>::run(x + chunk_offset<true>(i, contig, cpr, ldx), v[u]);
            else for (int j = 0; j < 8; j++) v[u][j] = 0.0f;
        }
#pragma unroll
        for (int u = 0; u < UQ; u++) {
            const int64_t i = base + u * 32 + lane;
            float m = 0.0f;
#pragma unroll
            for (int j = 0; j < 8; j++) m = fmaxf(m, fabsf(v[u][j]));
            const float s = fp8_scale(warp_max(m, 16));
            if (i < total) {
                if ((lane & 15) == 0) scales[i >> 4] = s;
                fp8_encode8(v[u], Recip(s), codes + i * 8, deq ? deq + i * 8 : nullptr);
            }
        }
    }
    pdl_trigger();                                // the next call may launch as this one drains
}

// ----------------------------------------------------- 128 x 128 blocks

// One CTA per (br x 128) block, br = min(128, rows); the block stays in
// registers in its input format (up to 8 chunks per thread) between the
// amax reduction and the encode.
template <typename T> struct Raw8;
template <> struct Raw8<float> {
    float4 a, b;
    __device__ __forceinline__ void load(const float* p) {
        a = __ldg(reinterpret_cast<const float4*>(p));
        b = __ldg(reinterpret_cast<const float4*>(p) + 1);
    }
    __device__ __forceinline__ void unpack(float v[8]) const {
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
};
template <> struct Raw8<uint16_t> {
    uint4 a;
    __device__ __forceinline__ void load(const uint16_t* p) { a = __ldg(reinterpret_cast<const uint4*>(p)); }
    __device__ __forceinline__ void unpack(float v[8]) const {
        const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int i = 0; i < 4; i++) {
            v[2 * i] = __uint_as_float(w[i] << 16);
            v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    }
};

template <typename T>
__global__ void __launch_bounds__(kThreads)
fp8_block_kernel(const T* __restrict__ x, int64_t rows, int64_t cols, int64_t ldx, int br,
                 uint8_t* __restrict__ codes, float* __restrict__ scales, float* __restrict__ deq) {
    pdl_wait();                                   // the previous kernel on the stream has finished
    __shared__ float red[kWarps];
    const int64_t nbc = cols / 128;
    const int64_t bi = blockIdx.x / nbc, bj = blockIdx.x % nbc;
    const int nchunks = br * 16;
    Raw8<T> raw[8];
#pragma unroll
    for (int u = 0; u < 8; u++) {
        const int j = threadIdx.x + u * kThreads;
        if (j < nchunks) raw[u].load(x + (bi * br + (j >> 4)) * ldx + bj * 128 + (j & 15) * 8);
    }
    float m = 0.0f;
#pragma unroll
    for (int u = 0; u < 8; u++) {
        const int j = threadIdx.x + u * kThreads;
        if (j < nchunks) {
            float v[8];
            raw[u].unpack(v);
#pragma unroll
            for (int e = 0; e < 8; e++) m = fmaxf(m, fabsf(v[e]));
        }
    }
    const float s = fp8_scale(block_max(m, red));
    if (threadIdx.x == 0) scales[blockIdx.x] = s;
    const Recip d(s);
#pragma unroll
    for (int u = 0; u < 8; u++) {
        const int j = threadIdx.x + u * kThreads;
        if (j < nchunks) {
            const int64_t r = bi * br + (j >> 4), c = bj * 128 + (j & 15) * 8;
            float v[8];
            raw[u].unpack(v);
            fp8_encode8(v, d, codes + r * cols + c, deq ? deq + r * cols + c : nullptr);
        }
    }
    pdl_trigger();                                // the next call may launch as this one drains
}

// ------------------------------------------------------------------ MXFP4

// 4 threads per 32-element block. scale = 2^(E-2) with E = floor(log2 amax)
// read from the exponent field; x / 2^(E-2) is exact as x * 2^(2-E).
template <typename T>
__global__ void __launch_bounds__(kThreads)
mxfp4_kernel(const T* __restrict__ x, int64_t rows, int64_t cols, int64_t ldx, bool contig,
             uint8_t* __restrict__ codes, uint8_t* __restrict__ e8m0, float* __restrict__ deq) {
    const int lane = threadIdx.x & 31;
    const int64_t cpr = cols / 8;
    const int64_t total = rows * cpr;
    const int64_t wbase = (((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5) * (32 * UQ);
    const int64_t wstride = (int64_t)gridDim.x * kThreads * UQ;
    for (int64_t base = wbase; base < total; base += wstride) {
        float v[UQ][8];
#pragma unroll
        for (int u = 0; u < UQ; u++) {
            const int64_t i = base + u * 32 + lane;
            if (i < total) Load8<T>::run(x + chunk_offset<true>(i, contig, cpr, ldx), v[u]);
            else for (int j = 0; j < 8; j++) v[u][j] = 0.0f;
        }
#pragma unroll
        for (int u = 0; u < UQ; u++) {
            const int64_t i = base + u * 32 + lane;
            float m = 0.0f;
#pragma unroll
            for (int j = 0; j < 8; j++) m = fmaxf(m, fabsf(v[u][j]));
            m = fmaxf(warp_max(m, 4), kAmaxMin);
            const int E = (int)((__float_as_uint(m) >> 23) & 0xFF) - 127;   // m is normal
            const float sc = __uint_as_float((uint32_t)(E - 2 + 127) << 23);
            const float inv = __uint_as_float((uint32_t)(127 + 2 - E) << 23);
            if (i < total) {
                const uint32_t packed = mxfp4_encode8<sizeof(T) == 2>(v[u], inv);
                reinterpret_cast<uint32_t*>(codes)[i] = packed;
                if (deq) {
                    float o[8];
#pragma unroll
                    for (int j = 0; j < 8; j++) o[j] = __fmul_rn(e2m1_value(packed >> (4 * j)), sc);
                    reinterpret_cast<float4*>(deq + i * 8)[0] = make_float4(o[0], o[1], o[2], o[3]);
                    reinterpret_cast<float4*>(deq + i * 8)[1] = make_float4(o[4], o[5], o[6], o[7]);
                }
                if ((lane & 3) == 0) e8m0[i >> 2] = (uint8_t)(E - 2 + 127);
            }
        }
    }
}

// ------------------------------------------------------------------ NVFP4

// One thread per 16-element block. g comes from the per-tensor partials (or
// a given amax); the block scale is E4M3(amax16 / 6 / g). A tensor has at most
// 128 block scales s = max(E4M3 value, 1e-12) * g, one per code: each CTA
// tabulates s and RN(1/s) once, so a block pays one table read instead of a
// correctly rounded reciprocal. I: the block index type (32 bits when the
// tensor allows).
template <typename T, typename I>
__global__ void __launch_bounds__(kThreads)
nvfp4_kernel(const T* __restrict__ x, int64_t rows, int64_t cols, int64_t ldx, bool contig,
             const float* __restrict__ partial, int nparts, const float* __restrict__ amax_in,
             uint8_t* __restrict__ codes, uint8_t* __restrict__ sb, float* __restrict__ g_out,
             float* __restrict__ deq) {
    __shared__ float red[kWarps];
    __shared__ float tab_s[128], tab_r[128];
    if (!partial) pdl_wait();                     // a given amax and x may be the previous kernel's output
    const float amax_t = partial ? reduce_partials(partial, nparts, red) : __ldg(amax_in);
    const float g = div_rn(fmaxf(amax_t, kAmaxMin), kFp8Max * kFp4Max);
    if (blockIdx.x == 0 && threadIdx.x == 0) *g_out = g;
    if (threadIdx.x < 128) {
        const float sv = __fmul_rn(fmaxf(e4m3_value(threadIdx.x), kAmaxMin), g);
        tab_s[threadIdx.x] = sv;
        tab_r[threadIdx.x] = __frcp_rn(sv);
    }
    __syncthreads();
    const Recip dg(g), d6(kFp4Max);
    const I bpr = (I)(cols / 16);
    const I total = (I)rows * bpr;
    const I stride = (I)gridDim.x * kThreads;
    for (I i = (I)blockIdx.x * kThreads + threadIdx.x; i < total; i += stride) {
        const T* p = x + (contig ? (int64_t)i * 16 : (int64_t)(i / bpr) * ldx + (int64_t)(i % bpr) * 16);
        float v[16];
        Load8<T>::run(p, v);
        Load8<T>::run(p + 8, v + 8);
        float m = 0.0f;
#pragma unroll
        for (int j = 0; j < 16; j++) m = fmaxf(m, fabsf(v[j]));
        // t = (amax16 / 6) / g, both quotients correctly rounded
        const float t = div1(div1(m, d6), dg);
        const uint32_t bcode = e4m3_code(t);                     // saturating, as the clamp-free page
        const uint2 packed = fp4_encode16(v, Recip(tab_s[bcode], tab_r[bcode]), deq ? deq + (int64_t)i * 16 : nullptr);
        reinterpret_cast<uint2*>(codes)[i] = packed;
        sb[i] = (uint8_t)bcode;
    }
    pdl_trigger();                                // the next call may launch as this one drains
}

// ------------------------------------------------- NVFP4, many tensors

// A decode step's activations (one small tensor per linear) quantized in two
// launches instead of two per tensor: kernel 1 reduces each tensor's amax in
// NV_SLICES partial maxima (one CTA per slice), kernel 2 walks the
// concatenation of all tensors' 16-element blocks, one per thread; each block
// looks up its tensor, reduces that tensor's partials to g and encodes as
// nvfp4_kernel does.
constexpr int NV_GROUP_MAX = 256;
constexpr int NV_SLICES = 4;

struct NvTensor {
    const void* x;                      // contiguous [rows, cols]
    uint8_t* codes;                     // [rows, cols/2]
    uint8_t* sb;                        // [rows, cols/16]
    float* g;                           // 1 fp32
    long long chunk_begin;              // first 8-element chunk of this tensor in the launch
    long long chunks;
};

struct NvGroup {
    NvTensor t[NV_GROUP_MAX];
    int count;
    long long total_chunks;
};

template <typename T>
__global__ void __launch_bounds__(kThreads)
nvfp4_group_amax_kernel(const __grid_constant__ NvGroup P, float* __restrict__ partial) {
    pdl_wait();                                   // the previous kernel on the stream has finished
    __shared__ float red[kWarps];
    const int ti = blockIdx.x / NV_SLICES, sl = blockIdx.x % NV_SLICES;
    const NvTensor& tn = P.t[ti];
    const T* x = static_cast<const T*>(tn.x);
    const long long cb = tn.chunks * sl / NV_SLICES, ce = tn.chunks * (sl + 1) / NV_SLICES;
    float m = 0.0f;
    for (long long i0 = cb + threadIdx.x; i0 < ce; i0 += (long long)U * kThreads) {
        float v[U][8];
#pragma unroll
        for (int u = 0; u < U; u++) {
            const long long i = i0 + (long long)u * kThreads;
            if (i < ce) Load8<T>::run(x + i * 8, v[u]);
            else for (int j = 0; j < 8; j++) v[u][j] = 0.0f;
        }
#pragma unroll
        for (int u = 0; u < U; u++)
#pragma unroll
            for (int j = 0; j < 8; j++) m = fmaxf(m, fabsf(v[u][j]));
    }
    m = block_max(m, red);
    if (threadIdx.x == 0) partial[blockIdx.x] = m;
    pdl_trigger();
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
nvfp4_group_encode_kernel(const __grid_constant__ NvGroup P, const float* __restrict__ partial) {
    pdl_wait();
    const Recip d6(kFp4Max);
    const long long total = P.total_chunks / 2;              // 16-element blocks (every tensor holds whole ones)
    for (long long i = (long long)blockIdx.x * kThreads + threadIdx.x; i < total; i += (long long)gridDim.x * kThreads) {
        const long long c = 2 * i;                            // first chunk of block i
        int lo = 0, hi = P.count - 1;                        // tensor of block i
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (P.t[mid].chunk_begin <= c) lo = mid; else hi = mid - 1;
        }
        const NvTensor& tn = P.t[lo];
        const long long li = (c - tn.chunk_begin) >> 1;      // block within the tensor
        float amax_t = 0.0f;
#pragma unroll
        for (int k = 0; k < NV_SLICES; k++) amax_t = fmaxf(amax_t, __ldg(partial + lo * NV_SLICES + k));
        const float g = div_rn(fmaxf(amax_t, kAmaxMin), kFp8Max * kFp4Max);
        if (li == 0) *tn.g = g;
        const Recip dg(g);
        float v[16];
        const T* p = static_cast<const T*>(tn.x) + li * 16;
        Load8<T>::run(p, v);
        Load8<T>::run(p + 8, v + 8);
        float m = 0.0f;
#pragma unroll
        for (int j = 0; j < 16; j++) m = fmaxf(m, fabsf(v[j]));
        const float t = div1(div1(m, d6), dg);
        const uint32_t bcode = e4m3_code(t);
        const float sv = __fmul_rn(fmaxf(e4m3_value(bcode), kAmaxMin), g);
        reinterpret_cast<uint2*>(tn.codes)[li] = fp4_encode16(v, Recip(sv), nullptr);
        tn.sb[li] = (uint8_t)bcode;
    }
    pdl_trigger();                                // the next call may launch as this one drains
}

// --------------------------------------------------------------- INT4 g128

// One CTA per (group of 128 rows) x (64 columns) tile of w[K, N]: the tile is
// staged in shared memory, 4 threads reduce each column's amax over 32 rows,
// then every (k-octet, column) pair packs eight 4-bit codes into one int32.
template <typename T>
__global__ void __launch_bounds__(kThreads)
int4_g128_kernel(const T* __restrict__ w, int64_t K, int64_t N, int64_t ldw,
                 int32_t* __restrict__ qweight, uint16_t* __restrict__ scale, float* __restrict__ deq) {
    pdl_wait();                                   // the previous kernel on the stream has finished
    __shared__ float tile[128][65];
    __shared__ float part[4][64];
    __shared__ float sc[64];
    const int64_t ncb = N / 64;
    const int64_t g = blockIdx.x / ncb, n0 = (blockIdx.x % ncb) * 64;
    // load 128 x 64 (8 chunks of 8 per row; 1024 chunks, 4 per thread)
#pragma unroll
    for (int u = 0; u < 4; u++) {
        const int j = threadIdx.x + u * kThreads;
        const int r = j >> 3, c = (j & 7) * 8;
        float v[8];
        Load8<T>::run(w + (g * 128 + r) * ldw + n0 + c, v);
#pragma unroll
        for (int e = 0; e < 8; e++) tile[r][c + e] = v[e];
    }
    __syncthreads();
    {
        const int c = threadIdx.x & 63, p = threadIdx.x >> 6;
        float m = 0.0f;
        for (int r = p * 32; r < p * 32 + 32; r++) m = fmaxf(m, fabsf(tile[r][c]));
        part[p][c] = m;
    }
    __syncthreads();
    if (threadIdx.x < 64) {
        const int c = threadIdx.x;
        const float m = fmaxf(fmaxf(part[0][c], part[1][c]), fmaxf(part[2][c], part[3][c]));
        const float sf = div_rn(fmaxf(m, kAmaxMin), 7.0f);
        const __nv_bfloat16 sb = __float2bfloat16_rn(sf);
        const uint16_t bits = __bfloat16_as_ushort(sb);
        scale[g * N + n0 + c] = bits;
        sc[c] = bf16_bits_to_f32(bits);
    }
    __syncthreads();
#pragma unroll
    for (int u = 0; u < 4; u++) {
        const int j = threadIdx.x + u * kThreads;        // 16 octets x 64 columns
        const int o = j >> 6, c = j & 63;
        const float s = sc[c];
        uint32_t word = 0;
#pragma unroll
        for (int e = 0; e < 8; e++) {
            const float val = tile[o * 8 + e][c];
            float q = rintf(div_rn(val, s));
            q = fminf(fmaxf(q, -8.0f), 7.0f);
            word |= ((uint32_t)(int)q & 0xFu) << (4 * e);
            if (deq) deq[(g * 128 + o * 8 + e) * N + n0 + c] = __fmul_rn(q, s);
        }
        qweight[(g * 16 + o) * N + n0 + c] = (int32_t)word;
    }
    pdl_trigger();                                // the next call may launch as this one drains
}

// ---------------------------------------------------------------- helpers

int amax_grid() { return num_sms() * 4; }

// Launch `kernel` so that it may start while the previous kernel on the stream
// finishes (it must call pdl_wait before consuming that kernel's results). Every
// quantizer's first kernel is launched this way and waits at its start, and every
// last kernel triggers at its end, so back-to-back calls (or a producer that
// triggers) overlap one call's launch and ramp with the previous one's tail
// (1024 x 1024 round trips 0.3-0.6 us faster, KV write 11.5 -> 11.1 us). The MXFP4
// encoder is the exception: launched this way it measured 17.2 -> 19.7 us at
// 8192 x 4096, so it keeps the plain launch.
template <typename... KArgs, typename... Args>
void launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Grid of a grid-stride kernel: one thread per unit of work, capped at
// per_sm CTAs per SM (the warp-uniform encoders run best with many small CTAs
// in flight; the two-pass per-tensor encoder with one wave).
int stream_grid(int64_t threads_needed, int per_sm = 4) {
    const int64_t ctas = (threads_needed + kThreads - 1) / kThreads;
    return (int)std::max<int64_t>(1, std::min<int64_t>(ctas, (int64_t)num_sms() * per_sm));
}
constexpr int kEncoderCtasPerSm = 16;     // FP8 1x128 (2048 x 4096 bf16: 16 per SM 7.55 us, 8 8.29, 32 8.61)
constexpr int kMxfp4CtasPerSm = 8;        // MXFP4 (8192 x 4096 bf16: 8 per SM 16.77 us, 16 16.91, 32 17.41)
constexpr int kNvfp4CtasPerSm = 4;       // the NVFP4 encoder's CTAs also build a scale table (8192 x 4096 bf16: 4 per SM 27.2 us, 6 27.3, 8 27.5, 16 28.2)

bool vec_ok(const void* x, int64_t ldx, int64_t cols, qz_dtype t) {
    const size_t es = t == QZ_F32 ? 4 : 2;
    return is_aligned(x, 16) && ((size_t)ldx * es) % 16 == 0 && cols % 8 == 0;
}

template <typename T, bool VEC>
void launch_tensor_amax(const void* x0, const void* x1, int ny, int64_t rows, int64_t cols, int64_t ldx,
                        bool contig, float* partial, cudaStream_t st) {
    dim3 grid(amax_grid(), ny);
    launch_dependent(amax_partial_kernel<T, VEC>, grid, dim3(kThreads), st, (const T*)x0, (const T*)x1, rows, cols,
                     ldx, contig, partial);
}

} // namespace

size_t ws_quantize_fp8_tensor(int64_t, int64_t) { return (size_t)amax_grid() * sizeof(float); }
size_t ws_quantize_nvfp4(int64_t, int64_t) { return (size_t)amax_grid() * sizeof(float); }
size_t ws_kv_write(int64_t) { return (size_t)2 * amax_grid() * sizeof(float); }

template <typename T>
static qz_status fp8_launch_t(const T* x, int64_t rows, int64_t cols, int64_t ldx, qz_fp8_gran gran,
                              uint8_t* codes, float* scales, float* deq, void* ws, cudaStream_t st,
                              bool vec) {
    const bool contig = (ldx == cols);
    switch (gran) {
    case QZ_FP8_PER_TENSOR: {
        float* partial = (float*)ws;
        const int np = amax_grid();
        const int64_t work = vec ? rows * cols / 8 : rows * cols;
        const float* none = nullptr;
        if (vec) {
            launch_tensor_amax<T, true>(x, x, 1, rows, cols, ldx, contig, partial, st);
            launch_dependent(fp8_tensor_encode_kernel<T, true, false>, dim3(stream_grid(work), 1), dim3(kThreads), st,
                             x, x, rows, cols, ldx, contig, (const float*)partial, np, none, none, codes, codes,
                             scales, scales, deq, deq);
        } else {
            launch_tensor_amax<T, false>(x, x, 1, rows, cols, ldx, contig, partial, st);
            launch_dependent(fp8_tensor_encode_kernel<T, false, false>, dim3(stream_grid(work), 1), dim3(kThreads),
                             st, x, x, rows, cols, ldx, contig, (const float*)partial, np, none, none, codes,
                             codes, scales, scales, deq, deq);
        }
        break;
    }
    case QZ_FP8_PER_ROW: {
        const int grid = (int)std::max<int64_t>(1, std::min<int64_t>((rows + kWarps - 1) / kWarps,
                                                                     (int64_t)num_sms() * 8));
        if (vec) launch_dependent(fp8_row_kernel<T, true>, dim3(grid), dim3(kThreads), st, x, rows, cols, ldx, codes, scales, deq);
        else launch_dependent(fp8_row_kernel<T, false>, dim3(grid), dim3(kThreads), st, x, rows, cols, ldx, codes, scales, deq);
        break;
    }
    case QZ_FP8_GROUP_1x128:
        launch_dependent(fp8_group_kernel<T>, dim3(stream_grid(rows * cols / 8, kEncoderCtasPerSm)), dim3(kThreads), st,
                         x, rows, cols, ldx, contig, codes, scales, deq);
        break;
    case QZ_FP8_BLOCK_128x128: {
        const int br = (int)std::min<int64_t>(128, rows);
        const int64_t nblocks = (rows / br) * (cols / 128);
        launch_dependent(fp8_block_kernel<T>, dim3((unsigned)nblocks), dim3(kThreads), st, x, rows, cols, ldx, br, codes,
                         scales, deq);
        break;
    }
    }
    return launch_status();
}

qz_status quantize_fp8_launch(const void* x, qz_dtype xt, int64_t rows, int64_t cols, int64_t ldx,
                              qz_fp8_gran gran, uint8_t* codes, float* scales, float* deq,
                              void* ws, size_t, cudaStream_t st) {
    const bool vec = vec_ok(x, ldx, cols, xt);
    if (xt == QZ_F32) return fp8_launch_t<float>((const float*)x, rows, cols, ldx, gran, codes, scales, deq, ws, st, vec);
    return fp8_launch_t<uint16_t>((const uint16_t*)x, rows, cols, ldx, gran, codes, scales, deq, ws, st, vec);
}

qz_status quantize_mxfp4_launch(const void* x, qz_dtype xt, int64_t rows, int64_t cols, int64_t ldx,
                                uint8_t* codes, uint8_t* e8m0, float* deq, cudaStream_t st) {
    const bool contig = (ldx == cols);
    const int grid = stream_grid(rows * cols / 8, kMxfp4CtasPerSm);
    if (xt == QZ_F32)
        mxfp4_kernel<float><<<grid, kThreads, 0, st>>>((const float*)x, rows, cols, ldx, contig, codes, e8m0, deq);
    else
        mxfp4_kernel<uint16_t><<<grid, kThreads, 0, st>>>((const uint16_t*)x, rows, cols, ldx, contig, codes, e8m0, deq);
    return launch_status();
}

template <typename T, typename I>
void launch_nvfp4_encode(const T* x, int64_t rows, int64_t cols, int64_t ldx, bool contig, const float* partial,
                         int np, const float* amax_in, uint8_t* codes, uint8_t* sb, float* g, float* deq,
                         cudaStream_t st) {
    const int grid = stream_grid(rows * cols / 16, kNvfp4CtasPerSm);
    launch_dependent(nvfp4_kernel<T, I>, dim3(grid), dim3(kThreads), st, x, rows, cols, ldx, contig, partial, np,
                     amax_in, codes, sb, g, deq);
}

template <typename T>
void launch_nvfp4(const T* x, int64_t rows, int64_t cols, int64_t ldx, bool contig, float* partial,
                  const float* amax_in, uint8_t* codes, uint8_t* sb, float* g, float* deq, cudaStream_t st) {
    const int np = amax_grid();
    if (partial) launch_tensor_amax<T, true>(x, x, 1, rows, cols, ldx, contig, partial, st);
    const int64_t blocks = rows * cols / 16;
    // 32-bit block indices while the last grid-stride step cannot overflow them
    if (blocks + (int64_t)stream_grid(blocks, kNvfp4CtasPerSm) * kThreads < ((int64_t)1 << 31))
        launch_nvfp4_encode<T, int>(x, rows, cols, ldx, contig, partial, np, amax_in, codes, sb, g, deq, st);
    else
        launch_nvfp4_encode<T, int64_t>(x, rows, cols, ldx, contig, partial, np, amax_in, codes, sb, g, deq, st);
}

qz_status quantize_nvfp4_launch(const void* x, qz_dtype xt, int64_t rows, int64_t cols, int64_t ldx,
                                uint8_t* codes, uint8_t* sb, float* g, const float* amax_in,
                                float* deq, void* ws, size_t, cudaStream_t st) {
    const bool contig = (ldx == cols);
    float* partial = amax_in ? nullptr : (float*)ws;
    if (xt == QZ_F32)
        launch_nvfp4<float>((const float*)x, rows, cols, ldx, contig, partial, amax_in, codes, sb, g, deq, st);
    else
        launch_nvfp4<uint16_t>((const uint16_t*)x, rows, cols, ldx, contig, partial, amax_in, codes, sb, g, deq, st);
    return launch_status();
}

size_t ws_quantize_nvfp4_grouped(int count) { return (size_t)count * NV_SLICES * sizeof(float); }

qz_status quantize_nvfp4_grouped_launch(const qz_nvfp4_tensor* tensors, int count, qz_dtype xt, void* ws,
                                        cudaStream_t st) {
    NvGroup P;
    P.count = count;
    long long total = 0;
    for (int i = 0; i < count; i++) {
        const qz_nvfp4_tensor& q = tensors[i];
        NvTensor& t = P.t[i];
        t.x = q.x;
        t.codes = q.codes;
        t.sb = q.scale_e4m3;
        t.g = q.global_scale;
        t.chunk_begin = total;
        t.chunks = q.rows * q.cols / 8;
        total += t.chunks;
    }
    P.total_chunks = total;
    float* partial = static_cast<float*>(ws);
    const int grid = stream_grid(total / 2, kEncoderCtasPerSm);
    if (xt == QZ_F32) {
        launch_dependent(nvfp4_group_amax_kernel<float>, dim3(count * NV_SLICES), dim3(kThreads), st, P, partial);
        launch_dependent(nvfp4_group_encode_kernel<float>, dim3(grid), dim3(kThreads), st, P, (const float*)partial);
    } else {
        launch_dependent(nvfp4_group_amax_kernel<uint16_t>, dim3(count * NV_SLICES), dim3(kThreads), st, P, partial);
        launch_dependent(nvfp4_group_encode_kernel<uint16_t>, dim3(grid), dim3(kThreads), st, P,
                         (const float*)partial);
    }
    return launch_status();
}

qz_status quantize_int4_launch(const void* w, qz_dtype wt, int64_t K, int64_t N, int64_t ldw,
                               int32_t* qweight, uint16_t* scale, float* deq, cudaStream_t st) {
    const int64_t nblocks = (K / 128) * (N / 64);
    if (wt == QZ_F32)
        launch_dependent(int4_g128_kernel<float>, dim3((unsigned)nblocks), dim3(kThreads), st, (const float*)w, K, N, ldw,
                         qweight, scale, deq);
    else
        launch_dependent(int4_g128_kernel<uint16_t>, dim3((unsigned)nblocks), dim3(kThreads), st, (const uint16_t*)w, K, N,
                         ldw, qweight, scale, deq);
    return launch_status();
}

qz_status kv_write_launch(const uint16_t* k, const uint16_t* v, int64_t n, uint8_t* kc, uint8_t* vc,
                          float* ks, float* vs, qz_scale_mode mode, void* ws, size_t, cudaStream_t st) {
    const int np = amax_grid();
    float* partial = (mode == QZ_SCALE_COMPUTE) ? (float*)ws : nullptr;
    // 3 encoder CTAs per SM and tensor: every CTA first reduces all partials,
    // so fewer, longer-lived CTAs measured faster (9.4 us at 4M elements per
    // tensor, against 10.8 with 4 per SM and 14.0 with 16)
    const dim3 grid(stream_grid(n / 8, 3), 2);
    if (partial) {
        const float* none = nullptr;
        float* nod = nullptr;
        launch_tensor_amax<uint16_t, true>(k, v, 2, 1, n, n, true, partial, st);
        launch_dependent(fp8_tensor_encode_kernel<uint16_t, true, false>, grid, dim3(kThreads), st, k, v, (int64_t)1,
                         n, n, true, (const float*)partial, np, none, none, kc, vc, ks, vs, nod, nod);
    } else {
        fp8_tensor_encode_kernel<uint16_t, true, true><<<grid, kThreads, 0, st>>>(
            k, v, 1, n, n, true, nullptr, np, ks, vs, kc, vc, nullptr, nullptr, nullptr, nullptr);
    }
    return launch_status();
}

} // namespace qz
