// quantize_next.cu -- the quantizer variants beyond the four base formats:
//  * INT4 with a zero point, one bf16 scale and one integer zero point per
//    128 rows of K ("量化部署实战", 格式速查: W4A16 "+ 零点"; "LLM 推理优化 ·
//    量化学习笔记" 5.1: q = clamp(round(x / s) + z, ...)).
//  * FP8 KV-cache writes with one scale per (batch, head) ("量化部署实战",
//    KV Cache 量化: the per_head function), computed or given (calibrated).
//  * K per channel with a zero point plus V per token ("量化部署实战", KV
//    Cache 量化: K is a constant bias per channel plus a small variation; the
//    zero point absorbs the bias; the KIVI split quantizes K per channel and V
//    per token). The cache stays E4M3: per channel (b, h, d) over the tokens,
//    z = fl(0.5 * fl(max + min)), r = fl(x - z), s = max(max |r|, 1e-12) / 448,
//    code = E4M3(r / s); dequant = fl(fl(value * s) + z).
//  * SmoothQuant statistics and factors ("量化：让每一步搬更少的字节", 路线二:
//    s_j = max|X_j|^a / max|W_j|^(1-a), a = 0.5), and INT8 per-row
//    quantization (per token for activations, per output channel for weights
//    stored as B^T) after dividing or multiplying by those factors
//    ("量化部署实战", 格式速查: W8A8 INT8, -128..127, per channel + per token;
//    "量化：让每一步搬更少的字节", 量化在做什么: s = amax / 127).
// All of them are HBM-bound: 16-byte loads of 8 elements per thread, amax and
// min/max reductions in registers and shared memory, deterministic two-pass
// reductions through the caller's workspace (no atomics, no zeroed memory).
#include "qz_internal.cuh"
#include "qz_next.cuh"

#include <algorithm>

namespace qz {

namespace {

constexpr int kT = 256;                 // threads per CTA
constexpr int kW = kT / 32;

__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
qz_status launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...) == cudaSuccess ? QZ_OK : QZ_ERR_CUDA;
}

__device__ __forceinline__ float cta_max(float v, float* red) {
    v = warp_max(v, 32);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    __syncthreads();
    if (l == 0) red[w] = v;
    __syncthreads();
    float r = red[0];
#pragma unroll
    for (int i = 1; i < kW; i++) r = fmaxf(r, red[i]);
    return r;
}

// E4M3 codes of 8 quotients v / d.s (correctly rounded, the sign of an exact
// zero kept), saturating at +-448 like the clamp; 8 bytes.
__device__ __forceinline__ uint2 e4m3x8(const float v[8], const Recip& d) {
    float y[8];
#pragma unroll
    for (int j = 0; j < 8; j++) y[j] = sign_of(div1(v[j], d), v[j]);
    uint32_t p[4];
#pragma unroll
    for (int j = 0; j < 4; j++) p[j] = e4m3x2(y[2 * j], y[2 * j + 1]);
    return make_uint2(__byte_perm(p[0], p[1], 0x5410), __byte_perm(p[2], p[3], 0x5410));
}

// ------------------------------------------------------- INT4 zero point

// One CTA per (128 rows of K) x (64 columns) tile of w[K, N], staged in shared
// memory; per column the range [min(min, 0), max(max, 0)] gives
// s = bf16(max(hi - lo, 1e-12) / 15) and z = clamp(rint(-lo / s), 0, 15); each
// (k-octet, column) pair packs eight codes clamp(rint(w / s) + z, 0, 15).
template <typename T>
__global__ void __launch_bounds__(kT)
int4_zp_kernel(const T* __restrict__ w, int64_t K, int64_t N, int64_t ldw, int32_t* __restrict__ qweight,
               uint16_t* __restrict__ scale, uint8_t* __restrict__ zero, float* __restrict__ deq) {
    pdl_wait();                                   // the previous kernel on the stream has finished
    __shared__ float tile[128][65];
    __shared__ float plo[4][64], phi[4][64];
    __shared__ float sc[64], zf[64];
    const int64_t ncb = N / 64;
    const int64_t g = blockIdx.x / ncb, n0 = (blockIdx.x % ncb) * 64;
#pragma unroll
    for (int u = 0; u < 4; u++) {
        const int j = threadIdx.x + u * kT;
        const int r = j >> 3, c = (j & 7) * 8;
        float v[8];
        Load8<T>::run(w + (g * 128 + r) * ldw + n0 + c, v);
#pragma unroll
        for (int e = 0; e < 8; e++) tile[r][c + e] = v[e];
    }
    __syncthreads();
    {
        const int c = threadIdx.x & 63, p = threadIdx.x >> 6;
        float lo = 0.0f, hi = 0.0f;
        for (int r = p * 32; r < p * 32 + 32; r++) {
            lo = fminf(lo, tile[r][c]);
            hi = fmaxf(hi, tile[r][c]);
        }
        plo[p][c] = lo;
        phi[p][c] = hi;
    }
    __syncthreads();
    if (threadIdx.x < 64) {
        const int c = threadIdx.x;
        const float lo = fminf(fminf(plo[0][c], plo[1][c]), fminf(plo[2][c], plo[3][c]));
        const float hi = fmaxf(fmaxf(phi[0][c], phi[1][c]), fmaxf(phi[2][c], phi[3][c]));
        const float sf = div_rn(fmaxf(__fsub_rn(hi, lo), kAmaxMin), 15.0f);
        const uint16_t bits = __bfloat16_as_ushort(__float2bfloat16_rn(sf));
        const float s = bf16_bits_to_f32(bits);
        const float z = fminf(fmaxf(rintf(div_rn(-lo, s)), 0.0f), 15.0f);
        scale[g * N + n0 + c] = bits;
        zero[g * N + n0 + c] = (uint8_t)(int)z;
        sc[c] = s;
        zf[c] = z;
    }
    __syncthreads();
#pragma unroll
    for (int u = 0; u < 4; u++) {
        const int j = threadIdx.x + u * kT;              // 16 octets x 64 columns
        const int o = j >> 6, c = j & 63;
        const float s = sc[c], z = zf[c];
        uint32_t word = 0;
#pragma unroll
        for (int e = 0; e < 8; e++) {
            float q = __fadd_rn(rintf(div_rn(tile[o * 8 + e][c], s)), z);
            q = fminf(fmaxf(q, 0.0f), 15.0f);
            word |= (uint32_t)(int)q << (4 * e);
            if (deq) deq[(g * 128 + o * 8 + e) * N + n0 + c] = __fmul_rn(__fsub_rn(q, z), s);
        }
        qweight[(g * 16 + o) * N + n0 + c] = (int32_t)word;
    }
    pdl_trigger();                                // the next call may launch as this one drains
}

// ------------------------------------------------------ FP8 KV per head

// Kernel 1: partial[y * chunks + x] = max |.| over chunk x of slice y (slices
// are the B*H heads of K, then those of V; each T*D elements, contiguous).
__global__ void __launch_bounds__(kT)
kv_head_amax_kernel(const uint16_t* __restrict__ k, const uint16_t* __restrict__ v, int64_t BH, int64_t L,
                    int chunks, float* __restrict__ partial) {
    pdl_wait();                                   // the previous kernel on the stream has finished
    __shared__ float red[kW];
    const int64_t y = blockIdx.y;
    const uint16_t* x = (y < BH ? k + y * L : v + (y - BH) * L);
    const int64_t n8 = L / 8;
    const int64_t b = n8 * blockIdx.x / chunks, e = n8 * (blockIdx.x + 1) / chunks;
    float m = 0.0f;
    for (int64_t i0 = b + threadIdx.x; i0 < e; i0 += 4 * kT) {
        float val[4][8];
#pragma unroll
        for (int u = 0; u < 4; u++) {
            const int64_t i = i0 + (int64_t)u * kT;
            if (i < e) Load8<uint16_t>::run(x + i * 8, val[u]);
            else for (int j = 0; j < 8; j++) val[u][j] = 0.0f;
        }
#pragma unroll
        for (int u = 0; u < 4; u++)
#pragma unroll
            for (int j = 0; j < 8; j++) m = fmaxf(m, fabsf(val[u][j]));
    }
    m = cta_max(m, red);
    if (threadIdx.x == 0) partial[y * chunks + blockIdx.x] = m;
    pdl_trigger();
}

// Kernel 2: each CTA reduces its slice's partials (or reads the given scale),
// and encodes its chunk; chunk 0 stores the slice's scale.
template <bool GIVEN>
__global__ void __launch_bounds__(kT)
kv_head_encode_kernel(const uint16_t* __restrict__ k, const uint16_t* __restrict__ v, int64_t BH, int64_t L,
                      int chunks, const float* __restrict__ partial, float* __restrict__ ks,
                      float* __restrict__ vs, uint8_t* __restrict__ kc, uint8_t* __restrict__ vc) {
    pdl_wait();
    const int64_t y = blockIdx.y;
    const bool isk = y < BH;
    const int64_t h = isk ? y : y - BH;
    const uint16_t* x = (isk ? k : v) + h * L;
    uint8_t* codes = (isk ? kc : vc) + h * L;
    float* sp = (isk ? ks : vs) + h;
    float s;
    if (GIVEN) {
        s = __ldg(sp);
    } else {
        float m = 0.0f;
        for (int i = 0; i < chunks; i++) m = fmaxf(m, __ldg(partial + y * chunks + i));
        s = div1(fmaxf(m, kAmaxMin), Recip(kFp8Max));
        if (blockIdx.x == 0 && threadIdx.x == 0) *sp = s;
    }
    const Recip d(s);
    const int64_t n8 = L / 8;
    const int64_t b = n8 * blockIdx.x / chunks, e = n8 * (blockIdx.x + 1) / chunks;
    for (int64_t i = b + threadIdx.x; i < e; i += kT) {
        float val[8];
        Load8<uint16_t>::run(x + i * 8, val);
        reinterpret_cast<uint2*>(codes)[i] = e4m3x8(val, d);
    }
    pdl_trigger();                                // the next call may launch as this one drains
}

// ------------------------------------ K per channel with a zero point

// Launch 1, K part: per head y and token chunk x, the min and max of every
// channel d over the chunk's tokens: partial[((y * tc + x) * 2 + {0 min, 1 max}) * D + d].
// Thread layout: D/8 channel octets x (256 / (D/8)) token lanes.
__device__ __forceinline__ void kzp_stats(const uint16_t* __restrict__ k, int64_t T, int D, int tc, int64_t y, int cx,
                                          float* __restrict__ partial, float* smn, float* smx) {
    const int oc = D / 8, lanes = kT / oc;
    const int o = threadIdx.x % oc, tl = threadIdx.x / oc;
    const int64_t t0 = T * cx / tc, t1 = T * (cx + 1) / tc;
    const uint16_t* x = k + y * T * D;
    float mn[8], mx[8];
#pragma unroll
    for (int j = 0; j < 8; j++) { mn[j] = INFINITY; mx[j] = -INFINITY; }
    if (tl < lanes) {
        for (int64_t t = t0 + tl; t < t1; t += 4 * lanes) {     // four token rows in flight
            float val[4][8];
#pragma unroll
            for (int u = 0; u < 4; u++)
                if (t + u * lanes < t1) Load8<uint16_t>::run(x + (t + u * lanes) * D + o * 8, val[u]);
#pragma unroll
            for (int u = 0; u < 4; u++)
                if (t + u * lanes < t1)
#pragma unroll
                    for (int j = 0; j < 8; j++) { mn[j] = fminf(mn[j], val[u][j]); mx[j] = fmaxf(mx[j], val[u][j]); }
        }
    }
#pragma unroll
    for (int j = 0; j < 8; j++) {
        smn[threadIdx.x * 8 + j] = mn[j];
        smx[threadIdx.x * 8 + j] = mx[j];
    }
    __syncthreads();
    if (threadIdx.x < D) {
        const int d = threadIdx.x, od = d / 8, jd = d % 8;
        float a = INFINITY, b = -INFINITY;
        for (int l = 0; l < lanes; l++) {
            a = fminf(a, smn[(l * oc + od) * 8 + jd]);
            b = fmaxf(b, smx[(l * oc + od) * 8 + jd]);
        }
        float* p = partial + (y * tc + cx) * 2 * D;
        p[d] = a;
        p[D + d] = b;
    }
}

// Launch 2: every CTA (token chunk x, head y) first folds the head's chunk
// minima and maxima into each channel's zero point and scale (the CTAs of
// chunk 0 store them), then encodes its tokens: code = E4M3(fl(x - z) / s).
__global__ void __launch_bounds__(kT)
kzp_encode_kernel(const uint16_t* __restrict__ k, int64_t T, int D, int tc, const float* __restrict__ partial,
                  float* __restrict__ k_scale, float* __restrict__ k_zero, uint8_t* __restrict__ codes) {
    __shared__ float zs[256], ss[256], rs[256];
    pdl_wait();
    const int64_t y = blockIdx.y;
    if (threadIdx.x < D) {
        const int d = threadIdx.x;
        float a = INFINITY, b = -INFINITY;
        for (int c = 0; c < tc; c++) {
            const float* p = partial + (y * tc + c) * 2 * D;
            a = fminf(a, __ldcg(p + d));
            b = fmaxf(b, __ldcg(p + D + d));
        }
        const float z = __fmul_rn(0.5f, __fadd_rn(b, a));
        // fl(x - z) is monotone in x, so the largest |fl(x - z)| sits at an end of the range
        const float amax = fmaxf(__fsub_rn(b, z), __fsub_rn(z, a));
        const float sv = div1(fmaxf(amax, kAmaxMin), Recip(kFp8Max));
        if (blockIdx.x == 0) {
            k_zero[y * D + d] = z;
            k_scale[y * D + d] = sv;
        }
        zs[d] = z;
        ss[d] = sv;
        rs[d] = __frcp_rn(sv);
    }
    __syncthreads();
    const int oc = D / 8, lanes = kT / oc;
    const int o = threadIdx.x % oc, tl = threadIdx.x / oc;
    if (tl >= lanes) return;
    const int64_t t0 = T * blockIdx.x / tc, t1 = T * (blockIdx.x + 1) / tc;
    const uint16_t* x = k + y * T * D;
    uint8_t* cy = codes + y * T * D;
    for (int64_t t = t0 + tl; t < t1; t += 4 * lanes) {          // four token rows in flight
        float val[4][8];
#pragma unroll
        for (int u = 0; u < 4; u++)
            if (t + u * lanes < t1) Load8<uint16_t>::run(x + (t + u * lanes) * D + o * 8, val[u]);
#pragma unroll
        for (int u = 0; u < 4; u++) {
            if (t + u * lanes >= t1) break;
            float yq[8];
#pragma unroll
            for (int j = 0; j < 8; j++) {
                const int d = o * 8 + j;
                const float r = __fsub_rn(val[u][j], zs[d]);
                yq[j] = sign_of(div1(r, Recip(ss[d], rs[d])), r);
            }
            uint32_t p[4];
#pragma unroll
            for (int j = 0; j < 4; j++) p[j] = e4m3x2(yq[2 * j], yq[2 * j + 1]);
            *reinterpret_cast<uint2*>(cy + (t + u * lanes) * D + o * 8) =
                make_uint2(__byte_perm(p[0], p[1], 0x5410), __byte_perm(p[2], p[3], 0x5410));
        }
    }
}

// V per token in one pass: D/8 threads per token row each hold 8 values; the
// row's amax is a shuffle over those threads, then each encodes its 8 values.
// CTA vb of nvb takes a grid-stride share of the rows.
template <int TPR>
__device__ __forceinline__ void v_token(const uint16_t* __restrict__ v, int64_t rows, uint8_t* __restrict__ codes,
                                        float* __restrict__ scales, int64_t vb, int64_t nvb) {
    constexpr int D = TPR * 8;
    const int64_t tid = vb * kT + threadIdx.x;
    const int64_t nthreads = nvb * kT;
    const int sub = threadIdx.x % TPR;
    for (int64_t i = tid; i < ((rows * TPR + kT - 1) / kT) * kT; i += nthreads) {   // warp-uniform trip count
        const int64_t r = i / TPR;
        const bool live = r < rows;
        float val[8];
        if (live) Load8<uint16_t>::run(v + r * D + sub * 8, val);
        else for (int j = 0; j < 8; j++) val[j] = 0.0f;
        float m = 0.0f;
#pragma unroll
        for (int j = 0; j < 8; j++) m = fmaxf(m, fabsf(val[j]));
#pragma unroll
        for (int o = TPR / 2; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        const float s = div1(fmaxf(m, kAmaxMin), Recip(kFp8Max));
        if (live) {
            reinterpret_cast<uint2*>(codes + r * D)[sub] = e4m3x8(val, Recip(s));
            if (sub == 0) scales[r] = s;
        }
    }
}

// Launch 1: the first tc * BH CTAs take the K statistics (chunk x, head y), the
// remaining ones encode V per token; the two parts are independent.
template <int TPR>
__global__ void __launch_bounds__(kT)
kzp_stats_v_kernel(const uint16_t* __restrict__ k, const uint16_t* __restrict__ v, int64_t BH, int64_t T, int tc,
                   float* __restrict__ partial, uint8_t* __restrict__ vc, float* __restrict__ v_scale) {
    __shared__ float smn[kT * 8], smx[kT * 8];
    pdl_wait();
    const int64_t kblocks = BH * tc;
    if ((int64_t)blockIdx.x < kblocks)
        kzp_stats(k, T, TPR * 8, tc, (int64_t)blockIdx.x / tc, (int)((int64_t)blockIdx.x % tc), partial, smn, smx);
    else
        v_token<TPR>(v, BH * T, vc, v_scale, (int64_t)blockIdx.x - kblocks, (int64_t)gridDim.x - kblocks);
    pdl_trigger();
}

// ------------------------------------------------ SmoothQuant statistics

// partial[x * cols + c] = max |x[r, c]| over the rows of chunk x; then
// col_amax_final_kernel folds the chunks. Threads own 8 consecutive columns.
template <typename T>
__global__ void __launch_bounds__(kT)
col_amax_partial_kernel(const T* __restrict__ x, int64_t rows, int64_t cols, int chunks, float* __restrict__ partial) {
    pdl_wait();                                   // the previous kernel on the stream has finished
    const int64_t c8 = (int64_t)blockIdx.y * kT + threadIdx.x;          // column octet
    if (c8 * 8 >= cols) return;
    const int64_t r0 = rows * blockIdx.x / chunks, r1 = rows * (blockIdx.x + 1) / chunks;
    float m[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    for (int64_t r = r0; r < r1; r++) {
        float val[8];
        Load8<T>::run(x + r * cols + c8 * 8, val);
#pragma unroll
        for (int j = 0; j < 8; j++) m[j] = fmaxf(m[j], fabsf(val[j]));
    }
    float4* out = reinterpret_cast<float4*>(partial + (int64_t)blockIdx.x * cols + c8 * 8);
    out[0] = make_float4(m[0], m[1], m[2], m[3]);
    out[1] = make_float4(m[4], m[5], m[6], m[7]);
    pdl_trigger();
}

__global__ void __launch_bounds__(kT)
col_amax_final_kernel(const float* __restrict__ partial, int64_t cols, int chunks, float* __restrict__ out) {
    pdl_wait();
    const int64_t c = (int64_t)blockIdx.x * kT + threadIdx.x;
    if (c >= cols) return;
    float m = 0.0f;
    for (int i = 0; i < chunks; i++) m = fmaxf(m, __ldg(partial + (int64_t)i * cols + c));
    out[c] = m;
}

// s = fl(sqrt(max(ax, 1e-12))) / fl(sqrt(max(aw, 1e-12))), all IEEE-rounded.
__global__ void __launch_bounds__(kT)
smooth_factors_kernel(const float* __restrict__ xm, const float* __restrict__ wm, int64_t n, float* __restrict__ s) {
    pdl_wait();                                   // the previous kernel on the stream has finished
    const int64_t j = (int64_t)blockIdx.x * kT + threadIdx.x;
    if (j >= n) return;
    const float ax = fmaxf(__ldg(xm + j), kAmaxMin), aw = fmaxf(__ldg(wm + j), kAmaxMin);
    s[j] = __fdiv_rn(__fsqrt_rn(ax), __fsqrt_rn(aw));
}

// ------------------------------------------------------- INT8 per row

// Rows of up to 8192 columns: one CTA per row, the row read once into
// registers (VPT values per thread), x' = x / f or x * f (IEEE rounded), the
// row's amax reduced across the CTA, then q = clamp(rint(x' / s), -128, 127)
// with s = max(amax, 1e-12) / 127 encoded from the registers.
template <int OP>
__device__ __forceinline__ void smooth8(float v[8], const float* __restrict__ f, int64_t c) {
    if (OP == QZ_SMOOTH_NONE) return;
    const float4 a = __ldg(reinterpret_cast<const float4*>(f + c));
    const float4 b = __ldg(reinterpret_cast<const float4*>(f + c) + 1);
    const float fv[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int j = 0; j < 8; j++) v[j] = (OP == QZ_SMOOTH_DIVIDE) ? __fdiv_rn(v[j], fv[j]) : __fmul_rn(v[j], fv[j]);
}

__device__ __forceinline__ void int8_encode8(const float v[8], const Recip& d, float s, int8_t* codes, float* deq) {
    uint32_t w[2] = {0u, 0u};
    float o[8];
#pragma unroll
    for (int j = 0; j < 8; j++) {
        const float q = fminf(fmaxf(rintf(div1(v[j], d)), -128.0f), 127.0f);
        w[j >> 2] |= ((uint32_t)(int)q & 0xFFu) << (8 * (j & 3));
        o[j] = __fmul_rn(q, s);
    }
    *reinterpret_cast<uint2*>(codes) = make_uint2(w[0], w[1]);
    if (deq) {
        reinterpret_cast<float4*>(deq)[0] = make_float4(o[0], o[1], o[2], o[3]);
        reinterpret_cast<float4*>(deq)[1] = make_float4(o[4], o[5], o[6], o[7]);
    }
}

template <typename T, int OP, int CPT>                // CPT: 8-element chunks per thread
__global__ void __launch_bounds__(kT)
int8_row_cta_kernel(const T* __restrict__ x, int64_t cols, const float* __restrict__ f,
                    int8_t* __restrict__ codes, float* __restrict__ scales, float* __restrict__ deq) {
    pdl_wait();                                   // the previous kernel on the stream has finished
    __shared__ float red[kW];
    const int64_t r = blockIdx.x;
    const T* xr = x + r * cols;
    float v[CPT][8];
#pragma unroll
    for (int u = 0; u < CPT; u++) {
        const int64_t c = ((int64_t)u * kT + threadIdx.x) * 8;
        if (c < cols) Load8<T>::run(xr + c, v[u]);
    }
    float m = 0.0f;
#pragma unroll
    for (int u = 0; u < CPT; u++) {
        const int64_t c = ((int64_t)u * kT + threadIdx.x) * 8;
        if (c < cols) {
            smooth8<OP>(v[u], f, c);
#pragma unroll
            for (int j = 0; j < 8; j++) m = fmaxf(m, fabsf(v[u][j]));
        }
    }
    const float s = div1(fmaxf(cta_max(m, red), kAmaxMin), Recip(127.0f));
    if (threadIdx.x == 0) scales[r] = s;
    const Recip d(s);
#pragma unroll
    for (int u = 0; u < CPT; u++) {
        const int64_t c = ((int64_t)u * kT + threadIdx.x) * 8;
        if (c < cols) int8_encode8(v[u], d, s, codes + r * cols + c, deq ? deq + r * cols + c : nullptr);
    }
    pdl_trigger();                                // the next call may launch as this one drains
}

// Wider rows: one warp per row, two passes (the second re-reads the row).
template <typename T, int OP>
__global__ void __launch_bounds__(kT)
int8_rows_kernel(const T* __restrict__ x, int64_t rows, int64_t cols, const float* __restrict__ f,
                 int8_t* __restrict__ codes, float* __restrict__ scales, float* __restrict__ deq) {
    pdl_wait();                                   // the previous kernel on the stream has finished
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * kT + threadIdx.x) >> 5;
    const int64_t nwarps = (int64_t)gridDim.x * kW;
    for (int64_t r = warp; r < rows; r += nwarps) {
        const T* xr = x + r * cols;
        float m = 0.0f;
        for (int64_t c = lane * 8; c < cols; c += 256) {
            float v[8];
            Load8<T>::run(xr + c, v);
            smooth8<OP>(v, f, c);
#pragma unroll
            for (int j = 0; j < 8; j++) m = fmaxf(m, fabsf(v[j]));
        }
        const float s = div1(fmaxf(warp_max(m, 32), kAmaxMin), Recip(127.0f));
        if (lane == 0) scales[r] = s;
        const Recip d(s);
        for (int64_t c = lane * 8; c < cols; c += 256) {
            float v[8];
            Load8<T>::run(xr + c, v);
            smooth8<OP>(v, f, c);
            int8_encode8(v, d, s, codes + r * cols + c, deq ? deq + r * cols + c : nullptr);
        }
    }
    pdl_trigger();                                // the next call may launch as this one drains
}

int kv_head_chunks(int64_t BH, int64_t L) {
    // about four CTAs per SM over both tensors, at least 4096 elements per CTA
    const int64_t want = std::max<int64_t>(1, (int64_t)num_sms() * 4 / std::max<int64_t>(1, 2 * BH));
    return (int)std::max<int64_t>(1, std::min<int64_t>(want, std::max<int64_t>(1, L / 4096)));
}

int kzp_chunks(int64_t BH, int64_t T) {
    const int64_t want = std::max<int64_t>(1, (int64_t)num_sms() * 2 / std::max<int64_t>(1, BH));
    return (int)std::max<int64_t>(1, std::min<int64_t>({want, (T + 15) / 16, (int64_t)64}));
}

int col_chunks(int64_t rows) { return (int)std::max<int64_t>(1, std::min<int64_t>(64, rows / 16)); }

} // namespace

// ------------------------------------------------------------------ host

size_t ws_kv_per_head(int64_t BH, int64_t L) { return (size_t)2 * BH * kv_head_chunks(BH, L) * sizeof(float); }
size_t ws_kv_channel_zp(int64_t BH, int64_t T, int64_t D) {
    return (size_t)BH * kzp_chunks(BH, T) * 2 * D * sizeof(float);
}
size_t ws_col_amax(int64_t rows, int64_t cols) { return (size_t)col_chunks(rows) * cols * sizeof(float); }

qz_status int4_zp_launch(const void* w, qz_dtype wt, int64_t K, int64_t N, int64_t ldw, int32_t* qweight,
                         uint16_t* scale, uint8_t* zero, float* deq, cudaStream_t st) {
    const int64_t nblocks = (K / 128) * (N / 64);
    if (wt == QZ_F32)
        QZ_TRY(launch_pdl(int4_zp_kernel<float>, dim3((unsigned)nblocks), dim3(kT), st, (const float*)w, K, N, ldw,
                          qweight, scale, zero, deq));
    else
        QZ_TRY(launch_pdl(int4_zp_kernel<uint16_t>, dim3((unsigned)nblocks), dim3(kT), st, (const uint16_t*)w, K, N, ldw,
                          qweight, scale, zero, deq));
    return launch_status();
}

qz_status kv_per_head_launch(const uint16_t* k, const uint16_t* v, int64_t BH, int64_t L, uint8_t* kc, uint8_t* vc,
                             float* ks, float* vs, qz_scale_mode mode, void* ws, cudaStream_t st) {
    const int chunks = kv_head_chunks(BH, L);
    const dim3 grid(chunks, (unsigned)(2 * BH));
    if (mode == QZ_SCALE_GIVEN) {
        QZ_TRY(launch_pdl(kv_head_encode_kernel<true>, grid, dim3(kT), st, k, v, BH, L, chunks, (const float*)nullptr,
                          ks, vs, kc, vc));
        return launch_status();
    }
    float* partial = (float*)ws;
    QZ_TRY(launch_pdl(kv_head_amax_kernel, grid, dim3(kT), st, k, v, BH, L, chunks, partial));
    QZ_TRY(launch_pdl(kv_head_encode_kernel<false>, grid, dim3(kT), st, k, v, BH, L, chunks, (const float*)partial,
                      ks, vs, kc, vc));
    return launch_status();
}

qz_status kv_channel_zp_launch(const uint16_t* k, const uint16_t* v, int64_t B, int64_t H, int64_t T, int64_t D,
                               uint8_t* kc, uint8_t* vc, float* k_scale, float* k_zero, float* v_scale, void* ws,
                               cudaStream_t st) {
    const int64_t BH = B * H;
    const int tc = kzp_chunks(BH, T);
    float* partial = (float*)ws;
    // one launch for K's statistics and V per token, one for K's scales and codes
    const int64_t vrows = BH * T;
    const int tpr = (int)(D / 8);
    const int64_t vblocks = std::max<int64_t>(1, std::min<int64_t>((vrows * tpr + kT - 1) / kT, (int64_t)num_sms() * 2));
    const dim3 g1((unsigned)(BH * tc + vblocks));
    qz_status s1;
    switch (tpr) {
    case 1: s1 = launch_pdl(kzp_stats_v_kernel<1>, g1, dim3(kT), st, k, v, BH, T, tc, partial, vc, v_scale); break;
    case 2: s1 = launch_pdl(kzp_stats_v_kernel<2>, g1, dim3(kT), st, k, v, BH, T, tc, partial, vc, v_scale); break;
    case 4: s1 = launch_pdl(kzp_stats_v_kernel<4>, g1, dim3(kT), st, k, v, BH, T, tc, partial, vc, v_scale); break;
    case 8: s1 = launch_pdl(kzp_stats_v_kernel<8>, g1, dim3(kT), st, k, v, BH, T, tc, partial, vc, v_scale); break;
    case 16: s1 = launch_pdl(kzp_stats_v_kernel<16>, g1, dim3(kT), st, k, v, BH, T, tc, partial, vc, v_scale); break;
    default: s1 = launch_pdl(kzp_stats_v_kernel<32>, g1, dim3(kT), st, k, v, BH, T, tc, partial, vc, v_scale); break;
    }
    QZ_TRY(s1);
    QZ_TRY(launch_pdl(kzp_encode_kernel, dim3(tc, (unsigned)BH), dim3(kT), st, k, T, (int)D, tc,
                      (const float*)partial, k_scale, k_zero, kc));
    return launch_status();
}

qz_status col_amax_launch(const void* x, qz_dtype xt, int64_t rows, int64_t cols, float* out, void* ws,
                          cudaStream_t st) {
    const int chunks = col_chunks(rows);
    const dim3 grid(chunks, (unsigned)((cols / 8 + kT - 1) / kT));
    float* partial = (float*)ws;
    if (xt == QZ_F32)
        QZ_TRY(launch_pdl(col_amax_partial_kernel<float>, grid, dim3(kT), st, (const float*)x, rows, cols, chunks, partial));
    else
        QZ_TRY(launch_pdl(col_amax_partial_kernel<uint16_t>, grid, dim3(kT), st, (const uint16_t*)x, rows, cols, chunks,
                          partial));
    QZ_TRY(launch_pdl(col_amax_final_kernel, dim3((unsigned)((cols + kT - 1) / kT)), dim3(kT), st,
                      (const float*)partial, cols, chunks, out));
    return launch_status();
}

qz_status smooth_factors_launch(const float* xm, const float* wm, int64_t n, float* s, cudaStream_t st) {
    QZ_TRY(launch_pdl(smooth_factors_kernel, dim3((unsigned)((n + kT - 1) / kT)), dim3(kT), st, xm, wm, n, s));
    return launch_status();
}

template <typename T, int OP>
qz_status launch_i8(const void* x, int64_t rows, int64_t cols, const float* f, int8_t* codes, float* scales,
                    float* deq, cudaStream_t st) {
    const int64_t cpt = (cols / 8 + kT - 1) / kT;               // chunks per thread, one CTA per row
    switch (cpt) {
    case 1: QZ_TRY(launch_pdl(int8_row_cta_kernel<T, OP, 1>, dim3((unsigned)rows), dim3(kT), st, (const T*)x, cols, f, codes, scales, deq)); break;
    case 2: QZ_TRY(launch_pdl(int8_row_cta_kernel<T, OP, 2>, dim3((unsigned)rows), dim3(kT), st, (const T*)x, cols, f, codes, scales, deq)); break;
    case 3: QZ_TRY(launch_pdl(int8_row_cta_kernel<T, OP, 3>, dim3((unsigned)rows), dim3(kT), st, (const T*)x, cols, f, codes, scales, deq)); break;
    case 4: QZ_TRY(launch_pdl(int8_row_cta_kernel<T, OP, 4>, dim3((unsigned)rows), dim3(kT), st, (const T*)x, cols, f, codes, scales, deq)); break;
    default: {
        const int grid = (int)std::max<int64_t>(1, std::min<int64_t>((rows + kW - 1) / kW, (int64_t)num_sms() * 8));
        QZ_TRY(launch_pdl(int8_rows_kernel<T, OP>, dim3(grid), dim3(kT), st, (const T*)x, rows, cols, f, codes, scales, deq));
    }
    }
    return launch_status();
}

qz_status int8_rows_launch(const void* x, qz_dtype xt, int64_t rows, int64_t cols, const float* f, int op,
                           int8_t* codes, float* scales, float* deq, cudaStream_t st) {
    if (rows > 0x7FFFFFFF) return QZ_ERR_SHAPE;
    if (xt == QZ_F32) {
        if (op == QZ_SMOOTH_NONE) return launch_i8<float, QZ_SMOOTH_NONE>(x, rows, cols, f, codes, scales, deq, st);
        if (op == QZ_SMOOTH_DIVIDE) return launch_i8<float, QZ_SMOOTH_DIVIDE>(x, rows, cols, f, codes, scales, deq, st);
        return launch_i8<float, QZ_SMOOTH_MULTIPLY>(x, rows, cols, f, codes, scales, deq, st);
    }
    if (op == QZ_SMOOTH_NONE) return launch_i8<uint16_t, QZ_SMOOTH_NONE>(x, rows, cols, f, codes, scales, deq, st);
    if (op == QZ_SMOOTH_DIVIDE) return launch_i8<uint16_t, QZ_SMOOTH_DIVIDE>(x, rows, cols, f, codes, scales, deq, st);
    return launch_i8<uint16_t, QZ_SMOOTH_MULTIPLY>(x, rows, cols, f, codes, scales, deq, st);
}

} // namespace qz
