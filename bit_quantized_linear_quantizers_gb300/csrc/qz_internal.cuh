// qz_internal.cuh -- device codecs and host helpers shared by the libqz kernels.
//
// Number formats ("量化部署实战", 格式速查; "量化：让每一步搬更少的字节",
// 新一代低位格式):
//   E4M3 (fn): 1 sign, 4 exponent (bias 7), 3 mantissa bits, max 448, no inf.
//   E2M1: 1 sign, 2 exponent, 1 mantissa bit: +-{0, .5, 1, 1.5, 2, 3, 4, 6}.
//   E8M0: an 8-bit biased exponent (bias 127), a pure power of two.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>

#include "../../include/qz.h"

namespace qz {

// The clamp floor of the fake-quant functions: the fp32 value nearest 1e-12.
// Return the status of `expr` from the calling function unless it is QZ_OK.
#define QZ_TRY(expr)                                   \
    do {                                               \
        const qz_status _s = (expr);                   \
        if (_s != QZ_OK) return _s;                    \
    } while (0)

constexpr float kAmaxMin = 1e-12f;
constexpr float kFp8Max = 448.0f;
constexpr float kFp4Max = 6.0f;

// ---------------------------------------------------------------- device

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b16) {
    return __uint_as_float(b16 << 16);
}

// Widen eight consecutive input elements (fp32 or bf16) to fp32.
template <typename T> struct Load8;
template <> struct Load8<float> {
    static __device__ __forceinline__ void run(const float* p, float v[8]) {
        float4 a = __ldg(reinterpret_cast<const float4*>(p));
        float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
};
template <> struct Load8<uint16_t> {
    static __device__ __forceinline__ void run(const uint16_t* p, float v[8]) {
        uint4 a = __ldg(reinterpret_cast<const uint4*>(p));
        uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int i = 0; i < 4; i++) {
            v[2 * i] = __uint_as_float(w[i] << 16);
            v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    }
};

__device__ __forceinline__ float load1(const float* p) { return __ldg(p); }
__device__ __forceinline__ float load1(const uint16_t* p) { return bf16_bits_to_f32(__ldg(p)); }

// x / s rounded once (IEEE round to nearest even): the codes depend on it.
__device__ __forceinline__ float div_rn(float x, float s) { return __fdiv_rn(x, s); }

// Correctly rounded quotients x / s for a whole scale unit, from r = RN(1/s):
// q0 = RN(x * r) is within one ulp of x / s, the remainder x - q0 * s is then
// exact (one fma), and the correction RN(q0 + rem * r) is the correctly
// rounded quotient (Markstein's theorem: P. Markstein, "Computation of
// elementary functions on the IBM RISC System/6000 processor", IBM J. Res.
// Dev. 34(1), 1990). The preconditions hold whenever the quotient can map to a
// non-zero code: the scales are >= 1e-12 / 2688 and the quotient and the
// remainder stay normal. An exactly zero x comes back as +0; callers that
// keep the sign of zero restore it (sign_of).
struct Recip {
    float s, r;
    __device__ __forceinline__ explicit Recip(float s_) {
        s = s_;
        r = __frcp_rn(s_);                     // correctly rounded reciprocal
    }
    __device__ __forceinline__ Recip(float s_, float r_) : s(s_), r(r_) {}   // r_ == RN(1 / s_)
};

// One correctly rounded quotient x / d.s (Markstein's correction step), x >= 0.
__device__ __forceinline__ float div1(float x, const Recip& d) {
    const float q0 = __fmul_rn(x, d.r);
    const float rem = __fmaf_rn(-q0, d.s, x);
    return __fmaf_rn(rem, d.r, q0);
}

// Two quotients at once with the paired fp32 instructions of sm_100+ (each
// lane rounds exactly as the scalar mul / fma): the same three steps as div1,
// the negation moved onto the scale (fma(q0, -s, x) == fma(-q0, s, x)).
__device__ __forceinline__ void div1x2(float a, float b, const Recip& d, float& qa, float& qb) {
    asm("{ .reg .b64 x, r2, ns2, q0, rem, q;\n\t"
        "mov.b64 x, {%2, %3};\n\t"
        "mov.b64 r2, {%4, %4};\n\t"
        "mov.b64 ns2, {%5, %5};\n\t"
        "mul.rn.f32x2 q0, x, r2;\n\t"
        "fma.rn.f32x2 rem, q0, ns2, x;\n\t"
        "fma.rn.f32x2 q, rem, r2, q0;\n\t"
        "mov.b64 {%0, %1}, q; }"
        : "=f"(qa), "=f"(qb) : "f"(a), "f"(b), "f"(d.r), "f"(-d.s));
}

// y with the sign bit of x (a non-zero quotient already has it; fixes -0).
__device__ __forceinline__ float sign_of(float y, float x) {
    return __uint_as_float(__float_as_uint(y) | (__float_as_uint(x) & 0x80000000u));
}

// Eight E2M1 codes (element j in bits 4j..4j+3) of quotients y[8], by the
// hardware conversion: round to nearest even, saturating at 6. The four code
// bytes are assembled inside one asm block (no widening or byte shuffles).
__device__ __forceinline__ uint32_t e2m1x8_rne(const float y[8]) {
    uint32_t w;
    asm("{ .reg .b8 a, b, c, d;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 a, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 c, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 d, %8, %7;\n\t"
        "mov.b32 %0, {a, b, c, d}; }"
        : "=r"(w)
        : "f"(y[0]), "f"(y[1]), "f"(y[2]), "f"(y[3]), "f"(y[4]), "f"(y[5]), "f"(y[6]), "f"(y[7]));
    return w;
}

// The pages' rule (first index of the minimum distance: ties go to the smaller
// magnitude) differs from round to nearest even only at exact midpoints, and
// only where round-to-even goes up: 0.75, 1.75 and 3.5 (0.25, 1.25, 2.5 and 5
// already round down to an even code); its sign bit is (y < 0), so an exact
// -0.0 encodes as +0. Both corrections come from a second round-to-nearest-even
// conversion, of p = pred(y) = RN(y - y * 2^-24) (one fma: the exact difference
// lies more than half an ulp below y and less than one, or exactly on pred(y)
// for a power of two; pred(-0) is +0). The two codes differ only beside a
// midpoint m: at y == m where round-to-even went up (the even code is wrong and
// p rounds down), and at y == succ(m) where round-to-even of m goes down (p == m
// rounds down wrongly and the odd code is right). Adjacent codes alternate in
// parity, so the odd code of a differing pair is the right one, and elsewhere
// the codes agree. Element j lands in bits 4j..4j+3.
__device__ __forceinline__ uint32_t e2m1x8_tiesdown(const float y[8]) {
    float p[8];
#pragma unroll
    for (int j = 0; j < 8; j += 2)                               // pred of two quotients per paired fma
        asm("{ .reg .b64 y2, c2, p2;\n\t"
            "mov.b64 y2, {%2, %3};\n\t"
            "mov.b64 c2, {%4, %4};\n\t"
            "fma.rn.f32x2 p2, y2, c2, y2;\n\t"
            "mov.b64 {%0, %1}, p2; }"
            : "=f"(p[j]), "=f"(p[j + 1]) : "f"(y[j]), "f"(y[j + 1]), "f"(-0x1.0p-24f));
    const uint32_t w1 = e2m1x8_rne(y), w2 = e2m1x8_rne(p);
    const uint32_t odd = (w1 & 0x11111111u) * 15u;               // nibbles of w1 with an odd code, all ones
    return w2 ^ ((w1 ^ w2) & odd);
}

// Two fp32 -> two E4M3 bytes, round to nearest even, saturating to +-448
// (the hardware conversion). Returns lo | hi << 8.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Value of one E4M3 byte as fp32 (exact; via the hardware E4M3 -> f16 conversion).
__device__ __forceinline__ float e4m3_value(uint32_t code) {
    uint32_t h2;
    uint16_t in = (uint16_t)(code & 0xFF);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
    return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFF)));
}

// E4M3 code of one fp32 (saturating at +-448).
__device__ __forceinline__ uint32_t e4m3_code(float y) { return e4m3x2(y, 0.0f) & 0xFF; }

// Value of a 4-bit E2M1 code (sign bit 3) as fp32; code 8 gives -0.0.
__device__ __forceinline__ float e2m1_value(uint32_t c) {
    uint32_t m = c & 7u, e = m >> 1, f = m & 1u;
    float v = (m < 2u) ? 0.5f * (float)f : __uint_as_float(((e + 126u) << 23) | (f << 22));
    return (c & 8u) ? -v : v;
}

// Encode one 16-element block to E2M1 with scale d.s (correctly rounded
// quotients, ties to the smaller magnitude); returns the 16 nibbles (element j
// at bit 4j of word j / 8); writes the dequantized block if asked.
__device__ __forceinline__ uint2 fp4_encode16(const float v[16], const Recip& d, float* deq) {
    float y[16];
#pragma unroll
    for (int j = 0; j < 16; j += 2) div1x2(v[j], v[j + 1], d, y[j], y[j + 1]);
    const uint2 packed = make_uint2(e2m1x8_tiesdown(y), e2m1x8_tiesdown(y + 8));
    if (deq) {
        float o[16];
#pragma unroll
        for (int j = 0; j < 16; j++) o[j] = __fmul_rn(e2m1_value((j < 8 ? packed.x : packed.y) >> (4 * (j & 7))), d.s);
#pragma unroll
        for (int q = 0; q < 4; q++) reinterpret_cast<float4*>(deq)[q] = make_float4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
    }
    return packed;
}

// NVFP4 block of 16 values with tensor scale g (dg = Recip(g), d6 = Recip(6)):
// the block scale code E4M3(amax16 / 6 / g) and the 16 E2M1 codes of v / s with
// s = max(E4M3 value, 1e-12) * g (element j at bit 4j of word j / 8).
__device__ __forceinline__ uint2 nvfp4_block16(const float v[16], float g, const Recip& dg, const Recip& d6,
                                               uint32_t& bcode) {
    float m = 0.0f;
#pragma unroll
    for (int j = 0; j < 16; j++) m = fmaxf(m, fabsf(v[j]));
    bcode = e4m3_code(div1(div1(m, d6), dg));
    const float sv = __fmul_rn(fmaxf(e4m3_value(bcode), kAmaxMin), g);
    return fp4_encode16(v, Recip(sv), nullptr);
}

// MXFP4: the E2M1 codes of 8 values of one 32-element block whose scale is
// 2^(E-2), given inv = 2^(2-E) (element j at bit 4j). y = RN(x * 2^(2-E) + 0):
// the power-of-two scaling, -0 -> +0 except where a negative product underflows
// to -0 (the tie rule below maps that to +0 as well); two lanes per paired fma.
// BF16IN (every x has at most 8 significant bits): y keeps x's 8 significant
// bits, so no y lies strictly between a midpoint and the fp32 value one ulp
// above it. Stepping every non-zero y one fp32 ulp toward zero therefore moves
// exact midpoints just below themselves (ties go down, the pages' rule) and
// changes no other code; the hardware's round-to-nearest-even then gives the
// exact codes. The step is RZ(y * (1 - 2^-24) + 0): the exact product lies less
// than one ulp below |y| (exactly one below a power of two, and for
// subnormals), so rounding toward zero lands on the neighbour toward zero; a
// zero of either sign becomes +0 (an exact -0 + +0 in RZ). Other inputs take
// the ties-down encoder.
template <bool BF16IN>
__device__ __forceinline__ uint32_t mxfp4_encode8(const float v[8], float inv) {
    float y[8];
#pragma unroll
    for (int j = 0; j < 8; j += 2)
        asm("{ .reg .b64 x2, s2, z2, r2;\n\t"
            "mov.b64 x2, {%2, %3}; mov.b64 s2, {%4, %4}; mov.b64 z2, {%5, %5};\n\t"
            "fma.rn.f32x2 r2, x2, s2, z2;\n\t"
            "mov.b64 {%0, %1}, r2; }"
            : "=f"(y[j]), "=f"(y[j + 1]) : "f"(v[j]), "f"(v[j + 1]), "f"(inv), "f"(0.0f));
    if constexpr (BF16IN) {
        float yd[8];
#pragma unroll
        for (int j = 0; j < 8; j += 2)
            asm("{ .reg .b64 y2, c2, z2, r2;\n\t"
                "mov.b64 y2, {%2, %3}; mov.b64 c2, {%4, %4}; mov.b64 z2, {%5, %5};\n\t"
                "fma.rz.f32x2 r2, y2, c2, z2;\n\t"
                "mov.b64 {%0, %1}, r2; }"
                : "=f"(yd[j]), "=f"(yd[j + 1]) : "f"(y[j]), "f"(y[j + 1]), "f"(0x1.fffffep-1f), "f"(0.0f));
        return e2m1x8_rne(yd);
    } else {
        return e2m1x8_tiesdown(y);
    }
}

__device__ __forceinline__ float warp_max(float v, int width) {
    for (int o = width / 2; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// ------------------------------------------------------------------ host

int num_sms();                         // SM count of the current device (cached)
qz_status launch_status();             // cudaGetLastError -> qz_status
bool is_aligned(const void* p, size_t a);
qz_status opt_in_smem(const void* fn, int bytes);   // thread-safe dynamic shared-memory opt-in

// Stream order of INT4 weights. The W4A16 kernels start under programmatic
// dependent launch: each lets the next kernel on the stream launch at its entry,
// and reads its weights (not its activations) before griddepcontrol.wait. An
// INT4 quantizer call lets its successor start only after its own wait, so its
// outputs can still be in flight when a W4A16 kernel starts only if that kernel
// follows it directly or through other W4A16 launches. Per device and stream,
// the library keeps the byte ranges of the last INT4 quantizer call; a W4A16
// call whose weights overlap them launches after all earlier work on the stream
// and then clears the record. Other launches only complete earlier work, so
// they leave the record as it is (at worst one later call waits needlessly).
struct Span {
    const void* p;
    size_t bytes;
};
struct Int4Writes {
    uint64_t gen;                      // changes with every noted call
    int n;                             // 0: nothing in flight
    Span s[3];
};
void note_int4_writes(cudaStream_t st, const Span* w, int n);   // n <= 3
Int4Writes int4_writes(cudaStream_t st);                         // current device
void clear_int4_writes(cudaStream_t st, uint64_t gen);           // unless noted again since gen

inline bool spans_overlap(const Span& a, const Span& b) {
    const uintptr_t a0 = (uintptr_t)a.p, b0 = (uintptr_t)b.p;
    return a.bytes && b.bytes && a0 < b0 + b.bytes && b0 < a0 + a.bytes;
}

// Does one W4A16 problem read (qweight int32 [K/8, N], scale bf16 [K/128, N],
// zero uint8 [K/128, N] or none) overlap the recorded ranges?
inline bool w4a16_reads_in_flight(const Int4Writes& rec, const void* qweight, const void* scale,
                                  const void* zero, int N, int K) {
    const size_t kn = (size_t)K * (size_t)N;
    const Span r[3] = {{qweight, kn / 2}, {scale, kn / 64}, {zero, zero ? kn / 128 : 0}};
    for (int i = 0; i < rec.n; i++)
        for (const Span& x : r)
            if (spans_overlap(rec.s[i], x)) return true;
    return false;
}

} // namespace qz

// Internal launchers (quantize.cu).
namespace qz {
size_t ws_quantize_fp8_tensor(int64_t rows, int64_t cols);
size_t ws_quantize_nvfp4(int64_t rows, int64_t cols);
size_t ws_quantize_nvfp4_grouped(int count);
constexpr int kNvfp4GroupMax = 256;
qz_status quantize_nvfp4_grouped_launch(const qz_nvfp4_tensor* tensors, int count, qz_dtype xt, void* ws,
                                        cudaStream_t st);
size_t ws_kv_write(int64_t n);

qz_status quantize_fp8_launch(const void* x, qz_dtype xt, int64_t rows, int64_t cols, int64_t ldx,
                              qz_fp8_gran gran, uint8_t* codes, float* scales, float* deq,
                              void* ws, size_t ws_bytes, cudaStream_t st);
qz_status quantize_mxfp4_launch(const void* x, qz_dtype xt, int64_t rows, int64_t cols, int64_t ldx,
                                uint8_t* codes, uint8_t* e8m0, float* deq, cudaStream_t st);
qz_status quantize_nvfp4_launch(const void* x, qz_dtype xt, int64_t rows, int64_t cols, int64_t ldx,
                                uint8_t* codes, uint8_t* sb, float* g, const float* amax_in,
                                float* deq, void* ws, size_t ws_bytes, cudaStream_t st);
qz_status quantize_int4_launch(const void* w, qz_dtype wt, int64_t K, int64_t N, int64_t ldw,
                               int32_t* qweight, uint16_t* scale, float* deq, cudaStream_t st);
qz_status kv_write_launch(const uint16_t* k, const uint16_t* v, int64_t n, uint8_t* kc, uint8_t* vc,
                          float* ks, float* vs, qz_scale_mode mode, void* ws, size_t ws_bytes,
                          cudaStream_t st);
} // namespace qz
