"""GPU parity of the NVFP4 and MXFP4 GEMMs (tcgen05 block-scaled FP4) against the
oracle's FP64 reference: |y_gpu - y_ref| <= 1e-3 * sum_k |a_ik * b_kj| plus half
a bf16 ulp of y_ref (the rounding of the bf16 output), on the exactly dequantized
operands (E2M1 x block scale (x tensor scale)). Operands come
from the oracle's quantizers; integer cases with unit scales must be exact."""
import numpy as np
import pytest
import torch

import oracle
import synthetic as syn
from gpu_util import assert_same_bytes, bf16_bits_to_f64, check_gemm, host

pytestmark = pytest.mark.gpu

REL = 1e-3


@pytest.fixture(scope="module")
def qz():
    import bit_quantized_linear_quantizers_gb300 as q
    return q


def dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def check(y_bits, y_ref, bound, what):
    check_gemm(y_bits, y_ref, bound, what, REL)


def inputs(M, N, K, seed):
    rng = np.random.default_rng(seed)
    a = rng.standard_normal((M, K)).astype(np.float32)
    a[:, rng.choice(K, max(1, K // 200), replace=False)] *= np.float32(30)
    bt = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    return syn.to_bf16_bits(a), syn.to_bf16_bits(bt)


def nv_run(qz, a, bt):
    ca, sa, ga, _ = oracle.quant_nvfp4(a, want_deq=False)
    cb, sb, gb, _ = oracle.quant_nvfp4(bt, want_deq=False)
    y = host(qz.qz_gemm_nvfp4(dev(ca), dev(sa), dev(np.float32([ga])), dev(cb), dev(sb), dev(np.float32([gb]))))
    return y, (ca, sa, ga, cb, sb, gb)


def mx_run(qz, a, bt):
    ca, ea, _ = oracle.quant_mxfp4(a, want_deq=False)
    cb, eb, _ = oracle.quant_mxfp4(bt, want_deq=False)
    y = host(qz.qz_gemm_mxfp4(dev(ca), dev(ea), dev(cb), dev(eb)))
    return y, (ca, ea, cb, eb)


def pack(codes):
    return (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)


@pytest.mark.parametrize("M", [128, 256, 640])
@pytest.mark.parametrize("fmt", ["nv", "mx"])
def test_fp4_gemm_integer_exact(qz, fmt, M):
    """Unit scales and E2M1 codes of small integers: an exact integer matmul, over one and
    several 128-row tiles."""
    rng = np.random.default_rng(1 + M)
    N, K = 256, 256
    mag = np.array([0, 2, 4, 5, 6, 7])                    # 0, 1, 2, 3, 4, 6
    ca = (rng.choice(mag, (M, K)) | (rng.integers(0, 2, (M, K)) << 3)).astype(np.uint8)
    cb = (rng.choice(mag, (N, K)) | (rng.integers(0, 2, (N, K)) << 3)).astype(np.uint8)
    va = np.vectorize(oracle.e2m1_decode)(ca)
    vb = np.vectorize(oracle.e2m1_decode)(cb)
    ref = (va @ vb.T).astype(np.float32)
    if fmt == "nv":
        one = 0x38
        y = host(qz.qz_gemm_nvfp4(dev(pack(ca)), dev(np.full((M, K // 16), one, np.uint8)),
                                  dev(np.float32([1.0])), dev(pack(cb)), dev(np.full((N, K // 16), one, np.uint8)),
                                  dev(np.float32([1.0]))))
    else:
        y = host(qz.qz_gemm_mxfp4(dev(pack(ca)), dev(np.full((M, K // 32), 127, np.uint8)),
                                  dev(pack(cb)), dev(np.full((N, K // 32), 127, np.uint8))))
    assert np.array_equal(bf16_bits_to_f64(y), bf16_bits_to_f64(syn.to_bf16_bits(ref)))


@pytest.mark.parametrize("M,N,K", [(128, 256, 256), (128, 256, 1024), (256, 512, 512), (384, 768, 256),
                                   (256, 256, 256), (640, 256, 512), (1152, 1024, 768)])
def test_nvfp4_gemm(qz, M, N, K):
    a, bt = inputs(M, N, K, seed=M + N + K)
    y, ops = nv_run(qz, a, bt)
    y_ref, bound = oracle.gemm_nvfp4(*ops)
    check(y, y_ref, bound, f"nvfp4 {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(128, 256, 256), (128, 256, 1024), (256, 512, 512), (384, 768, 256),
                                   (256, 256, 256), (640, 256, 512), (1152, 1024, 768)])
def test_mxfp4_gemm(qz, M, N, K):
    a, bt = inputs(M, N, K, seed=M + N + K + 1)
    y, ops = mx_run(qz, a, bt)
    y_ref, bound = oracle.gemm_mxfp4(*ops)
    check(y, y_ref, bound, f"mxfp4 {M}x{N}x{K}")


def test_fp4_gemm_scales_per_block(qz):
    """Distinct scales per (row, block) on both operands: a scale read from the wrong
    block or row shows up as a large error."""
    rng = np.random.default_rng(9)
    M, N, K = 256, 512, 512
    ca = rng.integers(0, 16, (M, K)).astype(np.uint8)
    cb = rng.integers(0, 16, (N, K)).astype(np.uint8)
    ea = rng.integers(120, 135, (M, K // 32)).astype(np.uint8)
    eb = rng.integers(120, 135, (N, K // 32)).astype(np.uint8)
    y = host(qz.qz_gemm_mxfp4(dev(pack(ca)), dev(ea), dev(pack(cb)), dev(eb)))
    y_ref, bound = oracle.gemm_mxfp4(pack(ca), ea, pack(cb), eb)
    check(y, y_ref, bound, "mx per-block scales")
    sa = rng.integers(0x20, 0x60, (M, K // 16)).astype(np.uint8)          # UE4M3 in [2^-4, 2^4)
    sb = rng.integers(0x20, 0x60, (N, K // 16)).astype(np.uint8)
    y = host(qz.qz_gemm_nvfp4(dev(pack(ca)), dev(sa), dev(np.float32([0.5])), dev(pack(cb)), dev(sb),
                              dev(np.float32([3.0]))))
    y_ref, bound = oracle.gemm_nvfp4(pack(ca), sa, 0.5, pack(cb), sb, 3.0)
    check(y, y_ref, bound, "nv per-block scales")


@pytest.mark.parametrize("fmt", ["nv", "mx"])
def test_fp4_gemm_full_size_sampled(qz, fmt):
    """Config 4 at full size (M=8192, N=4096, K=4096) in the bench's launch
    configuration, operands from the oracle's quantizers, sampled outputs."""
    a, bt = syn.fp4_gemm_inputs(seed=0)
    y, ops = (nv_run if fmt == "nv" else mx_run)(qz, a, bt)
    rng = np.random.default_rng(3)
    ii, jj = rng.integers(0, a.shape[0], 3000), rng.integers(0, bt.shape[0], 3000)
    ref = oracle.gemm_nvfp4 if fmt == "nv" else oracle.gemm_mxfp4
    y_ref, bound = ref(*ops, ii, jj)
    check(y[ii, jj], y_ref, bound, f"{fmt} full size")


# ------------------------------------------------- prepared scales, grouped decode

def relayout_reference(sf, K, nv):
    """The tensor cores' scale-factor order written out with numpy: per 128 rows and 4
    scales, byte (m%32)*16 + (m/32)*4 + k holds sf[m][4*kg + k]; padding rows are 0."""
    R, KS = sf.shape
    assert KS == K // (16 if nv else 32)
    rp = -(-R // 128) * 128
    pad = np.zeros((rp, KS), np.uint8)
    pad[:R] = sf
    out = np.zeros((rp // 128, KS // 4, 512), np.uint8)
    m = np.arange(128)
    for rb in range(rp // 128):
        for kg in range(KS // 4):
            for k in range(4):
                out[rb, kg, (m % 32) * 16 + (m // 32) * 4 + k] = pad[rb * 128 + m, 4 * kg + k]
    return out.ravel()


@pytest.mark.parametrize("nv", [True, False])
@pytest.mark.parametrize("rows", [1, 200, 256])
def test_prepare_fp4_scales_layout(qz, nv, rows):
    K = 512
    rng = np.random.default_rng(rows + nv)
    sf = rng.integers(0, 256, (rows, K // (16 if nv else 32)), dtype=np.uint8)
    got = host(qz.qz_prepare_fp4_scales(dev(sf), K, nv=nv))
    assert np.array_equal(got, relayout_reference(sf, K, nv))


def grouped_case(qz, shapes, seed):
    """Quantize each (M, N, K) with the oracle, re-lay B's scales on the GPU, run one
    grouped call; returns the problems (with sentinel-filled Y) and the oracle operands."""
    probs, ops = [], []
    for i, (M, N, K) in enumerate(shapes):
        a, bt = inputs(M, N, K, seed + i)
        ca, sa, ga, _ = oracle.quant_nvfp4(a, want_deq=False)
        cb, sb, gb, _ = oracle.quant_nvfp4(bt, want_deq=False)
        Y = torch.full((M + 1, N), -7.0, dtype=torch.bfloat16, device="cuda")   # row M: sentinel
        probs.append((dev(ca), dev(sa), dev(np.float32([ga])), dev(cb),
                      qz.qz_prepare_fp4_scales(dev(sb), K, nv=True), dev(np.float32([gb])), Y[:M]))
        ops.append((ca, sa, ga, cb, sb, gb, Y))
    qz.qz_gemm_nvfp4_grouped(probs)
    torch.cuda.synchronize()
    return ops


def test_nvfp4_grouped_mixed_decode_shapes(qz):
    """Partial 128-row tiles (M = 1, 37, 128) and different N and K in one launch; every
    output checked, and the row after each Y untouched."""
    shapes = [(1, 256, 256), (37, 512, 1024), (128, 256, 512), (64, 768, 256)]
    for (M, N, K), (ca, sa, ga, cb, sb, gb, Y) in zip(shapes, grouped_case(qz, shapes, 11)):
        y_ref, bound = oracle.gemm_nvfp4(ca, sa, ga, cb, sb, gb)
        yh = host(Y)
        check(yh[:M], y_ref, bound, f"grouped M={M} N={N} K={K}")
        assert np.all(bf16_bits_to_f64(yh[M]) == -7.0), "a padding row was stored"


def test_nvfp4_grouped_matches_single_call(qz):
    """At M = 128 the grouped call and qz_gemm_nvfp4 run the same tiles: equal outputs."""
    shapes = [(128, 512, 512)]
    (ca, sa, ga, cb, sb, gb, Y), = grouped_case(qz, shapes, 21)
    y_single = host(qz.qz_gemm_nvfp4(dev(ca), dev(sa), dev(np.float32([ga])), dev(cb), dev(sb),
                                     dev(np.float32([gb]))))
    assert np.array_equal(host(Y)[:128], y_single)


def test_nvfp4_grouped_more_than_one_launch(qz):
    """85 problems: two GEMM launches (72 problems fit one launch's parameters)."""
    shapes = [(8 + (i % 3), 256, 256) for i in range(85)]
    ops = grouped_case(qz, shapes, 31)
    for i in (0, 41, 79, 80, 84):
        (ca, sa, ga, cb, sb, gb, Y), (M, N, K) = ops[i], shapes[i]
        y_ref, bound = oracle.gemm_nvfp4(ca, sa, ga, cb, sb, gb)
        check(host(Y)[:M], y_ref, bound, f"problem {i}")


def test_nvfp4_grouped_qwen_layer(qz):
    """One Qwen3-0.6B layer's seven linears at 64 tokens (the decode-step configuration),
    weights as B^T, all outputs checked."""
    probs, refs = [], []
    for layer, name, A, w in syn.qwen3_decode_linears(layers=1, tokens=64, seed=2):
        K, N = w.shape
        bt = syn.to_bf16_bits(np.ascontiguousarray(w.T))
        ca, sa, ga, _ = oracle.quant_nvfp4(A, want_deq=False)
        cb, sb, gb, _ = oracle.quant_nvfp4(bt, want_deq=False)
        Y = torch.empty((64, N), dtype=torch.bfloat16, device="cuda")
        probs.append((dev(ca), dev(sa), dev(np.float32([ga])), dev(cb),
                      qz.qz_prepare_fp4_scales(dev(sb), K, nv=True), dev(np.float32([gb])), Y))
        refs.append((name,) + oracle.gemm_nvfp4(ca, sa, ga, cb, sb, gb))
    qz.qz_gemm_nvfp4_grouped(probs)
    for (name, y_ref, bound), p in zip(refs, probs):
        check(host(p[6]), y_ref, bound, f"qwen {name}")


# ---------------------------------------- NVFP4 GEMM with NVFP4 output

def test_nvfp4_gemm_quantized_output_exact_case(qz):
    """Unit scales and E2M1 codes of small integers make every sum exact, so the output
    the epilogue quantizes is the oracle's exact product rounded once to bf16: codes,
    block scales and the tensor scale bit-exact against the oracle's NVFP4 quantizer of
    that output with the same given amax (a value below the output's own amax, so
    some blocks saturate, and one above it)."""
    rng = np.random.default_rng(31)
    M, N, K = 256, 512, 256
    mag = np.array([0, 2, 4, 5, 6, 7])                    # 0, 1, 2, 3, 4, 6
    ca = (rng.choice(mag, (M, K)) | (rng.integers(0, 2, (M, K)) << 3)).astype(np.uint8)
    cb = (rng.choice(mag, (N, K)) | (rng.integers(0, 2, (N, K)) << 3)).astype(np.uint8)
    va = np.vectorize(oracle.e2m1_decode)(ca)
    vb = np.vectorize(oracle.e2m1_decode)(cb)
    ybf = syn.to_bf16_bits((va @ vb.T).astype(np.float32))
    one = 0x38
    ops = (dev(pack(ca)), dev(np.full((M, K // 16), one, np.uint8)), dev(np.float32([1.0])),
           dev(pack(cb)), dev(np.full((N, K // 16), one, np.uint8)), dev(np.float32([1.0])))
    amax = float(np.abs(bf16_bits_to_f64(ybf)).max())
    for given in (amax * 0.25, amax * 1.5):
        codes, sb, g = qz.qz_gemm_nvfp4_quant(*ops, dev(np.float32([given])))
        rc, rs, rg, _ = oracle.quant_nvfp4(ybf, amax_in=np.float32(given), want_deq=False)
        assert_same_bytes(host(codes), rc, f"codes, amax {given}")
        assert_same_bytes(host(sb), rs, f"block scales, amax {given}")
        assert_same_bytes(host(g).reshape(np.shape(rg)), np.asarray(rg, np.float32), f"tensor scale, amax {given}")
    assert qz.qz_device_error() == 0


@pytest.mark.parametrize("M,N,K", [(128, 256, 256), (384, 768, 512), (1152, 1024, 768), (8192, 4096, 4096)])
def test_nvfp4_gemm_quantized_output_matches_gemm_then_quantizer(qz, M, N, K):
    """Realistic operands over one tile, several tiles in both directions, more tiles
    than SMs, and the prefill shape: the fused codes, block scales and tensor scale
    equal qz_quantize_nvfp4 with the same given amax applied to the plain NVFP4 GEMM's
    bf16 output, bit for bit."""
    a, bt = inputs(M, N, K, seed=M + N)
    ca, sa, ga, _ = oracle.quant_nvfp4(a, want_deq=False)
    cb, sb, gb, _ = oracle.quant_nvfp4(bt, want_deq=False)
    ops = (dev(ca), dev(sa), dev(np.float32([ga])), dev(cb), dev(sb), dev(np.float32([gb])))
    y = qz.qz_gemm_nvfp4(*ops)
    amax = dev(np.float32([float(torch.max(torch.abs(y.float())))]))
    codes, scales, g = qz.qz_gemm_nvfp4_quant(*ops, amax)
    c2, s2, g2, _ = qz.qz_quantize_nvfp4(y, global_amax_in=amax)
    assert np.array_equal(host(codes), host(c2)), "codes differ from GEMM then quantizer"
    assert np.array_equal(host(scales), host(s2)), "block scales differ from GEMM then quantizer"
    assert np.array_equal(host(g), host(g2)), "tensor scale differs"
    assert qz.qz_device_error() == 0


# ---------------------------------------- MXFP4 GEMM with MXFP4 output

def test_mxfp4_gemm_quantized_output_exact_case(qz):
    """Unit scales and E2M1 codes of small integers make every sum exact: codes and E8M0
    scales bit-exact against the oracle's MXFP4 quantizer of the exact product rounded
    once to bf16."""
    rng = np.random.default_rng(37)
    M, N, K = 256, 512, 256
    mag = np.array([0, 2, 4, 5, 6, 7])                    # 0, 1, 2, 3, 4, 6
    ca = (rng.choice(mag, (M, K)) | (rng.integers(0, 2, (M, K)) << 3)).astype(np.uint8)
    cb = (rng.choice(mag, (N, K)) | (rng.integers(0, 2, (N, K)) << 3)).astype(np.uint8)
    va = np.vectorize(oracle.e2m1_decode)(ca)
    vb = np.vectorize(oracle.e2m1_decode)(cb)
    ybf = syn.to_bf16_bits((va @ vb.T).astype(np.float32))
    codes, e8 = qz.qz_gemm_mxfp4_quant(dev(pack(ca)), dev(np.full((M, K // 32), 127, np.uint8)),
                                       dev(pack(cb)), dev(np.full((N, K // 32), 127, np.uint8)))
    rc, re8, _ = oracle.quant_mxfp4(ybf, want_deq=False)
    assert_same_bytes(host(codes), rc, "codes")
    assert_same_bytes(host(e8), re8, "E8M0 scales")
    assert qz.qz_device_error() == 0


@pytest.mark.parametrize("M,N,K", [(128, 256, 256), (384, 768, 512), (1152, 1024, 768), (8192, 4096, 4096)])
def test_mxfp4_gemm_quantized_output_matches_gemm_then_quantizer(qz, M, N, K):
    """Realistic operands over one tile, several tiles, more tiles than SMs, and the
    prefill shape: the fused codes and E8M0 scales equal qz_quantize_mxfp4 applied to
    the plain MXFP4 GEMM's bf16 output, bit for bit."""
    a, bt = inputs(M, N, K, seed=M + N + 1)
    ca, ea, _ = oracle.quant_mxfp4(a, want_deq=False)
    cb, eb, _ = oracle.quant_mxfp4(bt, want_deq=False)
    ops = (dev(ca), dev(ea), dev(cb), dev(eb))
    y = qz.qz_gemm_mxfp4(*ops)
    codes, e8 = qz.qz_gemm_mxfp4_quant(*ops)
    c2, e2, _ = qz.qz_quantize_mxfp4(y)
    assert np.array_equal(host(codes), host(c2)), "codes differ from GEMM then quantizer"
    assert np.array_equal(host(e8), host(e2)), "E8M0 scales differ from GEMM then quantizer"
    assert qz.qz_device_error() == 0


@pytest.mark.parametrize("fmt", ["nv", "mx"])
def test_fused_output_feeds_the_next_layer(qz, fmt):
    """Two layers in a row: layer 1's fused FP4 output (codes, block scales and, for
    NVFP4, the tensor scale) is layer 2's A operand as written, with no bf16 tensor in
    between. Layer 1's codes equal the oracle quantizer of its bf16 output, and layer 2's
    output is within the GEMM bound of the oracle's GEMM on those codes."""
    M, K1, N1, N2 = 256, 512, 768, 512
    a, w1t = inputs(M, N1, K1, seed=41)
    _, w2t = inputs(M, N2, N1, seed=42)
    if fmt == "nv":
        ca, sa, ga, _ = oracle.quant_nvfp4(a, want_deq=False)
        c1, s1, g1, _ = oracle.quant_nvfp4(w1t, want_deq=False)
        c2, s2, g2, _ = oracle.quant_nvfp4(w2t, want_deq=False)
        l1 = (dev(ca), dev(sa), dev(np.float32([ga])), dev(c1), dev(s1), dev(np.float32([g1])))
        y1 = qz.qz_gemm_nvfp4(*l1)                              # layer 1's bf16 output, for its amax
        amax = float(torch.max(torch.abs(y1.float())))
        yc, ys, yg = qz.qz_gemm_nvfp4_quant(*l1, dev(np.float32([amax])))
        y2 = qz.qz_gemm_nvfp4(yc, ys, yg, dev(c2), dev(s2), dev(np.float32([g2])))
        rc, rs, rg, _ = oracle.quant_nvfp4(host(y1), amax_in=np.float32(amax), want_deq=False)
        assert_same_bytes(host(yc), rc, "layer-1 codes")
        assert_same_bytes(host(ys), rs, "layer-1 block scales")
        y_ref, bound = oracle.gemm_nvfp4(rc, rs, float(np.asarray(rg).ravel()[0]), c2, s2, g2)
    else:
        ca, ea, _ = oracle.quant_mxfp4(a, want_deq=False)
        c1, e1, _ = oracle.quant_mxfp4(w1t, want_deq=False)
        c2, e2, _ = oracle.quant_mxfp4(w2t, want_deq=False)
        l1 = (dev(ca), dev(ea), dev(c1), dev(e1))
        y1 = qz.qz_gemm_mxfp4(*l1)
        yc, ye = qz.qz_gemm_mxfp4_quant(*l1)
        y2 = qz.qz_gemm_mxfp4(yc, ye, dev(c2), dev(e2))
        rc, re8, _ = oracle.quant_mxfp4(host(y1), want_deq=False)
        assert_same_bytes(host(yc), rc, "layer-1 codes")
        assert_same_bytes(host(ye), re8, "layer-1 E8M0 scales")
        y_ref, bound = oracle.gemm_mxfp4(rc, re8, c2, e2)
    check(host(y2), y_ref, bound, f"{fmt} layer 2 on layer 1's fused output")
    assert qz.qz_device_error() == 0
